"""The integer-pipe division helpers that the finalize kernels use (csrc/divide.cuh), compiled
for the host with g++ and checked against exact rational arithmetic: RN64 of a quotient of two
binary64 magnitudes (division by an invariant integer with a precomputed reciprocal), RN32 of
a binary64 given as mantissa and exponent (normal, subnormal, overflow), RN64 of a Kulisch
digit value, and the binary32 split.  CPython's int / int is correctly rounded and numpy's
float32 conversion rounds to nearest even, so both serve as the exact references here."""
import math
import os
import shutil
import struct
import subprocess
from fractions import Fraction

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "bitwise_deterministic_shard_gb300", "csrc")


@pytest.fixture(scope="module")
def drv(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not available")
    exe = str(tmp_path_factory.mktemp("divide") / "drv")
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-I", CSRC, os.path.join(HERE, "divide_driver.cpp"),
                    "-o", exe], check=True)

    def run(mode, n):
        return subprocess.run([exe, str(mode), str(n)], capture_output=True, text=True, check=True).stdout.splitlines()
    return run


def test_div_rn64_is_correctly_rounded(drv):
    for line in drv(0, 60000):
        mn, en, md, ed, q, E, f = map(int, line.split())
        k = en - ed
        val = (mn << k) / md if k >= 0 else mn / (md << -k)
        m, e = math.frexp(val)
        assert (q, E) == (int(m * 2 ** 53), e - 53), line


def test_rn32_of_binary64(drv):
    for line in drv(1, 60000):
        q, E, neg, f = map(int, line.split())
        x = math.ldexp(q, E) * (-1 if neg else 1)
        with np.errstate(over="ignore"):
            ref = struct.unpack("<I", struct.pack("<f", np.float32(x)))[0]
        assert ref == f, line


def test_digits_rn64(drv):
    for line in drv(2, 20000):
        a, r = line.split("|")
        a = list(map(int, a.split()))
        nz, neg, m, e = map(int, r.split())
        S = sum(Fraction(v) * Fraction(2) ** (-320 + 32 * k) for k, v in enumerate(a))
        if S == 0:
            assert nz == 0, line
            continue
        mm, ee = math.frexp(abs(float(S)))
        assert (nz, neg, m, e) == (1, int(S < 0), int(mm * 2 ** 53), ee - 53), line


def test_f32_split(drv):
    for line in drv(3, 20000):
        b, m, e = map(int, line.split())
        x = struct.unpack("<f", struct.pack("<I", b))[0]
        assert 2 ** 52 <= m < 2 ** 53 and Fraction(m) * Fraction(2) ** e == Fraction(x), line


def test_binary32_numerator_division(drv):
    """div_f32_rn32 (two 32 x 32 products) equals the generic division, and RN32(RN64(w / d))
    computed exactly."""
    for k, line in enumerate(drv(4, 60000)):
        b, md, ed, fast, generic = map(int, line.split())
        assert fast == generic, line
        if k % 10 == 0:
            w = Fraction(struct.unpack("<f", struct.pack("<I", b))[0])
            d = Fraction(md) * Fraction(2) ** (ed)
            q = w / d
            q64 = q.numerator / q.denominator          # correctly rounded binary64
            ref = struct.unpack("<I", struct.pack("<f", np.float32(q64)))[0]
            assert fast == ref, line


def test_i128_rn64(drv):
    """RN64 of d0 + d1 2^32 + d2 2^64 (three lazy radix-2^32 digits as one 128-bit integer)
    times 2^lsb, the tensor-PV epilogue's form for the elements that touched no spill digit,
    against CPython's correctly rounded int -> float conversion."""
    for line in drv(5, 20000):
        a, r = line.split("|")
        d0, d1, d2, lsb = map(int, a.split())
        nz, neg, m, e = map(int, r.split())
        X = d0 + (d1 << 32) + (d2 << 64)
        if X == 0:
            assert nz == 0, line
            continue
        mm, ee = math.frexp(float(abs(X)))               # int -> float rounds to nearest even
        assert (nz, neg, m, e) == (1, int(X < 0), int(mm * 2 ** 53), ee - 53 + lsb), line


def test_direct_binary32_quotient(drv):
    """div_f32_rn32_direct (the dLogits fast path): whenever it reports success its bits equal
    the exact division's, and every fourth case is also checked against RN32(RN64(w / d))
    computed with CPython's exact arithmetic.  Quotients within about 2^-53 of a binary32
    half-way point must take the exact path, and for weights like the backward's
    (exponents in [-40, 0], divisors of ordinary size) the fallback stays rare."""
    taken = {0: [0, 0], 1: [0, 0], 2: [0, 0], 3: [0, 0]}
    for k, line in enumerate(drv(6, 80000)):
        b, md, ed, ok, fast, exact = map(int, line.split())
        kind = k % 4
        taken[kind][0] += 1
        taken[kind][1] += ok
        if ok:
            assert fast == exact, line
        if k % 4 == 0 or kind == 2:
            w = Fraction(struct.unpack("<f", struct.pack("<I", b))[0])
            q = w / (Fraction(md) * Fraction(2) ** ed)
            q64 = q.numerator / q.denominator
            assert exact == struct.unpack("<I", struct.pack("<f", np.float32(q64)))[0], line
            if kind == 2 and ok:   # certain only when far from the half-way point
                qf = Fraction(struct.unpack("<f", struct.pack("<I", fast))[0])
                assert abs(q - qf) < Fraction(struct.unpack("<f", struct.pack("<I", fast + 1))[0]) - qf, line
    assert taken[0][1] >= 0.999 * taken[0][0], taken      # exp-like weights: almost never the exact path
    assert taken[2][1] <= 0.01 * taken[2][0], taken       # near half-way points: the exact path


def test_direct_binary32_of_binary64_quotient(drv):
    """div_rn64_rn32_direct (the finalize epilogues' fast path): whenever it reports success its
    bits equal rn32_bits(div_rn64(...)), which every fourth case also checks against
    RN32(RN64(n / d)) from CPython's exact arithmetic; quotients within about 2^-53 of a binary32
    half-way point must take the exact path, exact quotients must not."""
    taken = [[0, 0] for _ in range(4)]
    for k, line in enumerate(drv(7, 80000)):
        mn, en, md, ed, neg, ok, fast, exact = map(int, line.split())
        kind = k % 4
        taken[kind][0] += 1
        taken[kind][1] += ok
        if ok:
            assert fast == exact, line
        if k % 4 == 0 or kind == 2:
            q = Fraction(mn) * Fraction(2) ** en / (Fraction(md) * Fraction(2) ** ed)
            q64 = q.numerator / q.denominator if abs(q) < 2 ** 1000 else float("inf")
            ref = struct.unpack("<I", struct.pack("<f", np.float32(-q64 if neg else q64)))[0]
            assert exact == ref, line
    assert taken[0][1] == taken[0][0], taken     # ordinary quotients: always direct here
    assert taken[2][1] == 0, taken               # near half-way points: always exact
    assert taken[3][1] == taken[3][0], taken     # exact quotients are decided directly


def test_fp32_pipe_quotient_with_certificate(drv):
    """fdiv::div_rn32 (the dLogits fast path on the FP32 pipe): whenever its certificate holds,
    its bits equal the exact division's (div_f32_rn32, itself pinned to exact rationals above),
    and every fourth case plus every near-half-way case is also checked against
    RN32(RN64(p / d)) from CPython's exact arithmetic.  Quotients within about 2^-53 of a
    binary32 half-way point must fail the certificate; for ordinary denominators it fails
    about once in 2^15 quotients."""
    taken = [[0, 0] for _ in range(4)]
    for k, line in enumerate(drv(8, 200000)):
        pb, db, ok, fast, exact = map(int, line.split())
        kind = k % 4
        taken[kind][0] += 1
        taken[kind][1] += ok
        if ok:
            assert fast == exact, line
        if k % 4 == 0 or kind == 2:
            p = Fraction(struct.unpack("<f", struct.pack("<I", pb))[0])
            d = Fraction(struct.unpack("<d", struct.pack("<Q", db))[0])
            q = p / d
            q64 = q.numerator / q.denominator                  # RN64 of the exact quotient
            assert exact == struct.unpack("<I", struct.pack("<f", np.float32(q64)))[0], line
    assert taken[0][1] >= 0.999 * taken[0][0], taken        # ordinary denominators: rarely exact
    assert taken[1][1] >= 0.95 * taken[1][0], taken         # the whole range (a few outside it)
    assert taken[2][1] <= 0.001 * taken[2][0], taken        # near half-way points: never certified
