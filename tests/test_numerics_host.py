"""The CUDA path's scalar numerics (csrc/numerics.cuh: exp32_det and its branch-free twin,
the correctly rounded binary32 of an exact int64 dot, digits -> binary64, log64_det),
compiled for the host with g++ through tests/cuda_host_shim.h, against the oracle, bit for
bit.  The oracle and the CUDA path share no code; this test feeds both the same inputs."""
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

from oracle import exact as E

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "bitwise_deterministic_shard_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"


@pytest.fixture(scope="module")
def drv(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None or not os.path.exists(os.path.join(CUDA_INC, "cuda_runtime.h")):
        pytest.skip("needs g++ and the CUDA headers")
    exe = str(tmp_path_factory.mktemp("numerics") / "drv")
    subprocess.run([cxx, "-std=c++17", "-O2", "-ffp-contract=off", "-I", CUDA_INC, "-I", HERE, "-I", CSRC,
                    "-include", "cuda_host_shim.h", os.path.join(HERE, "numerics_driver.cpp"), "-o", exe], check=True)

    def run(mode, data: np.ndarray, out_dtype, width):
        r = subprocess.run([exe, str(mode)], input=np.ascontiguousarray(data).tobytes(), capture_output=True,
                           check=True)
        return np.frombuffer(r.stdout, dtype=out_dtype).reshape(-1, width)
    return run


def test_exp32_det_equals_the_oracle(drv, oracle_native):
    rng = np.random.default_rng(51)
    x = np.concatenate([
        -rng.random(2_000_000) * 105.0,                                     # the whole range and past -104
        -rng.random(200_000) * 1e-3,                                        # near 0
        np.array([0.0, -0.0, -104.0, -103.97, -104.0001, -np.inf, -1e-45, -1.17549435e-38, np.nan]),
    ]).astype(np.float32)
    got = drv(0, x, np.uint32, 3)
    want = oracle_native.exp32_det_many(x).view(np.uint32)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan, 0], want[~nan])
    assert np.all(np.isnan(got[nan, 0].view(np.float32)))
    assert np.array_equal(got[~nan, 1], got[~nan, 0])                      # the branch-free twin
    # the split form the cross-entropy backward uses: exp32_det = p 2^k exactly for k >= -125,
    # which holds for every x down to about -86.6 (so all but the deepest weights)
    have = got[:, 2] != 0xFFFFFFFF
    assert np.array_equal(got[have, 2], want[have])
    assert np.all(have[~nan & (x >= -86.6)])


def test_cr32_scaled_is_the_correctly_rounded_binary32(drv):
    rng = np.random.default_rng(52)
    n = 60_000
    mag = rng.integers(0, 2 ** 62, n, dtype=np.int64) >> rng.integers(0, 62, n)
    T = np.where(rng.random(n) < 0.5, -mag, mag)
    T[:6] = [0, 1, -1, 2 ** 62, -(2 ** 62), 0x1000001]
    F = rng.integers(-200, 120, n).astype(np.int64)
    # the edges of the normal range: values just below / at / above 2^-126 and 2^128, ties included
    edge_T, edge_F = [], []
    for t in (2 ** 24 - 1, 2 ** 24, 2 ** 24 + 1, 2 ** 25 - 1, 2 ** 25 + 1, 2 ** 26 - 2, 3 * 2 ** 23,
              2 ** 40 - 2 ** 15, 2 ** 40 + 2 ** 16 + 1, 2 ** 62 - 1):
        top = t.bit_length() - 1
        for f in (-126 - top - 1, -126 - top, -126 - top + 1, 127 - top - 1, 127 - top, 127 - top + 1):
            for sgn in (1, -1):
                edge_T.append(sgn * t)
                edge_F.append(f)
    T = np.concatenate([T, np.asarray(edge_T, dtype=np.int64)])
    F = np.concatenate([F, np.asarray(edge_F, dtype=np.int64)])
    pairs = np.stack([T, F], axis=1).astype(np.int64)
    got = drv(1, pairs, np.uint32, 5)
    n_cvt = 0
    for (t, f), (a, b, sp, c, sc) in zip(pairs.tolist(), got.tolist()):
        want = np.float32(E.rn32(Fraction(t) * Fraction(2) ** f)).view(np.uint32)
        assert a == want, (t, f)
        if not sp:
            assert b == a, (t, f)                                           # fast twin where it claims the result
        if not sc:
            assert c == a, (t, f)                                           # conversion twin likewise
            n_cvt += 1
    assert n_cvt > len(pairs) // 3                                         # and it claims most of them


def test_digits_to_binary64(drv):
    """Digit arrays (canonical or plainly added) of values inside the contract's range: the
    top word stays below 2^31 in magnitude (NUM below 2^160, DEN below 2^32)."""
    rng = np.random.default_rng(53)
    for n, mode, e0 in ((15, 2, -320), (6, 3, -160)):
        a = rng.integers(-(2 ** 33), 2 ** 33, (3000, n), dtype=np.int64)
        a[:, n - 1] = rng.integers(-(2 ** 30), 2 ** 30, 3000)
        a[::3, n - 1] = 0
        a[::5, n - 2:] = 0
        a[::7] = 0
        a[1::7, : n - 1] = 0
        got = drv(mode, a, np.float64, 1)[:, 0]
        for row, g in zip(a.tolist(), got.tolist()):
            v = sum(Fraction(d) * Fraction(2) ** (e0 + 32 * k) for k, d in enumerate(row))
            assert g == E.rn64(v), row


def test_log64_det_equals_the_oracle(drv, oracle_native):
    rng = np.random.default_rng(54)
    d = np.concatenate([1.0 + rng.random(100_000) * 2 ** 31, 1.0 + rng.random(50_000),
                        np.array([1.0, 2.0, 1.5, np.sqrt(2.0), 2.0 ** 31, np.nextafter(1.0, 2.0)])])
    got = drv(4, d, np.float64, 1)[:, 0]
    assert np.array_equal(got.view(np.uint64), oracle_native.log64_det_many(d).view(np.uint64))


# ------------------------------------------------------- the exact score on the tensor cores
# (csrc/score_tc.cuh): a row's 26-bit fixed point X split into four balanced base-128 bf16
# slices; the seven diagonal sums A_c of slice products (what the MMAs accumulate, exact in
# f32) recombined into the int64 dot; rows outside the window corrected by their low limbs.

def _bf16_to_int(bits):
    return np.array(bits, dtype=np.uint32).__lshift__(16).view(np.float32).astype(np.int64)


def test_slices_recompose_the_fixed_point(drv):
    rng = np.random.default_rng(55)
    X = np.concatenate([rng.integers(-(2 ** 26) + 1, 2 ** 26, 200_000),
                        [0, 1, -1, 63, 64, -64, -65, 2 ** 26 - 1, -(2 ** 26) + 1]]).astype(np.int32)
    s = _bf16_to_int(drv(5, X, np.uint16, 4).astype(np.uint32))
    assert np.all(np.abs(s) <= 64)
    assert np.array_equal(s[:, 0] + s[:, 1] * 2 ** 7 + s[:, 2] * 2 ** 14 + s[:, 3] * 2 ** 21, X.astype(np.int64))


def test_diagonal_sums_recombine_to_the_exact_dot(drv):
    """Slices of random 26-bit rows (D = 128 and 256), the seven diagonal sums formed exactly,
    handed to combine_diag as the f32 values the tensor core holds: the int64 dot."""
    rng = np.random.default_rng(56)
    A_all, dots = [], []
    for D in (128, 256):
        for _ in range(40):
            q = rng.integers(-(2 ** 26) + 1, 2 ** 26, D).astype(np.int32)
            k = rng.integers(-(2 ** 26) + 1, 2 ** 26, D).astype(np.int32)
            if rng.random() < 0.3:
                q[rng.random(D) < 0.5] = 0
            sq = _bf16_to_int(drv(5, q, np.uint16, 4).astype(np.uint32))
            sk = _bf16_to_int(drv(5, k, np.uint16, 4).astype(np.uint32))
            A = [sum(int((sq[:, a] * sk[:, c - a]).sum()) for a in range(4) if 0 <= c - a < 4) for c in range(7)]
            assert max(abs(v) for v in A) <= 2 ** 22
            A_all.append(A)
            dots.append(int((q.astype(object) * k.astype(object)).sum()))
    T = drv(6, np.array(A_all, dtype=np.float32), np.int64, 1)[:, 0]
    assert [int(t) for t in T] == dots


def test_hi26_truncates_toward_zero(drv):
    rng = np.random.default_rng(57)
    x = (rng.standard_normal(50_000) * np.exp2(rng.integers(-40, 40, 50_000))).astype(np.float32)
    F = rng.integers(-180, 40, 50_000).astype(np.int32)
    emax = ((x.view(np.uint32) >> 23) & 0xFF).astype(np.int64)
    F = np.maximum(F, emax - 152).astype(np.int32)              # windows a row can have (|X| < 2^26)
    pairs = np.stack([x.view(np.int32), F], axis=1)
    got = drv(7, pairs, np.int32, 1)[:, 0]
    for xi, fi, g in zip(x.tolist(), F.tolist(), got.tolist()):
        v = Fraction(xi) / Fraction(2) ** fi
        assert g == (int(v) if v >= 0 else -int(-v)), (xi, fi)


def _row_limbs(x, F):
    """(X_hi, listed low limbs) of a row in window F per the score_tc.cuh definitions, or None
    for a deep row."""
    hi, lo = [], []
    for d, xv in enumerate(x.tolist()):
        v = Fraction(xv) / Fraction(2) ** F
        h = int(v) if v >= 0 else -int(-v)
        r = (v - h) * 2 ** 26
        if r.denominator != 1:
            return None
        hi.append(h)
        if r:
            lo.append((d, int(r)))
    return (hi, lo) if len(lo) <= 4 else None


def test_low_limb_correction_gives_the_exact_score(drv):
    """bf16-valued rows (8 significant bits) with a few elements scaled 2^-19 .. 2^-24 below
    the rest, so that their low bits fall under the 26-bit window as listed low limbs."""
    rng = np.random.default_rng(58)
    recs, want = [], []
    D = 128

    def bf16_row():
        r = rng.standard_normal(D).astype(np.float32)
        r = (r.view(np.uint32) & 0xFFFF0000).view(np.float32)
        idx = rng.choice(D, rng.integers(0, 5), replace=False)
        r[idx] = r[idx] * np.exp2(-rng.integers(19, 25, len(idx))).astype(np.float32)
        return r

    for _ in range(4000):
        if len(recs) >= 300:
            break
        q, k = bf16_row(), bf16_row()
        Fq = int(((q.view(np.uint32) >> 23) & 0xFF).max()) - 152
        Fk = int(((k.view(np.uint32) >> 23) & 0xFF).max()) - 152
        lq, lk = _row_limbs(q, Fq), _row_limbs(k, Fk)
        if lq is None or lk is None:
            continue
        Thh = sum(a * b for a, b in zip(lq[0], lk[0]))
        head = np.array([D, Fq, Fk, len(lq[1]), len(lk[1])], np.int32).tobytes() + np.int64(Thh).tobytes()
        body = q.tobytes() + k.tobytes() + np.array(lq[1] + lk[1], np.int32).reshape(-1).tobytes()
        recs.append(head + body)
        exact = sum((Fraction(a) * Fraction(b) for a, b in zip(q.tolist(), k.tolist())), Fraction(0))
        want.append(int(np.float32(E.rn32(exact)).view(np.uint32)))
    assert len(recs) >= 100
    got = drv(8, np.frombuffer(b"".join(recs), np.uint8), np.uint32, 1)[:, 0]
    assert got.tolist() == want
