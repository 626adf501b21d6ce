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
    got = drv(0, x, np.uint32, 2)
    want = oracle_native.exp32_det_many(x).view(np.uint32)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan, 0], want[~nan])
    assert np.all(np.isnan(got[nan, 0].view(np.float32)))
    assert np.array_equal(got[~nan, 1], got[~nan, 0])                      # the branch-free twin


def test_cr32_scaled_is_the_correctly_rounded_binary32(drv):
    rng = np.random.default_rng(52)
    n = 60_000
    mag = rng.integers(0, 2 ** 62, n, dtype=np.int64) >> rng.integers(0, 62, n)
    T = np.where(rng.random(n) < 0.5, -mag, mag)
    T[:6] = [0, 1, -1, 2 ** 62, -(2 ** 62), 0x1000001]
    F = rng.integers(-200, 120, n).astype(np.int64)
    pairs = np.stack([T, F], axis=1).astype(np.int64)
    got = drv(1, pairs, np.uint32, 3)
    for (t, f), (a, b, sp) in zip(pairs.tolist(), got.tolist()):
        want = np.float32(E.rn32(Fraction(t) * Fraction(2) ** f)).view(np.uint32)
        assert a == want, (t, f)
        if not sp:
            assert b == a, (t, f)                                           # fast twin where it claims the result


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
