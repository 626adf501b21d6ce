"""The exact accumulation of the cross-entropy denominator kernel (csrc/den_acc.cuh),
compiled for the host with g++: the six digits it leaves must hold exactly the sum of the
binary32 weights, whatever their exponents, for sequences long enough to force the private
64-bit word to be moved into the digits many times."""
import os
import shutil
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
    exe = str(tmp_path_factory.mktemp("denacc") / "drv")
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, os.path.join(HERE, "den_acc_driver.cpp"), "-o", exe],
                   check=True)
    return exe


def _sequences():
    rng = np.random.default_rng(12)
    seqs = [
        np.ones(5000, np.float32),                                        # w = 1: many flushes
        np.float32(1.0) - rng.random(3000).astype(np.float32) * 1e-3,
        np.exp(-rng.random(4000) * 30).astype(np.float32),               # both routes (2^-31 ~ e^-21.5)
        np.exp(-rng.random(4000) * 104).astype(np.float32),              # down to 2^-150
        np.array([2.0 ** -31, np.nextafter(np.float32(2.0 ** -31), 0), 2.0 ** -149, 2.0 ** -126,
                  np.float32(1.0), 0.0], np.float32),                    # the boundaries
        np.zeros(7, np.float32),
        rng.random(10000).astype(np.float32),
    ]
    return seqs


def test_den_digits_hold_the_exact_sum(drv):
    seqs = _sequences()
    text = "\n".join("\n".join(str(int(b)) for b in s.view(np.uint32)) + "\n" for s in seqs)
    out = subprocess.run([drv], input=text, capture_output=True, text=True, check=True).stdout.splitlines()
    assert len(out) == len(seqs)
    for s, line in zip(seqs, out):
        d = [int(v) for v in line.split()]
        got = sum(Fraction(v) * Fraction(2) ** (32 * k - 160) for k, v in enumerate(d))
        want = sum((Fraction(float(w)) for w in s), Fraction(0))
        assert got == want
