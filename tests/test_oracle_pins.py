"""Pins of the oracle against things other than itself (CPU only).

Each test ties some part of oracle/ to an independent fact: the IEEE conversions of numpy
and CPython, mpmath at high precision, closed forms of the softmax reduction, a naive
float64 softmax attention, torch's float64 cross-entropy, and the invariances that the
det-attn page ("Method", "Correctness") and the det-cross-entropy page ("Method",
"Correctness") state.  A plausible slip anywhere in the oracle (a dropped polynomial term,
a wrong sign, a transposed Q/K, a wrong GQA head map, a shifted digit exponent, a missing
rounding) breaks at least one of them; tests/test_oracle_mutations.py plants such slips
and checks that they are caught.
"""
import itertools
import math
import random
from fractions import Fraction

import mpmath as mp
import numpy as np
import pytest
import torch

from oracle import exact as E
import workloads as W


# ---------------------------------------------------------------------------- roundings

def test_rn32_matches_numpy_conversion():
    """RN32 of a double equals numpy's IEEE double->float conversion (normal, subnormal,
    halfway cases, overflow)."""
    rng = np.random.default_rng(0)
    xs = list(rng.standard_normal(3000) * np.exp2(rng.integers(-160, 130, 3000)))
    # exact halfway points between adjacent floats, both parities
    for _ in range(500):
        f = np.float32(rng.standard_normal() * 2.0 ** rng.integers(-140, 120))
        g = np.nextafter(f, np.float32(np.inf))
        xs.append((float(f) + float(g)) / 2)
    xs += [2.0 ** -150, 3 * 2.0 ** -151, 2.0 ** -149 * 0.75, 3.4028235677973366e38, 3.4028235e38 * 1.0000001]
    for x in xs:
        with np.errstate(over="ignore"):
            ref = float(np.float32(x))
        got = E.rn32(Fraction(x))
        assert got == ref and math.copysign(1, got) == math.copysign(1, ref), x


def test_rn64_matches_cpython_division():
    """RN64 of p/q equals CPython's correctly rounded int true division."""
    rng = random.Random(1)
    for _ in range(3000):
        p = rng.getrandbits(rng.randint(1, 400)) * rng.choice([-1, 1])
        q = rng.getrandbits(rng.randint(1, 400)) + 1
        try:
            ref = p / q
        except OverflowError:
            continue
        assert E.rn64(Fraction(p, q)) == ref


# ---------------------------------------------------------------------------- constants

def test_exp_constants_from_mpmath():
    mp.mp.prec = 300
    ln2 = mp.log(2)
    assert abs(mp.mpf(E.LN2.numerator) / E.LN2.denominator - ln2) < mp.mpf(2) ** -290
    assert E.EXP_L2E == float(np.float32(float(1 / ln2)))  # 1/ln2 is far from a float32 tie
    assert E.EXP_C1 == float.fromhex('0x1.62e4p-1')
    assert E.EXP_C2 == float(np.float32(float(ln2 - mp.mpf(E.EXP_C1))))
    for n in range(8):
        assert E.EXP_TAYLOR[n] == float(np.float32(1.0 / math.factorial(n)))


def test_log_constants_from_mpmath():
    mp.mp.prec = 300
    ln2 = mp.log(2)
    assert E.LOG_SQRT2 == float(mp.sqrt(2))
    assert abs(mp.mpf(E.LOG_LN2_HI) + mp.mpf(E.LOG_LN2_LO) - ln2) < mp.mpf(2) ** -95
    assert (Fraction(E.LOG_LN2_HI) * (1 << 42)).denominator == 1   # e*LN2_HI exact for |e| < 2**11


def test_default_scale_values():
    assert E.default_scale(64) == 0.125
    assert E.default_scale(128) == float.fromhex('0x1.6a09e6p-4')


# ---------------------------------------------------------------------------- exp / log

def test_exp32_det_special_values():
    assert E.exp32_det(0.0) == 1.0
    assert E.exp32_det(-0.0) == 1.0
    assert E.exp32_det(-104.5) == 0.0
    assert E.exp32_det(-1e30) == 0.0
    assert math.isnan(E.exp32_det(math.nan))
    assert E.exp32_det(-103.0) == 2.0 ** -149


def test_exp32_det_python_equals_c(oracle_native):
    rng = np.random.default_rng(2)
    xs = np.concatenate([-rng.random(4000).astype(np.float32) * 104, -rng.random(1000).astype(np.float32),
                         np.array([-0.3465736, -0.34657362, -87.33655, -87.33654, -103.97, -103.28], np.float32)])
    c = oracle_native.exp32_det_many(xs)
    for x, y in zip(xs, c):
        assert E.exp32_det(float(x)) == float(y), x


def test_exp32_det_ulp_sweep(oracle_native):
    """Error against the float64 exponential, in units of the binary32 spacing at the true
    value (2**-149 below the normal range), over every 16th binary32 in [-104, 0].  The
    full sweep of all 1.12e9 inputs gives 0.937 ulp."""
    lo, hi = 0x80000000, 0xC2D00000
    worst = 0.0
    for start in range(lo, hi + 1, 1 << 26):
        bits = np.arange(start, min(start + (1 << 26), hi + 1), 16, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        y = oracle_native.exp32_det_many(x).astype(np.float64)
        ref = np.exp(x.astype(np.float64))
        ulp = np.spacing(np.abs(ref.astype(np.float32))).astype(np.float64)
        worst = max(worst, float(np.max(np.abs(y - ref) / ulp)))
    assert worst < 1.0


def test_exp32_det_against_mpmath_points():
    mp.mp.prec = 120
    rng = np.random.default_rng(3)
    for x in (-rng.random(300) * 104).astype(np.float32):
        w = E.exp32_det(float(x))
        ref = mp.exp(mp.mpf(float(x)))
        ulp = float(np.spacing(np.float32(float(ref)))) if float(ref) > 0 else 2.0 ** -149
        assert abs(mp.mpf(w) - ref) <= 1.0 * ulp


def test_log64_det_against_mpmath(oracle_native):
    mp.mp.prec = 200
    rng = np.random.default_rng(4)
    xs = np.concatenate([1 + rng.random(3000) * 3, np.exp(rng.random(3000) * 22), np.arange(1, 200, dtype=np.float64),
                         2.0 ** np.arange(0, 31)])
    ys = oracle_native.log64_det_many(xs)
    worst = 0.0
    for x, y in zip(xs, ys):
        ref = mp.log(mp.mpf(float(x)))
        assert E.log64_det(float(x)) == float(y)
        if ref != 0:
            worst = max(worst, float(abs(mp.mpf(float(y)) - ref) / mp.mpf(float(np.spacing(float(ref))))))
    assert E.log64_det(1.0) == 0.0
    assert worst <= 2.0


# ---------------------------------------------------------------------------- scores

def _bf16_values(rng, n, spread=8):
    x = torch.tensor(rng.standard_normal(n) * np.exp2(rng.integers(-spread, spread, n)), dtype=torch.float32)
    return x.to(torch.bfloat16).float().numpy().astype(np.float64)


def test_score_single_term_is_exact_product():
    """D = 1: the dot is one product of two bf16 values (16 significant bits), exact in
    binary32, so d = q*k and s = RN32(scale*q*k)."""
    rng = np.random.default_rng(5)
    q, k = _bf16_values(rng, 2000), _bf16_values(rng, 2000)
    for a, b in zip(q, k):
        ref = np.float32(np.float32(a) * np.float32(b)) * np.float32(0.125)
        assert E.score([E.to_int149(a)], [E.to_int149(b)], 0.125) == float(ref)


def test_score_two_terms_single_rounding():
    """D = 2 with bf16 inputs: the float64 sum of the two exact products is exact when the
    exponents are close, so numpy's one conversion to float32 is the correct rounding."""
    rng = np.random.default_rng(6)
    q, k = _bf16_values(rng, 4000, 4).reshape(-1, 2), _bf16_values(rng, 4000, 4).reshape(-1, 2)
    s32 = float(np.float32(1 / math.sqrt(2)))
    for a, b in zip(q, k):
        dot64 = a[0] * b[0] + a[1] * b[1]
        ref = np.float32(np.float32(dot64) * np.float32(s32))
        assert E.score([E.to_int149(x) for x in a], [E.to_int149(x) for x in b], s32) == float(ref)


def test_score_against_mpmath_f32():
    """D = 8, f32 inputs over a wide exponent range: the exact dot from mpmath at 2000 bits,
    rounded once to 24 bits."""
    rng = np.random.default_rng(7)
    mp.mp.prec = 2000
    for _ in range(400):
        q = (rng.standard_normal(8) * np.exp2(rng.integers(-30, 30, 8))).astype(np.float32)
        k = (rng.standard_normal(8) * np.exp2(rng.integers(-30, 30, 8))).astype(np.float32)
        exact = mp.fsum(mp.mpf(float(a)) * mp.mpf(float(b)) for a, b in zip(q, k))
        with mp.workprec(24):
            d = float(+exact)   # unary plus rounds to the working precision, ties to even
        got = E.score([E.to_int149(float(a)) for a in q], [E.to_int149(float(b)) for b in k], 1.0)
        assert got == d


# ---------------------------------------------------------------------------- attention

def _naive64(Q, K, V, causal, scale):
    Q, K, V = (t.double() for t in (Q, K, V))
    rep = Q.shape[1] // K.shape[1]
    K, V = K.repeat_interleave(rep, 1), V.repeat_interleave(rep, 1)
    s = (Q @ K.transpose(-1, -2)) * scale
    if causal:
        S = s.shape[-1]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    return torch.softmax(s, -1) @ V


def test_tiny_exact_agrees_with_naive_float64_attention(oracle_native):
    """North-star agreement: the exact result equals a naive float64 softmax attention to
    1e-6 absolute on the tiny f32 workload."""
    w = W.tiny_exact()
    Q, K, V = w.tensors()
    A = oracle_native.Attn(Q, K, V, w.causal, w.scale)
    _, _, _, out = A.forward_rows()
    ref = _naive64(Q, K, V, w.causal, 0.125).reshape(-1, w.D).numpy()
    assert np.max(np.abs(out - ref)) < 1e-6


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_gqa_agrees_with_naive_float64(oracle_native, causal, dtype):
    Q, K, V = W.random_attn(8, 2, 4, 2, 48, 16, dtype, causal)
    A = oracle_native.Attn(Q, K, V, causal)
    _, _, _, out = A.forward_rows()
    ref = _naive64(Q, K, V, causal, float(np.float32(0.25))).reshape(-1, 16).numpy()
    assert np.max(np.abs(out - ref)) < 2e-6


def test_python_exact_agrees_with_naive_float64():
    Q, K, V = W.random_attn(9, 1, 2, 1, 12, 8, torch.bfloat16, True)
    out = E.det_attn(Q, K, V, causal=True)
    ref = _naive64(Q, K, V, True, E.default_scale(8)).numpy()
    assert np.max(np.abs(out - ref)) < 2e-6


def test_causal_row0_is_v0_exactly(oracle_native):
    Q, K, V = W.random_attn(10, 1, 2, 2, 24, 16, torch.bfloat16, True)
    _, _, _, out = oracle_native.Attn(Q, K, V, True).forward_rows()
    out = out.reshape(1, 2, 24, 16)
    assert np.array_equal(out[:, :, 0, :], V[:, :, 0, :].float().numpy())


def test_zero_queries_give_mean_of_v(oracle_native):
    """Q = 0: every score is +0, every weight 1, so o = RN32(RN64(RN64(sum_j v_j) / S));
    math.fsum is the correctly rounded float64 sum."""
    _, K, V = W.random_attn(11, 1, 1, 1, 40, 8, torch.float32, False)
    Q = torch.zeros(1, 1, 40, 8)
    _, _, _, out = oracle_native.Attn(Q, K, V, False).forward_rows()
    Vn = V.numpy()[0, 0]
    for d in range(8):
        ref = np.float32(math.fsum(Vn[:, d].astype(np.float64)) / 40.0)
        assert np.all(out[:, d] == ref)


def test_constant_power_of_two_values(oracle_native):
    Q, K, _ = W.random_attn(12, 1, 2, 2, 32, 8, torch.bfloat16, False)
    V = torch.full((1, 2, 32, 8), 0.375, dtype=torch.bfloat16)  # 3/8: NUM = 3/8 DEN exactly
    _, _, _, out = oracle_native.Attn(Q, K, V, False).forward_rows()
    assert np.all(out == np.float32(0.375))


def test_value_scaling_and_negation(oracle_native):
    Q, K, V = W.random_attn(13, 1, 2, 2, 32, 8, torch.float32, True)
    _, n1, d1, o1 = oracle_native.Attn(Q, K, V, True).forward_rows()
    _, n2, d2, o2 = oracle_native.Attn(Q, K, V * 64, True).forward_rows()
    _, n3, d3, o3 = oracle_native.Attn(Q, K, -V, True).forward_rows()
    assert np.array_equal(o2, o1 * 64)
    assert np.array_equal(o3, -o1)
    assert np.array_equal(d1, d2) and np.array_equal(d1, d3)
    tot, _ = oracle_native.normalize(n1 + n3, E.NUM_E0)
    assert not tot.any()


def test_single_key_returns_its_value(oracle_native):
    Q, K, V = W.random_attn(14, 1, 2, 2, 1, 16, torch.float32, False)
    _, _, _, out = oracle_native.Attn(Q, K, V, False).forward_rows()
    assert np.array_equal(out.reshape(2, 16), V.numpy().reshape(2, 16))


def test_digits_decode_to_exact_sums():
    """Canonical digits decode to the exact sums built independently from Fractions, and
    lie in the canonical ranges."""
    Q, K, V = W.random_attn(15, 1, 1, 1, 6, 4, torch.float32, False)
    P = E.AttnProblem(Q, K, V)
    m = P.rowmax()
    num, den, _ = P.accumulate(m)
    q, k, v = (E.decode(t)[0, 0] for t in (Q, K, V))
    for i in range(6):
        s = [E.score([E.to_int149(x) for x in q[i]], [E.to_int149(x) for x in k[j]], P.scale32) for j in range(6)]
        ws = [Fraction(E.exp32_det(E.rn32(Fraction(sj) - Fraction(float(m[0, 0, i]))))) for sj in s]
        assert max(ws) == 1
        assert E.digits_value(den[0, 0, i], E.DEN_E0) == sum(ws)
        for d in range(4):
            dg = num[0, 0, i, :, d]
            assert E.digits_value(dg, E.NUM_E0) == sum(wj * Fraction(float(v[j, d])) for j, wj in enumerate(ws))
            assert all(0 <= int(x) < 2 ** 32 for x in dg[:-1])


def test_normalize_of_digit_sums(oracle_native):
    rng = np.random.default_rng(16)
    a = rng.integers(0, 2 ** 32, size=(50, 15, 3), dtype=np.int64)
    b = rng.integers(0, 2 ** 32, size=(50, 15, 3), dtype=np.int64)
    a[:, 14, :] = rng.integers(-2 ** 40, 2 ** 40, size=(50, 3))
    b[:, 14, :] = rng.integers(-2 ** 40, 2 ** 40, size=(50, 3))
    tot, bad = oracle_native.normalize(a + b, E.NUM_E0)
    assert bad == 0
    for r in range(50):
        for c in range(3):
            want = E.canon_digits(E.digits_value(a[r, :, c], E.NUM_E0) + E.digits_value(b[r, :, c], E.NUM_E0),
                                  E.NUM_E0, 15)
            assert list(tot[r, :, c]) == want


def test_finalize_rounds_twice_as_stated():
    """o = RN32(RN64(RN64(NUM) / RN64(DEN))): CPython's float(Fraction) is correctly
    rounded, its float division is IEEE, numpy's float32 conversion rounds once."""
    rng = random.Random(17)
    for _ in range(300):
        num = Fraction(rng.getrandbits(120) - (1 << 119), 1 << rng.randint(100, 300))
        den = Fraction(rng.getrandbits(60) | 1, 1 << rng.randint(20, 150)) + 1
        ref = np.float32(float(num) / float(den))
        got = E.finalize_value(E.canon_digits(num, E.NUM_E0, 15), E.canon_digits(den, E.DEN_E0, 6))
        assert got == ref


# ---------------------------------------------------------------------------- invariance

def test_python_sharded_equals_fused_all_orders():
    Q, K, V = W.random_attn(18, 1, 2, 1, 10, 4, torch.bfloat16, False)
    fused = E.det_attn(Q, K, V)
    for order in itertools.permutations(range(3)):
        assert np.array_equal(E.det_attn_sharded(Q, K, V, [3, 3, 4], order=order).view(np.uint32),
                              fused.view(np.uint32))


def test_tiny_exact_sharded_all_24_orders_equal_fused(oracle_native):
    w = W.tiny_exact()
    Q, K, V = w.tensors()
    A = oracle_native.Attn(Q, K, V, w.causal, w.scale)
    m0, n0, d0, o0 = A.forward_rows()
    for sp, order in w.splits:
        bounds = np.cumsum([0] + sp)
        ms = [A.rowmax(bounds[k], bounds[k + 1])[0] for k in order]
        m = ms[0]
        for x in ms[1:]:
            m = np.maximum(m, x)
        assert np.array_equal(m, m0)
        num = sum(A.accumulate(m, bounds[k], bounds[k + 1])[0] for k in order)
        den = sum(A.accumulate(m, bounds[k], bounds[k + 1])[1] for k in order)
        num, _ = oracle_native.normalize(num, E.NUM_E0)
        den, _ = oracle_native.normalize(den, E.DEN_E0)
        assert np.array_equal(num, n0) and np.array_equal(den, d0)
        assert np.array_equal(oracle_native.finalize(num, den).view(np.uint32), o0.view(np.uint32))


def test_repeat_runs_identical(oracle_native):
    Q, K, V = W.random_attn(19, 1, 4, 2, 64, 32, torch.bfloat16, True)
    a = oracle_native.Attn(Q, K, V, True).forward_rows()
    b = oracle_native.Attn(Q, K, V, True).forward_rows(nthreads=3)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_rowmax_violation_is_reported(oracle_native):
    Q, K, V = W.random_attn(20, 1, 1, 1, 16, 8, torch.float32, False)
    A = oracle_native.Attn(Q, K, V)
    m, _ = A.rowmax()
    _, _, st = A.accumulate(m - 1.0)
    assert st & 2
    _, _, st = A.accumulate(m)
    assert st == 0


# ---------------------------------------------------------------------------- cross-entropy

def test_dce_matches_torch_cross_entropy(oracle_native):
    g = torch.Generator().manual_seed(21)
    x = torch.randn(64, 1000, generator=g) * 2
    t = torch.randint(0, 1000, (64,), generator=g)
    loss, denom, m, den, st = oracle_native.DCE(x).forward(t.numpy())
    ref = torch.nn.functional.cross_entropy(x.double(), t, reduction="none").numpy()
    assert st == 0
    assert np.max(np.abs(loss - ref)) < 2e-6
    lse = torch.logsumexp(x.double() - torch.tensor(m, dtype=torch.float64)[:, None], 1).exp().numpy()
    assert np.max(np.abs(denom / lse - 1)) < 1e-6


def test_dce_closed_forms(oracle_native):
    x = torch.full((3, 777), 1.25)
    loss, denom, *_ = oracle_native.DCE(x).forward(np.array([0, 5, 776]))
    assert np.all(denom == 777.0)
    assert np.all(loss == np.float32(E.log64_det(777.0)))
    x1 = torch.randn(5, 1)
    loss1, denom1, *_ = oracle_native.DCE(x1).forward(np.zeros(5, dtype=np.int64))
    assert np.all(loss1 == 0) and np.all(denom1 == 1)


def test_dce_splits_invariant_and_python_equal(oracle_native):
    g = torch.Generator().manual_seed(22)
    x = (torch.randn(6, 40, generator=g) * 2).to(torch.bfloat16)
    t = torch.randint(0, 40, (6,), generator=g)
    base = oracle_native.DCE(x).forward(t.numpy())
    for sp in ([20, 20], [10, 10, 10, 10], [1, 7, 32], [39, 1]):
        got = oracle_native.DCE(x).forward(t.numpy(), splits=sp)
        for a, b in zip(base[:4], got[:4]):
            assert np.array_equal(a, b)
    loss, denom, m, den = E.dce_forward(x, t.numpy(), splits=[13, 27])
    assert np.array_equal(loss, base[0]) and np.array_equal(denom, base[1]) and np.array_equal(den, base[3])


def test_dce_bad_target_flag(oracle_native):
    x = torch.randn(4, 10)
    loss, _, _, _, st = oracle_native.DCE(x).forward(np.array([0, 10, -1, 3]))
    assert st & 8
    assert np.isnan(loss[1]) and np.isnan(loss[2]) and not np.isnan(loss[0])
