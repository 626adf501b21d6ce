"""Planted mistakes: each test plants a plausible slip in the Python oracle (on the CPU,
through monkeypatch) and checks that an independent pin rejects the mutated oracle.  This
shows that the pins of tests/test_oracle_pins.py are sharp enough to catch a dropped term,
a wrong sign, a transposed operand, a wrong head map, an off-by-one mask, a shifted digit
exponent and a dropped digit."""
import math
from fractions import Fraction

import mpmath as mp
import numpy as np
import torch

from oracle import exact as E
import workloads as W


def _exp_within_one_ulp(fn) -> bool:
    with mp.workprec(120):
        rng = np.random.default_rng(30)
        for x in np.concatenate([(-rng.random(200) * 104), -rng.random(100)]).astype(np.float32):
            w = fn(float(x))
            ref = mp.exp(mp.mpf(float(x)))
            ulp = float(np.spacing(np.float32(float(ref)))) if float(ref) > 0 else 2.0 ** -149
            if abs(mp.mpf(w) - ref) > ulp:
                return False
    return True


def _naive64(Q, K, V, causal, scale):
    Q, K, V = (t.double() for t in (Q, K, V))
    rep = Q.shape[1] // K.shape[1]
    K, V = K.repeat_interleave(rep, 1), V.repeat_interleave(rep, 1)
    s = (Q @ K.transpose(-1, -2)) * scale
    if causal:
        S = s.shape[-1]
        s = s.masked_fill(torch.ones(S, S, dtype=torch.bool).triu(1), float("-inf"))
    return torch.softmax(s, -1) @ V


def _agrees_with_naive(Q, K, V, causal) -> bool:
    out = E.det_attn(Q, K, V, causal=causal)
    ref = _naive64(Q, K, V, causal, E.default_scale(Q.shape[-1])).numpy()
    return bool(np.max(np.abs(out - ref)) < 2e-6)


def test_unmutated_oracle_passes_the_checks_used_here():
    assert _exp_within_one_ulp(E.exp32_det)
    Q, K, V = W.random_attn(31, 1, 4, 2, 8, 8, torch.bfloat16, True)
    assert _agrees_with_naive(Q, K, V, True)


def test_dropped_taylor_term_is_caught(monkeypatch):
    monkeypatch.setattr(E, "EXP_TAYLOR", E.EXP_TAYLOR[:7] + [0.0])
    assert not _exp_within_one_ulp(E.exp32_det)


def test_wrong_reduction_sign_is_caught(monkeypatch):
    def bad_exp(x):
        if x < E.EXP_X_MIN:
            return 0.0
        fx = Fraction(x)
        k = round(E.rn32(fx * Fraction(E.EXP_L2E)))
        r1 = E.rn32(fx + k * Fraction(E.EXP_C1))     # sign slip
        r = E.rn32(Fraction(r1) - k * Fraction(E.EXP_C2))
        p = Fraction(E.EXP_TAYLOR[7])
        for n in range(6, -1, -1):
            p = Fraction(E.rn32(p * Fraction(r) + Fraction(E.EXP_TAYLOR[n])))
        return E.rn32(p * Fraction(2) ** k)
    assert not _exp_within_one_ulp(bad_exp)


def test_floor_instead_of_nearest_reduction_is_caught():
    def bad_exp(x):
        if x < E.EXP_X_MIN:
            return 0.0
        fx = Fraction(x)
        k = math.floor(E.rn32(fx * Fraction(E.EXP_L2E)))   # floor, not ties-to-even
        r1 = E.rn32(fx - k * Fraction(E.EXP_C1))
        r = E.rn32(Fraction(r1) - k * Fraction(E.EXP_C2))
        p = Fraction(E.EXP_TAYLOR[7])
        for n in range(6, -1, -1):
            p = Fraction(E.rn32(p * Fraction(r) + Fraction(E.EXP_TAYLOR[n])))
        return E.rn32(p * Fraction(2) ** k)
    assert not _exp_within_one_ulp(bad_exp)


def test_transposed_scores_are_caught(monkeypatch):
    def swapped(self, b, h, i, kv_lo, kv_hi):
        kk = self._k(b, self.kv_head(h))
        qq = self._q(b, h)
        return {j: E.score(kk[i], qq[j], self.scale32) for j in range(kv_lo, kv_hi) if self.valid(i, j)}
    monkeypatch.setattr(E.AttnProblem, "scores_row", swapped)
    Q, K, V = W.random_attn(32, 1, 2, 2, 8, 8, torch.float32, False)
    assert not _agrees_with_naive(Q, K, V, False)


def test_wrong_gqa_head_map_is_caught(monkeypatch):
    monkeypatch.setattr(E.AttnProblem, "kv_head", lambda self, h: h % self.Hkv)
    Q, K, V = W.random_attn(33, 1, 4, 2, 8, 8, torch.bfloat16, False)
    assert not _agrees_with_naive(Q, K, V, False)


def test_causal_off_by_one_is_caught(monkeypatch):
    monkeypatch.setattr(E.AttnProblem, "valid", lambda self, i, j: (not self.causal) or j < i)   # drops the diagonal key
    Q, K, V = W.random_attn(34, 1, 2, 2, 8, 8, torch.float32, True)
    assert not _agrees_with_naive(Q, K, V, True)


def test_shifted_digit_exponent_is_caught(monkeypatch):
    Q, K, V = W.random_attn(35, 1, 1, 1, 5, 4, torch.float32, False)
    monkeypatch.setattr(E, "NUM_E0", -321)   # digits written one bit too fine
    P = E.AttnProblem(Q, K, V)
    num, den, _ = P.accumulate(P.rowmax())
    monkeypatch.setattr(E, "NUM_E0", -320)   # ...and read at the contract's weight
    assert not _agrees_with_naive_out(E.finalize(num, den), Q, K, V)


def _agrees_with_naive_out(out, Q, K, V):
    ref = _naive64(Q, K, V, False, E.default_scale(Q.shape[-1])).numpy()
    return bool(np.max(np.abs(out - ref)) < 2e-6)


def test_dropped_top_digit_in_finalize_is_caught(monkeypatch):
    orig = E.finalize_value

    def bad(num_digits, den_digits):
        nd = list(num_digits)
        nd[10] = 0            # loses the digit of weight 2**0, where values near 1 live
        return orig(nd, den_digits)
    monkeypatch.setattr(E, "finalize_value", bad)
    Q, K, V = W.random_attn(36, 1, 1, 1, 6, 4, torch.float32, False)
    assert not _agrees_with_naive_out(E.det_attn(Q, K, V), Q, K, V)


# ---------------------------------------------------------------- cross-entropy backward

def _dce_backward_agrees_with_torch(oracle_native, reduction) -> bool:
    g = torch.Generator().manual_seed(41)
    x = torch.randn(10, 200, generator=g) * 2
    t = torch.randint(0, 200, (10,), generator=g)
    loss, denom, m, den, st = oracle_native.DCE(x).forward(t.numpy())
    up = torch.rand(10 if reduction == "none" else 1, generator=g).float() + 0.5
    grad = E.dce_backward(x, t.numpy(), m, denom, E.dce_go(up.numpy(), 10, reduction))
    x64 = x.double().requires_grad_(True)
    torch.nn.functional.cross_entropy(x64, t, reduction=reduction).backward(
        up.double() if reduction == "none" else up.double()[0])
    return bool(np.max(np.abs(grad - x64.grad.numpy())) < 2.0 ** -20)


def test_unmutated_backward_passes(oracle_native):
    for reduction in ("none", "sum", "mean"):
        assert _dce_backward_agrees_with_torch(oracle_native, reduction)


def test_one_hot_at_the_wrong_column_is_caught(monkeypatch, oracle_native):
    orig = E.dce_backward

    def bad(logits, targets, m, denom, go):
        return orig(logits, (np.asarray(targets) + 1) % np.asarray(logits).shape[1], m, denom, go)
    monkeypatch.setattr(E, "dce_backward", bad)
    assert not _dce_backward_agrees_with_torch(oracle_native, "none")


def test_mean_without_the_division_by_n_is_caught(monkeypatch, oracle_native):
    orig = E.dce_go

    def bad(grad, N, reduction):
        return orig(grad, N, "sum" if reduction == "mean" else reduction)
    monkeypatch.setattr(E, "dce_go", bad)
    assert not _dce_backward_agrees_with_torch(oracle_native, "mean")


def test_mean_over_n_minus_one_is_caught(monkeypatch):
    def bad(loss, reduction):
        L = np.asarray(loss, dtype=np.float32).reshape(-1)
        S = sum((Fraction(float(v)) for v in L), Fraction(0))
        return np.float32(float(S) / (len(L) - 1)) if reduction == "mean" else np.float32(float(S))
    monkeypatch.setattr(E, "dce_reduce", bad)
    # the printed-value pin of the reduction: mean of [1, 2, 4] is RN32(7/3) = 0x40155555
    got = E.dce_reduce(np.array([1, 2, 4], np.float32), "mean")
    assert np.float32(got).view(np.uint32) != np.uint32(0x40155555)
