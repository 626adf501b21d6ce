"""Pins of the oracle's cross-entropy backward and loss reductions (page "det-cross-entropy",
sections "API" and "Method": gradient softmax(x_i) - onehot(t_i), reduction "mean" / "sum" /
"none").  Each pin comes from outside the oracle's own formula: torch's float64 autograd,
printed hex values of the single-rounded quantities, invariants of softmax, or exact
rational arithmetic."""
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import exact as E


def f32_hex(h: str) -> np.float32:
    return np.frombuffer(struct.pack("<I", int(h, 16)), dtype=np.float32)[0]


def forward_state(oracle_native, x, t):
    loss, denom, m, den, st = oracle_native.DCE(x).forward(t.numpy())
    return loss, denom, m, st


@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
def test_backward_matches_torch_autograd(oracle_native, reduction):
    g = torch.Generator().manual_seed(31)
    x = torch.randn(12, 300, generator=g) * 2
    t = torch.randint(0, 300, (12,), generator=g)
    loss, denom, m, st = forward_state(oracle_native, x, t)
    up = torch.rand(12 if reduction == "none" else 1, generator=g).float() + 0.5
    go = E.dce_go(up.numpy(), 12, reduction)
    grad = E.dce_backward(x, t.numpy(), m, denom, go)
    x64 = x.double().requires_grad_(True)
    ref_loss = torch.nn.functional.cross_entropy(x64, t, reduction=reduction)
    ref_loss.backward(up.double() if reduction == "none" else up.double()[0])
    ref = x64.grad.numpy()
    # p carries exp32_det's error (a few ulp) and three single f32 roundings: relative to the
    # value off the target; p - 1 at the target is absolute (magnitude <= 1)
    onehot = np.zeros_like(ref, dtype=bool)
    onehot[np.arange(12), t.numpy()] = True
    rel = np.abs(grad[~onehot] - ref[~onehot]) / np.abs(ref[~onehot])
    assert rel.max() < 2.0 ** -20
    assert np.max(np.abs(grad[onehot] - ref[onehot])) < 2.0 ** -21
    small = np.abs(ref) < 1e-4   # entries the size of the page's gradient differences
    assert np.max(np.abs(grad[small] - ref[small])) < 1.2e-10


def test_uniform_logits_give_single_rounded_one_over_v(oracle_native):
    x = torch.full((3, 7), -2.5)
    t = torch.tensor([0, 3, 6])
    loss, denom, m, st = forward_state(oracle_native, x, t)
    assert np.all(denom == 7.0)
    grad = E.dce_backward(x, t.numpy(), m, denom, np.ones(3, dtype=np.float32))
    p = f32_hex("3e124925")           # RN32(RN64(1/7)): 0x3FC2492492492492 rounds to 0x3E124925
    pm1 = f32_hex("bf5b6db7")         # RN32(p - 1) = -0.857142865657806...
    for i, ti in enumerate([0, 3, 6]):
        for v in range(7):
            assert grad[i, v] == (pm1 if v == ti else p)


def test_single_class_gradient_is_zero(oracle_native):
    x = torch.randn(5, 1)
    t = torch.zeros(5, dtype=torch.int64)
    loss, denom, m, st = forward_state(oracle_native, x, t)
    grad = E.dce_backward(x, t.numpy(), m, denom, np.ones(5, dtype=np.float32))
    assert np.all(grad == 0)


def test_gradient_rows_sum_to_zero_within_rounding(oracle_native):
    g = torch.Generator().manual_seed(32)
    x = (torch.randn(8, 257, generator=g) * 3).to(torch.bfloat16)
    t = torch.randint(0, 257, (8,), generator=g)
    loss, denom, m, st = forward_state(oracle_native, x, t)
    grad = E.dce_backward(x, t.numpy(), m, denom, np.ones(8, dtype=np.float32)).astype(np.float64)
    assert np.max(np.abs(grad.sum(axis=1))) < 257 * 2.0 ** -24


def test_bad_target_subtracts_nothing(oracle_native):
    x = torch.randn(2, 9)
    t = torch.tensor([9, -1])
    loss, denom, m, st = forward_state(oracle_native, x, t)
    grad = E.dce_backward(x, t.numpy(), m, denom, np.ones(2, dtype=np.float32))
    assert np.all(grad > 0)
    assert abs(grad.astype(np.float64).sum(axis=1) - 1).max() < 9 * 2.0 ** -24


def test_reductions_are_exact_sums():
    tiny = np.float32(2.0 ** -30)
    vals = np.array([1.0, tiny, -1.0], dtype=np.float32)
    assert E.dce_reduce(vals, "sum") == tiny                 # a running f32 sum would give 0
    assert E.dce_reduce(vals[::-1], "sum") == tiny
    assert E.dce_reduce(np.array([1, 2, 4], np.float32), "mean") == f32_hex("40155555")   # RN32(7/3)
    assert np.isnan(E.dce_reduce(np.array([1, np.nan], np.float32), "mean"))
    g = np.random.default_rng(33)
    L = (g.random(1000) * 12).astype(np.float32)
    exact = sum(Fraction(float(v)) for v in L)
    assert E.dce_reduce(L, "sum") == np.float32(float(exact))
    assert abs(float(E.dce_reduce(L, "mean")) - float(exact) / 1000) <= 2.0 ** -23 * float(exact) / 1000
    perm = g.permutation(1000)
    assert E.dce_reduce(L[perm], "mean") == E.dce_reduce(L, "mean")


def test_vectorized_backward_equals_exact(oracle_native):
    g = torch.Generator().manual_seed(34)
    x = (torch.randn(5, 203, generator=g) * 4).to(torch.bfloat16)
    t = torch.tensor([0, 202, 17, -3, 99])
    loss, denom, m, st = forward_state(oracle_native, x, t)
    go = np.array([1.0, -0.5, 2.0, 0.25, 3.0], dtype=np.float32)
    a = E.dce_backward(x, t.numpy(), m, denom, go)
    b = oracle_native.dce_backward_many(x, t.numpy(), m, denom, go)
    assert np.array_equal(a, b)


def test_reduce_of_no_losses():
    assert E.dce_reduce(np.zeros(0, np.float32), "sum") == 0
    assert np.isnan(E.dce_reduce(np.zeros(0, np.float32), "mean"))
