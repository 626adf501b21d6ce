"""The oracle against values the pages print (fixtures under tests/golden/, each with its
citation).  CPU only."""
import os

import numpy as np
import pytest
import torch

from oracle import exact as E

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        lines = f.read().splitlines()
    for line in lines:
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "key":
            continue
        out[key] = [float(v) for v in vals] if len(vals) > 1 else float(vals[0])
    return out


def test_dce_matches_torch_within_the_printed_bounds(oracle_native):
    """Loss and mean-reduced gradient of the oracle against torch in float64 on a batch of the
    page's size (1,024 tokens; a 32,768-word vocabulary gives losses near 10), within the
    page's printed maxima; the loss and gradient are the same bytes for each vocab split."""
    g = _fixture("dce_torch_match.txt")
    N, V = int(g["tokens"]), 32768
    gen = torch.Generator().manual_seed(11)
    x = torch.randn(N, V, generator=gen) * 2.0
    t = torch.randint(0, V, (N,), generator=gen)
    D = oracle_native.DCE(x)
    loss, denom, m, den, st = D.forward(t.numpy())
    go = E.dce_go(np.ones(1, np.float32), N, "mean")
    grad = oracle_native.dce_backward_many(x, t.numpy(), m, denom, go)
    for n in g["vocab_splits"][1:]:
        splits = [V // int(n)] * int(n)
        l2, d2, m2, _, _ = D.forward(t.numpy(), splits=splits)
        assert np.array_equal(l2.view(np.uint32), loss.view(np.uint32)) and np.array_equal(d2, denom)
    x64 = x.double().requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(x64, t, reduction="none")
    assert 8.0 < float(ref.mean()) < 14.0                      # the page's loss magnitude
    assert float((torch.from_numpy(loss).double() - ref.detach()).abs().max()) <= g["loss_abs_max"]
    ref.mean().backward()
    assert float((torch.from_numpy(grad).double() - x64.grad).abs().max()) <= g["grad_abs_max"]
