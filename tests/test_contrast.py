"""Order-dependence contrasts (context only, CPU).

Page "det-attn", introduction and "Method": the usual float32 online-softmax combine of
KV shards (running max, exp rescale of the running sum and output) gives results whose
bits depend on how the keys are split and in which order the shards are merged, while
the exact digit composition gives one result for every split and order.  Page
"det-cross-entropy", "Correctness": a float32 logsumexp combine over vocabulary shards
changes the bits of some token losses as the split count varies (1, 2, 4, 8), the exact
path none.

The float32 combines below are a few lines of plain torch written for this contrast; they
are not part of the library.  The exact side is the oracle.
"""
import hashlib

import numpy as np
import pytest
import torch

import workloads as W
from oracle import native


@pytest.fixture(autouse=True)
def _one_thread():
    """One torch thread, so the float32 sums run in one fixed order (restored after)."""
    n = torch.get_num_threads()
    yield
    torch.set_num_threads(n)


def _sha(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def _f32_online_softmax(q, k, v, scale, bounds, order):
    """Flash-style float32 combine of per-shard (max, sum, output) states, shards merged in
    `order`; q, k, v float32 [S, D] of one head (non-causal)."""
    m = l = o = None
    for s in order:
        a, b = bounds[s]
        sc = (q @ k[a:b].T) * scale
        ms = sc.max(dim=1).values
        p = torch.exp(sc - ms[:, None])
        ls, os_ = p.sum(dim=1), p @ v[a:b]
        if m is None:
            m, l, o = ms, ls, os_
            continue
        mn = torch.maximum(m, ms)
        ca, cb = torch.exp(m - mn), torch.exp(ms - mn)
        l = l * ca + ls * cb
        o = o * ca[:, None] + os_ * cb[:, None]
        m = mn
    return (o / l[:, None]).numpy()


def _bounds(S, n):
    sp = W.equal_splits(S, n)
    b = np.cumsum([0] + sp)
    return [(int(b[i]), int(b[i + 1])) for i in range(n)]


def test_f32_online_softmax_changes_bits_across_shard_rotations_exact_does_not():
    Q, K, V = W.random_attn(31, 1, 1, 1, 256, 64, torch.float32, False)
    q, k, v = Q[0, 0], K[0, 0], V[0, 0]
    scale = float(np.float32(1.0 / 8.0))
    bounds = _bounds(256, 4)
    outs = [_f32_online_softmax(q, k, v, scale, bounds, [(r + j) % 4 for j in range(4)]) for r in range(4)]
    hashes = {_sha(o) for o in outs}
    drift = max(float(np.abs(o - outs[0]).max()) for o in outs)
    assert len(hashes) > 1, "the float32 combine happened to give one result for every rotation"
    assert 0 < drift < 1e-5   # small drift, on the order the page reports

    # exact: the digits of each shard, composed in every rotation, give one output
    A = native.Attn(Q, K, V, causal=False, scale=scale)
    m = None
    for a, b in bounds:
        mm, _ = A.rowmax(a, b)
        m = mm if m is None else np.maximum(m, mm)
    parts = [A.accumulate(m, a, b)[:2] for a, b in bounds]
    exact = set()
    for r in range(4):
        num = den = None
        for j in range(4):
            n_, d_ = parts[(r + j) % 4]
            num = n_.copy() if num is None else num + n_
            den = d_.copy() if den is None else den + d_
        exact.add(_sha(native.finalize(native.normalize(num, -320)[0], native.normalize(den, -160)[0])))
    _, _, _, fused = A.forward_rows()
    assert exact == {_sha(fused)}


def _f32_lse_loss(x, t, n):
    """Token losses from a float32 logsumexp combine over n equal vocabulary shards."""
    bounds = _bounds(x.shape[1], n)
    lse = None
    for a, b in bounds:
        ls = torch.logsumexp(x[:, a:b], dim=1)
        lse = ls if lse is None else torch.logaddexp(lse, ls)
    return (lse - x[torch.arange(x.shape[0]), t]).numpy()


def test_f32_logsumexp_changes_token_losses_across_splits_exact_does_not():
    g = torch.Generator().manual_seed(71)
    x = torch.randn(1024, 4096, generator=g) * 2
    t = torch.randint(0, 4096, (1024,), generator=g)
    base = _f32_lse_loss(x, t, 1)
    changed = np.zeros(1024, dtype=bool)
    for n in (2, 4, 8):
        changed |= _f32_lse_loss(x, t, n).view(np.uint32) != base.view(np.uint32)
    assert changed.sum() > 0, "no float32 loss changed bits across the splits"

    D = native.DCE(x)
    ref, *_ = D.forward(t.numpy())
    for n in (2, 4, 8):
        got, *_ = D.forward(t.numpy(), splits=W.equal_splits(4096, n))
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
