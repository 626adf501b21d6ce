"""GPU parity of the det-cross-entropy backward, the loss reductions and the autograd
wrapper, through the C ABI, against the oracle (oracle/exact.py and its vectorized twin in
oracle/native.py, pinned in test_dce_backward_oracle.py).

Every dLogits element and every reduced loss is compared bit for bit: the reading of the
det-cross-entropy page's backward fixes each rounding (f64 division, f32 subtraction of the
one-hot, f32 product with the upstream gradient), so the tolerance is zero.  bf16 logits get
bf16 gradients: the f32 dLogits rounded to nearest even, which the test takes with torch's
own conversion of the oracle's f32 values.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import exact as E

pytestmark = pytest.mark.gpu

cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


@pytest.fixture(scope="module")
def da():
    import bitwise_deterministic_shard_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def orc():
    from oracle import native
    native.build()
    return native


def _want(orc, x, t, rm, rd, go, dtype):
    w = torch.from_numpy(orc.dce_backward_many(x, t.cpu().numpy(), rm, rd, go))
    return w if dtype == torch.float32 else w.to(dtype)


def _assert_same(got, want, what):
    a, b = got.detach().cpu(), want.cpu()
    assert a.dtype == b.dtype, what
    ia = a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16)
    ib = b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16)
    if not torch.equal(ia, ib):
        d = (ia != ib).nonzero()
        raise AssertionError(f"{what}: {d.shape[0]} elements differ, first at {d[:5].tolist()}")


@cuda
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("reduction", ["none", "sum", "mean"])
@pytest.mark.parametrize("V", [1, 12, 517, 4096, 5003, 8200])   # 12, 4096, 8200: 16-byte rows (vector path)
def test_backward_matches_oracle(da, orc, dt, reduction, V):
    g = torch.Generator().manual_seed(60 + V)
    N = 37
    x = (torch.randn(N, V, generator=g) * 3).to(dt)
    t = torch.randint(0, V, (N,), generator=g)
    grad = torch.rand(N if reduction == "none" else 1, generator=g) * 2 - 0.5
    xd, td = x.cuda(), t.cuda()
    loss, m, denom = da.forward(xd, td)
    got = da.dce_backward(xd, td, m, denom, grad.cuda(), reduction)
    rl, rd, rm, rden, st = orc.DCE(x).forward(t.numpy())
    go = E.dce_go(grad.numpy(), N, reduction)
    _assert_same(got, _want(orc, x, t, rm, rd, go, dt), f"dLogits {dt} {reduction} V={V}")


@cuda
def test_backward_extreme_logits(da, orc):
    """Rows whose weights underflow, a -inf logit, a huge spread and the target at the max."""
    N, V = 6, 3001
    g = torch.Generator().manual_seed(71)
    x = torch.randn(N, V, generator=g)
    x[0] *= 200.0                      # most weights underflow to zero
    x[1, 5] = float("-inf")
    x[2] = 0.0                         # uniform row
    x[3, 17] = 1e30                    # one dominant logit, the target below
    x[4, ::7] = -1e30
    t = torch.tensor([3, 5, 0, 17, 1, V - 1])
    xd, td = x.cuda(), t.cuda()
    loss, m, denom = da.forward(xd, td)
    grad = torch.linspace(-2, 2, N)
    got = da.dce_backward(xd, td, m, denom, grad.cuda(), "none")
    rl, rd, rm, rden, st = orc.DCE(x).forward(t.numpy())
    go = E.dce_go(grad.numpy(), N, "none")
    _assert_same(got, _want(orc, x, t, rm, rd, go, torch.float32), "extreme rows")


@cuda
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_cross_entropy_autograd_split_invariant(da, orc, dt):
    g = torch.Generator().manual_seed(72)
    N, V = 29, 4099
    x = (torch.randn(N, V, generator=g) * 2).to(dt)
    t = torch.randint(0, V, (N,), generator=g)
    outs = []
    for splits in ([V], [2049, 2050], [1024, 1024, 1024, 1027]):
        for reduction in ("none", "sum", "mean"):
            xd = x.cuda().requires_grad_(True)
            loss = da.cross_entropy(xd, t.cuda(), reduction=reduction, splits=splits)
            up = torch.arange(1, N + 1, dtype=torch.float32, device="cuda") / 8 if reduction == "none" else None
            (loss.backward(up) if up is not None else loss.backward())
            outs.append((reduction, loss.detach().clone(), xd.grad.clone()))
    for reduction in ("none", "sum", "mean"):
        same = [o for o in outs if o[0] == reduction]
        for o in same[1:]:
            assert torch.equal(o[1], same[0][1]) and torch.equal(o[2], same[0][2]), reduction
    rl, rd, rm, rden, st = orc.DCE(x).forward(t.numpy())
    for reduction, loss, grad in outs[:3]:
        if reduction == "none":
            up = (torch.arange(1, N + 1, dtype=torch.float32) / 8).numpy()
            _assert_same(loss, torch.from_numpy(rl), "loss none")
        else:
            up = np.ones(1, dtype=np.float32)
            assert loss.dtype == torch.float32 and loss.dim() == 0
            _assert_same(loss.reshape(1), torch.tensor([E.dce_reduce(rl, reduction)]), f"loss {reduction}")
        go = E.dce_go(up, N, reduction)
        _assert_same(grad, _want(orc, x, t, rm, rd, go, dt), f"grad {reduction}")


@cuda
@pytest.mark.parametrize("n", [0, 1, 2, 255, 256, 257, 100003])
@pytest.mark.parametrize("reduction", ["sum", "mean"])
def test_reduce_matches_oracle(da, n, reduction):
    g = torch.Generator().manual_seed(73 + n)
    L = (torch.rand(n, generator=g) * 20).float()
    if n > 3:
        L[::97] *= 2.0 ** 60           # wide exponent spread: the exact sum differs from any fp order
        L[1::89] = 2.0 ** -100
    got = da.dce_reduce(L.cuda(), reduction)
    want = E.dce_reduce(L.numpy(), reduction)
    _assert_same(got.reshape(1), torch.tensor([want], dtype=torch.float32), f"{reduction} n={n}")
    perm = torch.randperm(n, generator=g)
    _assert_same(da.dce_reduce(L[perm].cuda(), reduction).reshape(1), got.reshape(1), "permuted")


@cuda
def test_reduce_nonfinite(da):
    inf, nan = float("inf"), float("nan")
    for vals in ([1.0, inf, 2.0], [-inf, 1.0], [inf, -inf], [1.0, nan], [3.4e38, 3.4e38]):
        L = torch.tensor(vals)
        for reduction in ("sum", "mean"):
            got = da.dce_reduce(L.cuda(), reduction).cpu()
            want = torch.tensor(E.dce_reduce(L.numpy(), reduction))
            assert (torch.isnan(got) and torch.isnan(want)) or torch.equal(got, want), (vals, reduction)


@cuda
def test_backward_argument_errors(da):
    x = torch.randn(4, 10, device="cuda")
    t = torch.tensor([0, 1, 2, 3], device="cuda")
    loss, m, denom = da.forward(x, t)
    with pytest.raises(da.DetAttnError):
        da.dce_backward(x, t, m, denom, torch.ones(3, device="cuda"), "none")
    with pytest.raises(da.DetAttnError):
        da.cross_entropy(x, t, reduction="avg")


@cuda
def test_vocab_sharded_backward_sampled_rows(da, orc):
    """The N4096 x V128256 f32 vocab-sharded workload: mean-reduced cross-entropy and its
    dLogits, split-invariant, and sampled rows against the oracle."""
    w = W.vocab_sharded_ce()
    x, t = w.tensors("cuda")
    grads = []
    for sp in (w.splits[0], w.splits[-1]):
        xd = x.clone().requires_grad_(True)
        loss = da.cross_entropy(xd, t, reduction="mean", splits=sp)
        loss.backward()
        grads.append((loss.detach(), xd.grad))
        del xd
    assert torch.equal(grads[0][0], grads[1][0]) and torch.equal(grads[0][1], grads[1][1])
    rows = np.arange(3, w.N, 64, dtype=np.int64)
    xs = x[torch.from_numpy(rows).cuda()].cpu()
    ts = t[torch.from_numpy(rows).cuda()].cpu()
    rl, rd, rm, rden, st = orc.DCE(xs).forward(ts.numpy())
    go = E.dce_go(np.ones(1, dtype=np.float32), w.N, "mean")[: len(rows)]
    want = _want(orc, xs, ts, rm, rd, go, torch.float32)
    _assert_same(grads[0][1][torch.from_numpy(rows).cuda()], want, "vocab-sharded sampled dLogits")
    # the det-cross-entropy page's match to torch: loss within 1.9e-6, gradient within 1.2e-10
    x64 = x.double().requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(x64, t)
    ref.backward()
    assert abs(float(grads[0][0]) - float(ref)) < 1.9e-6
    assert float((grads[0][1].double() - x64.grad).abs().max()) < 1.2e-10
