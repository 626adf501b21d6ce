"""Context-parallel composition with real collectives, on the CPU (gloo, world size 2).

Page "det-attn", section "Method": composing KV shards is an int64 addition of digit
arrays plus a max of the rowmax, bit-identical to the single-device result and the same
at every world size.  Here each gloo rank owns a contiguous KV shard, computes its shard
rowmax and digits with the oracle, and the ranks combine them with all_reduce(MAX) and
all_reduce(SUM) on int64 - the collectives a multi-GPU deployment would run.  The result
must equal the fused single-process result bit for bit, in either rank order.  A missing
or duplicated shard must change it (failure detection by comparison).  The vocab-parallel
cross-entropy (page "det-cross-entropy") is composed the same way at the end of the file.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import workloads as W


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, splits, reverse, outq):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import native
    import workloads as W
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    Q, K, V = W.random_attn(77, 1, 2, 1, 64, 16, torch.bfloat16, True)
    A = native.Attn(Q, K, V, causal=True)
    bounds = np.cumsum([0] + splits)
    shard = (world - 1 - rank) if reverse else rank
    lo, hi = int(bounds[shard]), int(bounds[shard + 1])
    m, _ = A.rowmax(lo, hi, nthreads=1)
    mt = torch.from_numpy(m.copy())
    dist.all_reduce(mt, op=dist.ReduceOp.MAX)
    num, den, st = A.accumulate(mt.numpy(), lo, hi, nthreads=1)
    nt, dt_ = torch.from_numpy(num.copy()), torch.from_numpy(den.copy())
    dist.all_reduce(nt, op=dist.ReduceOp.SUM)
    dist.all_reduce(dt_, op=dist.ReduceOp.SUM)
    numc, _ = native.normalize(nt.numpy(), -320)
    denc, _ = native.normalize(dt_.numpy(), -160)
    out = native.finalize(numc, denc)
    if rank == 0:
        outq.put((out, numc, denc, st))
    dist.destroy_process_group()


def _run(splits, reverse):
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, splits, reverse, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    return res


@pytest.fixture(scope="module")
def fused():
    from oracle import native
    Q, K, V = W.random_attn(77, 1, 2, 1, 64, 16, torch.bfloat16, True)
    return native.Attn(Q, K, V, causal=True).forward_rows()


@pytest.mark.parametrize("splits,reverse", [([32, 32], False), ([10, 54], True), ([63, 1], False)])
def test_gloo_allreduce_composition_equals_fused(fused, splits, reverse):
    out, num, den, st = _run(splits, reverse)
    assert st == 0
    assert np.array_equal(num, fused[1]) and np.array_equal(den, fused[2])
    assert np.array_equal(out.view(np.uint32), fused[3].view(np.uint32))


def test_missing_or_duplicated_shard_is_detected(fused):
    from oracle import native
    Q, K, V = W.random_attn(77, 1, 2, 1, 64, 16, torch.bfloat16, True)
    A = native.Attn(Q, K, V, causal=True)
    m = fused[0]
    n0, d0, _ = A.accumulate(m, 0, 32)
    n1, d1, _ = A.accumulate(m, 32, 64)
    good = native.finalize(native.normalize(n0 + n1, -320)[0], native.normalize(d0 + d1, -160)[0])
    assert np.array_equal(good.view(np.uint32), fused[3].view(np.uint32))
    missing = native.finalize(native.normalize(n0, -320)[0], native.normalize(d0, -160)[0])
    dup = native.finalize(native.normalize(n0 + n1 + n1, -320)[0], native.normalize(d0 + d1 + d1, -160)[0])
    assert not np.array_equal(missing, fused[3])
    assert not np.array_equal(dup, fused[3])


# ------------------------------------------------ vocab-parallel cross-entropy (gloo, 2 ranks)
#
# Page "det-cross-entropy", sections "Usage" and "Method": a vocab-parallel LM head keeps a
# column range of the logits per rank; the rowmax composes by max, the denominator digits by
# int64 addition, and finalize gives the loss; the gradient softmax - onehot of each rank's
# columns needs only the global rowmax and denominator.

def _dce_case():
    g = torch.Generator().manual_seed(78)
    x = torch.randn(24, 3001, generator=g) * 2
    t = torch.randint(0, 3001, (24,), generator=g)
    return x, t


def _dce_worker(rank, world, port, splits, outq):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from oracle import native
    from oracle import exact as E
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    x, t = _dce_case()
    D = native.DCE(x)
    bounds = np.cumsum([0] + splits)
    lo, hi = int(bounds[rank]), int(bounds[rank + 1])
    m, _ = D.rowmax(lo, hi, nthreads=1)
    mt = torch.from_numpy(m.copy())
    dist.all_reduce(mt, op=dist.ReduceOp.MAX)
    den, _ = D.denom_digits(mt.numpy(), lo, hi, nthreads=1)
    dt_ = torch.from_numpy(den.copy())
    dist.all_reduce(dt_, op=dist.ReduceOp.SUM)
    denc, _ = native.normalize(dt_.numpy(), -160)
    loss, denom, st = D.finalize(denc, t.numpy(), mt.numpy())
    go = E.dce_go(np.ones(1, np.float32), 24, "mean")
    grad = native.dce_backward_many(x[:, lo:hi], t.numpy() - lo, mt.numpy(), denom, go)
    parts = [None] * world
    dist.all_gather_object(parts, grad)
    if rank == 0:
        outq.put((loss, denom, np.concatenate(parts, axis=1), st))
    dist.destroy_process_group()


@pytest.mark.parametrize("splits", [[1500, 1501], [1, 3000]])
def test_gloo_vocab_parallel_cross_entropy_equals_single_process(splits):
    from oracle import native
    from oracle import exact as E
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_dce_worker, args=(r, 2, port, splits, q)) for r in range(2)]
    for p in procs:
        p.start()
    loss, denom, grad, st = q.get()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    x, t = _dce_case()
    rl, rd, rm, rden, st1 = native.DCE(x).forward(t.numpy())
    want = native.dce_backward_many(x, t.numpy(), rm, rd, E.dce_go(np.ones(1, np.float32), 24, "mean"))
    assert st == 0
    assert np.array_equal(loss.view(np.uint32), rl.view(np.uint32)) and np.array_equal(denom, rd)
    assert np.array_equal(grad.view(np.uint32), want.view(np.uint32))
