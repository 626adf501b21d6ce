"""Context-parallel composition around the GPU kernels (det-attn, introduction and "Method":
the output does not depend on how the keys are split over devices).

Two ranks share the one GPU of this machine; each holds every query row and one contiguous
key / value shard, runs its shard's rowmax and accumulate kernels, and the group composes
through torch.distributed (gloo, through host copies): a max all-reduce of the rowmax, an
int64 sum all-reduce of the digits.  No kernel waits on another rank's kernel: the ranks
meet only in the host-side collectives.  The output must equal det_attn over the whole
sequence bit for bit.  A second test poisons every key and value row outside a call's range
with NaN and checks that the kernels never read them (the context-parallel path presents a
shard at its global positions and relies on that)."""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
cuda = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, cuts, causal, outdir):
    import torch.distributed as dist
    import bitwise_deterministic_shard_gb300 as da
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    Q, K, V = W.random_attn(77, 1, 4, 2, 700, 128, torch.bfloat16, causal)
    lo, hi = cuts[rank], cuts[rank + 1]
    st = da.new_status()
    out = da.det_attn_cp(Q.cuda(), K[:, :, lo:hi].cuda().contiguous(), V[:, :, lo:hi].cuda().contiguous(), lo,
                         S_kv=K.shape[2], causal=causal, status=st)
    torch.cuda.synchronize()
    torch.save({"out": out.cpu(), "status": da.read_status(st)}, os.path.join(outdir, f"r{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


@cuda
@pytest.mark.parametrize("causal,cuts", [(True, [0, 300, 700]), (False, [0, 512, 700]), (True, [0, 0, 700])])
def test_context_parallel_two_ranks_equal_fused(causal, cuts):
    import torch.multiprocessing as mp
    import bitwise_deterministic_shard_gb300 as da
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_rank_main, args=(2, _free_port(), cuts, causal, d), nprocs=2, start_method="spawn")
        res = [torch.load(os.path.join(d, f"r{r}.pt")) for r in range(2)]
    Q, K, V = W.random_attn(77, 1, 4, 2, 700, 128, torch.bfloat16, causal)
    ref = da.det_attn(Q.cuda(), K.cuda(), V.cuda(), causal=causal).cpu()
    for r in res:
        assert r["status"] == 0
        assert torch.equal(r["out"], ref)


@cuda
@pytest.mark.parametrize("D,dt", [(128, torch.bfloat16), (64, torch.bfloat16), (256, torch.bfloat16),
                                  (128, torch.float32)])
def test_kernels_read_only_their_key_range(D, dt):
    import bitwise_deterministic_shard_gb300 as da
    Q, K, V = (t.cuda() for t in W.random_attn(78, 1, 2, 2, 400, D, dt, False))
    lo, hi = 130, 290
    Kp, Vp = K.clone(), V.clone()
    for X in (Kp, Vp):
        X[:, :, :lo] = float("nan")
        X[:, :, hi:] = float("nan")
    m = da.rowmax(Q, K, lo, hi)
    num, den = da.accumulate(Q, K, V, m, lo, hi)
    st = da.new_status()
    mp_ = da.rowmax(Q, Kp, lo, hi, status=st)
    nump, denp = da.accumulate(Q, Kp, Vp, m, lo, hi, status=st)
    torch.cuda.synchronize()
    assert da.read_status(st) == 0                  # no NaN row was read
    assert torch.equal(mp_, m) and torch.equal(nump, num) and torch.equal(denp, den)


def _vp_rank_main(rank, world, port, cuts, dt, outdir):
    import torch.distributed as dist
    import bitwise_deterministic_shard_gb300 as da
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    g = torch.Generator().manual_seed(81)
    x = (torch.randn(64, 3001, generator=g) * 2).to(dt)
    t = torch.randint(0, 3001, (64,), generator=g)
    t[5] = 3001                                          # a target outside the vocabulary
    lo, hi = cuts[rank], cuts[rank + 1]
    xl = x[:, lo:hi].cuda().contiguous().requires_grad_(True)
    st = da.new_status()
    loss_rows = da.dce_forward_vp(xl.detach(), t.cuda(), lo, 3001, status=st)[0]
    loss = da.cross_entropy_vp(xl, t.cuda(), lo, 3001, reduction="sum")
    loss.backward()
    torch.cuda.synchronize()
    torch.save({"rows": loss_rows.cpu(), "loss": loss.detach().cpu(), "grad": xl.grad.cpu(),
                "status": da.read_status(st)}, os.path.join(outdir, f"r{rank}.pt"))
    dist.barrier()
    dist.destroy_process_group()


@cuda
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_vocab_parallel_cross_entropy_two_ranks(dt):
    """Two ranks hold columns [0, 1400) and [1400, 3001) of the logits; the composed per-row
    losses, the summed loss and each rank's gradient columns equal the single-device
    cross-entropy bit for bit (det-cross-entropy, "Usage")."""
    import torch.multiprocessing as mp
    import bitwise_deterministic_shard_gb300 as da
    cuts = [0, 1400, 3001]
    with tempfile.TemporaryDirectory() as d:
        mp.start_processes(_vp_rank_main, args=(2, _free_port(), cuts, dt, d), nprocs=2, start_method="spawn")
        res = [torch.load(os.path.join(d, f"r{r}.pt")) for r in range(2)]
    g = torch.Generator().manual_seed(81)
    x = (torch.randn(64, 3001, generator=g) * 2).to(dt)
    t = torch.randint(0, 3001, (64,), generator=g)
    t[5] = 3001
    xd = x.cuda().requires_grad_(True)
    rows = da.dce_forward(x.cuda(), t.cuda())[0].cpu()
    ref = da.cross_entropy(xd, t.cuda(), reduction="sum")
    ref.backward()
    for r, rk in enumerate(res):
        assert rk["status"] == da.STATUS_BAD_TARGET
        assert torch.equal(rk["rows"].view(torch.int32), rows.view(torch.int32))   # NaN row included
        assert torch.equal(rk["loss"].view(torch.int32), ref.detach().cpu().view(torch.int32))
        assert torch.equal(rk["grad"], xd.grad.cpu()[:, cuts[r]:cuts[r + 1]])
