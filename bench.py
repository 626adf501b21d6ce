"""Benchmark of the exact, order-invariant softmax reduction on one GB300 (or N replicas).

Metric: exact attention MACs/s on the long-context causal workload (B1 H16 S4096 D128
bf16, 1% of K rows x8), MACs = B * Hq * P * 2D with P the unmasked (query, key) pairs.
A step is one pass of the whole attention path through the C ABI, the calls det_attn makes:
da_rowmax over all keys, then da_accumulate_finalize (exact NUM/DEN sums, normalized, rounded
and divided in the tensor-PV kernel's epilogue: the output is f32, no digits are stored).
Inputs are resident in HBM when the timed region starts; L2 is flushed (a 512 MiB write)
between timed steps, outside the per-step CUDA events.

Under torchrun (N > 1) every rank runs its own independent problem of the same shape
(weak scaling; the path partitions by (batch, head) with no exchange), the timed region
is bracketed by barriers, and rank 0 reports total MACs / max time over ranks.

--impl reference times the oracle (the exact C implementation, as it stands) on the host
cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes as C
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "exact attention MACs/s (S=4096,D=128,bf16) and % of binding INT/FP64 pipe peak"
UNIT = "MAC/s"


# DRAM bytes (read + write) of one accumulate launch at the metric workload: dram__bytes_read.sum +
# dram__bytes_write.sum (189.20 MB + 6.43 MB) of the 4-head case of the same kernel (`python bench.py
# --heads 4 --dce-rows 256 --steps 1 --warmup 1 --no-cpu-baseline --no-sharded` under ncu, -k
# regex:accumulate_tp -s 1 -c 1) scaled by 4 (the traffic is per head: the score cache, the V digit
# planes and the output of each head).  None whenever the kernel has changed since that capture.
ACC_TRAFFIC_PER_LAUNCH = 4 * (189_380_608 + 8_980_224)


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except OSError:
        return {}


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    def __init__(self, gpu_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={q}", "--format=csv,noheader",
                                       "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1].split()[0]))
                smax.append(float(parts[2].split()[0]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_sample(w, Q, K, V, rows_per_head: int, nthreads: int):
    """Time the oracle's fused pass on sampled query rows; returns (MACs, seconds, sample)."""
    from oracle import native
    native.build()
    A = native.Attn(Q, K, V, w.causal, w.scale)
    rng = np.random.default_rng(0)
    rows = []
    for h in range(w.Hq):
        for i in rng.choice(w.S, size=rows_per_head, replace=False):
            rows.append(h * w.S + int(i))
    rows = np.asarray(rows, dtype=np.int64)
    keys = (rows % w.S) + 1 if w.causal else np.full(len(rows), w.S)
    macs = int(keys.sum()) * 2 * w.D
    t0 = time.perf_counter()
    A.forward_rows(rows=rows, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return macs, dt, f"{len(rows)} query rows ({rows_per_head} per head, seeded), all their keys"


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = W.long_context_causal()
    Q, K, V = w.tensors("cpu")
    cores = os.cpu_count() or 1
    rows_per_head = args.ref_rows_step
    vals, secs = [], []
    for s in range(args.warmup + args.steps):
        macs, dt, sample = oracle_sample(w, Q, K, V, rows_per_head, cores)
        if s >= args.warmup:
            vals.append(macs / dt)
            secs.append(dt)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": statistics.median(secs) * 1e3,   # one timed step = one sample of the workload
            "ms_per_full_workload_extrapolated": w.attn_macs / v * 1e3,
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D, "causal": True,
                       "input_dtype": "bf16", "parallelism": "single GPU" if world == 1 else f"replicas x{world}",
                       "l2": "host oracle on sampled query rows (no device cache involved)",
                       "attn_macs_per_step": w.attn_macs, "pairs_per_step": w.pairs},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_dce(args, dev, stream):
    """The cross-entropy rows of the path on the vocab-sharded workload (N4096 x V128256 f32
    logits, resident in HBM; 2.1 GB, larger than L2, so no flush): per step the forward
    (dce_rowmax, dce_denom_digits, dce_finalize), the mean reduction and the backward
    (dce_backward), each bracketed by CUDA events on the launching stream.  HBM roofline per
    kernel: algorithmic bytes (logits read once per kernel; the backward also writes dLogits)
    over its event time."""
    import bitwise_deterministic_shard_gb300 as da
    L = da.lib()
    w = W.vocab_sharded_ce()
    if args.dce_rows != w.N:                   # smaller case of the same kernels (profiling)
        w.name = w.name.replace(f"N{w.N}", f"N{args.dce_rows}")
        w.N = args.dce_rows
    x, t = w.tensors(dev)
    M, _keep = da._matrix(x)
    N, V = w.N, w.V
    m = torch.empty(N, dtype=torch.float32, device=dev)
    den = torch.empty(N, 6, dtype=torch.int64, device=dev)
    loss = torch.empty(N, dtype=torch.float32, device=dev)
    denom = torch.empty(N, dtype=torch.float64, device=dev)
    red = torch.empty((), dtype=torch.float32, device=dev)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    dx = torch.empty_like(x)
    sp = C.c_void_p(stream.cuda_stream)

    def ptr(a):
        return C.c_void_p(a.data_ptr())

    def step(ev):
        ev[0].record(stream)
        assert L.dce_rowmax(C.byref(M), 0, V, ptr(m), None, sp) == 0
        ev[1].record(stream)
        assert L.dce_denom_digits(C.byref(M), ptr(m), 0, V, ptr(den), 0, None, sp) == 0
        ev[2].record(stream)
        assert L.dce_finalize(ptr(den), C.byref(M), ptr(t), ptr(m), ptr(loss), ptr(denom), None, sp) == 0
        assert L.dce_reduce(ptr(loss), N, 2, ptr(red), sp) == 0
        ev[3].record(stream)
        assert L.dce_backward(C.byref(M), ptr(t), ptr(m), ptr(denom), ptr(one), 2, ptr(dx), None, sp) == 0
        ev[4].record(stream)

    mk = lambda: [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for _ in range(args.warmup):
        step(mk())
    torch.cuda.synchronize()
    evs = [mk() for _ in range(args.steps)]
    for e in evs:
        step(e)
    torch.cuda.synchronize()
    ms = lambda a, b: statistics.mean(e[a].elapsed_time(e[b]) for e in evs)
    k = {"rowmax": ms(0, 1), "denom_digits": ms(1, 2), "finalize_reduce": ms(2, 3), "backward": ms(3, 4)}
    step_ms = ms(0, 4)
    nbytes = N * V * x.element_size()
    traffic = {"rowmax": nbytes, "denom_digits": nbytes, "backward": 2 * nbytes}
    peak = _peaks().get("hbm_gbs") or 6800.0
    roof = {kk: {"achieved_gbs": b / (k[kk] * 1e-3) / 1e9, "frac": b / (k[kk] * 1e-3) / 1e9 / peak,
                 "bytes": b} for kk, b in traffic.items()}
    out = {"workload": w.name, "tokens_per_s": N / (step_ms * 1e-3), "ms_per_step": step_ms,
           "kernels_ms": k, "hbm_roofline": roof, "hbm_peak_gbs": peak,
           "peak_basis": "measured copy bandwidth (MEASURED_PEAKS.json)" if _peaks().get("hbm_gbs")
           else "fallback 6.8 TB/s", "gpu_launches_per_step": 5}
    if not args.no_cpu_baseline:
        from oracle import native
        from oracle import exact as E
        native.build()
        rows = 512
        xs, ts = x[:rows].cpu(), t[:rows].cpu()
        t0 = time.perf_counter()
        rl, rd, rm, rden, st = native.DCE(xs).forward(ts.numpy())
        native.dce_backward_many(xs, ts.numpy(), rm, rd, E.dce_go(np.ones(1, np.float32), N, "mean")[:rows])
        dt = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": rows / dt, "unit": "tokens/s", "cores": native.default_threads(),
                               "kind": "oracle",
                               "sample": f"{rows} tokens x {V} logits: forward (exact C) and backward (numpy)",
                               "seconds": dt}
    return out


def run_ours(args, rank, world, local_rank):
    import bitwise_deterministic_shard_gb300 as da
    da.lib()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    w = W.long_context_causal()
    if args.heads != w.Hq:                     # smaller case of the same kernels (profiling)
        w.Hq = w.Hkv = args.heads
        w.name = w.name.replace("H16", f"H{args.heads}")
    if rank > 0:
        w.seed = w.seed + 1000 * rank          # an independent problem per rank
    Qh, Kh, Vh = w.tensors("cpu")
    Q, K, V = Qh.to(dev), Kh.to(dev), Vh.to(dev)
    P = da._Problem(Q, K, V, True, None)
    L = da.lib()
    ws = torch.empty(L.da_workspace_bytes(P.ref(), 1), dtype=torch.uint8, device=dev)
    kvws = torch.empty(L.da_kv_workspace_bytes(P.ref()), dtype=torch.uint8, device=dev)
    rows = w.B * w.Hq * w.S
    m = torch.empty(rows, dtype=torch.float32, device=dev)
    out = torch.empty(w.B, w.Hq, w.S, w.D, dtype=torch.float32, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    sp = C.c_void_p(stream.cuda_stream)

    def ptr(t):
        return C.c_void_p(t.data_ptr())

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        # pass 1: keys and values prepared once, rowmax, every exact score kept in the workspace's cache
        assert L.da_rowmax_cached(P.ref(), ptr(m), ptr(ws), ws.numel(), sp) == 0
        if ev:
            ev[1].record(stream)
        # pass 2: the exact sums from the cached scores with the global rowmax, finalized in the
        # tensor-PV kernel's epilogue (the calls da_det_attn makes)
        assert L.da_accumulate_finalize_cached(P.ref(), ptr(m), ptr(out), ptr(ws), ws.numel(), sp) == 0
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = Clocks(local_rank) if rank == 0 else None
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(args.steps):
        flush.zero_()
        step(evs[s])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t0
    ck = clocks.stop() if clocks else None
    k_rowmax = [e[0].elapsed_time(e[1]) for e in evs]
    k_acc = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    ms = statistics.mean(step_ms)
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    # --- end to end through the C ABI with host buffers (pinned): da_det_attn_host copies Q, K, V
    # up, runs det_attn and copies the output down, in groups of heads whose copies overlap the
    # kernels; the whole call is inside the timed region
    Qp, Kp, Vp = Qh.pin_memory(), Kh.pin_memory(), Vh.pin_memory()
    outp = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    hdesc = da._Desc()
    hdesc.q, hdesc.k, hdesc.v = da._host_tensor(Qp, "Q"), da._host_tensor(Kp, "K"), da._host_tensor(Vp, "V")
    hdesc.causal, hdesc.scale, hdesc.dev_status = 1, float("nan"), None
    e2e_groups = 4
    hws_bytes = int(L.da_det_attn_host_workspace_bytes(C.byref(hdesc), e2e_groups))
    hws = torch.empty(hws_bytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        assert L.da_det_attn_host(C.byref(hdesc), ptr(outp), e2e_groups, ptr(hws), hws_bytes, sp) == 0

    for _ in range(max(1, args.warmup)):
        flush.zero_()
        e2e_step()
    torch.cuda.synchronize()
    macs_step = w.attn_macs
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    assert torch.equal(outp, out.cpu())
    h2d = (Qh.numel() + Kh.numel() + Vh.numel()) * Qh.element_size()
    d2h = out.numel() * 4

    # --- the sharded path on the same workload: ring steps 1..32 as equal kv_splits through
    # da_det_attn_sharded (every shard's rowmax, compose_max, accumulate into one digit array, finalize)
    sharded = {}
    if not args.no_sharded:
        for splits, order in w.splits:
            n = len(splits)
            wsn = torch.empty(L.da_workspace_bytes(P.ref(), n), dtype=torch.uint8, device=dev)
            spv = (C.c_int64 * n)(*splits)
            ordv = (C.c_int32 * n)(*order)
            outs = torch.empty_like(out)

            def sh_step():
                assert L.da_det_attn_sharded(P.ref(), spv, n, ordv, ptr(outs), ptr(wsn), wsn.numel(), sp) == 0

            flush.zero_()
            sh_step()
            ts = []
            for _ in range(max(1, args.steps // 3)):
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                sh_step()
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b))
            torch.cuda.synchronize()
            assert torch.equal(outs, out), f"sharded ({n} splits) differs from the fused output"
            t_med = statistics.median(ts)
            sharded[str(n)] = {"ms": t_med, "macs_per_s": macs_step / (t_med * 1e-3), "bit_identical_to_fused": True}
            del wsn
    if rank != 0:
        return
    dce = run_dce(args, dev, stream)
    macs = w.attn_macs
    value = macs * world / (ms * 1e-3)
    e2e_val = macs * world / (statistics.mean(e2e_ms) * 1e-3)
    # Roofline of the dominant kernel (accumulate + finalize), on the algorithmic basis: per unmasked
    # (query, key) pair, D exact PV multiply-adds, 2 flop each (the pair's D score multiply-adds run
    # in pass 1, which hands the exact score over through the score cache), over the kernel's event
    # time, against the measured dense bf16 tensor peak (the exact products run on the tensor cores
    # as integer digit products).  Two further views:
    #  - mma_util: the MMA work the kernel actually issues for its digit decomposition (per 128-key tile
    #    of 16 query rows: 24 PV MMAs M128 N160 K16 and 8 DEN MMAs M128 N16 K16, plus 32 score MMAs
    #    M128 N64 K16 when the scores are recomputed instead of read from pass 1's cache) against the
    #    same peak;
    #  - int_pipe: the whole path's exact multiply-adds per second (D score + D PV per pair, each once,
    #    over the step time) against the integer pipe's rate of exact 32 x 32 -> 64-bit multiply-adds,
    #    measured by the library's probe kernel in this run (the metric's "% of binding INT pipe peak":
    #    what an exact integer-pipe implementation could reach at best).
    pk = _peaks()
    sm_clock = (ck or {}).get("sm_mhz") or pk.get("clocks_under_load", {}).get("sm_mhz_median") or 1447.0
    acc_ms = statistics.mean(k_acc)
    alg_macs = w.pairs * w.D                                             # per launch: PV
    achieved = 2.0 * alg_macs / (acc_ms * 1e-3) / 1e12                   # TFLOP/s
    cached = L.da_score_cache_bytes(P.ref()) > 0
    tile_macs = (0 if cached else 32 * 128 * 64 * 16) + 24 * 128 * 160 * 16 + 8 * 128 * 16 * 16
    tiles = w.B * w.Hq * sum(-(-min(w.S, 16 * (qi + 1)) // 128) for qi in range(-(-w.S // 16)))
    mma_tflops = 2.0 * tile_macs * tiles / (acc_ms * 1e-3) / 1e12
    peak = pk.get("bf16_tflops") or 1900.0
    peak_src = "measured burst bf16 (MEASURED_PEAKS.json)" if pk.get("bf16_tflops") else "fallback 1.9 PFLOP/s bf16"
    int_rate = da.probe_int_mac_rate()
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    int_pipe = {"achieved_exact_macs_per_s": macs / (ms * 1e-3),
                "peak_exact_macs_per_s": int_rate,
                "peak_per_clock_per_sm": int_rate / (n_sm * sm_clock * 1e6),
                "frac": macs / (ms * 1e-3) / int_rate,
                "basis": "the step's exact multiply-adds (D score + D PV per unmasked pair) over the step time",
                "peak_basis": "mad.wide.s32 (exact 32 x 32 -> 64-bit multiply-add) issue rate over all SMs, "
                              "measured by da_probe_int_mac in this run"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D, "causal": True,
                   "input_dtype": "bf16", "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed between timed steps (512 MiB write, outside the step events)",
                   "attn_macs_per_step": macs, "pairs_per_step": w.pairs},
        "kernels_ms": {"rowmax": statistics.mean(k_rowmax), "accumulate_finalize": acc_ms},
        "score_cache_bytes": int(L.da_score_cache_bytes(P.ref())),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": ACC_TRAFFIC_PER_LAUNCH if args.heads == 16 else None,
                     "kernel": "accumulate",
                     "algorithmic": f"{w.pairs} unmasked pairs x D exact PV multiply-adds x 2 flop per launch "
                                    "(the D score multiply-adds per pair run in pass 1)",
                     "peak_basis": peak_src, "sm_mhz": sm_clock,
                     "mma_util": {"achieved": mma_tflops, "frac": mma_tflops / peak,
                                  "basis": f"{tiles} key tiles x {tile_macs} bf16/f16 MACs per launch "
                                           "(the digit decomposition the kernel issues)"},
                     "int_pipe": int_pipe},
        "sharded": sharded,
        "clocks": ck,
        "e2e": {"value": e2e_val, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": statistics.mean(e2e_ms)},
        # per step: V columns, key + V prep, rowmax (storing scores), the work order (item keys,
        # classes, placement), accumulate
        "gpu_launches": 7 * args.steps,
        "dce": dce,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        macs_c, dt_c, sample = oracle_sample(w, Qh, Kh, Vh, args.ref_rows, os.cpu_count() or 1)
        line["cpu_baseline"] = {"value": macs_c / dt_c, "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle",
                                "sample": sample, "seconds": dt_c}
    print(json.dumps(line), flush=True)


def _sha(*ts) -> str:
    import hashlib
    h = hashlib.sha256()
    for t in ts:
        t = t.detach().cpu().contiguous()
        h.update((t.view(torch.int16) if t.dtype == torch.bfloat16 else t).numpy().tobytes())
    return h.hexdigest()


def _time_ms(fn, stream, flush, reps):
    fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


KERNEL_CALLS = ("rowmax", "accumulate_digits", "compose_max", "compose_add", "normalize", "finalize",
                "rowmax_d64", "accumulate_d64", "rowmax_d256", "accumulate_d256",
                "dce_rowmax", "dce_denom_digits", "dce_finalize", "dce_reduce", "dce_backward")


def run_kernels(args):
    """One JSON line per C-ABI call, each timed alone with CUDA events on the launching stream
    (L2 flushed before each timed call; median of --steps calls after --warmup): the
    device kernels it launches, its algorithmic bytes (inputs read once, outputs written once)
    or flops, and the achieved rate against the measured peak.  Attention calls run on the
    long-context causal shape (S4096, --heads heads; D = 64 and 256 variants of the same shape
    for the integer-pipe kernels), the digit calls on that shape's NUM/DEN digits, the
    cross-entropy calls on --dce-rows tokens of the vocab-sharded shape (V128256 f32)."""
    import bitwise_deterministic_shard_gb300 as da
    want = KERNEL_CALLS if args.kernels == "all" else tuple(args.kernels.split(","))
    bad = [k for k in want if k not in KERNEL_CALLS]
    if bad:
        raise SystemExit(f"unknown kernel call(s) {bad}; choose from {', '.join(KERNEL_CALLS)}")
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    pk = _peaks()
    hbm = pk.get("hbm_gbs") or 6800.0
    tfl = pk.get("bf16_tflops") or 1900.0

    def emit(call, launches, workload, ms, nbytes=None, flops=None, note=None):
        line = {"call": call, "kernels": launches, "workload": workload, "ms": ms}
        if nbytes is not None:
            line.update({"algorithmic_bytes": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,
                         "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm})
        if flops is not None:
            line.update({"algorithmic_flops": flops, "achieved_tflops": flops / (ms * 1e-3) / 1e12,
                         "bf16_frac": flops / (ms * 1e-3) / 1e12 / tfl})
        if note:
            line["note"] = note
        print(json.dumps(line), flush=True)

    def timed(fn):
        for _ in range(max(args.warmup - 1, 0)):
            fn()
        return _time_ms(fn, stream, flush, args.steps)

    def attn(D, heads):
        w = W.long_context_causal()
        w.D, w.Hq, w.Hkv = D, heads, heads
        w.name = f"long-context causal B1 H{heads} S4096 D{D} bf16, 1% of K rows x8"
        Q, K, V = w.tensors(dev)
        ws = torch.empty(da.workspace_bytes(Q, K, V, True), dtype=torch.uint8, device=dev)
        return w, Q, K, V, ws

    attn_calls = [k for k in want if not k.startswith("dce_")]
    if attn_calls:
        w, Q, K, V, ws = attn(128, args.heads)
        rows = w.B * w.Hq * w.S
        io = (Q.numel() + K.numel() + V.numel()) * 2
        m = da.rowmax(Q, K, causal=True, workspace=ws)
        if "rowmax" in want:
            t = timed(lambda: da.rowmax(Q, K, causal=True, out=m, workspace=ws))
            emit("rowmax", ["prep_kv_kernel", "rowmax_tc_kernel"], w.name, t, flops=w.pairs * w.D * 2,
                 note="flops: the pages' score work, P x D multiply-adds x 2")
        num = torch.empty(w.B, w.Hq, w.S, da.NUM_NDIG, w.D, dtype=torch.int64, device=dev)
        den = torch.empty(w.B, w.Hq, w.S, da.DEN_NDIG, dtype=torch.int64, device=dev)
        da.accumulate(Q, K, V, m, causal=True, num=num, den=den, workspace=ws)
        if "accumulate_digits" in want:
            t = timed(lambda: da.accumulate(Q, K, V, m, causal=True, num=num, den=den, workspace=ws))
            emit("accumulate_digits", ["prep_vcol_kernel", "prep_kv_kernel", "accumulate_tp_kernel"], w.name, t,
                 flops=w.pairs * 2 * w.D * 2, note="flops: P x 2D exact multiply-adds x 2; NUM/DEN digits written")
        digit_bytes = num.numel() * 8
        if "compose_max" in want:
            m2 = m.clone()
            t = timed(lambda: da.compose_max(m2, m))
            emit("compose_max", ["compose_max_kernel"], w.name + ": rowmax f32", t, nbytes=3 * m.numel() * 4,
                 note="input fits in L2: launch-bound")
        if "compose_add" in want or "normalize" in want:
            num2 = num.clone()
            if "compose_add" in want:
                t = timed(lambda: da.compose_add(num2, num))
                emit("compose_add", ["compose_add_kernel"], w.name + ": NUM digits", t, nbytes=3 * digit_bytes)
            if "normalize" in want:
                t = timed(lambda: da.normalize(num2))
                emit("normalize", ["normalize_kernel"], w.name + ": NUM digits", t, nbytes=2 * digit_bytes)
            del num2
        if "finalize" in want:
            out = torch.empty(w.B, w.Hq, w.S, w.D, dtype=torch.float32, device=dev)
            t = timed(lambda: da.finalize(num, den, out=out))
            emit("finalize", ["finalize_kernel"], w.name + ": NUM/DEN digits to f32", t,
                 nbytes=digit_bytes + den.numel() * 8 + out.numel() * 4)
            del out
        del num, den, Q, K, V, ws, m
        torch.cuda.empty_cache()
        for D, heads, acc_kernel in ((64, args.heads, "accumulate_tp_kernel"),
                                     (256, max(1, args.heads // 4), "accumulate_kernel")):
            if f"rowmax_d{D}" not in want and f"accumulate_d{D}" not in want:
                continue
            w, Q, K, V, ws = attn(D, heads)
            m = da.rowmax(Q, K, causal=True, workspace=ws)
            if f"rowmax_d{D}" in want:
                t = timed(lambda: da.rowmax(Q, K, causal=True, out=m, workspace=ws))
                emit(f"rowmax_d{D}", ["prep_kv_kernel", "rowmax_tc_kernel"], w.name, t, flops=w.pairs * w.D * 2)
            if f"accumulate_d{D}" in want:
                num = torch.empty(w.B, w.Hq, w.S, da.NUM_NDIG, w.D, dtype=torch.int64, device=dev)
                den = torch.empty(w.B, w.Hq, w.S, da.DEN_NDIG, dtype=torch.int64, device=dev)
                t = timed(lambda: da.accumulate(Q, K, V, m, causal=True, num=num, den=den, workspace=ws))
                emit(f"accumulate_d{D}", ["prep_vcol_kernel", "prep_kv_kernel", acc_kernel], w.name, t,
                     flops=w.pairs * 2 * w.D * 2)
                del num, den
            del Q, K, V, ws, m
            torch.cuda.empty_cache()
    dce_calls = [k for k in want if k.startswith("dce_")]
    if dce_calls:
        w = W.vocab_sharded_ce()
        w.N = args.dce_rows
        w.name = f"vocab-sharded cross-entropy N{w.N} V{w.V} f32"
        x, tg = w.tensors(dev)
        nb = x.numel() * 4
        m = da.dce_rowmax(x)
        den = da.dce_denom_digits(x, m)
        loss, denom = da.dce_finalize(den, x, tg, m)
        if "dce_rowmax" in want:
            t = timed(lambda: da.dce_rowmax(x, out=m))
            emit("dce_rowmax", ["dce_rowmax_kernel"], w.name, t, nbytes=nb + w.N * 4)
        if "dce_denom_digits" in want:
            t = timed(lambda: da.dce_denom_digits(x, m, den=den))
            emit("dce_denom_digits", ["dce_denom_kernel"], w.name, t, nbytes=nb + w.N * (4 + 48))
        if "dce_finalize" in want:
            t = timed(lambda: da.dce_finalize(den, x, tg, m))
            emit("dce_finalize", ["dce_finalize_kernel"], w.name, t, nbytes=w.N * (48 + 4 + 8 + 4 + 4 + 8),
                 note="per token: DEN digits, rowmax, target, target logit read; loss, denom written")
        if "dce_reduce" in want:
            t = timed(lambda: da.dce_reduce(loss, "mean"))
            emit("dce_reduce", ["dce_reduce_kernel"], w.name, t, nbytes=w.N * 4, note="launch-bound")
        if "dce_backward" in want:
            g = torch.ones((), dtype=torch.float32, device=dev)
            t = timed(lambda: da.dce_backward(x, tg, m, denom, g, reduction="mean"))
            emit("dce_backward", ["dce_backward_kernel"], w.name, t, nbytes=2 * nb + w.N * 16)


def run_configs(args):
    """One JSON line per workload of the pages: fused and sharded device times (CUDA events, L2
    flushed between calls), exact attention MACs/s, the oracle's host time and core count, SHA-256
    of the inputs and the output, and parity against the oracle (every row where the oracle
    finishes in seconds; sampled rows on the large non-causal workload)."""
    import bitwise_deterministic_shard_gb300 as da
    from oracle import native
    native.build()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    cores = native.default_threads()
    for w in (W.tiny_exact(), W.gqa_causal(), W.long_context_causal(), W.large_noncausal()):
        Qh, Kh, Vh = w.tensors("cpu")
        Q, K, V = Qh.to(dev), Kh.to(dev), Vh.to(dev)
        ws = torch.empty(da.workspace_bytes(Q, K, V, w.causal, w.scale, max(len(s) for s, _ in w.splits)),
                         dtype=torch.uint8, device=dev)
        out = torch.empty(w.B, w.Hq, w.S, w.D, dtype=torch.float32, device=dev)
        reps = 2 if w.S > 10000 else 5
        fused_ms = _time_ms(lambda: da.det_attn(Q, K, V, w.causal, w.scale, out=out, workspace=ws), stream, flush,
                            reps)
        fused = out.clone()
        sh = {}
        outs = torch.empty_like(out)
        for sp, order in w.splits:
            key = f"{len(sp)} splits"
            t = _time_ms(lambda: da.det_attn_sharded(Q, K, V, sp, w.causal, w.scale, order=order, out=outs,
                                                     workspace=ws), stream, flush, 1 if w.S > 10000 else 2)
            assert torch.equal(outs, fused), (w.name, len(sp), order)
            sh.setdefault(key, []).append(t)
        sharded = {k: {"compositions": len(v), "median_ms": statistics.median(v),
                       "macs_per_s": w.attn_macs / (statistics.median(v) * 1e-3), "bit_identical_to_fused": True}
                   for k, v in sh.items()}
        A = native.Attn(Qh, Kh, Vh, w.causal, w.scale)
        if w.S > 10000:   # 64 rows per head (spread over the sequence) plus the last 50 rows of head 0
            rows = sorted({h * w.S + int(i) for h in range(w.Hq) for i in np.linspace(0, w.S - 1, 64)} |
                          {w.S - 1 - i for i in range(50)})
            rows = np.asarray(rows, dtype=np.int64)
        else:
            rows = native.all_rows(w.B, w.Hq, w.S)
        keys = (rows % w.S) + 1 if w.causal else np.full(len(rows), w.S)
        t0 = time.perf_counter()
        _, _, _, ref = A.forward_rows(rows=rows)
        dt = time.perf_counter() - t0
        got = fused.reshape(-1, w.D)[torch.from_numpy(rows).to(dev)].cpu().numpy()
        equal = bool(np.array_equal(got.view(np.uint32), ref.view(np.uint32)))
        o_macs = int(keys.sum()) * 2 * w.D
        line = {"config": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D, "causal": w.causal,
                "dtype": str(w.dtype).replace("torch.", ""), "pairs": w.pairs, "attn_macs": w.attn_macs,
                "fused_ms": fused_ms, "fused_macs_per_s": w.attn_macs / (fused_ms * 1e-3), "sharded": sharded,
                "oracle": {"seconds": dt, "cores": cores, "rows": "all" if len(rows) == w.B * w.Hq * w.S
                           else f"{len(rows)} sampled rows", "macs_per_s": o_macs / dt,
                           "full_workload_seconds_extrapolated": w.attn_macs / (o_macs / dt)},
                "sha256": {"inputs": _sha(Qh, Kh, Vh), "output": _sha(fused)},
                "parity": ("bit-exact vs oracle" if equal else "MISMATCH") +
                          (" (every row)" if len(rows) == w.B * w.Hq * w.S else f" ({len(rows)} rows)")}
        print(json.dumps(line), flush=True)
        del Q, K, V, ws, out, outs, fused
        torch.cuda.empty_cache()
    # vocab-sharded cross-entropy
    w = W.vocab_sharded_ce()
    xh, th = w.tensors("cpu")
    x, t = xh.to(dev), th.to(dev)
    base = da.dce_forward(x, t)
    times = {}
    for sp in w.splits:
        times[f"{len(sp)} splits"] = _time_ms(lambda: da.dce_forward(x, t, splits=sp), stream, flush, 5)
        got = da.dce_forward(x, t, splits=sp)
        assert all(torch.equal(a_, b_) for a_, b_ in zip(base, got))
    t0 = time.perf_counter()
    rl, rd, rm, rden, _ = native.DCE(xh).forward(th.numpy())
    dt = time.perf_counter() - t0
    equal = bool(np.array_equal(base[0].cpu().numpy().view(np.uint32), rl.view(np.uint32)) and
                 np.array_equal(base[1].cpu().numpy(), rd))
    print(json.dumps({"config": w.name, "N": w.N, "V": w.V, "dtype": "float32",
                      "forward_ms_by_splits": times, "tokens_per_s": {k: w.N / (v * 1e-3) for k, v in times.items()},
                      "all_splits_bit_identical": True,
                      "oracle": {"seconds": dt, "cores": cores, "rows": "all", "tokens_per_s": w.N / dt},
                      "sha256": {"inputs": _sha(xh, th), "loss": _sha(base[0]), "denom": _sha(base[1])},
                      "parity": "bit-exact vs oracle (every token)" if equal else "MISMATCH"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-rows", type=int, default=3072,
                    help="cpu_baseline sample: query rows per head (about 10-20 s of the oracle on 16 cores)")
    ap.add_argument("--ref-rows-step", type=int, default=1024,
                    help="--impl reference: query rows per head in each timed step (a few seconds each)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sharded", action="store_true", help="skip the sharded ring-step timings")
    ap.add_argument("--configs", action="store_true",
                    help="per-workload table (fused / sharded times, oracle, SHA-256, parity) instead of the step")
    ap.add_argument("--kernels", nargs="?", const="all", default=None,
                    help="time each C-ABI call alone instead of the step: 'all' or a comma list of "
                         + ", ".join(KERNEL_CALLS))
    ap.add_argument("--heads", type=int, default=16, help="heads of the workload (16 = the metric workload)")
    ap.add_argument("--dce-rows", type=int, default=4096,
                    help="tokens of the cross-entropy leg (4096 = the vocab-sharded workload)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and args.impl == "ours":
        torch.distributed.init_process_group("nccl")
    elif world > 1:
        torch.distributed.init_process_group("gloo")
    if args.configs:
        run_configs(args)
        return
    if args.kernels:
        run_kernels(args)
        return
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
