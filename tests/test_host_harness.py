"""The benchmark's host side and the workloads, on the CPU: the seeded inputs are
deterministic and have the documented shapes, and the reference arm (the oracle on the host
cores) prints one JSON line with the benchmark contract's keys."""
import json
import os
import subprocess
import sys

import torch

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_workloads_are_seeded_and_shaped_as_documented():
    w = W.tiny_exact()
    a, b = w.tensors(), w.tensors()
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert a[0].shape == (1, 2, 128, 64) and a[0].dtype == torch.float32
    w = W.long_context_causal()
    assert (w.B, w.Hq, w.Hkv, w.S, w.D, w.dtype, w.causal) == (1, 16, 16, 4096, 128, torch.bfloat16, True)
    assert w.big_k_frac == 0.01 and w.pairs == 16 * 4096 * 4097 // 2
    assert [sum(s) for s, _ in w.splits] == [4096] * len(w.splits)
    assert [len(s) for s, _ in w.splits] == [1, 2, 4, 8, 16, 32]
    w = W.large_noncausal()
    assert (w.Hq, w.S, w.D, w.causal) == (56, 37810, 128, False)
    assert all(len(s) == 32 and sum(s) == 37810 for s, _ in w.splits)
    w = W.gqa_causal()
    assert (w.B, w.Hq, w.Hkv, w.S) == (2, 8, 2, 1024)
    c = W.vocab_sharded_ce()
    assert (c.N, c.V, c.dtype) == (4096, 128256, torch.float32)
    assert [len(s) for s in c.splits] == [1, 2, 4, 8] and all(sum(s) == 128256 for s in c.splits)


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                        "--ref-rows-step", "8"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == W.long_context_causal().name
