"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random tensors; it holds none of the method's arithmetic, so both
the CUDA path's callers and the oracle may take their inputs from it.  Every tensor is
drawn on the CPU from a torch.Generator in a fixed order (Q, K, V, then extras), in
float32 from N(0, 1), then cast to bfloat16 (round to nearest even) where asked.

Workload shapes follow the det-attn page (Q, K, V are [B, H, S, D]; GQA allowed; causal
and non-causal; f32 and bf16; D <= 256) and the det-cross-entropy page (logits [N, V],
int64 targets).  The long non-causal case takes its shape (one batch, 56 heads, sequence
37,810, head dimension 128) from the "Canonical Boundary" section of the
"Exact Numerical Contract" page; the values here are synthetic.
"""
from __future__ import annotations

import random
from dataclasses import dataclass, field

import torch


@dataclass
class AttnWorkload:
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    dtype: torch.dtype
    causal: bool
    seed: int
    scale: float | None = None          # None: RN32(1/sqrt(D))
    big_k_frac: float = 0.0             # fraction of K rows multiplied by 8
    splits: list = field(default_factory=list)   # list of (kv_splits, order) compositions

    @property
    def pairs(self) -> int:
        """Number of unmasked (query, key) pairs over all batches and query heads."""
        per = self.S * (self.S + 1) // 2 if self.causal else self.S * self.S
        return self.B * self.Hq * per

    @property
    def attn_macs(self) -> int:
        """Attention MACs, B * Hq * P * 2D (QK^T plus PV)."""
        return self.pairs * 2 * self.D

    def tensors(self, device="cpu"):
        g = torch.Generator().manual_seed(self.seed)
        Q = torch.randn(self.B, self.Hq, self.S, self.D, generator=g)
        K = torch.randn(self.B, self.Hkv, self.S, self.D, generator=g)
        V = torch.randn(self.B, self.Hkv, self.S, self.D, generator=g)
        if self.big_k_frac > 0:
            mask = torch.rand(self.B, self.Hkv, self.S, generator=g) < self.big_k_frac
            K = K.to(self.dtype)
            K[mask] = K[mask] * 8          # exact in bf16 and f32
        Q, K, V = Q.to(self.dtype), K.to(self.dtype), V.to(self.dtype)
        return Q.to(device), K.to(device), V.to(device)


def equal_splits(S: int, n: int) -> list:
    base, rem = divmod(S, n)
    return [base + (1 if i < rem else 0) for i in range(n)]


def _gqa_causal_splits():
    r = random.Random(2)
    out = []
    for n in (4, 8):
        sp = equal_splits(1024, n)
        for _ in range(8):
            order = list(range(n))
            r.shuffle(order)
            out.append((sp, order))
    return out


def _large_noncausal_splits():
    r = random.Random(4)
    cuts = sorted(r.sample(range(1, 37810), 31))
    b = [0] + cuts + [37810]
    sp = [b[i + 1] - b[i] for i in range(32)]
    order = list(range(32))
    r.shuffle(order)
    return [(sp, order)]


def tiny_exact():
    import itertools
    perms = [([32] * 4, list(p)) for p in itertools.permutations(range(4))]
    return AttnWorkload("tiny exact check B1 H2 S128 D64 f32", 1, 2, 2, 128, 64, torch.float32, False, 0,
                        scale=0.125, splits=perms)


def gqa_causal():
    return AttnWorkload("GQA causal B2 Hq8 Hkv2 S1024 D128 bf16", 2, 8, 2, 1024, 128, torch.bfloat16, True, 2,
                        splits=_gqa_causal_splits())


def long_context_causal():
    return AttnWorkload("long-context causal B1 H16 S4096 D128 bf16, 1% of K rows x8", 1, 16, 16, 4096, 128,
                        torch.bfloat16, True, 3, big_k_frac=0.01,
                        splits=[(equal_splits(4096, n), list(range(n))) for n in (1, 2, 4, 8, 16, 32)])


def large_noncausal():
    return AttnWorkload("large non-causal B1 H56 S37810 D128 bf16", 1, 56, 56, 37810, 128, torch.bfloat16, False, 4,
                        splits=_large_noncausal_splits())


@dataclass
class DCEWorkload:
    name: str
    N: int
    V: int
    dtype: torch.dtype
    seed: int
    sigma: float = 2.0
    splits: list = field(default_factory=list)

    def tensors(self, device="cpu"):
        g = torch.Generator().manual_seed(self.seed)
        logits = (torch.randn(self.N, self.V, generator=g) * self.sigma).to(self.dtype)
        targets = torch.randint(0, self.V, (self.N,), generator=g, dtype=torch.int64)
        return logits.to(device), targets.to(device)


def vocab_sharded_ce():
    return DCEWorkload("vocab-sharded cross-entropy N4096 V128256 f32", 4096, 128256, torch.float32, 5,
                       splits=[equal_splits(128256, n) for n in (1, 2, 4, 8)])


def random_attn(seed, B, Hq, Hkv, S, D, dtype, causal, spread=1.0):
    """Small random case; `spread` > 1 widens the exponent range of the inputs."""
    g = torch.Generator().manual_seed(seed)
    out = []
    for h in (Hq, Hkv, Hkv):
        x = torch.randn(B, h, S, D, generator=g)
        if spread != 1.0:
            x = x * torch.exp2((torch.rand(B, h, S, D, generator=g) - 0.5) * spread)
        out.append(x.to(dtype))
    return tuple(out)
