"""GPU parity: the CUDA path through the C ABI against the oracle, bit for bit.

The oracle (oracle/native.py, the exact C implementation; oracle/exact.py pins it) and
the CUDA kernels share no code; both take their inputs from workloads/.  Every floating-
point output is compared with torch.equal / bit patterns (the contract fixes every
rounding, so the tolerance is zero); digits are compared exactly.  Sizes: small cases that
span several tiles with ragged tails, every workload of the det-attn and det-cross-entropy
pages at full size (every row of the long-context and cross-entropy workloads; sampled and
out-of-window rows of the large non-causal one, whose full oracle run would take hours),
and the edge cases (empty key ranges, one key, GQA, strided views, f32 and bf16).
"""
import itertools
import random

import numpy as np
import pytest
import torch

import workloads as W

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


def _bits(x):
    x = x.detach().cpu().contiguous() if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x))
    return x.view(torch.int32) if x.dtype == torch.float32 else x


def assert_bits_equal(a, b, what=""):
    a, b = _bits(a), _bits(b)
    if not torch.equal(a, b):
        diff = (a != b).nonzero()
        raise AssertionError(f"{what}: {diff.shape[0]} elements differ, first at {diff[:5].tolist()}")


def flat_rows(B, H, S, rows_bhi):
    return np.asarray([(b * H + h) * S + i for b, h, i in rows_bhi], dtype=np.int64)


def run_full(da, Q, K, V, causal, scale=None, status=None):
    dev = torch.device("cuda")
    Qd, Kd, Vd = Q.to(dev), K.to(dev), V.to(dev)
    m = da.rowmax(Qd, Kd, causal=causal, scale=scale, status=status)
    num, den = da.accumulate(Qd, Kd, Vd, m, causal=causal, scale=scale, status=status)
    out = da.finalize(num, den)
    fused = da.det_attn(Qd, Kd, Vd, causal=causal, scale=scale, status=status)
    torch.cuda.synchronize()
    return m, num, den, out, fused


CASES = [
    # (B, Hq, Hkv, S, D, dtype, causal)
    (1, 2, 2, 37, 8, torch.bfloat16, False),
    (1, 2, 1, 130, 64, torch.bfloat16, True),
    (2, 4, 2, 200, 128, torch.bfloat16, True),
    (1, 3, 3, 97, 100, torch.bfloat16, False),
    (1, 2, 2, 70, 256, torch.bfloat16, True),
    (1, 2, 1, 90, 64, torch.float32, False),
    (1, 2, 2, 66, 128, torch.float32, True),
    # causal, 15 query tiles of 16 rows (ragged last tile): the pass-2 work order splits the
    # pair beside the middle tile into two single-tile CTAs and leaves the middle one whole
    (1, 2, 2, 235, 128, torch.bfloat16, True),
    (1, 1, 1, 1, 16, torch.bfloat16, False),
    (1, 2, 2, 65, 200, torch.float32, False),
]


@cuda
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}Hq{c[1]}Hkv{c[2]}S{c[3]}D{c[4]}{str(c[5])[6:]}{'c' if c[6] else ''}")
def test_small_cases_match_oracle(da, orc, case):
    B, Hq, Hkv, S, D, dt, causal = case
    Q, K, V = W.random_attn(1000 + S + D, B, Hq, Hkv, S, D, dt, causal)
    st = da.new_status()
    m, num, den, out, fused = run_full(da, Q, K, V, causal, status=st)
    assert da.read_status(st) == 0
    A = orc.Attn(Q, K, V, causal)
    m_o, num_o, den_o, out_o = A.forward_rows()
    assert_bits_equal(m.reshape(-1), m_o, "rowmax")
    assert torch.equal(den.cpu().reshape(-1, 6), torch.from_numpy(den_o)), "DEN digits"
    assert torch.equal(num.cpu().reshape(-1, 15, D), torch.from_numpy(num_o)), "NUM digits"
    assert_bits_equal(out.reshape(-1, D), out_o, "output")
    assert_bits_equal(fused, out, "fused vs composed")


@cuda
def test_wide_exponent_inputs_take_the_exact_fallbacks(da, orc):
    """Rows whose elements span more than the fixed-point window (the Kulisch score
    fallback), tiny V elements and tiny weights (the atomic spill paths)."""
    Q, K, V = W.random_attn(7, 1, 2, 2, 150, 64, torch.bfloat16, False, spread=60.0)
    K = K.clone()
    K[0, 0, 3] *= 2 ** 40      # a key far above the others: tiny weights for the rest
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    st = da.new_status()
    out = da.det_attn(Qd, Kd, Vd, status=st)
    torch.cuda.synchronize()
    _, num_o, den_o, out_o = orc.Attn(Q, K, V).forward_rows()
    assert da.read_status(st) & ~1 == 0
    assert_bits_equal(out.reshape(-1, 64), out_o, "output")


@cuda
@pytest.mark.parametrize("causal", [False, True])
def test_rows_outside_the_fast_window_match_oracle(da, orc, causal):
    """Rows with one element 20 to 40 binades below the row maximum do not fit the 26-bit
    fixed point of the tensor-core path; their pairs take the deferred exact dot (52-bit
    window, one warp or one thread per pair).  Every third Q and K row is made such a row,
    so some pairs have both rows outside."""
    g = torch.Generator().manual_seed(70 + causal)
    Q, K, V = (torch.randn(1, 2, 150, 128, generator=g) for _ in range(3))
    for X in (Q, K):
        for r in range(0, 150, 3):
            X[:, :, r, r % 128] *= 2.0 ** -(20 + r % 21)
    Q, K, V = Q.to(torch.bfloat16), K.to(torch.bfloat16), V.to(torch.bfloat16)
    st = da.new_status()
    m, num, den, out, fused = run_full(da, Q, K, V, causal, status=st)
    assert da.read_status(st) == 0
    m_o, num_o, den_o, out_o = orc.Attn(Q, K, V, causal).forward_rows()
    assert_bits_equal(m.reshape(-1), m_o, "rowmax")
    assert torch.equal(num.cpu().reshape(-1, 15, 128), torch.from_numpy(num_o)), "NUM digits"
    assert torch.equal(den.cpu().reshape(-1, 6), torch.from_numpy(den_o)), "DEN digits"
    assert_bits_equal(fused.reshape(-1, 128), out_o, "output")


@cuda
@pytest.mark.parametrize("D", [64, 128, 256])
def test_extreme_digit_patterns_match_oracle(da, orc, D):
    """Every element has all eight significand bits set, exponents spread to the edge of
    the 26-bit fixed-point window: the tensor-core digit slices take their largest values,
    so the diagonal sums reach the top of their exactness bound."""
    g = torch.Generator().manual_seed(60 + D)

    def draw(h, S):
        e = torch.randint(-18, 1, (1, h, S, D), generator=g).float()
        sign = torch.randint(0, 2, (1, h, S, D), generator=g).float() * 2 - 1
        return (sign * (2.0 - 2.0 ** -7) * torch.exp2(e)).to(torch.bfloat16)

    Q, K = draw(2, 70), draw(2, 70)
    V = torch.randn(1, 2, 70, D, generator=g).to(torch.bfloat16)
    out = da.det_attn(Q.cuda(), K.cuda(), V.cuda(), causal=True)
    m = da.rowmax(Q.cuda(), K.cuda(), causal=True)
    A = orc.Attn(Q, K, V, causal=True)
    m_o, _, _, out_o = A.forward_rows()
    assert_bits_equal(m.reshape(-1), m_o, "rowmax")
    assert_bits_equal(out.reshape(-1, D), out_o, "output")


@cuda
def test_tiny_exact_fused_and_all_24_orders(da, orc):
    w = W.tiny_exact()
    Q, K, V = w.tensors("cuda")
    fused = da.det_attn(Q, K, V, causal=w.causal, scale=w.scale)
    _, _, _, ref = orc.Attn(Q.cpu(), K.cpu(), V.cpu(), w.causal, w.scale).forward_rows()
    assert_bits_equal(fused.reshape(-1, w.D), ref, "tiny fused vs oracle")
    for sp, order in w.splits:
        out = da.det_attn_sharded(Q, K, V, sp, causal=w.causal, scale=w.scale, order=order)
        assert torch.equal(out, fused), order
    # a physical permutation of the K/V blocks (allowed: non-causal)
    perm = torch.cat([torch.arange(96, 128), torch.arange(0, 32), torch.arange(64, 96), torch.arange(32, 64)])
    outp = da.det_attn(Q, K[:, :, perm], V[:, :, perm], causal=False, scale=w.scale)
    assert torch.equal(outp, fused)


@cuda
def test_gqa_causal_splits_and_oracle(da, orc):
    w = W.gqa_causal()
    Q, K, V = w.tensors("cuda")
    fused = da.det_attn(Q, K, V, causal=True)
    torch.cuda.synchronize()
    _, _, _, ref = orc.Attn(Q.cpu(), K.cpu(), V.cpu(), True).forward_rows()
    assert_bits_equal(fused.reshape(-1, w.D), ref, "GQA causal fused vs oracle")
    for sp, order in w.splits:
        out = da.det_attn_sharded(Q, K, V, sp, causal=True, order=order)
        assert torch.equal(out, fused), (sp, order)


def rows_outside_window(X):
    """Indices of the rows of X ([rows, D] float32 values) that do not fit the 26-bit
    fixed-point window of the tensor-core score path: some element is not a multiple of
    2^(emax - 152), emax the row's largest biased exponent.  Such rows take the exact
    low-limb or general dot, so the tests pick them out on purpose."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    e = (X.view(np.uint32) >> 23) & 0xFF
    F = np.maximum(e.max(axis=1), 1).astype(np.int64) - 152
    scaled = X.astype(np.float64) * np.exp2(-F.astype(np.float64))[:, None]
    return np.nonzero((scaled != np.floor(scaled)).any(axis=1))[0]


@cuda
def test_long_context_ring_steps_and_full_oracle(da, orc):
    """The metric workload at full size: every one of the 65,536 query rows against the
    oracle (rowmax and output), so the rare exact paths (rows outside the fixed-point window,
    rows whose maximum comes from a x8 key and their spill-slot products, several CTAs per
    SM in turn) are checked under full-size contention; then ring steps 1 to 32 against the
    fused result."""
    w = W.long_context_causal()
    Q, K, V = w.tensors("cuda")
    st = da.new_status()
    m = da.rowmax(Q, K, causal=True, status=st)
    fused = da.det_attn(Q, K, V, causal=True, status=st)
    torch.cuda.synchronize()
    assert da.read_status(st) == 0
    A = orc.Attn(Q.cpu(), K.cpu(), V.cpu(), True)
    m_o, _, _, ref = A.forward_rows()
    assert_bits_equal(m.reshape(-1), m_o, "long-context rowmax vs oracle (all rows)")
    assert_bits_equal(fused.reshape(-1, w.D), ref, "long-context output vs oracle (all rows)")
    # the rare paths really occur in this workload
    assert len(rows_outside_window(Q.float().cpu().reshape(-1, w.D).numpy())) > 0
    Kb = K.float().cpu().reshape(w.Hkv, w.S, w.D).abs().amax(dim=2)
    assert int((Kb > 8).sum()) > 0
    for sp, order in w.splits:
        out = da.det_attn_sharded(Q, K, V, sp, causal=True, order=order)
        assert torch.equal(out, fused), len(sp)


@cuda
def test_large_noncausal_unequal_splits_and_sampled_oracle(da, orc):
    """Large non-causal workload at full size (B1 H56 S37810 D128 bf16; S is no tile
    multiple): the fused call, the 32 unequal random splits composed in a random order, and
    against the oracle sampled rows (4 per head, the last row) plus up to 64 query rows that
    lie outside the fixed-point window (picked deterministically from the inputs)."""
    w = W.large_noncausal()
    Q, K, V = w.tensors("cuda")
    st = da.new_status()
    fused = da.det_attn(Q, K, V, status=st)
    torch.cuda.synchronize()
    assert da.read_status(st) == 0
    (sp, order), = w.splits
    assert sum(sp) == w.S and len(sp) == 32
    out = da.det_attn_sharded(Q, K, V, sp, order=order, status=st)
    torch.cuda.synchronize()
    assert da.read_status(st) == 0
    assert torch.equal(out, fused)
    del out
    rng = random.Random(4)
    rows = [(0, h, i) for h in range(w.Hq) for i in rng.sample(range(w.S), 4)] + [(0, w.Hq - 1, w.S - 1)]
    fl = flat_rows(1, w.Hq, w.S, rows)
    wide = rows_outside_window(Q.float().cpu().reshape(-1, w.D).numpy())
    assert len(wide) > 0
    fl = np.unique(np.concatenate([fl, wide[np.linspace(0, len(wide) - 1, min(64, len(wide))).astype(np.int64)]]))
    A = orc.Attn(Q.cpu(), K.cpu(), V.cpu(), False)
    _, _, _, ref = A.forward_rows(rows=fl)
    got = fused.reshape(-1, w.D)[torch.from_numpy(fl).cuda()]
    assert_bits_equal(got, ref, "large non-causal sampled and out-of-window rows vs oracle")


@cuda
def test_long_context_shard_digits_compose_to_fused_digits(da):
    """accumulate per shard into separate arrays + compose_add + normalize equals the
    fused digits (det-attn "Method": an int64 add of digit arrays)."""
    w = W.long_context_causal()
    Q, K, V = w.tensors("cuda")
    Q, K, V = Q[:, :4, :1024], K[:, :4, :1024], V[:, :4, :1024]
    m = da.rowmax(Q, K, causal=True)
    num0, den0 = da.accumulate(Q, K, V, m, causal=True)
    parts = [da.accumulate(Q, K, V, m, lo, lo + 256, causal=True) for lo in (768, 0, 512, 256)]
    num, den = parts[0][0].clone(), parts[0][1].clone()
    for n_, d_ in parts[1:]:
        da.compose_add(num, n_)
        da.compose_add(den, d_)
    da.normalize(num)
    da.normalize(den)
    assert torch.equal(num, num0) and torch.equal(den, den0)
    ms = [da.rowmax(Q, K, lo, lo + 256, causal=True) for lo in (512, 0, 768, 256)]
    mm = ms[0].clone()
    for x in ms[1:]:
        da.compose_max(mm, x)
    assert torch.equal(mm, m)


@cuda
def test_repeat_runs_bitwise_identical(da):
    w = W.long_context_causal()
    Q, K, V = w.tensors("cuda")
    a = da.det_attn(Q, K, V, causal=True)
    b = da.det_attn(Q, K, V, causal=True)
    assert torch.equal(a, b)


@cuda
def test_strided_nhd_views(da, orc):
    """Q/K/V as [B, S, H, D] projections viewed as [B, H, S, D] (non-contiguous heads)."""
    g = torch.Generator().manual_seed(44)
    qkv = torch.randn(1, 77, 3, 4, 64, generator=g).to(torch.bfloat16)
    Q, K, V = (qkv[:, :, t].transpose(1, 2) for t in range(3))
    out = da.det_attn(Q.cuda(), K.cuda(), V.cuda())
    _, _, _, ref = orc.Attn(Q, K, V).forward_rows()
    assert_bits_equal(out.reshape(-1, 64), ref, "strided")


@cuda
@pytest.mark.parametrize("case", [
    # (B, Hq, Hkv, S, D, dtype, causal, spread): every D <= 128 takes the 128-wide tensor-PV
    # kernel, which finalizes in its epilogue (the digit path stores NUM and finalizes apart)
    (1, 2, 2, 200, 128, torch.bfloat16, True, 1.0),
    (2, 4, 2, 300, 128, torch.float32, False, 1.0),
    (1, 2, 1, 150, 100, torch.bfloat16, True, 1.0),
    (1, 2, 2, 170, 128, torch.bfloat16, False, 60.0),
    (1, 2, 2, 90, 64, torch.bfloat16, False, 1.0),
])
def test_accumulate_finalize_equals_the_digit_path(da, orc, case):
    """The fused pass 2 (NUM digits never stored) against accumulate + finalize, bit for
    bit, and against the oracle."""
    B, Hq, Hkv, S, D, dt, causal, spread = case
    Q, K, V = W.random_attn(90 + S, B, Hq, Hkv, S, D, dt, causal, spread=spread)
    if spread != 1.0:
        K = K.clone()
        K[0, 0, 5] *= 2 ** 40   # tiny weights for the other keys: the spill slots
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    st = da.new_status()
    m = da.rowmax(Qd, Kd, causal=causal, status=st)
    fused = da.accumulate_finalize(Qd, Kd, Vd, m, causal=causal, status=st)
    num, den = da.accumulate(Qd, Kd, Vd, m, causal=causal, status=st)
    ref = da.finalize(num, den)
    torch.cuda.synchronize()
    assert_bits_equal(fused, ref, "fused vs digits")
    assert da.read_status(st) & ~1 == 0
    _, _, _, out_o = orc.Attn(Q, K, V, causal=causal).forward_rows()
    assert_bits_equal(fused.reshape(-1, D), out_o, "fused vs oracle")


@cuda
def test_empty_and_edge_ranges(da, orc):
    Q, K, V = W.random_attn(45, 1, 2, 2, 50, 32, torch.bfloat16, False)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    m = da.rowmax(Qd, Kd, 10, 10)
    assert torch.all(m == float("-inf"))
    mfull = da.rowmax(Qd, Kd)
    num, den = da.accumulate(Qd, Kd, Vd, mfull, 20, 20)
    assert not num.any() and not den.any()
    # a shard of one key
    n1, d1 = da.accumulate(Qd, Kd, Vd, mfull, 49, 50)
    A = orc.Attn(Q, K, V)
    mo, _ = A.rowmax()
    no, do, _ = A.accumulate(mo, 49, 50)
    assert torch.equal(n1.cpu().reshape(-1, 15, 32), torch.from_numpy(no))
    assert torch.equal(d1.cpu().reshape(-1, 6), torch.from_numpy(do))
    # causal: a shard that lies entirely after some queries contributes nothing to them
    Qc, Kc, Vc = W.random_attn(46, 1, 1, 1, 64, 16, torch.bfloat16, True)
    mc = da.rowmax(Qc.cuda(), Kc.cuda(), 32, 64, causal=True)
    assert torch.all(mc[0, 0, :32] == float("-inf"))
    mo2, _ = orc.Attn(Qc, Kc, Vc, True).rowmax(32, 64)
    assert_bits_equal(mc.reshape(-1), mo2, "causal shard rowmax")


@cuda
@pytest.mark.parametrize("D", [64, 128])
def test_key_ranges_at_and_beyond_the_tensor_pv_limit(da, orc, D):
    """65,536 keys (512 key tiles) is the longest range the tensor-PV kernel takes, with the
    score cache and the fused finalize; one key tile more sends the call to the integer-pipe
    kernel (digits in device memory, then finalize).  Both, and a sharded call whose shards
    lie on either side of the limit, equal the oracle bit for bit."""
    g = torch.Generator().manual_seed(60 + D)
    Sq = 24
    for Skv in (65536, 65536 + 131):
        Q = torch.randn(1, 1, Sq, D, generator=g).to(torch.bfloat16)
        K = torch.randn(1, 1, Skv, D, generator=g).to(torch.bfloat16)
        V = torch.randn(1, 1, Skv, D, generator=g).to(torch.bfloat16)
        Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
        out = da.det_attn(Qd, Kd, Vd)
        _, _, _, ref = orc.Attn(Q, K, V).forward_rows()
        assert_bits_equal(out.reshape(-1, D), ref, f"{Skv} keys, D = {D}")
        if Skv > 65536:
            assert torch.equal(da.det_attn_sharded(Qd, Kd, Vd, [131, 65536]), out)
            assert torch.equal(da.det_attn_sharded(Qd, Kd, Vd, [65536, 131]), out)


@cuda
def test_status_bits(da):
    Q, K, V = W.random_attn(47, 1, 1, 1, 40, 16, torch.bfloat16, False)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    m = da.rowmax(Qd, Kd)
    st = da.new_status()
    da.accumulate(Qd, Kd, Vd, m - 1.0, status=st)
    torch.cuda.synchronize()
    assert da.read_status(st) & da.STATUS_ROWMAX_VIOLATION
    st2 = da.new_status()
    Qn = Qd.clone()
    Qn[0, 0, 5, 3] = float("inf")
    da.rowmax(Qn, Kd, status=st2)
    torch.cuda.synchronize()
    assert da.read_status(st2) & da.STATUS_NONFINITE


@cuda
def test_host_argument_errors(da):
    Q, K, V = (t.cuda() for t in W.random_attn(48, 1, 2, 2, 16, 16, torch.bfloat16, True))
    with pytest.raises(da.DetAttnError):
        da.det_attn_sharded(Q, K, V, [8, 9], causal=True)        # splits do not sum to S
    with pytest.raises(da.DetAttnError):
        da.det_attn_sharded(Q, K, V, [8, 8], causal=True, order=[0, 0])
    with pytest.raises(da.DetAttnError):
        da.det_attn(Q, K[:, :, :8], V[:, :, :8], causal=True)   # causal needs Sq == Skv
    with pytest.raises(da.DetAttnError):
        da.det_attn(Q.cpu(), K, V)                               # no CPU path


# ------------------------------------------------------------------------ cross-entropy

@cuda
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_dce_small_matches_oracle(da, orc, dt):
    g = torch.Generator().manual_seed(50)
    x = (torch.randn(33, 1001, generator=g) * 3).to(dt)
    t = torch.randint(0, 1001, (33,), generator=g)
    for splits in ([1001], [500, 501], [1, 333, 667]):
        loss, denom, m, den = da.dce_forward(x.cuda(), t.cuda(), splits=splits)
        rl, rd, rm, rden, st = orc.DCE(x).forward(t.numpy(), splits=splits)
        assert_bits_equal(m, rm, "m")
        assert torch.equal(den.cpu(), torch.from_numpy(rden))
        assert_bits_equal(loss, rl, "loss")
        assert torch.equal(denom.cpu(), torch.from_numpy(rd))


@cuda
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,V,splits", [
    (64, 65613, [65613]),              # eight CTAs per row (one cluster), a ragged last share
    (64, 65613, [30001, 35612]),       # four and eight per shard, shares off the 16-byte grid
    (300, 40000, [40000]),             # four per row (152 SMs)
])
def test_dce_denominator_rows_split_over_clusters(da, orc, dt, N, V, splits):
    """Few rows of many columns: the denominator splits each row over a cluster of CTAs and
    adds their digit sums through distributed shared memory; digits, loss and denominator
    equal the oracle's bit for bit."""
    g = torch.Generator().manual_seed(51 + N)
    x = (torch.randn(N, V, generator=g) * 2).to(dt)
    t = torch.randint(0, V, (N,), generator=g)
    loss, denom, m, den = da.dce_forward(x.cuda(), t.cuda(), splits=splits)
    rl, rd, rm, rden, st = orc.DCE(x).forward(t.numpy(), splits=splits)
    assert_bits_equal(m, rm, "m")
    assert torch.equal(den.cpu(), torch.from_numpy(rden))
    assert_bits_equal(loss, rl, "loss")
    assert torch.equal(denom.cpu(), torch.from_numpy(rd))


@cuda
def test_vocab_sharded_splits_and_oracle(da, orc):
    w = W.vocab_sharded_ce()
    x, t = w.tensors("cuda")
    base = da.dce_forward(x, t)
    for sp in w.splits[1:]:
        got = da.dce_forward(x, t, splits=sp)
        for a, b in zip(base, got):
            assert torch.equal(a, b), len(sp)
    D = orc.DCE(x.cpu())
    rl, rd, rm, rden, st = D.forward(t.cpu().numpy())                  # every token
    assert_bits_equal(base[2], rm, "vocab-sharded rowmax")
    assert torch.equal(base[3].cpu(), torch.from_numpy(rden)), "vocab-sharded denominator digits"
    assert_bits_equal(base[0], rl, "vocab-sharded loss")
    assert torch.equal(base[1].cpu(), torch.from_numpy(rd))
    ref = torch.nn.functional.cross_entropy(x.double(), t, reduction="none")
    assert float((base[0].double() - ref).abs().max()) < 2e-6


@cuda
def test_dce_bad_target(da):
    x = torch.randn(4, 100, device="cuda")
    t = torch.tensor([0, 100, -1, 99], device="cuda")
    st = da.new_status()
    loss, denom, _, _ = da.dce_forward(x, t, status=st)
    torch.cuda.synchronize()
    assert da.read_status(st) & da.STATUS_BAD_TARGET
    assert torch.isnan(loss[1]) and torch.isnan(loss[2]) and not torch.isnan(loss[0])


@cuda
def test_packed_forms_equal_scalar_on_every_bit_pattern(da):
    """The cross-entropy kernels take two adjacent logits at once on the packed FP32 lanes: on
    all 2^32 binary32 bit patterns the packed exponential (reduction, polynomial, exponent;
    arguments clamped as the kernels clamp) and the backward's packed quotient and residual
    estimate equal the scalar forms bit for bit (the scalar forms are the ones the host tests
    pin to the oracle and to exact rationals).  A packed multiply feeding a packed add, fused
    by the compiler, fails the first on 79 patterns."""
    assert da.probe_packed(0, 0, 1 << 32) == 0
    assert da.probe_packed(0, 0xC2D00000 - 7, 15) == 0   # an odd count around -104
    assert da.probe_packed(1, 0, 1 << 32) == 0


@cuda
def test_bounded_wait_gives_up_and_reports_timeout(da, orc):
    """A kernel waits on an mbarrier phase that nothing completes, through the bounded wait
    every pipelined kernel uses: the wait gives up after its limit, the status word carries
    STATUS_TIMEOUT, and the context stays usable for the next call."""
    st = da.new_status()
    assert da.probe_bounded_wait(st) == da.STATUS_TIMEOUT
    Q, K, V = W.random_attn(49, 1, 2, 2, 40, 128, torch.bfloat16, True)
    out = da.det_attn(Q.cuda(), K.cuda(), V.cuda(), causal=True)
    _, _, _, ref = orc.Attn(Q, K, V, True).forward_rows()
    assert_bits_equal(out.reshape(-1, 128), ref, "after a timed-out wait")


@cuda
@pytest.mark.parametrize("causal", [False, True])
def test_score_cache_rare_paths_match_oracle(da, orc, causal):
    """det_attn at D = 128 (score cache, tensor-PV accumulate, finalize in the epilogue) on the
    inputs that reach its rare paths: a key far above the others (tiny weights for every
    other key: the spill slot and the whole-row canonical path), V columns with one huge
    element (the rest of the column falls below its fixed-point window: the listed V-bad
    keys and the touched-column canonical path), and wide-exponent rows."""
    Q, K, V = W.random_attn(311 + causal, 1, 2, 2, 300, 128, torch.bfloat16, causal, spread=20.0)
    K, V = K.clone(), V.clone()
    K[0, 0, 7] *= 2 ** 30
    K[0, 1, 200] *= 2 ** 25
    for d in (0, 17, 64, 127):
        V[0, :, 11 + d, d] = 2.0 ** 30
    st = da.new_status()
    out = da.det_attn(Q.cuda(), K.cuda(), V.cuda(), causal=causal, status=st)
    sh = da.det_attn_sharded(Q.cuda(), K.cuda(), V.cuda(), [100, 77, 123], causal=causal, order=[1, 2, 0], status=st)
    torch.cuda.synchronize()
    _, _, _, out_o = orc.Attn(Q, K, V, causal=causal).forward_rows()
    assert da.read_status(st) & ~1 == 0
    assert_bits_equal(out.reshape(-1, 128), out_o, "output")
    assert_bits_equal(sh, out, "sharded vs fused")


@cuda
@pytest.mark.parametrize("case", [
    # (B, Hq, Hkv, S, D, dtype, causal, ngroups, pinned)
    (2, 4, 2, 200, 128, torch.bfloat16, True, 3, True),
    (1, 4, 4, 150, 128, torch.bfloat16, False, 8, False),
    (1, 2, 1, 90, 64, torch.float32, True, 1, True),
])
def test_host_buffer_entry_point_equals_det_attn(da, case):
    """da_det_attn_host (host inputs and output, copies overlapped with the kernels in groups of
    (batch, KV head) units) against det_attn on device copies, bit for bit, for even and uneven
    groups, pinned and pageable host memory, GQA and f32."""
    B, Hq, Hkv, S, D, dt, causal, ngroups, pinned = case
    Q, K, V = W.random_attn(500 + S, B, Hq, Hkv, S, D, dt, causal)
    if pinned:
        Q, K, V = Q.pin_memory(), K.pin_memory(), V.pin_memory()
    got = da.det_attn_host(Q, K, V, causal=causal, ngroups=ngroups)
    ref = da.det_attn(Q.cuda(), K.cuda(), V.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert got.device.type == "cpu"
    assert_bits_equal(got, ref.cpu(), "host entry point vs det_attn")
