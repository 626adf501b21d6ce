"""The static-scratch cross-entropy entry point (for callers that cannot allocate device
memory) against the allocating entry points, through the C ABI, on two calls in a row.

This file is collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It passes both alone in a fresh process (the first
call looks up the scratch address) and after the other tests.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_static_scratch_forward_matches_allocating_path_twice(oracle_native):
    import bitwise_deterministic_shard_gb300 as da
    g = torch.Generator().manual_seed(91)
    cases = [((torch.randn(300, 5000, generator=g) * 2).float(), 5000),
             ((torch.randn(77, 1234, generator=g) * 3).to(torch.bfloat16), 1234)]
    for x, V in cases:                       # two calls in a row, different sizes and dtypes
        t = torch.randint(0, V, (x.shape[0],), generator=g)
        x, t = x.cuda(), t.cuda()
        st = da.new_status()
        loss, denom = da.dce_forward_static(x, t, status=st)
        ref_loss, ref_denom, _, _ = da.dce_forward(x, t)
        torch.cuda.synchronize()
        assert da.read_status(st) == 0
        assert torch.equal(loss, ref_loss)   # the contract fixes every rounding: zero tolerance
        assert torch.equal(denom, ref_denom)
        o_loss, o_denom, _, _, _ = oracle_native.DCE(x).forward(t.cpu().numpy())
        assert torch.equal(loss.cpu(), torch.from_numpy(o_loss))
        assert torch.equal(denom.cpu(), torch.from_numpy(o_denom))


@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_static_scratch_rejects_too_many_rows():
    import bitwise_deterministic_shard_gb300 as da
    x = torch.zeros(da.STATIC_MAX_ROWS + 1, 2, device="cuda")
    t = torch.zeros(da.STATIC_MAX_ROWS + 1, dtype=torch.int64, device="cuda")
    with pytest.raises(da.DetAttnError, match="workspace"):
        da.dce_forward_static(x, t)
