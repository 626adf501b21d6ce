"""Host-side argument checks of the Python binding, on the CPU: the CUDA-tensor check is
stubbed out and the library replaced by a stand-in that fails if called, so every case must be
rejected by the binding itself before any launch."""
import pytest
import torch

import bitwise_deterministic_shard_gb300 as da


@pytest.fixture
def nolib(monkeypatch):
    monkeypatch.setattr(da, "_cuda", lambda t, name: None)

    def forbidden():
        raise AssertionError("the library was reached")
    monkeypatch.setattr(da, "lib", forbidden)


def _state(N=4, V=10):
    x = torch.zeros(N, V)
    return x, torch.zeros(N, dtype=torch.int64), torch.zeros(N), torch.ones(N, dtype=torch.float64)


@pytest.mark.parametrize("bad", ["m_dtype", "m_len", "denom_dtype", "denom_len", "targets_len", "grad_len",
                                 "reduction"])
def test_dce_backward_rejects_bad_state(nolib, bad):
    x, t, m, d = _state()
    g = torch.ones(4)
    red = "none"
    if bad == "m_dtype":
        m = m.double()
    elif bad == "m_len":
        m = torch.zeros(3)
    elif bad == "denom_dtype":
        d = d.float()
    elif bad == "denom_len":
        d = torch.ones(5, dtype=torch.float64)
    elif bad == "targets_len":
        t = torch.zeros(2, dtype=torch.int64)
    elif bad == "grad_len":
        g = torch.ones(3)
    else:
        red = "avg"
    with pytest.raises(da.DetAttnError):
        da.dce_backward(x, t, m, d, g, red)


def test_dce_finalize_and_denom_reject_bad_state(nolib):
    x, t, m, d = _state()
    with pytest.raises(da.DetAttnError):
        da.dce_finalize(torch.zeros(4, 5, dtype=torch.int64), x, t, m)              # den is [N, 6]
    with pytest.raises(da.DetAttnError):
        da.dce_finalize(torch.zeros(4, 6, dtype=torch.int64), x, t, m.double())
    with pytest.raises(da.DetAttnError):
        da.dce_denom_digits(x, torch.zeros(3))
    with pytest.raises(da.DetAttnError):
        da.dce_reduce(torch.zeros(4), "none")
    with pytest.raises(da.DetAttnError):
        da.cross_entropy(x, t, reduction="avg")


def test_accumulate_finalize_rejects_a_bad_rowmax(monkeypatch):
    monkeypatch.setattr(da, "_cuda", lambda t, name: None)
    Q = torch.zeros(1, 2, 8, 128)
    with pytest.raises(da.DetAttnError):
        da.accumulate_finalize(Q, Q, Q, torch.zeros(15))
    with pytest.raises(da.DetAttnError):
        da.accumulate_finalize(Q, Q, Q, torch.zeros(16, dtype=torch.float64))


def test_static_forward_rejects_bad_targets(nolib):
    x, t, _, _ = _state()
    with pytest.raises(da.DetAttnError):
        da.dce_forward_static(x, torch.zeros(3, dtype=torch.int64))
    with pytest.raises(da.DetAttnError):
        da.dce_forward_static(x.double(), t)                     # f32 and bf16 logits only


class _Recorder:
    """Stands in for the library: records each call's name and arguments, returns DA_OK."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def f(*args):
            self.calls.append((name, args))
            return 0
        return f


@pytest.fixture
def recorder(monkeypatch):
    monkeypatch.setattr(da, "_cuda", lambda t, name: None)
    monkeypatch.setattr(da, "_stream", lambda: None)
    rec = _Recorder()
    monkeypatch.setattr(da, "lib", lambda: rec)
    return rec


def test_static_forward_reaches_the_library(recorder):
    x = torch.zeros(5, 7, dtype=torch.bfloat16)
    loss, denom = da.dce_forward_static(x, torch.arange(5, dtype=torch.int32))
    assert [c[0] for c in recorder.calls] == ["dce_forward_static"]
    M = recorder.calls[0][1][0]._obj
    assert (M.rows, M.cols, M.row_stride, M.dtype) == (5, 7, 7, 1)
    assert loss.shape == (5,) and loss.dtype == torch.float32
    assert denom.shape == (5,) and denom.dtype == torch.float64


@pytest.mark.parametrize("bad", ["dtype", "len", "noncontig"])
def test_denom_digits_checks_a_caller_den(nolib, bad):
    x, t, m, _ = _state()
    den = {"dtype": torch.zeros(4, 6, dtype=torch.int32), "len": torch.zeros(4, 5, dtype=torch.int64),
           "noncontig": torch.zeros(6, 4, dtype=torch.int64).t()}[bad]
    with pytest.raises(da.DetAttnError):
        da.dce_denom_digits(x, m, den=den, add_into=True)


@pytest.mark.parametrize("fn,dtype", [("compose_max", torch.float32), ("compose_add", torch.int64)])
def test_compose_checks_both_operands(nolib, fn, dtype):
    f = getattr(da, fn)
    dst = torch.zeros(8, dtype=dtype)
    other = torch.float32 if dtype == torch.int64 else torch.int64
    for src in (torch.zeros(7, dtype=dtype), torch.zeros(8, dtype=other), torch.zeros(16, dtype=dtype)[::2]):
        with pytest.raises(da.DetAttnError):
            f(dst, src)
    with pytest.raises(da.DetAttnError):
        f(torch.zeros(8, dtype=other), torch.zeros(8, dtype=other))


def test_outputs_and_state_are_checked(nolib):
    Q = torch.zeros(1, 2, 8, 16)
    with pytest.raises(da.DetAttnError):
        da.det_attn(Q, Q, Q, out=torch.zeros(1, 2, 8, 15))
    with pytest.raises(da.DetAttnError):
        da.rowmax(Q, Q, out=torch.zeros(1, 2, 7))
    with pytest.raises(da.DetAttnError):
        da.accumulate(Q, Q, Q, torch.zeros(1, 2, 8), num=torch.zeros(1, 2, 8, 15, 16, dtype=torch.int32))
    with pytest.raises(da.DetAttnError):
        da.accumulate(Q, Q, Q, torch.zeros(1, 2, 7))
    num = torch.zeros(1, 2, 8, 15, 16, dtype=torch.int64)
    with pytest.raises(da.DetAttnError):
        da.finalize(num, torch.zeros(1, 2, 8, 5, dtype=torch.int64))
    with pytest.raises(da.DetAttnError):
        da.finalize(num, torch.zeros(1, 2, 8, 6, dtype=torch.int64), out=torch.zeros(1, 2, 8, 16, dtype=torch.float64))
    with pytest.raises(da.DetAttnError):
        da.normalize(num.float())
    with pytest.raises(da.DetAttnError):
        da.dce_rowmax(torch.zeros(4, 10), out=torch.zeros(3))
    with pytest.raises(da.DetAttnError):
        da.det_attn(Q, Q, Q, status=torch.zeros(1, dtype=torch.int64))


def test_det_attn_host_rejects_bad_host_tensors():
    """The host-buffer entry point's binding checks its tensors before any CUDA call: host
    memory, [B, H, S, D], contiguous; ngroups >= 1."""
    import bitwise_deterministic_shard_gb300 as da
    Q = torch.zeros(1, 2, 8, 16, dtype=torch.bfloat16)
    with pytest.raises(da.DetAttnError):
        da.det_attn_host(Q.transpose(2, 3), Q, Q, device="cuda:0")      # not contiguous
    with pytest.raises(da.DetAttnError):
        da.det_attn_host(Q[0], Q, Q, device="cuda:0")                    # not 4-dimensional
    with pytest.raises(da.DetAttnError):
        da.det_attn_host(Q, Q, Q, ngroups=0, device="cuda:0")
    with pytest.raises(da.DetAttnError):
        da.det_attn_host(Q.half(), Q.half(), Q.half(), device="cuda:0")  # f16 is not a supported dtype
