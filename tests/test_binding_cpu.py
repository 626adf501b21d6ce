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
