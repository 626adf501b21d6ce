"""The C-ABI library loads without a GPU and exports every entry point that
include/detattn.h declares (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "detattn.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int64_t|int|size_t|char\s*\*|const char\s*\*)\s*\**\s*(\w+)\s*\(", txt, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def libpath():
    from bitwise_deterministic_shard_gb300 import build
    return build.build()


def test_header_declares_the_page_api():
    names = _declared()
    for n in ("da_rowmax", "da_accumulate", "da_finalize", "da_det_attn", "da_det_attn_sharded", "da_compose_max",
              "da_compose_add", "da_normalize", "dce_rowmax", "dce_denom_digits", "dce_finalize"):
        assert n in names


def test_library_exports_every_declared_symbol(libpath):
    lib = ctypes.CDLL(libpath)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_only_calls(libpath):
    lib = ctypes.CDLL(libpath)
    lib.da_status_string.restype = ctypes.c_char_p
    assert lib.da_abi_version() == 3
    assert lib.da_status_string(0) == b"ok"
    assert lib.da_status_string(5).startswith(b"workspace")


def test_argument_checks_reject_before_any_launch(libpath):
    """Host validation returns codes without touching a GPU (null / bad shapes)."""
    import bitwise_deterministic_shard_gb300 as da
    L = da.lib()
    R = lambda d, lo, hi: L.da_rowmax(d, lo, hi, None, None, 0, None)
    assert R(None, 0, 0) == 1                                               # null descriptor
    d = da._Desc()
    for t in (d.q, d.k, d.v):
        t.ptr = 4096                                                        # never dereferenced: rejected first
        t.dtype, t.B, t.H, t.S, t.D = 1, 1, 2, 8, 300                      # D > 256
        t.stride[3] = 1
    assert R(ctypes.byref(d), 0, 8) == 2
    for t in (d.q, d.k, d.v):
        t.D = 64
    d.k.H = d.v.H = 3                                                       # Hq % Hkv != 0
    assert R(ctypes.byref(d), 0, 8) == 2
    d.k.H = d.v.H = 1
    d.v.dtype = 0                                                           # mixed dtypes
    assert R(ctypes.byref(d), 0, 8) == 3
    d.v.dtype = 1
    d.causal, d.k.S, d.v.S = 1, 9, 9                                        # causal needs Sq == Skv
    assert R(ctypes.byref(d), 0, 9) == 1
    d.causal = 0
    assert R(ctypes.byref(d), 5, 3) == 1                                    # kv_hi < kv_lo
    d.k.S = d.v.S = 8
    assert R(ctypes.byref(d), 0, 8) == 1                                    # m is null
    assert L.da_kv_workspace_bytes(ctypes.byref(d)) > 0
    assert L.da_det_attn_sharded(ctypes.byref(d), (ctypes.c_int64 * 2)(4, 4), 2, None, None, None, 0, None) == 1
    assert L.da_normalize(None, 4, 7, 1, None, None) == 1                  # ndig must be 15 or 6


def test_new_entry_points_reject_before_any_launch(libpath):
    """da_accumulate_finalize, dce_backward and dce_reduce validate on the host first."""
    import bitwise_deterministic_shard_gb300 as da
    L = da.lib()
    d = da._Desc()
    for t in (d.q, d.k, d.v):
        t.ptr = 4096
        t.dtype, t.B, t.H, t.S, t.D = 1, 1, 2, 8, 128
        t.stride[3] = 1
    assert L.da_accumulate_finalize(None, None, None, None, 0, None) == 1        # null descriptor
    assert L.da_accumulate_finalize(ctypes.byref(d), None, None, None, 0, None) == 1   # null m / out
    assert L.da_accumulate_finalize(ctypes.byref(d), 4096, 8192, None, 0, None) == 5   # no workspace
    M = da._Matrix()
    M.ptr, M.dtype, M.rows, M.cols, M.row_stride = 4096, 0, 4, 10, 10
    assert L.dce_backward(ctypes.byref(M), None, None, None, None, 3, None, None, None) == 1    # reduction 0..2
    assert L.dce_backward(ctypes.byref(M), None, None, None, None, 0, None, None, None) == 1    # null pointers
    M.row_stride = 5
    assert L.dce_backward(ctypes.byref(M), 8, 4, 8, 4, 0, 4, None, None) == 2                   # row stride < cols
    assert L.dce_reduce(None, 4, 0, None, None) == 1                                             # "none" is not a reduction
    assert L.dce_reduce(None, -1, 1, 4096, None) == 1
    assert L.dce_reduce(None, 4, 2, 4096, None) == 1                                             # null losses
    assert L.dce_reduce(4098, 4, 2, 4096, None) == 4                                             # misaligned


def test_probe_arguments_rejected_before_any_launch(libpath):
    import bitwise_deterministic_shard_gb300 as da
    L = da.lib()
    assert L.da_probe_int_mac(-1, 4, None, None) == 1
    assert L.da_probe_int_mac(8, 0, None, None) == 1
    assert L.da_probe_int_mac(8, 4, None, None) == 1                        # null sink
    assert L.da_probe_int_mac(8, 4, ctypes.c_void_p(4100), None) == 4      # misaligned sink
    assert L.da_probe_bounded_wait(None, None) == 1
    assert L.da_probe_packed(0, 0, -1, ctypes.c_void_p(4096), None) == 1
    assert L.da_probe_packed(0, 0, (1 << 32) + 1, ctypes.c_void_p(4096), None) == 1
    assert L.da_probe_packed(2, 0, 8, ctypes.c_void_p(4096), None) == 1
    assert L.da_probe_packed(-1, 0, 8, ctypes.c_void_p(4096), None) == 1
    assert L.da_probe_packed(1, 0, 8, None, None) == 1
    assert L.da_probe_packed(1, 0, 8, ctypes.c_void_p(4100), None) == 4
    assert L.da_probe_int_mac_per_thread_iter() == 32
    assert "da_probe_int_mac_per_thread_iter" in _declared()
