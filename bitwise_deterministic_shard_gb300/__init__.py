"""Python binding of libdetattn, the C ABI of the exact, order-invariant softmax reduction.

Argument marshalling only: every step of the computation runs in the CUDA kernels behind
include/detattn.h.  PyTorch supplies device memory and the current stream.  There is no
CPU fallback: if the library is not built, or a tensor is not on a CUDA device, the call
raises.

Names follow the pages: det-attn ("API": det_attn, rowmax, accumulate, finalize,
det_attn_sharded) and det-cross-entropy ("API": rowmax, denom_digits, finalize; here
dce_rowmax, dce_denom_digits, dce_finalize).
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdetattn.so")

NUM_NDIG, DEN_NDIG = 15, 6
NUM_E0, DEN_E0 = -320, -160
STATUS_NONFINITE, STATUS_ROWMAX_VIOLATION, STATUS_DIGIT_HEADROOM, STATUS_BAD_TARGET, STATUS_TIMEOUT = 1, 2, 4, 8, 16


class DetAttnError(RuntimeError):
    pass


class _Tensor(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("dtype", C.c_int32), ("B", C.c_int64), ("H", C.c_int64), ("S", C.c_int64),
                ("D", C.c_int64), ("stride", C.c_int64 * 4)]


class _Desc(C.Structure):
    _fields_ = [("q", _Tensor), ("k", _Tensor), ("v", _Tensor), ("causal", C.c_int32), ("scale", C.c_float),
                ("dev_status", C.c_void_p)]


class _Matrix(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("dtype", C.c_int32), ("rows", C.c_int64), ("cols", C.c_int64),
                ("row_stride", C.c_int64)]


_lib = None
_P, _I64, _I32 = C.c_void_p, C.c_int64, C.c_int


def lib():
    """The loaded libdetattn.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise DetAttnError(f"{LIB_PATH} is missing: build it with "
                               "`python -m bitwise_deterministic_shard_gb300.build` (needs nvcc)")
        L = C.CDLL(LIB_PATH)
        L.da_abi_version.restype = C.c_int
        L.da_status_string.argtypes = [C.c_int]
        L.da_status_string.restype = C.c_char_p
        D = C.POINTER(_Desc)
        M = C.POINTER(_Matrix)
        L.da_kv_workspace_bytes.argtypes = [D]
        L.da_kv_workspace_bytes.restype = C.c_size_t
        L.da_rowmax.argtypes = [D, _I64, _I64, _P, _P, C.c_size_t, _P]
        L.da_accumulate.argtypes = [D, _P, _I64, _I64, _P, _P, _I32, _P, C.c_size_t, _P]
        L.da_compose_max.argtypes = [_P, _P, _I64, _P]
        L.da_compose_add.argtypes = [_P, _P, _I64, _P]
        L.da_normalize.argtypes = [_P, _I64, _I32, _I64, _P, _P]
        L.da_finalize.argtypes = [_P, _P, _I64, _I64, _I64, _I64, _P, _P, _P]
        L.da_workspace_bytes.argtypes = [D, _I32]
        L.da_workspace_bytes.restype = C.c_size_t
        L.da_det_attn.argtypes = [D, _P, _P, C.c_size_t, _P]
        L.da_det_attn_host_workspace_bytes.argtypes = [D, _I32]
        L.da_det_attn_host_workspace_bytes.restype = C.c_size_t
        L.da_det_attn_host.argtypes = [D, _P, _I32, _P, C.c_size_t, _P]
        L.da_score_cache_bytes.argtypes = [D]
        L.da_score_cache_bytes.restype = C.c_size_t
        L.da_rowmax_cached.argtypes = [D, _P, _P, C.c_size_t, _P]
        L.da_accumulate_finalize_cached.argtypes = [D, _P, _P, _P, C.c_size_t, _P]
        L.da_accumulate_finalize.argtypes = [D, _P, _P, _P, C.c_size_t, _P]
        L.da_det_attn_sharded.argtypes = [D, _P, _I32, _P, _P, _P, C.c_size_t, _P]
        L.dce_rowmax.argtypes = [M, _I64, _I64, _P, _P, _P]
        L.dce_denom_digits.argtypes = [M, _P, _I64, _I64, _P, _I32, _P, _P]
        L.dce_finalize.argtypes = [_P, M, _P, _P, _P, _P, _P, _P]
        L.dce_backward.argtypes = [M, _P, _P, _P, _P, _I32, _P, _P, _P]
        L.dce_reduce.argtypes = [_P, _I64, _I32, _P, _P]
        L.dce_forward_static.argtypes = [M, _P, _P, _P, _P, _P]
        L.dce_finalize_shard.argtypes = [_P, M, _I64, _I64, _P, _P, _P, _P, _P, _P]
        L.dce_backward_shard.argtypes = [M, _I64, _P, _P, _P, _P, _I32, _P, _P, _P]
        L.da_probe_int_mac.argtypes = [_I64, _I32, _P, _P]
        L.da_probe_int_mac_per_thread_iter.restype = C.c_int64
        L.da_probe_bounded_wait.argtypes = [_P, _P]
        L.da_probe_packed.argtypes = [_I32, C.c_uint32, _I64, _P, _P]
        for f in ("da_rowmax", "da_accumulate", "da_compose_max", "da_compose_add", "da_normalize", "da_finalize",
                  "da_det_attn", "da_det_attn_host", "da_det_attn_sharded", "da_accumulate_finalize", "dce_rowmax", "dce_denom_digits", "dce_finalize",
                  "dce_backward", "dce_reduce", "dce_forward_static", "da_probe_int_mac", "da_probe_bounded_wait",
                  "da_probe_packed",
                  "dce_finalize_shard", "dce_backward_shard", "da_rowmax_cached", "da_accumulate_finalize_cached"):
            getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def _check(code: int, what: str):
    if code != 0:
        raise DetAttnError(f"{what}: {lib().da_status_string(code).decode()} (code {code})")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return 0
    if t.dtype == torch.bfloat16:
        return 1
    raise DetAttnError(f"unsupported dtype {t.dtype}: f32 and bf16 only")


def _cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise DetAttnError(f"{name} must be a CUDA tensor (there is no CPU path)")


def _tensor(t: torch.Tensor, name: str) -> _Tensor:
    _cuda(t, name)
    if t.dim() != 4:
        raise DetAttnError(f"{name} must be [B, H, S, D]")
    if t.stride(3) != 1:
        t = t.contiguous()
    x = _Tensor()
    x.ptr = t.data_ptr()
    x.dtype = _dtype_code(t)
    x.B, x.H, x.S, x.D = t.shape
    for i in range(4):
        x.stride[i] = t.stride(i)
    return x


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _sptr(status):
    """Pointer of an optional device status word: a CUDA int32 tensor of at least one element."""
    if status is None:
        return None
    _cuda(status, "status")
    if status.dtype != torch.int32 or status.numel() < 1:
        raise DetAttnError("status must be a CUDA int32 tensor (see new_status())")
    return C.c_void_p(status.data_ptr())


def _out(t, dtype, shape, device, name):
    """A caller-supplied output (or in-place state): allocated when None, else checked for
    device, dtype, element count and contiguity.  Never copied, since the kernels write it."""
    n = 1
    for x in shape:
        n *= int(x)
    if t is None:
        return torch.empty(*shape, dtype=dtype, device=device)
    _cuda(t, name)
    if t.dtype != dtype or t.numel() != n or not t.is_contiguous() or t.device != torch.device(device):
        raise DetAttnError(f"{name} must be a contiguous {dtype} tensor of {n} elements on {device}")
    return t


class _Problem:
    """Keeps the tensors alive while their descriptor is in use."""

    def __init__(self, Q, K, V, causal, scale, status=None):
        self.keep = [t if t.stride(3) == 1 else t.contiguous() for t in (Q, K, V)]
        Q, K, V = self.keep
        self.desc = _Desc()
        self.desc.q, self.desc.k, self.desc.v = _tensor(Q, "Q"), _tensor(K, "K"), _tensor(V, "V")
        self.desc.causal = 1 if causal else 0
        self.desc.scale = math.nan if scale is None else float(scale)
        self.desc.dev_status = _sptr(status)
        self.B, self.Hq, self.Sq, self.D = Q.shape
        self.Skv = K.shape[2]
        self.device = Q.device

    def ref(self):
        return C.byref(self.desc)


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word for the `status=` arguments."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def read_status(status: torch.Tensor) -> int:
    return int(status.item())


def workspace_bytes(Q, K, V, causal=False, scale=None, nsplits=1) -> int:
    P = _Problem(Q, K, V, causal, scale)
    return int(lib().da_workspace_bytes(P.ref(), nsplits))


def _workspace(P: _Problem, nsplits: int, ws):
    need = int(lib().da_workspace_bytes(P.ref(), nsplits))
    if ws is None or ws.numel() * ws.element_size() < need:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=P.device)
    return ws


def _kv_workspace(P: _Problem, ws):
    need = int(lib().da_kv_workspace_bytes(P.ref()))
    if ws is None or ws.numel() * ws.element_size() < need:
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=P.device)
    return ws


def det_attn(Q, K, V, causal=False, scale=None, out=None, workspace=None, status=None):
    """Fused deterministic attention (det-attn "API": det_attn); f32 output [B, Hq, Sq, D]."""
    P = _Problem(Q, K, V, causal, scale, status)
    out = _out(out, torch.float32, (P.B, P.Hq, P.Sq, P.D), P.device, "out")
    ws = _workspace(P, 1, workspace)
    _check(lib().da_det_attn(P.ref(), _ptr(out), _ptr(ws), ws.numel(), _stream()), "det_attn")
    return out


def _host_tensor(t: torch.Tensor, name: str) -> _Tensor:
    """Descriptor of a contiguous host [B, H, S, D] tensor (the host-buffer entry point)."""
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise DetAttnError(f"{name} must be a host (CPU) tensor for det_attn_host")
    if t.dim() != 4 or not t.is_contiguous():
        raise DetAttnError(f"{name} must be a contiguous [B, H, S, D] host tensor")
    x = _Tensor()
    x.ptr = t.data_ptr()
    x.dtype = _dtype_code(t)
    x.B, x.H, x.S, x.D = t.shape
    for i in range(4):
        x.stride[i] = t.stride(i)
    return x


def det_attn_host(Q, K, V, causal=False, scale=None, out=None, ngroups=4, workspace=None, status=None,
                  device=None):
    """det_attn on HOST tensors through da_det_attn_host: Q, K, V contiguous CPU tensors
    [B, H, S, D] (pinned memory lets the copies overlap the kernels), the f32 output a CPU
    tensor [B, Hq, Sq, D] (pinned when allocated here).  The copies and the kernels run in
    `ngroups` groups of (batch, KV head) units on `device` (default: the current CUDA device);
    the call returns when the output is in host memory.  Bit-identical to det_attn."""
    desc = _Desc()
    desc.q, desc.k, desc.v = _host_tensor(Q, "Q"), _host_tensor(K, "K"), _host_tensor(V, "V")
    if int(ngroups) < 1:
        raise DetAttnError("ngroups must be at least 1")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    desc.causal = 1 if causal else 0
    desc.scale = math.nan if scale is None else float(scale)
    desc.dev_status = _sptr(status)
    B, Hq, Sq, D = Q.shape
    if out is None:
        out = torch.empty(B, Hq, Sq, D, dtype=torch.float32).pin_memory()
    elif (out.device.type != "cpu" or out.dtype != torch.float32 or tuple(out.shape) != (B, Hq, Sq, D)
          or not out.is_contiguous()):
        raise DetAttnError("out must be a contiguous f32 host tensor [B, Hq, Sq, D]")
    need = int(lib().da_det_attn_host_workspace_bytes(C.byref(desc), int(ngroups)))
    if need == 0 and B * Sq > 0:
        raise DetAttnError("det_attn_host: invalid shapes, dtypes or ngroups")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        _check(lib().da_det_attn_host(C.byref(desc), _ptr(out), int(ngroups), _ptr(workspace), need, _stream()),
               "det_attn_host")
        torch.cuda.current_stream().synchronize()
    return out


def score_cache_bytes(Q, K, V, causal=False, scale=None) -> int:
    """Bytes of the score cache det_attn keeps in its workspace (0 when it recomputes scores)."""
    P = _Problem(Q, K, V, causal, scale)
    return int(lib().da_score_cache_bytes(P.ref()))


def accumulate_finalize(Q, K, V, rowmax, causal=False, scale=None, out=None, workspace=None, status=None):
    """Pass 2 and finalize over all keys with the global rowmax: the f32 output [B, Hq, Sq, D],
    equal bit for bit to finalize(*accumulate(Q, K, V, rowmax, 0, Skv)); the tensor-PV kernel
    finalizes in its epilogue, so the NUM digits are never stored."""
    P = _Problem(Q, K, V, causal, scale, status)
    _cuda(rowmax, "rowmax")
    if rowmax.dtype != torch.float32 or rowmax.numel() != P.B * P.Hq * P.Sq:
        raise DetAttnError("rowmax must be f32 [B, Hq, Sq]")
    out = _out(out, torch.float32, (P.B, P.Hq, P.Sq, P.D), P.device, "out")
    ws = _workspace(P, 1, workspace)
    _check(lib().da_accumulate_finalize(P.ref(), _ptr(rowmax.contiguous()), _ptr(out), _ptr(ws), ws.numel(),
                                        _stream()), "accumulate_finalize")
    return out


def det_attn_sharded(Q, K, V, kv_splits, causal=False, scale=None, order=None, out=None, workspace=None,
                     status=None):
    """KV-shard composition (det-attn "API": det_attn_sharded), bit-identical to det_attn
    for any kv_splits and any visiting order."""
    P = _Problem(Q, K, V, causal, scale, status)
    n = len(kv_splits)
    splits = (C.c_int64 * n)(*[int(x) for x in kv_splits])
    ordv = None if order is None else (C.c_int32 * n)(*[int(x) for x in order])
    out = _out(out, torch.float32, (P.B, P.Hq, P.Sq, P.D), P.device, "out")
    ws = _workspace(P, n, workspace)
    _check(lib().da_det_attn_sharded(P.ref(), splits, n, ordv, _ptr(out), _ptr(ws), ws.numel(), _stream()),
           "det_attn_sharded")
    return out


def _all_reduce(t, op, group):
    """In-place all-reduce over the process group: on the device with NCCL, through a host copy
    with a CPU backend (gloo).  MAX of f32 and SUM of int64 are exact, so the result does not
    depend on the reduction order."""
    import torch.distributed as dist
    if dist.get_backend(group) == "nccl":
        dist.all_reduce(t, op=op, group=group)
        return t
    h = t.cpu()
    dist.all_reduce(h, op=op, group=group)
    t.copy_(h)
    return t


def det_attn_cp(Q, K, V, kv_lo, S_kv=None, causal=False, scale=None, group=None, status=None):
    """Context-parallel det-attn (det-attn, introduction and "Method": the output is the same
    whether the sequence lives on one device or is split over many).  This rank holds every
    query row Q [B, Hq, Sq, D] and the keys and values [kv_lo, kv_lo + K.shape[2]) of a
    sequence of S_kv keys (S_kv = Sq when causal).  The rank runs pass 1 over its keys, the
    group takes the max all-reduce of the f32 rowmax; the rank runs pass 2 with that global
    rowmax, the group sums the canonical int64 NUM / DEN digits (exact, any order); every
    rank then normalizes and finalizes on its GPU.  The f32 output [B, Hq, Sq, D] equals
    det_attn over the whole sequence bit for bit, for any split of the keys over the ranks.

    The shard is presented to the kernels at its global key positions (causal masking uses
    them); the kernels read key / value rows of their range only.  Collectives: NCCL on device
    tensors, or any CPU backend through host copies."""
    import torch.distributed as dist
    P = _Problem(Q, K, V, causal, scale, status)
    S_kv = P.Sq if S_kv is None else int(S_kv)
    n_local = P.keep[1].shape[2]
    kv_lo = int(kv_lo)
    kv_hi = kv_lo + n_local
    if P.keep[2].shape[2] != n_local or kv_lo < 0 or kv_hi > S_kv:
        raise DetAttnError("the key / value shard must lie inside [0, S_kv) and K, V must hold the same rows")
    for t, x in ((P.desc.k, P.keep[1]), (P.desc.v, P.keep[2])):
        if n_local > 0:
            t.ptr = x.data_ptr() - kv_lo * x.stride(2) * x.element_size()   # row kv_lo at the shard's first row
        else:   # an empty shard holds no storage; the kernels read no key row of an empty range
            t.ptr = P.keep[0].data_ptr()
        t.S = S_kv
    L = lib()
    kvws = torch.empty(max(int(L.da_kv_workspace_bytes(P.ref())), 1), dtype=torch.uint8, device=P.device)
    m = torch.empty(P.B, P.Hq, P.Sq, dtype=torch.float32, device=P.device)
    _check(L.da_rowmax(P.ref(), kv_lo, kv_hi, _ptr(m), _ptr(kvws), kvws.numel(), _stream()), "rowmax")
    _all_reduce(m, dist.ReduceOp.MAX, group)
    num = torch.empty(P.B, P.Hq, P.Sq, NUM_NDIG, P.D, dtype=torch.int64, device=P.device)
    den = torch.empty(P.B, P.Hq, P.Sq, DEN_NDIG, dtype=torch.int64, device=P.device)
    _check(L.da_accumulate(P.ref(), _ptr(m), kv_lo, kv_hi, _ptr(num), _ptr(den), 0, _ptr(kvws), kvws.numel(),
                           _stream()), "accumulate")
    _all_reduce(num, dist.ReduceOp.SUM, group)
    _all_reduce(den, dist.ReduceOp.SUM, group)
    normalize(num, status, ndig=NUM_NDIG)
    normalize(den, status, ndig=DEN_NDIG)
    return finalize(num, den, status=status)


def rowmax(Q, K, kv_lo=0, kv_hi=None, causal=False, scale=None, out=None, status=None, workspace=None):
    """Per-query rowmax over keys [kv_lo, kv_hi) (det-attn "API": rowmax); f32 [B, Hq, Sq].
    Shards combine with compose_max (or torch.maximum)."""
    P = _Problem(Q, K, K, causal, scale, status)
    kv_hi = P.Skv if kv_hi is None else kv_hi
    m = _out(out, torch.float32, (P.B, P.Hq, P.Sq), P.device, "out")
    ws = _kv_workspace(P, workspace)
    _check(lib().da_rowmax(P.ref(), kv_lo, kv_hi, _ptr(m), _ptr(ws), ws.numel(), _stream()), "rowmax")
    return m


def accumulate(Q, K, V, m, kv_lo=0, kv_hi=None, causal=False, scale=None, num=None, den=None, add_into=False,
               status=None, workspace=None):
    """Exact NUM/DEN digits of keys [kv_lo, kv_hi) with the global rowmax m (det-attn "API":
    accumulate).  Returns (num int64 [B,Hq,Sq,15,D], den int64 [B,Hq,Sq,6]), canonical."""
    P = _Problem(Q, K, V, causal, scale, status)
    kv_hi = P.Skv if kv_hi is None else kv_hi
    num = _out(num, torch.int64, (P.B, P.Hq, P.Sq, NUM_NDIG, P.D), P.device, "num")
    den = _out(den, torch.int64, (P.B, P.Hq, P.Sq, DEN_NDIG), P.device, "den")
    _cuda(m, "rowmax")
    if m.dtype != torch.float32 or m.numel() != P.B * P.Hq * P.Sq:
        raise DetAttnError("rowmax must be f32 [B, Hq, Sq]")
    m = m.contiguous()
    ws = _kv_workspace(P, workspace)
    _check(lib().da_accumulate(P.ref(), _ptr(m), kv_lo, kv_hi, _ptr(num), _ptr(den), 1 if add_into else 0,
                               _ptr(ws), ws.numel(), _stream()), "accumulate")
    return num, den


def _inplace_pair(dst, src, dtype, what):
    """dst and src of one composition: CUDA tensors of `dtype` on one device, equal element
    counts, both contiguous (dst is written in place, so it cannot be copied)."""
    _cuda(dst, f"{what} dst")
    _cuda(src, f"{what} src")
    if dst.dtype != dtype or src.dtype != dtype:
        raise DetAttnError(f"{what}: dst and src must both be {dtype}")
    if dst.numel() != src.numel():
        raise DetAttnError(f"{what}: dst has {dst.numel()} elements, src {src.numel()}")
    if dst.device != src.device:
        raise DetAttnError(f"{what}: dst and src are on different devices")
    if not dst.is_contiguous() or not src.is_contiguous():
        raise DetAttnError(f"{what}: dst and src must be contiguous")


def compose_max(dst, src):
    """dst = max(dst, src) elementwise (shard rowmax composition), in place."""
    _inplace_pair(dst, src, torch.float32, "compose_max")
    _check(lib().da_compose_max(_ptr(dst), _ptr(src), dst.numel(), _stream()), "compose_max")
    return dst


def compose_add(dst, src):
    """dst += src elementwise (int64 digit composition), in place."""
    _inplace_pair(dst, src, torch.int64, "compose_add")
    _check(lib().da_compose_add(_ptr(dst), _ptr(src), dst.numel(), _stream()), "compose_add")
    return dst


def normalize(digits, status=None, ndig=None):
    """Canonical form, in place, of NUM [..., 15, D] or DEN [..., 6] digit arrays.  ndig (15 or
    6) names the kind; without it a 5-dimensional array is NUM [B, Hq, Sq, 15, D] and a 4- or
    2-dimensional one DEN [B, Hq, Sq, 6] / [N, 6]."""
    _cuda(digits, "digits")
    if digits.dtype != torch.int64 or not digits.is_contiguous() or digits.dim() < 1:
        raise DetAttnError("digits must be a contiguous int64 tensor")
    if ndig is None:
        if digits.dim() == 5:
            ndig = NUM_NDIG
        elif digits.dim() in (2, 4):
            ndig = DEN_NDIG
        else:
            raise DetAttnError("pass ndig=15 (NUM) or ndig=6 (DEN) for this shape")
    if ndig == NUM_NDIG:
        if digits.dim() < 2 or digits.shape[-2] != NUM_NDIG:
            raise DetAttnError("NUM digits must be laid out [..., 15, D]")
        inner = digits.shape[-1]
    elif ndig == DEN_NDIG:
        if digits.shape[-1] != DEN_NDIG:
            raise DetAttnError("DEN digits must be laid out [..., 6]")
        inner = 1
    else:
        raise DetAttnError("ndig must be 15 (NUM) or 6 (DEN)")
    nrows = digits.numel() // (ndig * inner)
    _check(lib().da_normalize(_ptr(digits), nrows, ndig, inner, _sptr(status), _stream()), "normalize")
    return digits


def finalize(num, den, out=None, status=None):
    """Digits -> f32 output (det-attn "API": finalize): RN32(RN64(RN64(NUM)/RN64(DEN)))."""
    _cuda(num, "num")
    if num.dim() != 5 or num.shape[3] != NUM_NDIG:
        raise DetAttnError("num must be int64 [B, Hq, Sq, 15, D]")
    B, H, S, _, D = num.shape
    num = _out(num, torch.int64, tuple(num.shape), num.device, "num")
    den = _out(den, torch.int64, (B, H, S, DEN_NDIG), num.device, "den")
    out = _out(out, torch.float32, (B, H, S, D), num.device, "out")
    _check(lib().da_finalize(_ptr(num), _ptr(den), B, H, S, D, _ptr(out), _sptr(status), _stream()), "finalize")
    return out


def _matrix(x: torch.Tensor) -> tuple[_Matrix, torch.Tensor]:
    _cuda(x, "logits")
    if x.dim() != 2:
        raise DetAttnError("logits must be [N, V]")
    if x.stride(1) != 1:
        x = x.contiguous()
    m = _Matrix()
    m.ptr = x.data_ptr()
    m.dtype = _dtype_code(x)
    m.rows, m.cols = x.shape
    m.row_stride = x.stride(0)
    return m, x


def dce_rowmax(logits, v_lo=0, v_hi=None, out=None, status=None):
    """Per-token max over the vocab range [v_lo, v_hi) (det-cross-entropy "API": rowmax)."""
    M, keep = _matrix(logits)
    v_hi = M.cols if v_hi is None else v_hi
    m = _out(out, torch.float32, (M.rows,), logits.device, "out")
    _check(lib().dce_rowmax(C.byref(M), v_lo, v_hi, _ptr(m), _sptr(status), _stream()), "dce_rowmax")
    return m


def _vec(t, dtype, n, name):
    """A per-row input: a CUDA tensor of the given dtype and element count, made contiguous."""
    _cuda(t, name)
    if t.dtype != dtype or t.numel() != n:
        raise DetAttnError(f"{name} must be a {dtype} tensor of {n} elements")
    return t.contiguous()


def dce_denom_digits(logits, m, v_lo=0, v_hi=None, den=None, add_into=False, status=None):
    """Exact denominator digits over [v_lo, v_hi) with the global rowmax m
    (det-cross-entropy "API": denom_digits); int64 [N, 6]."""
    M, keep = _matrix(logits)
    m = _vec(m, torch.float32, M.rows, "rowmax")
    v_hi = M.cols if v_hi is None else v_hi
    if den is None:
        den = torch.empty(M.rows, DEN_NDIG, dtype=torch.int64, device=logits.device)
    else:   # written in place (and read with add_into): checked, never copied
        _cuda(den, "den")
        if den.dtype != torch.int64 or den.numel() != M.rows * DEN_NDIG or not den.is_contiguous():
            raise DetAttnError(f"den must be a contiguous torch.int64 tensor of {M.rows * DEN_NDIG} elements")
    _check(lib().dce_denom_digits(C.byref(M), _ptr(m), v_lo, v_hi, _ptr(den), 1 if add_into else 0, _sptr(status),
                                  _stream()), "dce_denom_digits")
    return den


def dce_finalize(den, logits, targets, m, status=None):
    """(loss f32 [N], denom f64 [N]) from composed digits (det-cross-entropy "API": finalize)."""
    M, keep = _matrix(logits)
    den = _vec(den, torch.int64, M.rows * DEN_NDIG, "den")
    m = _vec(m, torch.float32, M.rows, "rowmax")
    targets = _vec(targets.to(torch.int64), torch.int64, M.rows, "targets")
    loss = torch.empty(M.rows, dtype=torch.float32, device=logits.device)
    denom = torch.empty(M.rows, dtype=torch.float64, device=logits.device)
    _check(lib().dce_finalize(_ptr(den), C.byref(M), _ptr(targets), _ptr(m), _ptr(loss), _ptr(denom), _sptr(status),
                              _stream()), "dce_finalize")
    return loss, denom


def dce_forward(logits, targets, splits=None, status=None):
    """Vocab-sharded composition (det-cross-entropy "Usage"): rowmax by max, digits by add,
    finalize.  Returns (loss, denom, m, den)."""
    V = logits.shape[1]
    splits = [V] if splits is None else list(splits)
    bounds, lo = [], 0
    for n in splits:
        bounds.append((lo, lo + n))
        lo += n
    if lo != V:
        raise DetAttnError("vocab splits must sum to V")
    m = dce_rowmax(logits, *bounds[0], status=status)
    if len(bounds) > 1:
        tmp = torch.empty_like(m)
        for a, b in bounds[1:]:
            compose_max(m, dce_rowmax(logits, a, b, out=tmp, status=status))
    den = None
    for k, (a, b) in enumerate(bounds):
        den = dce_denom_digits(logits, m, a, b, den=den, add_into=k > 0, status=status)
    loss, denom = dce_finalize(den, logits, targets, m, status=status)
    return loss, denom, m, den


_REDUCTIONS = {"none": 0, "sum": 1, "mean": 2}


def dce_backward(logits, targets, m, denom, grad, reduction="none", status=None):
    """Deterministic dLogits of the cross-entropy loss from forward's state (m, denom):
    RN32(go_i * RN32(RN32(RN64(w / denom_i)) - onehot)), w = exp32_det(RN32(x - m_i));
    go_i = grad[i] ("none"), grad ("sum"), RN32(RN64(grad / N)) ("mean").  Returns a tensor
    shaped like logits, of its dtype."""
    M, keep = _matrix(logits)
    if reduction not in _REDUCTIONS:
        raise DetAttnError("reduction must be 'none', 'sum' or 'mean'")
    red = _REDUCTIONS[reduction]
    grad = grad.to(torch.float32).reshape(-1).contiguous()
    if grad.numel() != (M.rows if red == 0 else 1):
        raise DetAttnError("grad must have one entry per row for reduction='none', else one entry")
    targets = _vec(targets.to(torch.int64), torch.int64, M.rows, "targets")
    m = _vec(m, torch.float32, M.rows, "rowmax")
    denom = _vec(denom, torch.float64, M.rows, "denom")
    out = torch.empty((M.rows, M.cols), dtype=logits.dtype, device=logits.device)
    _check(lib().dce_backward(C.byref(M), _ptr(targets), _ptr(m), _ptr(denom), _ptr(grad), red, _ptr(out),
                              _sptr(status), _stream()), "dce_backward")
    return out


def dce_reduce(loss, reduction="mean"):
    """sum / mean of the f32 losses through their exact (Kulisch) sum, independent of the
    rows' order: RN32(RN64(S)) / RN32(RN64(RN64(S) / N))."""
    _cuda(loss, "loss")
    if reduction not in ("sum", "mean"):
        raise DetAttnError("reduction must be 'sum' or 'mean'")
    loss = loss.to(torch.float32).contiguous()
    out = torch.empty((), dtype=torch.float32, device=loss.device)
    _check(lib().dce_reduce(_ptr(loss), loss.numel(), _REDUCTIONS[reduction], _ptr(out), _stream()), "dce_reduce")
    return out


def forward(logits, targets, splits=None, status=None):
    """Fused cross-entropy forward (det-cross-entropy "API": forward): (loss [N], rowmax [N],
    denom [N]), the state the backward reuses.  Vocab splits compose by max and digit add."""
    loss, denom, m, den = dce_forward(logits, targets, splits=splits, status=status)
    return loss, m, denom


class _CrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, targets, reduction, splits, status):
        loss, m, denom = forward(logits, targets, splits=splits, status=status)
        ctx.save_for_backward(logits, targets, m, denom)
        ctx.reduction, ctx.status = reduction, status
        return loss if reduction == "none" else dce_reduce(loss, reduction)

    @staticmethod
    def backward(ctx, grad_out):
        logits, targets, m, denom = ctx.saved_tensors
        g = dce_backward(logits, targets, m, denom, grad_out.detach(), ctx.reduction, status=ctx.status)
        return g, None, None, None, None


def cross_entropy(logits, targets, reduction="mean", splits=None, status=None):
    """Bitwise-deterministic cross-entropy with autograd (det-cross-entropy "API":
    cross_entropy(logits, targets, reduction)).  Loss and dLogits are the same bytes for any
    vocab split (splits: column counts summing to V) and any run.  logits: [N, V] f32 or bf16
    on the GPU; targets: [N] integer."""
    if reduction not in _REDUCTIONS:
        raise DetAttnError("reduction must be 'none', 'sum' or 'mean'")
    return _CrossEntropy.apply(logits, targets, reduction, splits, status)


def dce_forward_vp(logits, targets, v_base, v_total, group=None, status=None):
    """Vocabulary-parallel cross-entropy forward (det-cross-entropy, "Usage": the vocabulary
    sharded over ranks composes by max and digit add).  This rank holds logits [N, cols], the
    columns [v_base, v_base + cols) of a vocabulary of v_total; targets [N] are global column
    indices.  The group takes a max all-reduce of the rowmax and an int64 sum all-reduce of
    the denominator digits; each rank finalizes the rows whose target it holds (the others
    add +0) and a sum all-reduce of the f32 losses (one nonzero term per row) completes the
    loss.  Returns (loss [N], rowmax [N], denom [N]), equal bit for bit on every rank to the
    single-device forward over the whole vocabulary."""
    import torch.distributed as dist
    M, keep = _matrix(logits)
    targets = _vec(targets.to(torch.int64), torch.int64, M.rows, "targets")
    m = dce_rowmax(logits, status=status)
    _all_reduce(m, dist.ReduceOp.MAX, group)
    den = dce_denom_digits(logits, m, status=status)
    _all_reduce(den, dist.ReduceOp.SUM, group)
    normalize(den, status, ndig=DEN_NDIG)
    loss = torch.empty(M.rows, dtype=torch.float32, device=logits.device)
    denom = torch.empty(M.rows, dtype=torch.float64, device=logits.device)
    _check(lib().dce_finalize_shard(_ptr(den), C.byref(M), int(v_base), int(v_total), _ptr(targets), _ptr(m),
                                    _ptr(loss), _ptr(denom), _sptr(status), _stream()), "dce_finalize_shard")
    _all_reduce(loss, dist.ReduceOp.SUM, group)
    return loss, m, denom


def dce_backward_vp(logits, targets, v_base, m, denom, grad, reduction="none", status=None):
    """dLogits of this rank's vocabulary columns from the composed forward state (m, denom):
    the same bytes as the matching columns of dce_backward over the whole vocabulary."""
    M, keep = _matrix(logits)
    if reduction not in _REDUCTIONS:
        raise DetAttnError("reduction must be 'none', 'sum' or 'mean'")
    red = _REDUCTIONS[reduction]
    grad = grad.to(torch.float32).reshape(-1).contiguous()
    if grad.numel() != (M.rows if red == 0 else 1):
        raise DetAttnError("grad must have one entry per row for reduction='none', else one entry")
    targets = _vec(targets.to(torch.int64), torch.int64, M.rows, "targets")
    m = _vec(m, torch.float32, M.rows, "rowmax")
    denom = _vec(denom, torch.float64, M.rows, "denom")
    out = torch.empty((M.rows, M.cols), dtype=logits.dtype, device=logits.device)
    _check(lib().dce_backward_shard(C.byref(M), int(v_base), _ptr(targets), _ptr(m), _ptr(denom), _ptr(grad), red,
                                    _ptr(out), _sptr(status), _stream()), "dce_backward_shard")
    return out


class _CrossEntropyVP(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, targets, v_base, v_total, reduction, group, status):
        loss, m, denom = dce_forward_vp(logits, targets, v_base, v_total, group=group, status=status)
        ctx.save_for_backward(logits, targets, m, denom)
        ctx.v_base, ctx.reduction, ctx.status = v_base, reduction, status
        return loss if reduction == "none" else dce_reduce(loss, reduction)

    @staticmethod
    def backward(ctx, grad_out):
        logits, targets, m, denom = ctx.saved_tensors
        g = dce_backward_vp(logits, targets, ctx.v_base, m, denom, grad_out.detach(), ctx.reduction,
                            status=ctx.status)
        return g, None, None, None, None, None, None


def cross_entropy_vp(logits, targets, v_base, v_total, reduction="mean", group=None, status=None):
    """Vocabulary-parallel cross_entropy with autograd: the loss is the same bytes on every rank
    as cross_entropy over the whole vocabulary, and each rank's dLogits are the same bytes as
    that call's columns [v_base, v_base + cols)."""
    if reduction not in _REDUCTIONS:
        raise DetAttnError("reduction must be 'none', 'sum' or 'mean'")
    return _CrossEntropyVP.apply(logits, targets, v_base, v_total, reduction, group, status)


STATIC_MAX_ROWS = 65536


def dce_forward_static(logits, targets, status=None):
    """Cross-entropy forward through the static-scratch entry point, for callers that
    cannot allocate device memory for the intermediates (the rowmax and the denominator
    digits live in a fixed device array of STATIC_MAX_ROWS rows inside the library; only
    loss and denom are returned in new tensors here).  Equal bit for bit to dce_forward
    without splits.  Calls that overlap on the GPU race on the shared array."""
    M, keep = _matrix(logits)
    targets = _vec(targets.to(torch.int64), torch.int64, M.rows, "targets")
    loss = torch.empty(M.rows, dtype=torch.float32, device=logits.device)
    denom = torch.empty(M.rows, dtype=torch.float64, device=logits.device)
    _check(lib().dce_forward_static(C.byref(M), _ptr(targets), _ptr(loss), _ptr(denom), _sptr(status), _stream()),
           "dce_forward_static")
    return loss, denom


def probe_bounded_wait(status=None):
    """Run the bounded-wait probe (a wait nothing ends; it gives up after about 2 s and
    reports STATUS_TIMEOUT); returns the status word after synchronizing."""
    st = new_status() if status is None else status
    _check(lib().da_probe_bounded_wait(_sptr(st), _stream()), "probe_bounded_wait")
    torch.cuda.current_stream().synchronize()
    return read_status(st)


def probe_packed(which, lo_bits, count):
    """Number of binary32 bit patterns in [lo_bits, lo_bits + count) whose packed two-lane
    result differs from the scalar one in any bit (0 expected): which 0 the exponential, 1 the
    backward's quotient."""
    out = torch.zeros(1, dtype=torch.int64, device="cuda")
    _check(lib().da_probe_packed(which, lo_bits & 0xFFFFFFFF, count, _ptr(out), _stream()), "probe_packed")
    return int(out.item())


def probe_int_mac_rate(iters=4096, nblocks=None):
    """Exact 32 x 32 -> 64-bit multiply-adds per second over the whole GPU (the integer
    pipe's rate for exact products), timed with CUDA events on the current stream."""
    dev = torch.cuda.current_device()
    if nblocks is None:
        nblocks = 4 * torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(1, dtype=torch.int64, device="cuda")
    L = lib()
    _check(L.da_probe_int_mac(16, nblocks, _ptr(sink), _stream()), "probe_int_mac")   # warm-up
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s = torch.cuda.current_stream()
    a.record(s)
    _check(L.da_probe_int_mac(iters, nblocks, _ptr(sink), _stream()), "probe_int_mac")
    b.record(s)
    b.synchronize()
    macs = iters * nblocks * 512 * int(L.da_probe_int_mac_per_thread_iter())
    return macs / (a.elapsed_time(b) * 1e-3)
