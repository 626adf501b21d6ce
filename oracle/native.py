"""ctypes front of the C oracle (detattn_oracle.c).  TEST INFRASTRUCTURE ONLY.

The C oracle computes the same definition as oracle/exact.py, independently written, fast
enough for whole rows of the full-size workloads.  build() compiles it with the host C
compiler; -ffp-contract=off keeps every binary32/binary64 operation a single IEEE
operation (no fused multiply-add unless the source writes fmaf).  dce_backward_many is the
cross-entropy gradient of oracle/exact.py vectorized with numpy on top of the C exp32_det
(pinned equal to the exact rational version in tests/test_dce_backward_oracle.py).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "detattn_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libdetattn_oracle.so")
_lib = None

NUM_NDIG, DEN_NDIG = 15, 6
P = C.c_void_p
I64 = C.c_int64


def build(force: bool = False) -> str:
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                               "-pthread", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        L = _lib
        L.or_exp32_det.argtypes = [C.c_float]
        L.or_exp32_det.restype = C.c_float
        L.or_log64_det.argtypes = [C.c_double]
        L.or_log64_det.restype = C.c_double
        L.or_attn_rowmax.argtypes = [P, P, C.c_int] + [I64] * 6 + [P, P, C.c_int, C.c_float, I64, I64, P, I64, P,
                                                                  C.c_int]
        L.or_attn_accumulate.argtypes = [P, P, P, C.c_int] + [I64] * 6 + [P, P, P, C.c_int, C.c_float, P, I64, I64,
                                                                         P, I64, P, P, C.c_int]
        L.or_finalize.argtypes = [P, P, I64, I64, P]
        L.or_normalize.argtypes = [P, I64, C.c_int, I64, C.c_int]
        L.or_dce_rowmax.argtypes = [P, C.c_int, I64, I64, I64, I64, I64, P, I64, P, C.c_int]
        L.or_dce_denom.argtypes = [P, C.c_int, I64, I64, I64, P, I64, I64, P, I64, P, C.c_int]
        L.or_dce_finalize.argtypes = [P, P, C.c_int, I64, I64, P, P, P, I64, P, P]
        L.or_exp32_det_many.argtypes = [P, P, I64]
        L.or_log64_det_many.argtypes = [P, P, I64]
        for f in ("or_attn_rowmax", "or_attn_accumulate", "or_finalize", "or_normalize", "or_dce_rowmax",
                  "or_dce_denom", "or_dce_finalize"):
            getattr(L, f).restype = C.c_int
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _host(t):
    """torch tensor / numpy array -> (contiguous numpy buffer, dtype code, element strides).
    bf16 is carried as its uint16 bit pattern (dtype code 1), f32 as float32 (code 0)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                a = t.view(torch.int16).numpy().view(np.uint16)
                code = 1
            else:
                a = t.float().numpy()
                code = 0
            return np.ascontiguousarray(a), code
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(t, dtype=np.float32))
    return a, 0


def _strides(a: np.ndarray):
    return np.array([s // a.itemsize for s in a.strides], dtype=np.int64)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def exp32_det(x: float) -> float:
    return float(lib().or_exp32_det(float(x)))


def log64_det(d: float) -> float:
    return float(lib().or_log64_det(float(d)))


def exp32_det_many(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().or_exp32_det_many(_ptr(x), _ptr(y), x.size)
    return y


def log64_det_many(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib().or_log64_det_many(_ptr(x), _ptr(y), x.size)
    return y


def all_rows(B, H, S) -> np.ndarray:
    return np.arange(B * H * S, dtype=np.int64)


class Attn:
    """Exact det-attn over host copies of Q, K, V ([B,H,S,D], f32 or bf16)."""

    def __init__(self, Q, K, V, causal=False, scale=None):
        self.q, self.dtype = _host(Q)
        self.k, dk = _host(K)
        self.v, dv = _host(V)
        assert self.dtype == dk == dv, "Q, K, V must share one dtype"
        self.B, self.Hq, self.Sq, self.D = self.q.shape
        _, self.Hkv, self.Skv, _ = self.k.shape
        self.causal = int(bool(causal))
        import math
        self.scale32 = float(np.float32(1.0 / math.sqrt(self.D) if scale is None else scale))

    def _shape(self):
        return (self.B, self.Hq, self.Hkv, self.Sq, self.Skv, self.D)

    def rowmax(self, kv_lo=0, kv_hi=None, rows=None, nthreads=None):
        kv_hi = self.Skv if kv_hi is None else kv_hi
        rows = all_rows(self.B, self.Hq, self.Sq) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        m = np.empty(len(rows), dtype=np.float32)
        st = lib().or_attn_rowmax(_ptr(self.q), _ptr(self.k), self.dtype, *self._shape(), _ptr(_strides(self.q)),
                                  _ptr(_strides(self.k)), self.causal, self.scale32, kv_lo, kv_hi, _ptr(rows),
                                  len(rows), _ptr(m), nthreads or default_threads())
        return m, st

    def accumulate(self, m_rows, kv_lo=0, kv_hi=None, rows=None, nthreads=None):
        kv_hi = self.Skv if kv_hi is None else kv_hi
        rows = all_rows(self.B, self.Hq, self.Sq) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        m_rows = np.ascontiguousarray(m_rows, dtype=np.float32).reshape(-1)
        assert len(m_rows) == len(rows)
        num = np.empty((len(rows), NUM_NDIG, self.D), dtype=np.int64)
        den = np.empty((len(rows), DEN_NDIG), dtype=np.int64)
        st = lib().or_attn_accumulate(_ptr(self.q), _ptr(self.k), _ptr(self.v), self.dtype, *self._shape(),
                                      _ptr(_strides(self.q)), _ptr(_strides(self.k)), _ptr(_strides(self.v)),
                                      self.causal, self.scale32, _ptr(m_rows), kv_lo, kv_hi, _ptr(rows), len(rows),
                                      _ptr(num), _ptr(den), nthreads or default_threads())
        return num, den, st

    def forward_rows(self, rows=None, nthreads=None):
        """Fused two-pass result for the listed rows: (m, num, den, out)."""
        m, _ = self.rowmax(rows=rows, nthreads=nthreads)
        num, den, _ = self.accumulate(m, rows=rows, nthreads=nthreads)
        return m, num, den, finalize(num, den)


def finalize(num: np.ndarray, den: np.ndarray) -> np.ndarray:
    num = np.ascontiguousarray(num, dtype=np.int64)
    den = np.ascontiguousarray(den, dtype=np.int64)
    n, nd, D = num.shape
    out = np.empty((n, D), dtype=np.float32)
    lib().or_finalize(_ptr(num), _ptr(den), n, D, _ptr(out))
    return out


def normalize(dg: np.ndarray, e0: int) -> tuple[np.ndarray, int]:
    """Canonical form of digit arrays laid out [n, ndig, inner] (inner = D for NUM, 1 for
    DEN).  The input may be the plain int64 sum of canonical arrays."""
    a = np.ascontiguousarray(dg, dtype=np.int64).copy()
    if a.ndim == 2:
        n, nd, inner = a.shape[0], a.shape[1], 1
    else:
        n, nd, inner = a.shape[0], a.shape[1], int(np.prod(a.shape[2:]))
    bad = lib().or_normalize(_ptr(a), n, nd, inner, e0)
    return a, bad


class DCE:
    """Exact det-cross-entropy over a host copy of logits [N, V] (f32 or bf16)."""

    def __init__(self, logits):
        self.x, self.dtype = _host(logits)
        self.N, self.V = self.x.shape

    def rows(self, rows=None):
        return np.arange(self.N, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)

    def rowmax(self, v_lo=0, v_hi=None, rows=None, nthreads=None):
        v_hi = self.V if v_hi is None else v_hi
        rows = self.rows(rows)
        m = np.empty(len(rows), dtype=np.float32)
        st = lib().or_dce_rowmax(_ptr(self.x), self.dtype, self.N, self.V, self.V, v_lo, v_hi, _ptr(rows), len(rows),
                                 _ptr(m), nthreads or default_threads())
        return m, st

    def denom_digits(self, m_rows, v_lo=0, v_hi=None, rows=None, nthreads=None):
        v_hi = self.V if v_hi is None else v_hi
        rows = self.rows(rows)
        m_rows = np.ascontiguousarray(m_rows, dtype=np.float32)
        den = np.empty((len(rows), DEN_NDIG), dtype=np.int64)
        st = lib().or_dce_denom(_ptr(self.x), self.dtype, self.N, self.V, self.V, _ptr(m_rows), v_lo, v_hi, _ptr(rows),
                                len(rows), _ptr(den), nthreads or default_threads())
        return den, st

    def finalize(self, den, targets, m_rows, rows=None):
        rows = self.rows(rows)
        den = np.ascontiguousarray(den, dtype=np.int64)
        tg = np.ascontiguousarray(targets, dtype=np.int64)
        m_rows = np.ascontiguousarray(m_rows, dtype=np.float32)
        loss = np.empty(len(rows), dtype=np.float32)
        denom = np.empty(len(rows), dtype=np.float64)
        st = lib().or_dce_finalize(_ptr(den), _ptr(self.x), self.dtype, self.V, self.V, _ptr(tg), _ptr(m_rows),
                                   _ptr(rows), len(rows), _ptr(loss), _ptr(denom))
        return loss, denom, st

    def forward(self, targets, splits=None, rows=None, nthreads=None):
        """Vocab-sharded composition: rowmax by max, digits by add, finalize."""
        rows = self.rows(rows)
        splits = [self.V] if splits is None else list(splits)
        bounds, lo = [], 0
        for n in splits:
            bounds.append((lo, lo + n))
            lo += n
        m = None
        for a, b in bounds:
            mm, _ = self.rowmax(a, b, rows, nthreads)
            m = mm if m is None else np.maximum(m, mm)
        den = None
        for a, b in bounds:
            dd, _ = self.denom_digits(m, a, b, rows, nthreads)
            den = dd if den is None else den + dd
        den, _ = normalize(den, -160)
        tg = np.asarray(targets, dtype=np.int64)[rows]
        loss, denom, st = self.finalize(den, tg, m, rows)
        return loss, denom, m, den, st


def dce_backward_many(logits, targets, m, denom, go) -> np.ndarray:
    """The cross-entropy dLogits of oracle.exact.dce_backward, vectorized over whole rows:
    numpy float32 subtraction and multiplication round once each, float64 division once,
    and the weights come from this module's C exp32_det (equal to the exact one)."""
    from .exact import decode
    X = decode(logits).astype(np.float32)
    N, V = X.shape
    xr = X - np.asarray(m, dtype=np.float32)[:, None]
    xr = np.where(xr > 0, np.float32(0), xr).astype(np.float32)
    w = exp32_det_many(xr.reshape(-1)).reshape(N, V).astype(np.float32)
    p = (w.astype(np.float64) / np.asarray(denom, dtype=np.float64)[:, None]).astype(np.float32)
    t = np.asarray(targets, dtype=np.int64)
    hit = (np.arange(V)[None, :] == t[:, None])
    g = np.where(hit, p - np.float32(1), p).astype(np.float32)
    return (np.asarray(go, dtype=np.float32)[:, None] * g).astype(np.float32)
