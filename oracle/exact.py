"""Exact reference for the order-invariant softmax reduction (TEST INFRASTRUCTURE ONLY).

This module is the oracle: a plain, slow, obviously exact CPU restatement of what
det-attn and det-cross-entropy compute.  Only the test-suite, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does.

Every real number here is held exactly: an f32 / bf16 input x is the integer
x * 2**149 (every finite f32 is a multiple of 2**-149), a product of two of them is an
integer over 2**298, and every rounding is written out from the IEEE 754 definition
(round to nearest, ties to even, gradual underflow) on Python Fractions.

Sources (page title, section):
  * "det-attn" model card, section "Method": rowmax_i = max_j(scale*Q_i.K_j);
    num_id = sum_j exp(s_ij - rowmax_i) V_jd; den_i = sum_j exp(s_ij - rowmax_i),
    accumulated exactly in a Kulisch long accumulator of signed int64 digits; KV shards
    compose by max and by digit add.
  * "det-attn", section "API": rowmax / accumulate / finalize / det_attn_sharded.
  * "det-attn", section "Correctness" and "Requirements and limits": causal and
    non-causal, MHA and GQA, f32 and bf16 inputs, D <= 256, f32 output.
  * "det-cross-entropy" model card, sections "Usage", "API", "Method": per-token
    rowmax over a vocab range, exact denominator digits, finalize to (loss, denom); the
    gradient softmax(x_i) - onehot(t_i) from the forward's state and the loss reductions
    "none" / "sum" / "mean" of cross_entropy.

The pages leave the roundings open.  The readings taken here (score = correctly rounded
f32 of the exact dot, then one f32 multiply by the scale; a fixed f32 exp routine; digits
in radix 2**32; finalize rounds NUM and DEN to f64, divides, rounds to f32) are the
numerical contract the CUDA path must meet bit for bit.  Parity status: pinned (see
tests/test_oracle_pins.py, tests/test_dce_backward_oracle.py and tests/test_golden.py;
tests/test_oracle_mutations.py shows the pins reject planted slips); nothing in this
module is "parity unpinned".
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

# ----------------------------------------------------------------------------------------
# IEEE 754 binary rounding, written from the definition.
# ----------------------------------------------------------------------------------------

def _floor_log2(a: Fraction) -> int:
    """Largest e with 2**e <= a, for a > 0 (exact)."""
    n, d = a.numerator, a.denominator
    e = n.bit_length() - d.bit_length()
    # now 2**(e-1) < a < 2**(e+1); fix up exactly
    if e >= 0:
        if n < (d << e):
            e -= 1
    else:
        if (n << -e) < d:
            e -= 1
    return e


def round_binary(q: Fraction, prec: int, emin: int, emax: int) -> float:
    """Round exact rational q to the binary format (prec significand bits, exponent range
    [emin, emax], gradual underflow) with round-to-nearest-ties-to-even.  Returns the
    result as a Python float (exact: both f32 and f64 values are doubles); overflow gives
    +-inf.  An exact zero gives +0.0 (callers that need a signed zero handle it)."""
    if q == 0:
        return 0.0
    neg = q < 0
    a = -q if neg else q
    e = _floor_log2(a)
    qe = max(e, emin) - (prec - 1)           # exponent of the unit in the last place
    scaled = a / Fraction(2) ** qe if qe >= 0 else a * (1 << -qe)
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and (n & 1)):
        n += 1
    # n may have reached 2**prec (carry into the next binade): still exact below.
    if n.bit_length() + qe > emax + 1:
        r = math.inf
    else:
        r = math.ldexp(float(n), qe)   # n <= 2**prec <= 2**53: exact
    return -r if neg else r


def rn32(q) -> float:
    """RN32: nearest binary32, ties to even, subnormals down to 2**-149."""
    return round_binary(Fraction(q), 24, -126, 127)


def rn64(q) -> float:
    """RN64: nearest binary64, ties to even, subnormals down to 2**-1074."""
    return round_binary(Fraction(q), 53, -1022, 1023)


# ----------------------------------------------------------------------------------------
# Input decoding (det-attn, "Correctness": f32 and bf16 inputs).
# ----------------------------------------------------------------------------------------

SCALE_POW = 149  # every finite binary32 is an integer multiple of 2**-149


def decode(t) -> np.ndarray:
    """Tensor (torch f32/bf16 or numpy f32) -> numpy float64 array of the exact values.
    bf16 is the upper half of a binary32, so widening is exact; f32 -> f64 is exact."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu").float().numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float32).astype(np.float64)


def to_int149(x: float) -> int:
    """Exact integer x * 2**149 for a finite binary32 value x."""
    f = Fraction(x) * (1 << SCALE_POW)
    assert f.denominator == 1, "value is not a binary32"
    return f.numerator


# ----------------------------------------------------------------------------------------
# Fixed constants of the contract, each computed here from its mathematical definition.
# ----------------------------------------------------------------------------------------

def _ln2_fraction(bits: int = 320) -> Fraction:
    """ln 2 = sum_{k>=1} 1 / (k 2**k); the tail after n terms is below 2**-n."""
    s = Fraction(0)
    for k in range(1, bits + 1):
        s += Fraction(1, k << k)
    return s


LN2 = _ln2_fraction()
# exp routine (Cody-Waite reduction, "Software Manual for the Elementary Functions",
# Cody & Waite 1980, plus a degree-7 Taylor polynomial), every step rounded to binary32.
EXP_X_MIN = -104.0                       # below: e^x < 2**-150, returns +0
EXP_L2E = rn32(1 / LN2)                  # RN32(log2 e)
EXP_C1 = float(Fraction(math.floor(LN2 * (1 << 16) + Fraction(1, 2)), 1 << 16))  # ln2 to 16 bits
EXP_C2 = rn32(LN2 - Fraction(EXP_C1))    # RN32(ln2 - C1)
EXP_TAYLOR = [rn32(Fraction(1, math.factorial(n))) for n in range(8)]  # RN32(1/n!), n = 0..7

# log routine for the cross-entropy finalize (binary64, no fused multiply-add): argument
# reduction to [sqrt(1/2), sqrt(2)], the atanh series log f = 2 sum u^(2n+1)/(2n+1) with
# u = (f-1)/(f+1), ten terms after the first, then + e*ln2 in a two-part constant.
LOG_SQRT2 = rn64(Fraction(math.isqrt(2 << 200), 1 << 100))  # RN64(sqrt 2); sqrt to 100 bits
LOG_LN2_HI = float(Fraction(math.floor(LN2 * (1 << 42)), 1 << 42))  # ln2 truncated to 42 bits
LOG_LN2_LO = rn64(LN2 - Fraction(LOG_LN2_HI))
LOG_COEF = [1.0 / (2 * n + 1) for n in range(1, 11)]  # RN64(1/(2n+1)), n = 1..10

# Kulisch digit layout (det-attn "Method": signed int64 digits over the full exponent
# range).  value = sum_k digit_k * 2**(E0 + 32 k); digits 0..n-2 in [0, 2**32), the top
# digit signed (the canonical form, unique for every value).
NUM_E0, NUM_NDIG = -320, 15
DEN_E0, DEN_NDIG = -160, 6


def default_scale(D: int) -> float:
    """Default softmax scale, RN32(1/sqrt(D)) with 1/sqrt(D) taken in binary64."""
    return float(np.float32(1.0 / math.sqrt(D)))


# ----------------------------------------------------------------------------------------
# The routines of the contract.
# ----------------------------------------------------------------------------------------

def exp32_det(x: float) -> float:
    """Fixed binary32 exp for x <= 0 (det-attn "Method": the weight exp(s_ij - rowmax_i)).
    Every operation is one RN32 rounding of its exact result; fma rounds once."""
    if x != x:
        return x
    if x < EXP_X_MIN:
        return 0.0
    fx = Fraction(x)
    t = rn32(fx * Fraction(EXP_L2E))
    k = round(t)                                   # ties to even
    r1 = rn32(fx - k * Fraction(EXP_C1))          # fma(-k, C1, x)
    r = rn32(Fraction(r1) - k * Fraction(EXP_C2))  # fma(-k, C2, r1)
    p = Fraction(EXP_TAYLOR[7])
    for n in range(6, -1, -1):
        p = Fraction(rn32(p * Fraction(r) + Fraction(EXP_TAYLOR[n])))  # fma(p, r, c_n)
    return rn32(p * Fraction(2) ** k)


def log64_det(d: float) -> float:
    """Fixed binary64 natural log of a positive finite normal d (det-cross-entropy "Method":
    loss = logsumexp - x_target).  Python float operations are IEEE binary64 RN, so each
    line below is one rounding; nothing is fused."""
    f, e = math.frexp(d)       # d = f * 2**e, f in [0.5, 1)
    f, e = f * 2.0, e - 1      # f in [1, 2)
    if f > LOG_SQRT2:
        f, e = f * 0.5, e + 1  # f in (sqrt(1/2), sqrt(2)]
    a = f - 1.0                # exact (Sterbenz)
    b = f + 1.0
    u = a / b
    u2 = u * u
    p = LOG_COEF[9]
    for n in range(8, -1, -1):
        p = p * u2 + LOG_COEF[n]
    t1 = u2 * p
    t2 = u * t1
    lf = (u + t2) * 2.0
    fe = float(e)
    return fe * LOG_LN2_HI + (fe * LOG_LN2_LO + lf)


def canon_digits(value: Fraction, e0: int, ndig: int) -> list[int]:
    """Canonical radix-2**32 digits of an exact value that is a multiple of 2**e0."""
    n = value * Fraction(2) ** (-e0)
    assert n.denominator == 1, "value below the digit range"
    n = n.numerator
    out = []
    for _ in range(ndig - 1):
        out.append(n & 0xFFFFFFFF)
        n >>= 32                 # floor division: arithmetic shift
    assert -(1 << 63) <= n < (1 << 63), "top digit out of int64 range"
    out.append(n)
    return out


def digits_value(digits, e0: int) -> Fraction:
    """Exact value of a (not necessarily canonical) digit list."""
    return sum(Fraction(int(dg)) * Fraction(2) ** (e0 + 32 * k) for k, dg in enumerate(digits))


def normalize_digits(digits, e0: int) -> list[int]:
    return canon_digits(digits_value(digits, e0), e0, len(digits))


# ----------------------------------------------------------------------------------------
# det-attn: rowmax, accumulate, finalize, and their compositions.
# ----------------------------------------------------------------------------------------

def _rowdata(X: np.ndarray) -> list[list[int]]:
    return [[to_int149(float(v)) for v in row] for row in X]


def score(qrow_int, krow_int, scale32: float) -> float:
    """s_ij = RN32(scale32 * RN32(sum_d q_id k_jd)): the exact dot rounded once, then one
    binary32 multiply by the scale (det-attn "Method": "Scores are per-(i, j)")."""
    dot = sum(a * b for a, b in zip(qrow_int, krow_int))
    d = rn32(Fraction(dot, 1 << (2 * SCALE_POW)))   # exact zero -> +0, tiny negative -> -0
    if not math.isfinite(d):
        return d * scale32
    prod = Fraction(scale32) * Fraction(d)
    if prod == 0:   # IEEE: an exact zero product carries the XOR of the operand signs
        return -0.0 if (math.copysign(1.0, scale32) * math.copysign(1.0, d)) < 0 else 0.0
    return rn32(prod)


class AttnProblem:
    """Q [B,Hq,Sq,D], K/V [B,Hkv,Skv,D] as exact values, with GQA head grouping
    hk = h // (Hq // Hkv) (contiguous groups) and the causal mask j <= i."""

    def __init__(self, Q, K, V, causal: bool = False, scale: float | None = None):
        self.Q, self.K, self.V = decode(Q), decode(K), decode(V)
        B, Hq, Sq, D = self.Q.shape
        Bk, Hkv, Skv, Dk = self.K.shape
        assert Bk == B and Dk == D and self.V.shape == self.K.shape
        assert Hq % Hkv == 0
        if causal:
            assert Sq == Skv
        self.B, self.Hq, self.Hkv, self.Sq, self.Skv, self.D = B, Hq, Hkv, Sq, Skv, D
        self.causal = causal
        self.scale32 = default_scale(D) if scale is None else float(np.float32(scale))
        self._qi, self._ki, self._vi = {}, {}, {}

    def _q(self, b, h):
        if (b, h) not in self._qi:
            self._qi[(b, h)] = _rowdata(self.Q[b, h])
        return self._qi[(b, h)]

    def _k(self, b, hk):
        if (b, hk) not in self._ki:
            self._ki[(b, hk)] = _rowdata(self.K[b, hk])
        return self._ki[(b, hk)]

    def _v(self, b, hk):
        if (b, hk) not in self._vi:
            self._vi[(b, hk)] = _rowdata(self.V[b, hk])
        return self._vi[(b, hk)]

    def kv_head(self, h: int) -> int:
        return h // (self.Hq // self.Hkv)

    def valid(self, i: int, j: int) -> bool:
        return (not self.causal) or j <= i

    def scores_row(self, b, h, i, kv_lo, kv_hi):
        qr = self._q(b, h)[i]
        kk = self._k(b, self.kv_head(h))
        return {j: score(qr, kk[j], self.scale32) for j in range(kv_lo, kv_hi) if self.valid(i, j)}

    # det-attn API "rowmax(Q, K, ..., kv_lo, kv_hi)": per-query max over a key range.
    def rowmax(self, kv_lo=0, kv_hi=None) -> np.ndarray:
        kv_hi = self.Skv if kv_hi is None else kv_hi
        m = np.full((self.B, self.Hq, self.Sq), -np.inf, dtype=np.float32)
        for b in range(self.B):
            for h in range(self.Hq):
                for i in range(self.Sq):
                    s = self.scores_row(b, h, i, kv_lo, kv_hi)
                    if s:
                        mx = max(s.values())
                        m[b, h, i] = 0.0 if mx == 0 else mx   # -0 -> +0
        return m

    # det-attn API "accumulate(Q, K, V, rowmax, ...)": exact NUM/DEN digits of a shard.
    def accumulate(self, m, kv_lo=0, kv_hi=None):
        kv_hi = self.Skv if kv_hi is None else kv_hi
        num = np.zeros((self.B, self.Hq, self.Sq, NUM_NDIG, self.D), dtype=np.int64)
        den = np.zeros((self.B, self.Hq, self.Sq, DEN_NDIG), dtype=np.int64)
        violation = False
        for b in range(self.B):
            for h in range(self.Hq):
                vv = self._v(b, self.kv_head(h))
                for i in range(self.Sq):
                    mi = float(m[b, h, i])
                    s = self.scores_row(b, h, i, kv_lo, kv_hi)
                    acc = [0] * self.D
                    dsum = 0
                    for j, sij in s.items():
                        if math.isfinite(mi) and math.isfinite(sij):
                            x = rn32(Fraction(sij) - Fraction(mi))
                        else:
                            x = sij - mi   # non-finite: outside the contract, flagged
                        if x > 0:
                            violation = True
                            x = 0.0
                        w = exp32_det(x)
                        wi = to_int149(w)
                        dsum += wi
                        row = vv[j]
                        for d in range(self.D):
                            acc[d] += wi * row[d]
                    for d in range(self.D):
                        num[b, h, i, :, d] = canon_digits(Fraction(acc[d], 1 << (2 * SCALE_POW)), NUM_E0, NUM_NDIG)
                    den[b, h, i, :] = canon_digits(Fraction(dsum, 1 << SCALE_POW), DEN_E0, DEN_NDIG)
        return num, den, violation


def finalize_value(num_digits, den_digits) -> float:
    """o = RN32(RN64(RN64(NUM) / RN64(DEN))) (det-attn API "finalize": compose digits to
    the f32 output)."""
    n64 = rn64(digits_value(num_digits, NUM_E0))
    d64 = rn64(digits_value(den_digits, DEN_E0))
    if d64 == 0.0:
        return math.nan if n64 == 0.0 else math.copysign(math.inf, n64)
    q = rn64(Fraction(n64) / Fraction(d64))
    o = rn32(q)
    if o == 0.0 and q < 0:
        o = -0.0
    return o


def finalize(num: np.ndarray, den: np.ndarray) -> np.ndarray:
    B, H, S, _, D = num.shape
    out = np.zeros((B, H, S, D), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                for d in range(D):
                    out[b, h, i, d] = finalize_value(num[b, h, i, :, d], den[b, h, i, :])
    return out


def compose_max(parts):
    out = parts[0].copy()
    for p in parts[1:]:
        out = np.maximum(out, p)
    return out


def compose_add(parts):
    """Elementwise digit add, then canonical form (det-attn "Method": an int64 add of
    digit arrays)."""
    tot = [np.asarray(p, dtype=object) for p in parts]
    s = tot[0]
    for p in tot[1:]:
        s = s + p
    return s


def normalize_num(num_obj) -> np.ndarray:
    a = np.asarray(num_obj, dtype=object)
    B, H, S, ND, D = a.shape
    out = np.zeros(a.shape, dtype=np.int64)
    for b in range(B):
        for h in range(H):
            for i in range(S):
                for d in range(D):
                    out[b, h, i, :, d] = normalize_digits(list(a[b, h, i, :, d]), NUM_E0)
    return out


def normalize_den(den_obj) -> np.ndarray:
    a = np.asarray(den_obj, dtype=object)
    out = np.zeros(a.shape, dtype=np.int64)
    for idx in np.ndindex(*a.shape[:-1]):
        out[idx] = normalize_digits(list(a[idx]), DEN_E0)
    return out


def det_attn(Q, K, V, causal=False, scale=None):
    """Fused two-pass reduction over the whole key range (det-attn API "det_attn")."""
    P = AttnProblem(Q, K, V, causal, scale)
    m = P.rowmax()
    num, den, _ = P.accumulate(m)
    return finalize(num, den)


def det_attn_sharded(Q, K, V, kv_splits, causal=False, scale=None, order=None):
    """KV-shard composition (det-attn API "det_attn_sharded"): rowmax of every shard
    composed by max, then digits of every shard (with the global rowmax) composed by add,
    then finalize.  `order` permutes the shard visiting order."""
    P = AttnProblem(Q, K, V, causal, scale)
    bounds, lo = [], 0
    for n in kv_splits:
        bounds.append((lo, lo + n))
        lo += n
    assert lo == P.Skv
    order = list(range(len(bounds))) if order is None else list(order)
    m = compose_max([P.rowmax(*bounds[k]) for k in order])
    parts = [P.accumulate(m, *bounds[k]) for k in order]
    num = normalize_num(compose_add([p[0] for p in parts]))
    den = normalize_den(compose_add([p[1] for p in parts]))
    return finalize(num, den)


# ----------------------------------------------------------------------------------------
# det-cross-entropy: rowmax, denominator digits, finalize.
# ----------------------------------------------------------------------------------------

def dce_rowmax(logits, v_lo, v_hi) -> np.ndarray:
    """m_i = max_{v in [v_lo, v_hi)} x_iv (det-cross-entropy API "rowmax"); -0 -> +0,
    empty range -> -inf."""
    X = decode(logits)
    N = X.shape[0]
    m = np.full(N, -np.inf, dtype=np.float32)
    if v_hi > v_lo:
        mx = X[:, v_lo:v_hi].max(axis=1)
        m = np.where(mx == 0, 0.0, mx).astype(np.float32)
    return m


def dce_denom_digits(logits, m, v_lo, v_hi) -> tuple[np.ndarray, bool]:
    """Exact digits of den_i = sum_v exp32_det(RN32(x_iv - m_i)) over [v_lo, v_hi)
    (det-cross-entropy API "denom_digits")."""
    X = decode(logits)
    N = X.shape[0]
    out = np.zeros((N, DEN_NDIG), dtype=np.int64)
    violation = False
    for i in range(N):
        mi = float(m[i])
        tot = 0
        for v in range(v_lo, v_hi):
            x = rn32(Fraction(float(X[i, v])) - Fraction(mi))
            if x > 0:
                violation = True
                x = 0.0
            tot += to_int149(exp32_det(x))
        out[i] = canon_digits(Fraction(tot, 1 << SCALE_POW), DEN_E0, DEN_NDIG)
    return out, violation


def dce_finalize(den, logits, targets, m):
    """(loss, denom): denom_i = RN64(den_i); loss_i = RN32(RN64(log64_det(denom_i) +
    RN64(m_i - x_{i,t_i}))) (det-cross-entropy API "finalize").  A target outside [0, V)
    gives NaN and the bad-target flag."""
    X = decode(logits)
    N, Vn = X.shape
    loss = np.zeros(N, dtype=np.float32)
    denom = np.zeros(N, dtype=np.float64)
    bad = False
    for i in range(N):
        d64 = rn64(digits_value(den[i], DEN_E0))
        denom[i] = d64
        t = int(targets[i])
        if t < 0 or t >= Vn:
            bad = True
            loss[i] = np.nan
            continue
        diff = rn64(Fraction(float(m[i])) - Fraction(float(X[i, t])))
        loss[i] = rn32(Fraction(log64_det(d64) + diff)) if d64 > 0 else np.float32(np.inf)
    return loss, denom, bad


def dce_forward(logits, targets, splits=None):
    """Vocab-sharded composition (det-cross-entropy "Usage"): rowmax by max, digits by
    add, finalize."""
    X = decode(logits)
    Vn = X.shape[1]
    if splits is None:
        splits = [Vn]
    bounds, lo = [], 0
    for n in splits:
        bounds.append((lo, lo + n))
        lo += n
    m = compose_max([dce_rowmax(X, a, b) for a, b in bounds])
    den = normalize_den(compose_add([dce_denom_digits(X, m, a, b)[0] for a, b in bounds]))
    loss, denom, _ = dce_finalize(den, X, targets, m)
    return loss, denom, m, den


# ----------------------------------------------------------------------------------------
# det-cross-entropy: backward and reductions ("API": cross_entropy(logits, targets,
# reduction) with a deterministic dLogits; "Method": the gradient softmax(x_i) -
# onehot(t_i)).  The pages fix the gradient's value and that it reuses forward's
# (loss, rowmax, denom); they do not print its rounding sequence.  Reading: each step is
# one IEEE rounding of its exact result, in this order:
#   w_iv = exp32_det(RN32(x_iv - m_i))                  (the forward's weights)
#   p_iv = RN32(RN64(w_iv / denom_i))                   (denom_i = RN64(den_i), f64)
#   g_iv = RN32(p_iv - [v == t_i])
#   dLogits_iv = RN32(go_i * g_iv)
# with go_i the upstream gradient of loss_i: grad[i] ("none"), grad ("sum"),
# RN32(RN64(grad / N)) ("mean").  A target outside [0, V) subtracts nothing.
# Reductions: "sum" = RN32(RN64(S)), "mean" = RN32(RN64(RN64(S) / N)), S the exact sum of
# the f32 losses (a NaN loss makes the result NaN).
# ----------------------------------------------------------------------------------------

def dce_go(grad, N: int, reduction: str) -> np.ndarray:
    """Per-row upstream gradient go_i of the loss for the given reduction."""
    g = np.asarray(grad, dtype=np.float32).reshape(-1)
    if reduction == "none":
        return g.astype(np.float32)
    if reduction == "sum":
        return np.full(N, g[0], dtype=np.float32)
    if reduction == "mean":
        return np.full(N, np.float32(float(g[0]) / N), dtype=np.float32)
    raise ValueError(reduction)


def dce_backward(logits, targets, m, denom, go) -> np.ndarray:
    """dLogits (float32 [N, V]) of the cross-entropy loss, in the reading above."""
    X = decode(logits)
    N, Vn = X.shape
    out = np.zeros((N, Vn), dtype=np.float32)
    one = np.float32(1.0)
    for i in range(N):
        mi = float(m[i])
        d64 = float(denom[i])
        t = int(targets[i])
        gi = np.float32(go[i])
        for v in range(Vn):
            x = float(X[i, v])
            if np.isfinite(x) and np.isfinite(mi):
                xr = rn32(Fraction(x) - Fraction(mi))
            else:
                xr = float(np.float32(x) - np.float32(mi))   # IEEE inf / NaN arithmetic
            if xr > 0:
                xr = 0.0                                      # above the rowmax: clamped as in forward
            w = exp32_det(xr)
            p = np.float32(w / d64)             # Python float division is RN64; np.float32 is RN32
            g = p - one if v == t else p        # float32 arithmetic: one RN32
            out[i, v] = gi * g
    return out


def dce_reduce(loss, reduction: str) -> np.float32:
    """sum / mean of the f32 losses through their exact sum."""
    L = np.asarray(loss, dtype=np.float32).reshape(-1)
    if np.isnan(L).any():
        return np.float32(np.nan)
    if np.isinf(L).any():
        return np.float32(np.sum(L.astype(np.float64)))   # +inf, or NaN for +inf and -inf
    S = sum((Fraction(float(x)) for x in L), Fraction(0))
    s64 = rn64(S)
    if reduction == "sum":
        return np.float32(s64)
    if reduction == "mean":
        if len(L) == 0:
            return np.float32(np.nan)                     # 0 / 0: IEEE division gives NaN
        return np.float32(s64 / len(L))
    raise ValueError(reduction)
