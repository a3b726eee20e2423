"""Plain, slow, fp64 CPU reference of one MoE FFN layer forward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py``'s CPU-baseline / reference legs, never by the product path.

What the layer computes ("MOE推理流程解析", sections 一, 二 and 三):

* the router scores every expert for every token, and top-k keeps the chosen
  experts' indices and weights (section 三);
* each chosen expert processes the token vector independently, and the layer
  output is the routing-weighted sum over the chosen set (section 一, the toy
  four-expert example);
* assignments are grouped per expert into contiguous matrices, each row
  keeping its source token id; the combine multiplies each expert result by
  its routing weight and sums the contributions of the same token
  (section 二, the 4-token / 4-expert top-2 worked example);
* shared experts process every token whatever the router scores (section 一).

Readings taken where the page leaves a step open (each is argued in the
design notes of the repository):

* softmax over all E logits, then top-k, then the kept weights are divided by
  their sum (section 九 speaks of re-normalising the remaining weights);
* experts ranked by logit, ties to the lower index; slots ordered by
  descending weight;
* rows inside an expert's matrix in ascending token order (section 二: E1
  receives T1, T2, T3; E2 receives T3, T4);
* the expert FFN is SwiGLU: down( SiLU(x·W_gᵀ) ⊙ (x·W_uᵀ) ); the page only
  says each expert applies its activation and output projection (section 三);
* the shared expert is added with weight 1;
* FP8 weights are OCP E4M3 ("fn": max 448, no infinities) times a per-expert,
  per-output-channel fp32 scale ("MoE 推理部署", section 专家量化: scales are
  per expert).
* MXFP4 weights follow the OCP Microscaling (MX) format that the same
  section names: blocks of 32 consecutive weights along the reduction index
  share one UE8M0 scale 2^(s-127), each weight an FP4 E2M1 code; two codes
  per byte, the even element in the low nibble; the scales of an expert
  matrix stored reduction-block-major, [K/32, rows].

Everything is computed in float64 from the exact stored input values.
"""

from __future__ import annotations

import itertools
from typing import Callable, Optional, Tuple

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# Storage formats, decoded from their definitions
# ---------------------------------------------------------------------------

def _bf16_formula(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.int64) & 0xFFFF
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    exp = (b >> 7) & 0xFF
    frac = (b & 0x7F).astype(F64)
    normal = sign * np.ldexp(1.0 + frac / 128.0, (exp - 127).astype(np.int64))
    sub = sign * np.ldexp(frac / 128.0, -126)
    special = np.where(frac == 0, sign * np.inf, np.nan)
    out = np.where(exp == 0, sub, np.where(exp == 255, special, normal))
    return out.astype(F64)


def decode_bf16(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64.

    bfloat16 is the upper half of an IEEE-754 binary32: 1 sign bit, 8 exponent
    bits (bias 127), 7 fraction bits.  Exponent 0 encodes zero / subnormals
    (value = fraction/128 * 2^-126), exponent 255 encodes inf / NaN.
    The formula is evaluated once for all 65536 patterns, then looked up.
    """
    return _BF16_TABLE[np.asarray(bits).astype(np.int64) & 0xFFFF]


def _e4m3_formula(bits) -> np.ndarray:
    b = np.asarray(bits).astype(np.int64) & 0xFF
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    exp = (b >> 3) & 0xF
    frac = (b & 0x7).astype(F64)
    normal = sign * np.ldexp(1.0 + frac / 8.0, (exp - 7).astype(np.int64))
    sub = sign * np.ldexp(frac / 8.0, -6)
    out = np.where(exp == 0, sub, normal)
    out = np.where((exp == 15) & (frac == 7), np.nan, out)
    return out.astype(F64)


def decode_e4m3(bits) -> np.ndarray:
    """OCP FP8 E4M3 ("fn" flavour) bit patterns (uint8) -> float64.

    1 sign bit, 4 exponent bits (bias 7), 3 fraction bits.  Exponent 0 encodes
    zero / subnormals (value = fraction/8 * 2^-6).  There are no infinities:
    exponent 15 with fraction 7 is NaN, every other code is finite, so the
    largest magnitude is 2^8 * 1.75 = 448.
    The formula is evaluated once for all 256 codes, then looked up.
    """
    return _E4M3_TABLE[np.asarray(bits).astype(np.int64) & 0xFF]


with np.errstate(invalid="ignore"):
    _BF16_TABLE = _bf16_formula(np.arange(1 << 16))
    _E4M3_TABLE = _e4m3_formula(np.arange(1 << 8))


def _e2m1_formula(code) -> np.ndarray:
    c = np.asarray(code).astype(np.int64) & 0xF
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    frac = (c & 0x1).astype(F64)
    normal = sign * np.ldexp(1.0 + frac / 2.0, (exp - 1).astype(np.int64))
    sub = sign * (frac / 2.0)
    return np.where(exp == 0, sub, normal).astype(F64)


_E2M1_TABLE = _e2m1_formula(np.arange(16))


def decode_e2m1(codes) -> np.ndarray:
    """OCP FP4 E2M1 codes (0..15) -> float64.

    1 sign bit, 2 exponent bits (bias 1), 1 fraction bit; exponent 0 encodes
    zero and the subnormal 0.5.  No infinities or NaN: the magnitudes are
    0, 0.5, 1, 1.5, 2, 3, 4, 6.  Evaluated once for the 16 codes."""
    return _E2M1_TABLE[np.asarray(codes).astype(np.int64) & 0xF]


def decode_ue8m0(s) -> np.ndarray:
    """OCP UE8M0 scale bytes -> float64: 2^(s - 127); 0xFF is NaN."""
    b = np.asarray(s).astype(np.int64) & 0xFF
    with np.errstate(invalid="ignore"):
        return np.where(b == 0xFF, np.nan, np.ldexp(1.0, b - 127)).astype(F64)


def unpack_fp4(packed) -> np.ndarray:
    """[..., n/2] bytes -> [..., n] FP4 codes: byte i holds element 2i in its
    low nibble and element 2i+1 in its high nibble."""
    b = np.asarray(packed).astype(np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def decode_mxfp4(packed, scales) -> np.ndarray:
    """One MXFP4 matrix -> float64 [rows, K]: packed codes [rows, K/2],
    scales [K/32, rows] (one UE8M0 byte per 32 consecutive weights of a row):
    w[o, i] = decode_e2m1(code[o, i]) * decode_ue8m0(scale[i // 32, o])."""
    codes = unpack_fp4(packed)
    K = codes.shape[-1]
    if K % 32:
        raise ValueError("MXFP4 rows hold whole 32-element blocks")
    per_elem = np.repeat(decode_ue8m0(scales), 32, axis=0)  # [K, rows]
    return decode_e2m1(codes) * per_elem.T


def _to_f64(arr, fmt: str) -> np.ndarray:
    if fmt == "f32":
        return np.asarray(arr, dtype=np.float32).astype(F64)
    if fmt == "bf16":
        return decode_bf16(arr)
    if fmt == "f64":
        return np.asarray(arr, dtype=F64)
    raise ValueError(f"unknown storage format {fmt!r}")


class ExpertWeights:
    """Per-expert weights, decoded to float64 one expert at a time.

    Layout (output-major, the reduction index contiguous):
      w_gate, w_up : [E, ffn, d]      w_down : [E, d, ffn]
    ``fmt`` is "f32" (float32 arrays), "bf16" (uint16 bit patterns),
    "fp8" (uint8 E4M3 codes with fp32 scales s_gate, s_up [E, ffn] and
    s_down [E, d]: weight = decode_e4m3(code) * scale[e, output_channel]) or
    "mxfp4" (packed FP4 codes w_gate, w_up [E, ffn, d/2], w_down [E, d,
    ffn/2] with UE8M0 block scales s_gate, s_up [E, d/32, ffn], s_down
    [E, ffn/32, d]: decode_mxfp4 per expert matrix).
    """

    def __init__(self, fmt, w_gate, w_up, w_down, s_gate=None, s_up=None, s_down=None):
        self.fmt = fmt
        self.w_gate, self.w_up, self.w_down = w_gate, w_up, w_down
        self.s_gate, self.s_up, self.s_down = s_gate, s_up, s_down
        self.E = int(np.shape(w_gate)[0])
        if fmt in ("fp8", "mxfp4") and (s_gate is None or s_up is None or s_down is None):
            raise ValueError(f"{fmt} expert weights need their scales")

    def get(self, e: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
        if self.fmt == "fp8":
            wg = decode_e4m3(self.w_gate[e]) * np.asarray(self.s_gate[e], F64)[:, None]
            wu = decode_e4m3(self.w_up[e]) * np.asarray(self.s_up[e], F64)[:, None]
            wd = decode_e4m3(self.w_down[e]) * np.asarray(self.s_down[e], F64)[:, None]
            return wg, wu, wd
        if self.fmt == "mxfp4":
            return (decode_mxfp4(self.w_gate[e], self.s_gate[e]), decode_mxfp4(self.w_up[e], self.s_up[e]),
                    decode_mxfp4(self.w_down[e], self.s_down[e]))
        return (_to_f64(self.w_gate[e], self.fmt), _to_f64(self.w_up[e], self.fmt),
                _to_f64(self.w_down[e], self.fmt))


# ---------------------------------------------------------------------------
# FP8 activations for the routed experts' gate/up matrices (optional mode)
# ---------------------------------------------------------------------------

# Finite non-negative E4M3 magnitudes, indexed by code 0x00..0x7E (0x7F is
# NaN).  They increase with the code, so the nearest code is found by search.
_E4M3_POS = _E4M3_TABLE[:0x7F]


def round_to_e4m3(v) -> np.ndarray:
    """float32 values -> E4M3 codes (uint8): round to the nearest E4M3 value,
    ties to the code with an even mantissa (round-half-to-even, the IEEE
    default carried to the 8-bit grid), magnitudes beyond 448 clamped to 448
    ("saturate to finite").  Zero keeps its sign bit."""
    v = np.asarray(v, dtype=np.float32).astype(F64)
    a = np.minimum(np.abs(v), 448.0)
    hi = np.clip(np.searchsorted(_E4M3_POS, a, side="left"), 0, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(v), code | 0x80, code)
    return code.astype(np.uint8)


def quantize_rows_e4m3(x) -> Tuple[np.ndarray, np.ndarray]:
    """Per-row FP8 quantisation of activations (float32 arithmetic, the
    values the device computes): scale s_t = max_i |x[t, i]| / 448 (1 for an
    all-zero row), codes q[t, i] = round_to_e4m3(x[t, i] / s_t).
    Returns (codes uint8 [T, d], scales float32 [T]).  ``x`` holds exact
    stored values (bf16 values are exact in float32)."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=1)
    s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    q = (x32 / s[:, None]).astype(np.float32)
    return round_to_e4m3(q), s


def dequantize_rows_e4m3(codes, scales) -> np.ndarray:
    """codes [T, d] uint8, scales [T] float32 -> float64 values code * scale."""
    return decode_e4m3(codes) * np.asarray(scales, F64)[:, None]


# ---------------------------------------------------------------------------
# Router: scores, softmax, top-k, renormalisation (section 三; section 九)
# ---------------------------------------------------------------------------

def router_logits(x: np.ndarray, w_router: np.ndarray, bias: Optional[np.ndarray] = None) -> np.ndarray:
    """l[t, e] = sum_i x[t, i] * W_r[e, i] (+ b[e]): one score per expert per
    token (section 三: the router first produces a score for every eligible
    expert).  The optional bias is added before the softmax."""
    x = np.asarray(x, F64)
    w = np.asarray(w_router, F64)
    logits = x @ w.T
    if bias is not None:
        logits = logits + np.asarray(bias, F64)[None, :]
    return logits


def softmax(logits: np.ndarray) -> np.ndarray:
    """Row-wise softmax over all experts, shifted by the row maximum."""
    z = np.asarray(logits, F64)
    z = z - z.max(axis=-1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=-1, keepdims=True)


def topk_renorm(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Keep the k highest-scoring experts per token and their renormalised
    weights (section 三: top-k keeps the chosen indices and their weights;
    section 九: the remaining weights are re-normalised).

    p = softmax(l) over all E; S = the k experts with the largest l (ties: the
    lower expert index first); w_j = p_{S_j} / sum_{e in S} p_e.
    Returns idx int32 [T, k] and w float64 [T, k], slots in descending weight.
    """
    logits = np.asarray(logits, F64)
    T, E = logits.shape
    if not 1 <= k <= E:
        raise ValueError("need 1 <= k <= E")
    p = softmax(logits)
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=F64)
    for t in range(T):
        # descending logit; equal logits keep ascending expert order
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))
        chosen = order[:k]
        kept = np.array([p[t, e] for e in chosen], dtype=F64)
        idx[t] = chosen
        w[t] = kept / kept.sum()
    return idx, w


def topk_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Per token: (k-th largest logit) - ((k+1)-th largest logit); +inf when
    k == E.  A small gap means several expert sets are equally valid answers
    under rounding, so tests treat such tokens separately."""
    logits = np.asarray(logits, F64)
    T, E = logits.shape
    if k >= E:
        return np.full(T, np.inf)
    s = -np.sort(-logits, axis=1)
    return s[:, k - 1] - s[:, k]


# ---------------------------------------------------------------------------
# Dispatch: grouping assignments into per-expert matrices (section 二, 三)
# ---------------------------------------------------------------------------

def permutation_maps(idx: np.ndarray, E: int):
    """Group the T*k assignments by expert (section 二) and record the inverse
    map used by the combine (section 三).

    counts[e]        number of assignments to expert e (an expert batch counts
                     assignments, not unique tokens);
    offsets[e]       start row of expert e's matrix, offsets[E] = T*k;
    perm_token[r]    source token id kept beside row r;
    inv_row[t, j]    the row that holds assignment (t, slot j).
    Inside an expert's matrix the rows are in ascending token order.
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            if not 0 <= e < E:
                raise ValueError("expert index out of range")
            counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:E].copy()
    perm_token = np.empty(T * k, dtype=np.int64)
    inv_row = np.empty((T, k), dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            r = fill[e]
            fill[e] += 1
            perm_token[r] = t
            inv_row[t, j] = r
    return (counts.astype(np.int32), offsets.astype(np.int32),
            perm_token.astype(np.int32), inv_row.astype(np.int32))


# ---------------------------------------------------------------------------
# Expert FFN (section 三: activation and output projection)
# ---------------------------------------------------------------------------

def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + e^-z), written to avoid overflow of e^-z."""
    z = np.asarray(z, F64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def swiglu_expert(x_rows: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray,
                  act8: bool = False) -> np.ndarray:
    """One expert on a matrix of rows: (SiLU(X W_gᵀ) ⊙ (X W_uᵀ)) W_dᵀ.
    ``act8``, the FP8-activation mode: both products take E4M3 activations
    quantised per row (quantize_rows_e4m3): the rows X before the gate and up
    products, and the rows of h = SiLU(g) ⊙ u (rounded to float32, the
    quantiser's input precision) before the down product."""
    x_rows = np.asarray(x_rows, F64)
    if act8:
        x_rows = dequantize_rows_e4m3(*quantize_rows_e4m3(x_rows))
    g = x_rows @ np.asarray(wg, F64).T
    u = x_rows @ np.asarray(wu, F64).T
    h = silu(g) * u
    if act8:
        h = dequantize_rows_e4m3(*quantize_rows_e4m3(h.astype(np.float32)))
    return h @ np.asarray(wd, F64).T


def shared_expert(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray) -> np.ndarray:
    """Always-on shared expert: every token, whatever the router scores
    (section 一), added with weight 1."""
    return swiglu_expert(x, wg, wu, wd)


# ---------------------------------------------------------------------------
# Layer forward, two independent formulations
# ---------------------------------------------------------------------------

def moe_forward_per_token(x, w_router, experts: ExpertWeights, k: int, bias=None,
                          shared: Optional[Tuple] = None, routing=None,
                          tokens=None, act8: bool = False):
    """Formulation (i), the plain definition (section 一): for each token,
    out_t = sum over its chosen experts e of w_{t,e} * FFN_e(x_t)
            (+ shared FFN(x_t)).

    ``routing`` = (idx, w) overrides the router (used to evaluate the layer
    under a given expert choice); ``tokens`` restricts the computation to a
    subset of token ids (rows of the result follow that subset).  ``act8``:
    the routed experts run in the FP8-activation mode of swiglu_expert (the
    router and the shared expert see x itself).
    Returns (out [n, d], idx, w) in float64.
    """
    x = np.asarray(x, F64)
    if routing is None:
        sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
        idx, w = topk_renorm(router_logits(x[sel], w_router, bias), k)
    else:
        idx, w = routing
        idx = np.asarray(idx)
        w = np.asarray(w, F64)
        if tokens is not None:
            idx, w = idx[np.asarray(tokens)], w[np.asarray(tokens)]
    sel = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    d = x.shape[1]
    out = np.zeros((len(sel), d), dtype=F64)
    cache = {}
    for n, t in enumerate(sel):
        for j in range(idx.shape[1]):
            e = int(idx[n, j])
            if e not in cache:
                cache[e] = experts.get(e)
            wg, wu, wd = cache[e]
            out[n] += w[n, j] * swiglu_expert(x[t:t + 1], wg, wu, wd, act8=act8)[0]
        if shared is not None:
            out[n] += shared_expert(x[t:t + 1], *shared)[0]
    return out, idx, w


def moe_forward_grouped(x, w_router, experts: ExpertWeights, k: int, bias=None,
                        shared: Optional[Tuple] = None, routing=None,
                        expert_hook: Optional[Callable] = None, act8: bool = False):
    """Formulation (ii), the grouped execution of section 二/三: sort the
    assignments by expert (a stable sort keeps ascending token order inside
    each expert), run one matrix per expert, then scatter each result back to
    its source token, scaled by its routing weight.

    ``expert_hook(e)`` is called before each expert's matrix (the CPU
    baseline uses it to exclude per-expert weight decoding from timing).
    Returns (out [T, d], idx, w) in float64.
    """
    x = np.asarray(x, F64)
    T, d = x.shape
    if routing is None:
        idx, w = topk_renorm(router_logits(x, w_router, bias), k)
    else:
        idx, w = np.asarray(routing[0]), np.asarray(routing[1], F64)
    kk = idx.shape[1]
    flat_e = idx.reshape(-1).astype(np.int64)
    flat_t = np.repeat(np.arange(T), kk)
    flat_w = w.reshape(-1)
    order = np.argsort(flat_e, kind="stable")
    out = np.zeros((T, d), dtype=F64)
    bounds = np.searchsorted(flat_e[order], np.arange(experts.E + 1))
    for e in range(experts.E):
        rows = order[bounds[e]:bounds[e + 1]]
        if rows.size == 0:
            continue
        if expert_hook is not None:
            wg, wu, wd = expert_hook(e)
        else:
            wg, wu, wd = experts.get(e)
        y = swiglu_expert(x[flat_t[rows]], wg, wu, wd, act8=act8)
        np.add.at(out, flat_t[rows], flat_w[rows, None] * y)
    if shared is not None:
        out += shared_expert(x, *shared)
    return out, idx, w


def brute_force_topk_sets(logits: np.ndarray, k: int):
    """For tiny E: the k-subset with the largest total softmax probability,
    found by enumerating every k-subset (used only to pin ``topk_renorm``)."""
    p = softmax(logits)
    T, E = p.shape
    best = []
    for t in range(T):
        sets = list(itertools.combinations(range(E), k))
        totals = [sum(p[t, e] for e in s) for s in sets]
        best.append(set(sets[int(np.argmax(totals))]))
    return best
