"""CPU oracle for the Beam MoE sublayer -- TEST INFRASTRUCTURE ONLY.

Plain, slow, FP64 NumPy restatement of what the layer computes. Only the
tests, the package's smoke check and the benchmark's CPU-baseline leg may use
it; the product path never imports it. It shares no code with the CUDA path.

Sources (release pages about the model, cited by title and section):
  [P1] "Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文"
       sections 专家混合模型 (experts, router), 残差流 (residual stream,
       FP32 steps, pre/post norm).
  [P3] tech.fxxz.com article on the Beam release, sections 混合专家系统 and
       残差流设计 (a machine-translated copy of [P1]).
  [P4] "Welcome Beam: a 501B open model you can own, customize, and scale"
       (English excerpt: layer counts, experts, residual step weights).
  [P5] "Reflection 放出 501B 的 Beam 权重：四套精度、滑动窗口和一场榜单落差"
       section "config.json 里还有六处能直接抄的细节" (n_group 8,
       topk_group 4, norm_topk_prob true, routed_scaling_factor 2.5).

Readings where the pages leave a step open (the E4M3, NVFP4 and attention
sections below list their own):
  * scaling: the combine weights are multiplied by 2.5 ([P1] 专家混合模型,
    [P5] routed_scaling_factor); [P3] "缩小为 2.5" is a garbled translation.
  * normalisation divides by the sum of the 8 selected sigmoid scores, with
    no epsilon.
  * a router-logit bias, when given, is added before the sigmoid, so it
    changes selection and weights alike.
  * ties: lower expert index first, lower group index first.
  * decisions (group ranking, expert ranking) are taken on FP32 scores, the
    router's precision on the pages ([P1] 残差流: the router runs in FP32);
    the group score is the FP32 sum of the two largest FP32 scores.
  * SwiGLU: silu(x W_g^T) * (x W_u^T), then W_d.
  * RMSNorm: v / sqrt(mean(v^2) + eps) * gain, eps = 1e-6, plain
    multiplicative gain.
  * post-norm applies to the combined MoE output before the 1/sqrt(k) weight.
  * the pre-norm output is rounded to BF16, the activation dtype the expert
    matmuls consume.

Everything is FP64 except the FP32 rounding of the router scores (above) and
the BF16 rounding of the pre-norm output.

Every function has a pin -- tests/test_oracle_pins.py, test_oracle_fp8_pins.py,
test_oracle_nvfp4_pins.py and test_oracle_attn_pins.py -- that checks it
against something other than itself (closed forms, hand-worked examples,
brute force, exactly representable cases and library routines).
"""
from __future__ import annotations

import math
from typing import Callable, Optional, Tuple

import numpy as np

F64 = np.float64
F32 = np.float32


# ----------------------------------------------------------------------------
# elementwise helpers
# ----------------------------------------------------------------------------
def bf16_round(a) -> np.ndarray:
    """Round to the nearest BF16 value (ties to even); returns float32 values.

    BF16 keeps the top 16 bits of an IEEE float32. Finite inputs only.
    """
    u = np.ascontiguousarray(np.asarray(a, dtype=F32)).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(F32)


def sigmoid(z: np.ndarray) -> np.ndarray:
    """Logistic function 1 / (1 + e^-z), FP64."""
    z = np.asarray(z, dtype=F64)
    return 1.0 / (1.0 + np.exp(-z))


def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z), FP64."""
    z = np.asarray(z, dtype=F64)
    return z * sigmoid(z)


def rms_norm(v: np.ndarray, gain: Optional[np.ndarray] = None,
             eps: float = 1e-6) -> np.ndarray:
    """Row-wise RMSNorm: v / sqrt(mean(v^2) + eps) * gain ([P1] 残差流: every
    sublayer is normalised before and after)."""
    v = np.asarray(v, dtype=F64)
    ms = np.mean(v * v, axis=-1, keepdims=True)
    out = v / np.sqrt(ms + eps)
    if gain is not None:
        out = out * np.asarray(gain, dtype=F64)
    return out


# ----------------------------------------------------------------------------
# router ([P1] 专家混合模型; [P5] config fields)
# ----------------------------------------------------------------------------
def router_scores(x: np.ndarray, w_router: np.ndarray,
                  bias: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Sigmoid scores for every expert.

    logit[t,e] = sum_j x[t,j] * w_router[e,j] (+ bias[e]); s = sigmoid(logit).
    Returns (s64 [T,E] FP64, s32 [T,E] FP32 rounding of s64).
    """
    x = np.asarray(x, dtype=F64)
    w = np.asarray(w_router, dtype=F64)
    logits = x @ w.T
    if bias is not None:
        logits = logits + np.asarray(bias, dtype=F64)[None, :]
    s64 = sigmoid(logits)
    return s64, s64.astype(F32)


def group_scores(s32: np.ndarray, n_group: int) -> np.ndarray:
    """Score of each group: FP32 sum of its two largest FP32 scores
    (of its only score when a group has one expert)."""
    T, E = s32.shape
    gsize = E // n_group
    sg = np.asarray(s32, dtype=F32).reshape(T, n_group, gsize)
    srt = -np.sort(-sg, axis=-1)           # descending within each group
    if gsize == 1:
        return srt[..., 0].copy()
    return (srt[..., 0] + srt[..., 1]).astype(F32)   # float32 addition


def _rank_desc(values: np.ndarray) -> np.ndarray:
    """Indices sorting one row by value descending, ties by lower index."""
    idx = np.arange(values.shape[-1])
    return np.lexsort((idx, -values.astype(F64)))


def group_limited_topk(s32: np.ndarray, n_group: int, topk_group: int,
                       top_k: int) -> dict:
    """Group-limited selection ([P1] 专家混合模型).

    1. split the E experts into n_group consecutive groups;
    2. rank the groups by the sum of their two best scores, keep topk_group;
    3. among the experts of the kept groups, take the top_k best scores.
    Output order: descending score, ties by lower expert index.

    Returns dict with
      idx         [T, top_k] int32 selected experts in output order
      kept        [T, topk_group] int32 kept groups in rank order
      gscore      [T, n_group] float32 group scores
      group_margin  [T] float64: 4th-best minus 5th-best group score (inf if
                    every group is kept)
      topk_margin   [T] float64: k-th selected minus best unselected
                    candidate score (inf if no candidate is left out)
    """
    s32 = np.asarray(s32, dtype=F32)
    T, E = s32.shape
    assert E % n_group == 0
    gsize = E // n_group
    assert 1 <= topk_group <= n_group and 1 <= top_k <= topk_group * gsize
    gs = group_scores(s32, n_group)
    idx = np.empty((T, top_k), dtype=np.int32)
    kept = np.empty((T, topk_group), dtype=np.int32)
    gmar = np.full(T, np.inf)
    kmar = np.full(T, np.inf)
    for t in range(T):
        gorder = _rank_desc(gs[t])
        kept[t] = gorder[:topk_group]
        if topk_group < n_group:
            gmar[t] = float(gs[t, gorder[topk_group - 1]]) - float(gs[t, gorder[topk_group]])
        cand = np.concatenate([np.arange(g * gsize, (g + 1) * gsize)
                               for g in sorted(kept[t])])
        corder = cand[_rank_desc(s32[t, cand])]
        idx[t] = corder[:top_k]
        if len(corder) > top_k:
            kmar[t] = float(s32[t, corder[top_k - 1]]) - float(s32[t, corder[top_k]])
    return dict(idx=idx, kept=kept, gscore=gs, group_margin=gmar,
                topk_margin=kmar)


def combine_weights(s: np.ndarray, idx: np.ndarray, scale: float) -> np.ndarray:
    """w[t,j] = scale * s[t, idx[t,j]] / sum_i s[t, idx[t,i]]  ([P1] 专家混合模型:
    normalised router weights, multiplied by 2.5; [P5] norm_topk_prob,
    routed_scaling_factor)."""
    s = np.asarray(s, dtype=F64)
    sel = np.take_along_axis(s, np.asarray(idx, dtype=np.int64), axis=1)
    return scale * sel / sel.sum(axis=1, keepdims=True)


def route(x, w_router, bias, n_group, topk_group, top_k, scale) -> dict:
    """Scores, group-limited selection and combine weights for every token."""
    s64, s32 = router_scores(x, w_router, bias)
    sel = group_limited_topk(s32, n_group, topk_group, top_k)
    sel["weights"] = combine_weights(s64, sel["idx"], scale)
    sel["s64"] = s64
    sel["s32"] = s32
    return sel


def near_ties(sel: dict, margin: float = 1e-5) -> np.ndarray:
    """Tokens whose group or top-k boundary is closer than `margin` in FP32
    score: another correct FP32 evaluation may pick the other side there."""
    return (sel["group_margin"] < margin) | (sel["topk_margin"] < margin)


# ----------------------------------------------------------------------------
# permutation (token -> expert order)
# ----------------------------------------------------------------------------
def permutation(idx: np.ndarray, E: int) -> dict:
    """Token-expert pairs grouped by expert, stable in pair order p = t*k + j.

    Returns counts [E], offsets [E+1], row_pair [T*k] (the pair at each row of
    the expert-ordered layout).
    """
    flat = np.asarray(idx, dtype=np.int64).ravel()
    row_pair = np.argsort(flat, kind="stable").astype(np.int64)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return dict(counts=counts, offsets=offsets, row_pair=row_pair)


# ----------------------------------------------------------------------------
# experts ([P1] 专家混合模型: each expert a SwiGLU MLP; [P1] 残差流: SwiGLU
# product in FP32 -- the oracle keeps FP64)
# ----------------------------------------------------------------------------
def swiglu_expert(x_rows: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray,
                  w_down: np.ndarray) -> np.ndarray:
    """y = (silu(x W_g^T) * (x W_u^T)) W_d^T for rows x [n,H];
    w_gate, w_up [I,H]; w_down [H,I]."""
    x = np.asarray(x_rows, dtype=F64)
    g = x @ np.asarray(w_gate, dtype=F64).T
    u = x @ np.asarray(w_up, dtype=F64).T
    a = silu(g) * u
    return a @ np.asarray(w_down, dtype=F64).T


def moe_combine(x: np.ndarray, idx: np.ndarray, weights: np.ndarray,
                get_expert: Callable[[int], tuple]) -> np.ndarray:
    """out[t] = sum_j weights[t,j] * f_{idx[t,j]}(x[t]), expert by expert
    ([P1] 专家混合模型: expert outputs combined with the normalised weights)."""
    x = np.asarray(x, dtype=F64)
    T = x.shape[0]
    out = np.zeros((T, x.shape[1]), dtype=F64)
    idx = np.asarray(idx)
    for e in np.unique(idx):
        tok, slot = np.nonzero(idx == e)
        wg, wu, wd = get_expert(int(e))
        y = swiglu_expert(x[tok], wg, wu, wd)
        out[tok] += weights[tok, slot][:, None] * y
    return out


# ----------------------------------------------------------------------------
# residual stream ([P1] 残差流; [P4] residual paragraph)
# ----------------------------------------------------------------------------
def residual_coeffs(k: int) -> Tuple[float, float]:
    """(sqrt((k-1)/k), 1/sqrt(k)): keep weight and add weight at step k."""
    if k < 2:
        raise ValueError("residual step k must be >= 2 (the embedding is step 1)")
    return math.sqrt((k - 1) / k), 1.0 / math.sqrt(k)


def residual_step(h_prev, sub_out, k: int, gain=None, eps: float = 1e-6,
                  apply_norm: bool = True) -> np.ndarray:
    """h_k = sqrt((k-1)/k) h_{k-1} + (1/sqrt(k)) * n, n = RMSNorm(sub_out)
    (or sub_out itself when apply_norm is False)."""
    a, b = residual_coeffs(k)
    n = rms_norm(sub_out, gain, eps) if apply_norm else np.asarray(sub_out, F64)
    return a * np.asarray(h_prev, dtype=F64) + b * n


# ----------------------------------------------------------------------------
# dense SwiGLU MLP of the first layers ([P1] 专家混合模型: the first 3 layers use
# a dense SwiGLU MLP; [P1] 残差流: normalised before and after, scaled residual)
# ----------------------------------------------------------------------------
def dense_mlp_forward(x_in, w_gate, w_up, w_down, *, eps=1e-6, pre_norm=False,
                      pre_gain=None, residual_k=0, post_gain=None) -> dict:
    """x = pre_norm ? bf16(RMSNorm(x_in)) : x_in; y = SwiGLU MLP of x;
    h = residual step at k (when residual_k >= 2). w_gate, w_up [I,H];
    w_down [H,I]; the intermediate size I is a parameter (not on the pages)."""
    x_in = np.asarray(x_in, dtype=F64)
    x = bf16_round(rms_norm(x_in, pre_gain, eps)).astype(F64) if pre_norm else x_in
    y = swiglu_expert(x, w_gate, w_up, w_down)
    h = residual_step(x_in, y, residual_k, post_gain, eps, True) if residual_k else None
    return dict(x=x, out=y, h=h)


# ----------------------------------------------------------------------------
# the whole sublayer
# ----------------------------------------------------------------------------
def moe_forward(x_in, w_router, bias, get_expert, *, n_group=8, topk_group=4,
                top_k=8, scale=2.5, eps=1e-6, pre_norm=False, pre_gain=None,
                residual_k=0, post_gain=None, routing: Optional[dict] = None) -> dict:
    """The MoE sublayer as the pages state it.

    x_in: layer input [T,H] (h_{k-1} when pre_norm or residual_k >= 2).
    get_expert(e) -> (w_gate [I,H], w_up [I,H], w_down [H,I]).
    routing: optional dict with 'idx' and 'weights' to use instead of the
    oracle's own routing (to compare experts and combine on near-tie tokens).
    Returns dict(x, sel, out, h).
    """
    x_in = np.asarray(x_in, dtype=F64)
    x = bf16_round(rms_norm(x_in, pre_gain, eps)).astype(F64) if pre_norm else x_in
    sel = route(x, w_router, bias, n_group, topk_group, top_k, scale)
    use = routing if routing is not None else sel
    out = moe_combine(x, use["idx"], use["weights"], get_expert)
    h = None
    if residual_k:
        h = residual_step(x_in, out, residual_k, post_gain, eps, True)
    return dict(x=x, sel=sel, out=out, h=h)


# ----------------------------------------------------------------------------
# FP8 expert weights ([P5] section 四套权重的账，自己算一遍: the FP8 checkpoint
# stores every linear weight except lm_head, the embedding and the router
# ("mlp.gate") as F8_E4M3 and is a dynamic FP8 quantisation; [P1] 专家混合模型:
# an FP8 checkpoint exists beside the BF16 one).
#
# Readings where the pages leave the format open:
#   * element type E4M3 in the OCP "E4M3FN" form: 4 exponent bits (bias 7),
#     3 mantissa bits, subnormals, largest finite value 448, no infinities;
#     conversion rounds to nearest, ties to even, and saturates at +-448.
#   * weights: one FP32 scale per output row (static, from the row's absolute
#     maximum); activations: one FP32 scale per token row, computed at run
#     time from that row ("dynamic"). The same row quantiser serves both:
#       amax = max_j |v_j|;  scale = fp32(amax / 448);  inv = fp32(448 / amax)
#       code_j = E4M3(fp32(v_j * inv))       (scale = inv = 1 for a zero row)
#     and a row is dequantised as E4M3 value * scale.
#   * the expert input x is the BF16 pre-norm output, quantised per token;
#     the SwiGLU output A is rounded to BF16 (the activation dtype) and then
#     quantised per token-expert pair, before the down projection.
#   * the router stays unquantised (FP32 weight, FP32 scores).
# ----------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_round(v) -> np.ndarray:
    """Nearest E4M3 value (ties to even) of each finite input, saturating at
    +-448; returned as float64. Spacing is 2^(e-3) in the binade [2^e, 2^(e+1))
    for e >= -6 and 2^-9 below 2^-6 (subnormals)."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    _, ex = np.frexp(a)                     # a = m * 2^ex, m in [0.5, 1)
    e = np.maximum(ex - 1, -6)              # binade exponent, subnormals share -6
    q = np.ldexp(1.0, e - 3)                # spacing of the grid there
    r = np.round(a / q) * q                 # np.round: halves go to even
    r = np.where(a == 0, 0.0, r)
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def e4m3_encode(v) -> np.ndarray:
    """Byte codes (sign | exponent << 3 | mantissa) of values already on the
    E4M3 grid (|v| <= 448)."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    sign = np.signbit(v).astype(np.uint8) << np.uint8(7)
    _, ex = np.frexp(a)
    e_unb = ex - 1
    normal = a >= 2.0 ** -6
    m_norm = np.where(normal, a / np.ldexp(1.0, np.where(normal, e_unb, 0)) - 1.0, 0.0) * 8.0
    m_sub = a / 2.0 ** -9
    mant = np.where(normal, m_norm, m_sub)
    expo = np.where(normal, e_unb + 7, 0)
    assert np.all(mant == np.round(mant)) and np.all((mant >= 0) & (mant <= 7)), "value off the E4M3 grid"
    assert np.all((expo >= 0) & (expo <= 15)), "value out of E4M3 range"
    return sign | (expo.astype(np.uint8) << np.uint8(3)) | mant.astype(np.uint8)


def _e4m3_value(c: np.ndarray) -> np.ndarray:
    """Value of each E4M3 byte code (int64 array): sign bit 7, exponent bits
    3..6 (bias 7; 0 = subnormal, m * 2^-9), mantissa bits 0..2; S.1111.111
    is NaN."""
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return s * val


_E4M3_TABLE = _e4m3_value(np.arange(256, dtype=np.int64))


def e4m3_decode(codes) -> np.ndarray:
    """Values of E4M3 byte codes as float64 (NaN for S.1111.111), looked up
    in the table of all 256 codes' values."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def quantize_rows_e4m3(a) -> Tuple[np.ndarray, np.ndarray]:
    """Per-row E4M3 quantisation with an FP32 scale (reading above).

    a: [R, K] FP32-representable values (BF16 weights or activations).
    Returns (codes [R, K] uint8, scale [R] float32)."""
    a32 = np.asarray(a, dtype=F32)
    amax = np.max(np.abs(a32), axis=-1)
    nz = amax > 0
    safe = np.where(nz, amax, F32(1.0)).astype(F32)
    scale = np.where(nz, safe / F32(E4M3_MAX), F32(1.0)).astype(F32)   # IEEE FP32 division
    inv = np.where(nz, F32(E4M3_MAX) / safe, F32(1.0)).astype(F32)
    v = (a32 * inv[..., None]).astype(F32)                             # one FP32 rounding
    return e4m3_encode(e4m3_round(v)), scale


def dequantize_rows_e4m3(codes, scale) -> np.ndarray:
    """E4M3 value * row scale, FP64."""
    return e4m3_decode(codes) * np.asarray(scale, dtype=F64)[..., None]


def swiglu_act_fp8(x_rows, gate_q, up_q) -> np.ndarray:
    """SwiGLU activation of an FP8 expert before its BF16 rounding: x rows
    (BF16 values) quantised per row, g = x W_g^T and u = x W_u^T on the
    dequantised operands, a = silu(g) * u (FP64).
    gate_q, up_q: (codes [I,H], scale [I])."""
    qx, sx = quantize_rows_e4m3(x_rows)
    xd = dequantize_rows_e4m3(qx, sx)
    g = xd @ dequantize_rows_e4m3(*gate_q).T
    u = xd @ dequantize_rows_e4m3(*up_q).T
    return silu(g) * u


def swiglu_expert_fp8(x_rows, gate_q, up_q, down_q) -> np.ndarray:
    """One expert on FP8 weights: a = swiglu_act_fp8, rounded to BF16 and
    quantised per row, then y = a W_d^T on the dequantised operands (FP64).
    down_q: (codes [H,I], scale [H])."""
    a = bf16_round(swiglu_act_fp8(x_rows, gate_q, up_q))
    qa, sa = quantize_rows_e4m3(a)
    return dequantize_rows_e4m3(qa, sa) @ dequantize_rows_e4m3(*down_q).T


def moe_combine_fp8(x: np.ndarray, idx: np.ndarray, weights: np.ndarray,
                    get_expert_q: Callable[[int], tuple]) -> np.ndarray:
    """out[t] = sum_j weights[t,j] * f8_{idx[t,j]}(x[t]) with the FP8 experts
    (swiglu_expert_fp8), expert by expert."""
    x = np.asarray(x, dtype=F64)
    out = np.zeros((x.shape[0], x.shape[1]), dtype=F64)
    idx = np.asarray(idx)
    weights = np.asarray(weights, dtype=F64)
    for e in np.unique(idx):
        tok, slot = np.nonzero(idx == e)
        y = swiglu_expert_fp8(x[tok], *get_expert_q(int(e)))
        out[tok] += weights[tok, slot][:, None] * y
    return out


def moe_forward_fp8(x_in, w_router, bias, get_expert_q, *, n_group=8, topk_group=4,
                    top_k=8, scale=2.5, eps=1e-6, pre_norm=False, pre_gain=None,
                    residual_k=0, post_gain=None, routing: Optional[dict] = None) -> dict:
    """The MoE sublayer with FP8 expert weights: routing as in moe_forward
    (unquantised router), each selected expert through swiglu_expert_fp8,
    combine, post-norm and residual as in moe_forward.
    get_expert_q(e) -> (gate_q, up_q, down_q), each (codes, row scales)."""
    x_in = np.asarray(x_in, dtype=F64)
    x = bf16_round(rms_norm(x_in, pre_gain, eps)).astype(F64) if pre_norm else x_in
    sel = route(x, w_router, bias, n_group, topk_group, top_k, scale)
    use = routing if routing is not None else sel
    out = moe_combine_fp8(x, use["idx"], use["weights"], get_expert_q)
    h = residual_step(x_in, out, residual_k, post_gain, eps, True) if residual_k else None
    return dict(x=x, sel=sel, out=out, h=h)


# ----------------------------------------------------------------------------
# NVFP4 expert weights ([P5] section 四套权重的账，自己算一遍: the NVFP4
# checkpoint packs every routed-expert weight as two 4-bit values per byte
# (U8 count = half the expert parameters) and keeps the rest in BF16; its
# section 上手前的五个坑: NVFP4 is packed by modelopt and runs on the FP4
# tensor-core path of Blackwell; [P1] 专家混合模型: NVFP4 stores most
# parameters in 4 bits for Blackwell GPUs).
#
# Readings where the pages leave the format open:
#   * element type E2M1: sign bit 3, exponent bits 1..2 (bias 1), mantissa
#     bit 0, values 0, 0.5, 1, 1.5, 2, 3, 4, 6; round to nearest, ties to
#     even, saturate at +-6; two per byte, the even element in the low nibble.
#   * 16 consecutive elements along K share a block scale stored as E4M3
#     (one byte); a second FP32 scale covers a group of rows: one expert
#     matrix for weights (static), one row for activations (dynamic, run
#     time). Supporting arithmetic: the NVFP4 checkpoint's disk size
#     (293.63 GB) equals its listed U8 + BF16 + F32 bytes (262.79 GB) plus one
#     byte per 16 routed-expert weights (30.83 GB) to within 0.02 GB.
#   * quantiser, in FP32 with IEEE division, for a group with largest
#     magnitude amax (g = 1 for an all-zero group) and each 16-block b:
#       g   = amax / 2688                      (2688 = 6 * 448)
#       s_b = E4M3(amax_b / (6 * g))           (block scale, <= 448)
#       q_i = E2M1(v_i * (1 / (s_b * g)))      (q = 0 where s_b = 0)
#     and an element is dequantised as E2M1 value * s_b * g.
#   * x (BF16, after the optional pre-norm) is quantised per token; the
#     SwiGLU output A is rounded to BF16 and quantised per (token, expert)
#     row, as for FP8; the router stays FP32.
# ----------------------------------------------------------------------------
E2M1_MAX = 6.0
NVFP4_BLOCK = 16


def e2m1_round(v) -> np.ndarray:
    """Nearest E2M1 value (ties to even mantissa), saturating at +-6; float64.
    Grid spacing 0.5 below 2, 1 in [2, 4), 2 in [4, 6]."""
    v = np.asarray(v, dtype=F64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    e = np.clip(ex - 1, 0, 2)                 # binade [2^e, 2^(e+1)); 0.5-steps below 2
    q = np.ldexp(1.0, e - 1)                  # spacing: 0.5, 1, 2
    r = np.round(a / q) * q                   # np.round: halves go to even
    r = np.minimum(np.where(a == 0, 0.0, r), E2M1_MAX)
    return np.copysign(r, v)


_E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_encode(v) -> np.ndarray:
    """4-bit codes (sign << 3 | magnitude index) of values on the E2M1 grid."""
    v = np.asarray(v, dtype=F64)
    mag = np.abs(v)
    idx = np.searchsorted(_E2M1_VALUES, mag)
    assert np.all(_E2M1_VALUES[np.minimum(idx, 7)] == mag), "value off the E2M1 grid"
    return (np.signbit(v).astype(np.uint8) << np.uint8(3)) | idx.astype(np.uint8)


def e2m1_decode(codes) -> np.ndarray:
    """Values of 4-bit E2M1 codes: exponent field e (bits 1..2), mantissa m
    (bit 0): e = 0 gives m * 0.5, else (1 + m/2) * 2^(e-1)."""
    c = np.asarray(codes, dtype=np.int64) & 0xF
    e = (c >> 1) & 0x3
    m = c & 0x1
    val = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.ldexp(1.0, e - 1))
    return np.where(c & 0x8, -val, val)


def pack_e2m1(codes) -> np.ndarray:
    """[..., K] 4-bit codes -> [..., K/2] bytes, the even element in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed) -> np.ndarray:
    """[..., K/2] bytes -> [..., K] 4-bit codes."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def quantize_nvfp4(a, rows_per_group: int):
    """NVFP4 quantisation (reading above) of rows a [R, K] (K % 16 == 0)
    whose consecutive groups of rows_per_group rows share the FP32 scale.
    Returns (packed codes [R, K/2] uint8, block scales [R, K/16] uint8 E4M3
    codes, group scales [R / rows_per_group] float32)."""
    a32 = np.asarray(a, dtype=F32)
    R, K = a32.shape
    assert K % NVFP4_BLOCK == 0 and R % rows_per_group == 0
    G = R // rows_per_group
    amax = np.max(np.abs(a32).reshape(G, -1), axis=1)
    g = np.where(amax > 0, amax / F32(2688.0), F32(1.0)).astype(F32)
    g_row = np.repeat(g, rows_per_group)
    blocks = a32.reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK)
    amax_b = np.max(np.abs(blocks), axis=2)
    six_g = (F32(6.0) * g_row).astype(F32)
    sb_val = e4m3_round((amax_b / six_g[:, None]).astype(F32))
    sb_code = e4m3_encode(sb_val)
    denom = (sb_val.astype(F32) * g_row[:, None]).astype(F32)
    with np.errstate(divide="ignore"):
        inv = np.where(sb_val > 0, F32(1.0) / np.where(sb_val > 0, denom, F32(1.0)),
                       F32(0.0)).astype(F32)
    v = (blocks * inv[:, :, None]).astype(F32)
    codes = e2m1_encode(e2m1_round(v)).reshape(R, K)
    return pack_e2m1(codes), sb_code, g


def dequantize_nvfp4(packed, block_scales, group_scales, rows_per_group: int) -> np.ndarray:
    """E2M1 value * E4M3 block scale * FP32 group scale, FP64 [R, K]."""
    vals = e2m1_decode(unpack_e2m1(packed))
    R, K = vals.shape
    sb = e4m3_decode(block_scales)
    g = np.repeat(np.asarray(group_scales, dtype=F64), rows_per_group)
    return (vals.reshape(R, K // NVFP4_BLOCK, NVFP4_BLOCK) * sb[:, :, None]
            * g[:, None, None]).reshape(R, K)


def swiglu_act_nvfp4(x_rows, gate_q, up_q) -> np.ndarray:
    """SwiGLU activation of an NVFP4 expert before its BF16 rounding: x rows
    quantised per row (NVFP4, group = one row), g and u on the dequantised
    operands, a = silu(g) * u (FP64). gate_q, up_q: (packed [I,H/2], block
    scales [I,H/16], group scale [1]) of one expert matrix."""
    xd = dequantize_nvfp4(*quantize_nvfp4(x_rows, 1), 1)
    I = gate_q[0].shape[0]
    g = xd @ dequantize_nvfp4(*gate_q, I).T
    u = xd @ dequantize_nvfp4(*up_q, I).T
    return silu(g) * u


def swiglu_expert_nvfp4(x_rows, gate_q, up_q, down_q) -> np.ndarray:
    """One NVFP4 expert: a = swiglu_act_nvfp4 rounded to BF16, quantised per
    row (NVFP4), y = a W_d^T on the dequantised operands (FP64)."""
    a = bf16_round(swiglu_act_nvfp4(x_rows, gate_q, up_q))
    ad = dequantize_nvfp4(*quantize_nvfp4(a, 1), 1)
    H = down_q[0].shape[0]
    return ad @ dequantize_nvfp4(*down_q, H).T


def moe_combine_nvfp4(x, idx, weights, get_expert_q) -> np.ndarray:
    """out[t] = sum_j weights[t,j] * f4_{idx[t,j]}(x[t]) (swiglu_expert_nvfp4)."""
    x = np.asarray(x, dtype=F64)
    out = np.zeros((x.shape[0], x.shape[1]), dtype=F64)
    idx = np.asarray(idx)
    weights = np.asarray(weights, dtype=F64)
    for e in np.unique(idx):
        tok, slot = np.nonzero(idx == e)
        out[tok] += weights[tok, slot][:, None] * swiglu_expert_nvfp4(x[tok], *get_expert_q(int(e)))
    return out


# ----------------------------------------------------------------------------
# attention sublayer ([P1] section 注意力: 52 decoder layers, hidden 5120;
# sliding-window attention over the last 512 tokens, every sixth layer and
# the last attend to the full context; sliding layers use RoPE, global
# layers none but multiply each query by (1 + (pos + 1) / 2048) ** 0.1;
# grouped-query attention with 48 query heads and 8 key/value heads, RMSNorm
# on queries and keys; a learned sigmoid gate computed from the layer input
# scales every channel of every head before the output projection.
# [P1] 残差流: normalised before and after, the scaled residual step; RoPE and
# the query scaling run in FP32. [P5] config.json: head_dim 128,
# sliding_window 512, rope_theta 10000 on the sliding layers.)
#
# Readings where the pages leave a step open:
#   * the window holds the current token and the 511 before it (key j is seen
#     by query i when 0 <= i - j < 512); attention is causal;
#   * softmax scale 1/sqrt(head_dim);
#   * q_norm / k_norm: RMSNorm over the 128 channels of each head with a
#     128-wide gain shared by the heads (eps 1e-6), applied before RoPE;
#   * RoPE: rotate-half form over all 128 channels, frequency
#     theta^(-2i/128) for channel pairs (i, i + 64), position = token index;
#   * the global query scale multiplies the normalised query (pos = token
#     index, 0-based);
#   * query head h uses key/value head h // 6;
#   * the gate is sigmoid(x W_g^T), x the pre-normed layer input, one value
#     per (head, channel);
#   * projections have no bias; Q, K, V and the gate come from one fused
#     weight [W_q; W_k; W_v; W_g] of (48 + 8 + 8 + 48) * 128 rows;
#   * Q, K, V enter the attention rounded to BF16 (the activation dtype) and
#     the gated attention output is rounded to BF16 before the output
#     projection.
# ----------------------------------------------------------------------------
def rope_rotate(v, pos, theta: float = 10000.0) -> np.ndarray:
    """RoPE, rotate-half form, on the last dimension (size d) of v [..., T, d]
    for positions pos [T] (FP64)."""
    v = np.asarray(v, dtype=F64)
    d = v.shape[-1]
    half = d // 2
    inv_freq = theta ** (-np.arange(half, dtype=F64) * 2.0 / d)
    ang = np.asarray(pos, dtype=F64)[:, None] * inv_freq[None, :]
    cos, sin = np.cos(ang), np.sin(ang)
    x1, x2 = v[..., :half], v[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def global_query_scale(pos) -> np.ndarray:
    """(1 + (pos + 1) / 2048) ** 0.1 per position (FP64)."""
    return (1.0 + (np.asarray(pos, dtype=F64) + 1.0) / 2048.0) ** 0.1


def attention_core(q, k, v, window: int, q_pos=None) -> np.ndarray:
    """softmax(q k^T / sqrt(d) + mask) v per head with the causal (and, when
    window > 0, sliding-window) mask; q [nq, Tq, d] at positions q_pos
    (default 0..Tq-1), k and v [nkv, T, d] at positions 0..T-1; query head h
    reads key/value head h // (nq // nkv). FP64."""
    q, k, v = (np.asarray(a, dtype=F64) for a in (q, k, v))
    nq, Tq, d = q.shape
    T = k.shape[1]
    group = nq // k.shape[0]
    i = (np.arange(Tq) if q_pos is None else np.asarray(q_pos))[:, None]
    j = np.arange(T)[None, :]
    allowed = j <= i
    if window > 0:
        allowed &= (i - j) < window
    out = np.empty_like(q)
    for h in range(nq):
        s = q[h] @ k[h // group].T / math.sqrt(d)
        s = np.where(allowed, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        out[h] = (p / p.sum(axis=1, keepdims=True)) @ v[h // group]
    return out


def attention_forward(h_in, w_qkvg, w_o, q_gain, k_gain, *, n_q=48, n_kv=8, head_dim=128,
                      window=512, rope_theta=10000.0, eps=1e-6, pre_norm=True, pre_gain=None,
                      residual_k=0, post_gain=None, query_rows=None) -> dict:
    """The attention sublayer for one sequence of T tokens at positions 0..T-1.

    h_in [T, H] (h_{k-1}; used as x itself when pre_norm is False);
    w_qkvg [(n_q + 2 n_kv + n_q) * head_dim, H]; w_o [H, n_q * head_dim];
    q_gain, k_gain [head_dim]. window > 0: sliding layer with RoPE;
    window == 0: global layer with the query scale. query_rows: compute the
    outputs of these token rows only (keys and values of every token).
    Returns dict(x, q, k, v, gate, attn (gated, BF16-rounded), out, h) over
    the output rows."""
    h_in = np.asarray(h_in, dtype=F64)
    T, H = h_in.shape
    rows = np.arange(T) if query_rows is None else np.asarray(query_rows)
    x = bf16_round(rms_norm(h_in, pre_gain, eps)).astype(F64) if pre_norm else h_in
    w = np.asarray(w_qkvg, dtype=F64)
    dq, dkv = n_q * head_dim, n_kv * head_dim
    qg = x[rows] @ np.concatenate([w[:dq], w[dq + 2 * dkv:]]).T          # q and gate rows
    kv = x @ w[dq:dq + 2 * dkv].T
    q = qg[:, :dq].reshape(len(rows), n_q, head_dim).transpose(1, 0, 2)
    k = kv[:, :dkv].reshape(T, n_kv, head_dim).transpose(1, 0, 2)
    v = kv[:, dkv:].reshape(T, n_kv, head_dim).transpose(1, 0, 2)
    gate = sigmoid(qg[:, dq:])                                  # [rows, n_q * head_dim]
    q = rms_norm(q, q_gain, eps)
    k = rms_norm(k, k_gain, eps)
    if window > 0:
        q = rope_rotate(q, rows, rope_theta)
        k = rope_rotate(k, np.arange(T), rope_theta)
    else:
        q = q * global_query_scale(rows)[None, :, None]
    q, k, v = (bf16_round(a).astype(F64) for a in (q, k, v))
    o = attention_core(q, k, v, window, q_pos=rows)              # [n_q, rows, d]
    attn = bf16_round(o.transpose(1, 0, 2).reshape(len(rows), dq) * gate).astype(F64)
    out = attn @ np.asarray(w_o, dtype=F64).T
    hk = (residual_step(h_in[rows], out, residual_k, post_gain, eps, True)
          if residual_k else None)
    return dict(x=x, q=q, k=k, v=v, gate=gate, attn=attn, out=out, h=hk)
