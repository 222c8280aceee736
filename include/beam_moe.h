/*
 * beam_moe.h -- C ABI of the Beam MoE sublayer on one B300 (sm_103a).
 *
 * The operation, as the release pages state it:
 *   [P1] "Reflection 发布 Beam 501B 开源模型，支持 1M tokens 上下文",
 *        section 专家混合模型: sigmoid router over all experts, 8 groups of
 *        32, keep the 4 groups with the best sum of their two top scores,
 *        top-8 experts inside them, no shared expert, each expert a SwiGLU
 *        MLP (intermediate 2560), outputs combined with the normalised
 *        router weights multiplied by 2.5;
 *        section 残差流: the embedding is step 1; step k keeps the stream
 *        with weight sqrt((k-1)/k) and adds the sublayer output with weight
 *        1/sqrt(k); every sublayer is normalised before and after; router,
 *        SwiGLU product and normalisation run in FP32.
 *   [P5] "Reflection 放出 501B 的 Beam 权重：四套精度、滑动窗口和一场榜单落差",
 *        section "config.json 里还有六处能直接抄的细节": n_group 8,
 *        topk_group 4, norm_topk_prob true, routed_scaling_factor 2.5; and
 *        the FP32 router weight (the quantisers skip "mlp.gate").
 *
 * Conventions for every entry point:
 *   - All pointers are DEVICE pointers owned by the caller (inputs, outputs
 *     and workspace) unless stated otherwise. The library never allocates
 *     device memory in these calls.
 *   - Tensors are dense row-major. Weight matrices use the nn.Linear layout
 *     [out_features, in_features]. Every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *     enqueued asynchronously; nothing synchronises the host.
 *   - Argument errors are reported synchronously through the return value
 *     (nothing is enqueued then). Errors inside kernels (a bounded wait that
 *     timed out) set a per-device flag read back by beam_status().
 *   - beam_last_error_string() describes the last failure of the calling
 *     host thread.
 *   - An empty batch (T = 0) is valid everywhere: size and layout queries
 *     answer, the calls check their other arguments and return BEAM_OK
 *     without enqueuing work (pointers may then be NULL), except
 *     beam_ep_dispatch, which zeroes its send counts.
 */
#ifndef BEAM_MOE_H_
#define BEAM_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BEAM_OK = 0,
  BEAM_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misalignment, k < 2 */
  BEAM_ERR_UNSUPPORTED = 2,  /* shape outside what the kernels implement */
  BEAM_ERR_WORKSPACE = 3,    /* workspace smaller than beam_moe_workspace_size() */
  BEAM_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
  BEAM_ERR_TIMEOUT = 5,      /* a device-side bounded wait gave up */
  BEAM_ERR_DEVICE_FLAG = 6   /* another device-side error flag was set */
} beam_status_t;

/* beam_moe_params.flags */
#define BEAM_FLAG_PRE_NORM 1      /* input is h_{k-1}; RMSNorm it (FP32) into BF16 x first */
#define BEAM_FLAG_FP32_OUT 2      /* `out` is FP32 (only without the residual step) */
#define BEAM_FLAG_RETURN_SCORES 4 /* beam_moe_route also writes the sigmoid scores */
#define BEAM_FLAG_FP8_EXPERTS 8   /* workspace also holds the E4M3 activations of the
                                     FP8 expert path (beam_moe_forward_fp8 and
                                     beam_dense_mlp_forward_fp8 require this bit) */
#define BEAM_FLAG_NVFP4_EXPERTS 16 /* workspace laid out for the NVFP4 expert path
                                      (beam_*_forward_nvfp4 require this bit; it
                                      excludes BEAM_FLAG_FP8_EXPERTS) */
#define BEAM_FLAG_PREFILL_WEIGHT_MAJOR 32 /* many tokens per expert: run the expert
                                      GEMMs on the weight-major kernel with token
                                      tiles of 128 instead of the 2-SM (BF16/E4M3) or
                                      token-major (NVFP4) kernels; same results within
                                      FP32 rounding, for cross-checks (part of the
                                      workspace layout: size it with the same flags) */

/* Shape and hyper-parameters of one MoE sublayer call.
 *   T           tokens in the batch (0 is allowed: nothing is enqueued)
 *   H           hidden size (5120 for Beam); multiple of 128, at most 8192
 *   E           experts (256 for Beam); multiple of 32, at most 256
 *   I           expert SwiGLU intermediate size (2560); multiple of 128
 *   n_group     expert groups (8); E / n_group must be 32, or n_group must equal
 *               topk_group (all groups kept: plain top-k)
 *   topk_group  groups kept per token (4)
 *   top_k       experts per token (8); 1..32 and <= topk_group * E / n_group
 *   routed_scale  factor on the normalised weights (2.5)
 *   rms_eps     RMSNorm epsilon (1e-6)
 *   residual_k  0: no residual step (out = combined MoE output); >= 2: the
 *               step index k of the scaled residual update; out = h_k
 *   flags       BEAM_FLAG_* bits
 */
typedef struct {
  int T, H, E, I, n_group, topk_group, top_k;
  float routed_scale;
  float rms_eps;
  int residual_k;
  int flags;
} beam_moe_params;

/* Bytes of device workspace that beam_moe_route / beam_moe_forward need for
 * these parameters (0 when the parameters are invalid; see
 * beam_last_error_string()). The same workspace may be reused by successive
 * calls on one stream; calls that overlap in time need separate workspaces. */
size_t beam_moe_workspace_size(const beam_moe_params* p);

/* Router only ([P1] 专家混合模型; [P5] config fields).
 *   x          [T,H] bf16: layer input (h_{k-1} when BEAM_FLAG_PRE_NORM)
 *   w_router   [E,H] fp32 router weight
 *   logit_bias [E] fp32 added to the logits before the sigmoid, or NULL
 *   pre_gain   [H] fp32 gain of the pre-norm, or NULL (= 1); used only
 *              with BEAM_FLAG_PRE_NORM
 *   topk_idx   [T,top_k] int32 out: selected experts, by descending score,
 *              ties to the lower expert index
 *   topk_w     [T,top_k] fp32 out: routed_scale * s / (sum of the selected s)
 *   scores     [T,E] fp32 out (sigmoid scores) when BEAM_FLAG_RETURN_SCORES,
 *              else ignored (may be NULL)
 * Scores are FP32: logits accumulate x (bf16 -> fp32) times w_router in FP32
 * (for T >= 512 and E == 256 on the tensor cores, with w_router split
 * exactly into three BF16 pieces so every product is exact in FP32).
 * Group score = FP32 sum of the group's two largest scores; groups rank by
 * it (ties to the lower group index). */
beam_status_t beam_moe_route(const beam_moe_params* p, const void* x,
                             const float* w_router, const float* logit_bias,
                             const float* pre_gain, int32_t* topk_idx, float* topk_w,
                             float* scores, void* workspace, size_t workspace_bytes,
                             void* stream);

/* The whole MoE sublayer ([P1] 专家混合模型 and 残差流):
 *   x = BEAM_FLAG_PRE_NORM ? bf16(RMSNorm(x_in) * pre_gain) : x_in
 *   route x (as beam_moe_route)
 *   y_e = (silu(x W_gate[e]^T) * (x W_up[e]^T)) W_down[e]^T for each selected
 *         expert, BF16 operands, FP32 accumulation, SwiGLU product in FP32,
 *         the intermediate rounded to BF16 before the down projection
 *   o   = sum_j topk_w[t,j] * y_{topk_idx[t,j]}   (FP32 expert outputs summed in
 *         FP32 by the down projection's epilogue with L2 reductions, in an order
 *         that varies from run to run)
 *   out = residual_k >= 2 ? bf16(sqrt((k-1)/k) x_in + RMSNorm(o) * post_gain / sqrt(k))
 *                         : o (bf16, or fp32 with BEAM_FLAG_FP32_OUT)
 * Arguments:
 *   x_in       [T,H] bf16
 *   w_router   [E,H] fp32;  logit_bias [E] fp32 or NULL
 *   w_gate     [E,I,H] bf16; w_up [E,I,H] bf16; w_down [E,H,I] bf16
 *   pre_gain   [H] fp32 or NULL (= 1);  post_gain [H] fp32 or NULL (= 1)
 *   out        [T,H] bf16 (fp32 with BEAM_FLAG_FP32_OUT); must not alias x_in
 *   topk_idx, topk_w  optional outputs as in beam_moe_route (NULL: kept in the
 *              workspace)
 * Token-to-expert order inside the workspace is stable (by token, then slot).
 * Routing (topk_idx, topk_w) is bit-reproducible; o is reproducible to FP32
 * rounding (the order of the 8 additions varies), so an output element can
 * differ by one BF16 rounding step between runs. */
beam_status_t beam_moe_forward(const beam_moe_params* p, const void* x_in,
                               const float* w_router, const float* logit_bias,
                               const void* w_gate, const void* w_up, const void* w_down,
                               const float* pre_gain, const float* post_gain, void* out,
                               int32_t* topk_idx, float* topk_w, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Dense SwiGLU MLP sublayer of the first layers ([P1] 专家混合模型: the first 3
 * of the 52 layers use a dense SwiGLU MLP instead of the experts; 残差流: normalised
 * before and after, scaled residual). The pages do not give its intermediate
 * size, so I is a parameter.
 *   T, H, I     tokens, hidden (multiple of 128, at most 8192), intermediate
 *               (multiple of 128)
 *   rms_eps, residual_k, flags  as in beam_moe_params (flags: PRE_NORM,
 *               FP32_OUT, FP8_EXPERTS, NVFP4_EXPERTS, PREFILL_WEIGHT_MAJOR)
 */
typedef struct {
  int T, H, I;
  float rms_eps;
  int residual_k;
  int flags;
} beam_dense_params;

/* Workspace bytes for beam_dense_mlp_forward (0 on invalid parameters). */
size_t beam_dense_workspace_size(const beam_dense_params* p);

/* Byte offsets of the dense MLP's workspace buffers, in the order and with
 * the meaning of beam_moe_workspace_layout (one expert, top_k = 1). Writes
 * min(n, 25) entries and returns how many it wrote (0 on invalid
 * parameters). Diagnostic. */
int beam_dense_workspace_layout(const beam_dense_params* p, size_t* offsets, int n);

/*   x = BEAM_FLAG_PRE_NORM ? bf16(RMSNorm(x_in) * pre_gain) : x_in
 *   y = (silu(x W_gate^T) * (x W_up^T)) W_down^T  (BF16 operands, FP32
 *       accumulation, SwiGLU product in FP32 rounded to BF16)
 *   out = residual_k >= 2 ? bf16(sqrt((k-1)/k) x_in + RMSNorm(y) * post_gain / sqrt(k))
 *                         : y (bf16, or fp32 with BEAM_FLAG_FP32_OUT)
 *   x_in [T,H] bf16; w_gate, w_up [I,H] bf16; w_down [H,I] bf16;
 *   pre_gain, post_gain [H] fp32 or NULL; out [T,H]. Runs on the same expert
 *   GEMM kernels as beam_moe_forward, as one expert that every token uses. */
beam_status_t beam_dense_mlp_forward(const beam_dense_params* p, const void* x_in,
                                     const void* w_gate, const void* w_up, const void* w_down,
                                     const float* pre_gain, const float* post_gain, void* out,
                                     void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) expert weights.
 * [P5] section 四套权重的账，自己算一遍: the FP8 checkpoint stores every linear
 * weight except lm_head, the embedding and the router ("mlp.gate") as
 * F8_E4M3, a dynamic FP8 quantisation; [P1] 专家混合模型 lists the FP8
 * checkpoint beside the BF16 one. The pages fix neither the scale
 * granularity nor the rounding; this library takes one FP32 scale per row:
 *   amax = max_j |v_j|;  scale = amax / 448;  inv = 448 / amax  (FP32 IEEE
 *   division; scale = inv = 1 for an all-zero row)
 *   code_j = E4M3(v_j * inv)  (FP32 product, round to nearest even, saturate
 *                              at +-448; E4M3 = OCP E4M3FN: bias 7,
 *                              subnormals, no infinities)
 * and dequantises a row as E4M3 value * scale. Weights carry one scale per
 * output row (static); activations are quantised per row at run time.
 * ------------------------------------------------------------------------- */

/* Row quantiser: q[r,:] = E4M3 codes of src[r,:], scale[r] as above.
 *   src    [rows, K] bf16 (device);  q [rows, K] uint8 out;  scale [rows] fp32 out
 *   K      multiple of 16; rows >= 0 (0: nothing is enqueued)
 * Used once to quantise expert weights: for W_gate / W_up [E,I,H] call it
 * with rows = E*I, K = H; for W_down [E,H,I] with rows = E*H, K = I. */
beam_status_t beam_quantize_e4m3_rows(const void* src, long long rows, int K, void* q,
                                      float* scale, void* stream);

/* The MoE sublayer with E4M3 expert weights. As beam_moe_forward except:
 *   x (BF16, after the optional pre-norm) is quantised per token;
 *   g = (sx q_x) . (s_g q_g)^T, u likewise, on the E4M3 tensor cores with FP32
 *   accumulation, the scales applied to the FP32 accumulators;
 *   A = bf16(silu(g) * u) is quantised per (token, expert) row;
 *   y_e = (sa q_A) . (s_d q_d)^T; combine, post-norm and residual as in
 *   beam_moe_forward. The router is unquantised (FP32 weight, FP32 scores).
 * Arguments as beam_moe_forward, with each expert weight given as codes and
 * row scales:
 *   wq_gate, wq_up [E,I,H] uint8;  ws_gate, ws_up [E*I] fp32
 *   wq_down [E,H,I] uint8;         ws_down [E*H] fp32
 * p->flags must include BEAM_FLAG_FP8_EXPERTS (and the workspace must be
 * sized with it). */
beam_status_t beam_moe_forward_fp8(const beam_moe_params* p, const void* x_in,
                                   const float* w_router, const float* logit_bias,
                                   const void* wq_gate, const float* ws_gate,
                                   const void* wq_up, const float* ws_up,
                                   const void* wq_down, const float* ws_down,
                                   const float* pre_gain, const float* post_gain, void* out,
                                   int32_t* topk_idx, float* topk_w, void* workspace,
                                   size_t workspace_bytes, void* stream);

/* The dense SwiGLU MLP with E4M3 weights (the FP8 checkpoint quantises the
 * dense layers too): as beam_dense_mlp_forward with x quantised per token
 * and A per token, as in beam_moe_forward_fp8.
 *   wq_gate, wq_up [I,H] uint8, ws_gate, ws_up [I] fp32;
 *   wq_down [H,I] uint8, ws_down [H] fp32.
 * p->flags must include BEAM_FLAG_FP8_EXPERTS. */
beam_status_t beam_dense_mlp_forward_fp8(const beam_dense_params* p, const void* x_in,
                                         const void* wq_gate, const float* ws_gate,
                                         const void* wq_up, const float* ws_up,
                                         const void* wq_down, const float* ws_down,
                                         const float* pre_gain, const float* post_gain,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         void* stream);

/* ---------------------------------------------------------------------------
 * NVFP4 expert weights.
 * [P5] section 四套权重的账，自己算一遍: the NVFP4 checkpoint packs every
 * routed-expert weight as two 4-bit values per byte (its U8 count is half
 * the expert parameters) and keeps the rest in BF16; section 上手前的五个坑:
 * NVFP4 is packed by modelopt and runs on the FP4 tensor-core path. The
 * pages fix neither block size nor scale types; this library reads them as:
 *   elements E2M1 (0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives), two per byte,
 *   the even element in the low nibble; one E4M3 block scale per 16
 *   elements along K; one FP32 scale per group of rows (an expert matrix
 *   for weights, one row for activations). In FP32 with IEEE division:
 *     g = amax_group / 2688;  s_b = E4M3(amax_b / (6 g));
 *     q_i = E2M1(v_i * (1 / (s_b g)))   (round to nearest even, saturating;
 *                                        q = 0 where s_b = 0)
 *   and v is dequantised as E2M1(q) * s_b * g.
 * Block-scale layout ("SF groups"): one 512-byte group per 128-row tile and
 * K = 64 step, group index (r / 128) * (K / 64) + k / 64, byte
 * (r % 32) * 16 + ((r % 128) / 32) * 4 + (k % 64) / 16. A matrix of R rows
 * (R a multiple of 128) and K columns has R * K / 16 bytes of scales.
 * ------------------------------------------------------------------------- */

/* NVFP4 quantiser: rows x K bf16 (device) -> codes [rows, K/2] uint8, block
 * scales [rows * K / 16] uint8 in the SF-group layout above, group scales
 * [rows / rows_per_group] fp32. rows must be a multiple of 128 and of
 * rows_per_group, K a multiple of 64. Expert weights: W_gate / W_up [E,I,H]
 * with rows = E*I, K = H, rows_per_group = I (one scale per expert matrix);
 * W_down [E,H,I] with rows = E*H, K = I, rows_per_group = H. */
beam_status_t beam_quantize_nvfp4(const void* src, long long rows, int K, int rows_per_group,
                                  void* codes, void* block_scales, float* group_scales,
                                  void* stream);

/* The MoE sublayer with NVFP4 expert weights: as beam_moe_forward_fp8 with
 * E4M3 replaced by NVFP4 -- x quantised per token, the BF16 SwiGLU output per
 * (token, expert) row, the FP4 tensor cores (kind::mxf4nvf4 with the E4M3
 * block scales) accumulating in FP32, group scales applied to the FP32
 * accumulators. Each expert weight is (codes, block scales, per-expert FP32
 * scale) as beam_quantize_nvfp4 writes them:
 *   wq_gate, wq_up [E,I,H/2] uint8; wsf_gate, wsf_up [E*I*H/16] uint8;
 *   wg_gate, wg_up [E] fp32; wq_down [E,H,I/2]; wsf_down [E*H*I/16];
 *   wg_down [E]. H and I must be multiples of 256; p->flags must include
 * BEAM_FLAG_NVFP4_EXPERTS. */
beam_status_t beam_moe_forward_nvfp4(const beam_moe_params* p, const void* x_in,
                                     const float* w_router, const float* logit_bias,
                                     const void* wq_gate, const void* wsf_gate, const float* wg_gate,
                                     const void* wq_up, const void* wsf_up, const float* wg_up,
                                     const void* wq_down, const void* wsf_down, const float* wg_down,
                                     const float* pre_gain, const float* post_gain, void* out,
                                     int32_t* topk_idx, float* topk_w, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* The dense SwiGLU MLP with NVFP4 weights (one expert: the group scales are
 * one float each). p->flags must include BEAM_FLAG_NVFP4_EXPERTS. */
beam_status_t beam_dense_mlp_forward_nvfp4(const beam_dense_params* p, const void* x_in,
                                           const void* wq_gate, const void* wsf_gate,
                                           const float* wg_gate, const void* wq_up,
                                           const void* wsf_up, const float* wg_up,
                                           const void* wq_down, const void* wsf_down,
                                           const float* wg_down, const float* pre_gain,
                                           const float* post_gain, void* out, void* workspace,
                                           size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * Attention sublayer ([P1] section 注意力: 52 layers, hidden 5120; sliding
 * window of 512 tokens on most layers with RoPE, full context on every sixth
 * layer and the last with each query multiplied by (1 + (pos+1)/2048)^0.1;
 * grouped-query attention, 48 query heads and 8 key/value heads, RMSNorm on
 * queries and keys; a sigmoid gate computed from the layer input scales every
 * head channel before the output projection. [P1] 残差流: normalised before
 * and after, the scaled residual step, RoPE and the query scaling in FP32.
 * [P5] config.json: head_dim 128, sliding_window 512, rope_theta 10000.)
 * One sequence of T tokens at positions 0..T-1 (prefill):
 *   x      = PRE_NORM ? bf16(RMSNorm(h_in) * pre_gain) : h_in
 *   [q|k|v|g] = x W_qkvg^T   (FP32 accumulation)
 *   q, k   = RMSNorm over each head's 128 channels * q_gain / k_gain (FP32),
 *            then RoPE (rotate-half, theta^(-2i/128), window > 0) or, for
 *            window == 0, q *= (1 + (t+1)/2048)^0.1; q, k, v rounded to BF16
 *   o_h    = softmax(q_h k_{h/(nq/nkv)}^T / sqrt(128) + mask) v_{h/(nq/nkv)},
 *            mask: causal, and 0 <= i - j < window when window > 0
 *   a      = bf16(o * sigmoid(g))   (per head and channel)
 *   y      = a W_o^T                (FP32)
 *   out    = residual_k >= 2 ? bf16(sqrt((k-1)/k) h_in + RMSNorm(y) * post_gain / sqrt(k))
 *                            : y (bf16, or fp32 with BEAM_FLAG_FP32_OUT)
 * ------------------------------------------------------------------------- */
typedef struct {
  int T;            /* tokens of the sequence (>= 0) */
  int H;            /* hidden size (5120); multiple of 256, at most 8192 */
  int n_q, n_kv;    /* query / key-value heads (48 / 8); n_q % n_kv == 0, n_q + n_kv even */
  int head_dim;     /* 128 (the only supported value) */
  int window;       /* sliding window (512), or 0 for a global layer */
  float rope_theta; /* 10000 */
  float rms_eps;    /* 1e-6 */
  int residual_k;   /* 0 (no residual) or the step k >= 2 */
  int flags;        /* BEAM_FLAG_PRE_NORM, BEAM_FLAG_FP32_OUT */
} beam_attn_params;

/* Workspace bytes for beam_attention_forward (0 on invalid parameters). */
size_t beam_attention_workspace_size(const beam_attn_params* p);

/* Byte offsets of the attention workspace buffers (diagnostic): 0 pre-normed
 * x [T,H] bf16, 1 fused projection [T,(2nq+2nkv)*128] fp32, 2 Q [nq][Tp][128]
 * bf16, 3 K [nkv][Tp][128] bf16, 4 V transposed [nkv][128][Tp] bf16, 5 RoPE
 * (cos, sin) table [T][64] fp32 pairs (sliding-window layers; empty for
 * global ones; the gate logits are read from the fused projection), 6 gated
 * attention output [T][nq*128] bf16, 7 output projection [T,H] fp32, 8-10
 * GEMM work lists and counts; Tp = T rounded up to 128. Writes min(n, 11)
 * entries and returns how many it wrote. */
int beam_attention_workspace_layout(const beam_attn_params* p, size_t* offsets, int n);

/* Arguments (device pointers, 16-byte aligned):
 *   h_in    [T,H] bf16
 *   w_qkvg  [(2 n_q + 2 n_kv) * 128, H] bf16: rows W_q (n_q*128), W_k, W_v
 *           (n_kv*128 each), W_g (n_q*128)
 *   w_o     [H, n_q * 128] bf16
 *   q_gain, k_gain [128] fp32 or NULL (= 1); pre_gain, post_gain [H] fp32 or NULL
 *   out     [T,H] bf16 (fp32 with BEAM_FLAG_FP32_OUT); must not alias h_in */
beam_status_t beam_attention_forward(const beam_attn_params* p, const void* h_in,
                                     const void* w_qkvg, const void* w_o, const float* q_gain,
                                     const float* k_gain, const float* pre_gain,
                                     const float* post_gain, void* out, void* workspace,
                                     size_t workspace_bytes, void* stream);

/* One scaled residual update ([P1] 残差流):
 *   h_out = bf16( sqrt((k-1)/k) * h_prev + (1/sqrt(k)) * n ),
 *   n = apply_norm ? RMSNorm(sub_out) * post_gain : sub_out   (FP32 math)
 *   h_prev  [T,H] bf16;  sub_out [T,H] bf16, or fp32 when sub_out_is_fp32
 *   post_gain [H] fp32 or NULL (= 1);  k >= 2 (the embedding is step 1)
 *   h_out   [T,H] bf16; may alias h_prev (each element is read before it is
 *           written by the same thread) but not sub_out.
 * H must be a multiple of 8. */
beam_status_t beam_residual_step(const void* h_prev, const void* sub_out, int T, int H,
                                 int k, const float* post_gain, float eps, int apply_norm,
                                 int sub_out_is_fp32, void* h_out, void* stream);

/* Synchronises `stream`, then reads and clears the calling device's error
 * flag: BEAM_OK, BEAM_ERR_TIMEOUT or BEAM_ERR_DEVICE_FLAG (or BEAM_ERR_CUDA
 * if the synchronisation itself failed). */
beam_status_t beam_status(void* stream);

/* Human-readable description of the calling thread's last failure. The
 * string stays valid until the next call on the same thread. */
const char* beam_last_error_string(void);

/* Router for callers that cannot allocate device memory.
 *
 * The pages have no counterpart to this entry point: it is an interface
 * choice of this library. Some programs that call the router cannot allocate:
 * hosts that hand all of a GPU's memory to their own pool at start-up and
 * forbid further cudaMalloc, and plug-ins inside such hosts that are given
 * no allocator and no workspace. beam_moe_route needs a caller workspace;
 * this variant needs none and allocates nothing (no cudaMalloc, cudaFree or
 * allocating library call). Its scratch -- the router's partial logits and,
 * with BEAM_FLAG_PRE_NORM, the normalised x -- is a fixed array of
 * BEAM_ROUTE_STATIC_SCRATCH_BYTES inside the library, which every GPU that
 * loads the library holds until the process exits.
 *
 * Arguments, results and errors are those of beam_moe_route (same kernels,
 * same K-slicing, so the results are identical), without the workspace.
 * Scratch needed: KS*T*E*4 bytes (rounded up to 256) for the partial logits,
 * where KS is the number of K-slices the router uses for this T (many for a
 * few tokens, one for thousands), plus T*H*2 bytes with BEAM_FLAG_PRE_NORM,
 * plus E*3H*2 bytes for the split router weight and its work list when the
 * router runs on the tensor cores (T >= 512). A call needing more returns
 * BEAM_ERR_UNSUPPORTED with a message that gives the bytes needed; nothing is
 * enqueued then. For the Beam shapes (H=5120, E=256, 148 SMs) that allows
 * T <= 409 with pre-norm and T <= 511 without.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it with the
 * ID of the device's context; a call that finds a different context current
 * (after a cudaDeviceReset, for instance) looks the address up again. Make
 * the first call on a device, and the first after a reset, before any stream
 * capture. All calls on a device share the one
 * array and it keeps the last call's contents; every call writes each scratch
 * byte it later reads, so nothing needs clearing between calls. Calls whose
 * work overlaps on the GPU (other streams, other host threads) race on the
 * array: the caller must order them. */
#define BEAM_ROUTE_STATIC_SCRATCH_BYTES (8u << 20)
beam_status_t beam_moe_route_static(const beam_moe_params* p, const void* x,
                                    const float* w_router, const float* logit_bias,
                                    const float* pre_gain, int32_t* topk_idx, float* topk_w,
                                    float* scores, void* stream);

/* ---------------------------------------------------------------------------
 * Expert parallelism ([P1] section 多 GPU 和多节点: each expert lives on one
 * device and the device count divides the 256 experts; [P1] 专家混合模型 and
 * 残差流 for what each step computes). P ranks, rank d owning experts
 * [d E/P, (d+1) E/P). A rank routes its own tokens (beam_moe_route; the
 * router weight is replicated), beam_ep_dispatch orders the token-expert
 * pairs for sending, the caller exchanges them (an all-to-all of its own
 * choosing), each owner runs beam_moe_forward_routed on the rows it
 * received, the outputs travel back in the same order, and beam_ep_combine
 * finishes the sublayer on the source rank.
 * ------------------------------------------------------------------------ */

/* The sublayer with the routing given instead of computed: the permutation,
 * the expert GEMMs, the weighted combine and the output or post-norm +
 * residual of beam_moe_forward, for BF16 experts.
 *   p          T rows ("tokens"), E = the experts in w_gate/w_up/w_down,
 *              top_k slots per row; flags PRE_NORM / FP32_OUT as in
 *              beam_moe_forward (FP8_EXPERTS and NVFP4_EXPERTS are refused)
 *   x_in       [T,H] bf16 (normalised first with BEAM_FLAG_PRE_NORM)
 *   topk_idx   [T,top_k] int32 expert of each slot, in [0, E); an index
 *              outside it sets the device error flag (BEAM_ERR_DEVICE_FLAG
 *              from beam_status) and its slot is dropped
 *   topk_w     [T,top_k] fp32 combine weight of each slot
 *   the rest as in beam_moe_forward; workspace: beam_moe_workspace_size(p).
 * An expert owner calls it with its received rows, their local expert ids,
 * weights 1, top_k = 1, BEAM_FLAG_FP32_OUT and no residual: out[r] is then
 * the FP32 output of row r's expert. */
beam_status_t beam_moe_forward_routed(const beam_moe_params* p, const void* x_in,
                                      const int32_t* topk_idx, const float* topk_w,
                                      const void* w_gate, const void* w_up, const void* w_down,
                                      const float* pre_gain, const float* post_gain, void* out,
                                      void* workspace, size_t workspace_bytes, void* stream);

/* Orders a rank's token-expert pairs for sending: by expert (so by owning
 * rank), stable by pair p = t*top_k + j.
 *   p          the layer (T, H, E, I, top_k as for beam_moe_route);
 *              n_ranks divides E
 *   x          [T,H] bf16 rows to send (the normalised x when the layer
 *              pre-norms: beam_moe_route writes it to workspace entry 0)
 *   topk_idx   [T,top_k] int32 global expert ids, in [0, E)
 *   send_x     [T*top_k,H] bf16 out: x of each pair, in send order
 *   send_expert [T*top_k] int32 out: global expert of each sent row
 *   pair_row   [T*top_k] int32 out: send position of pair p
 *   send_counts [n_ranks] int32 out: rows for each rank (contiguous blocks
 *              in rank order)
 *   workspace  beam_moe_workspace_size(p) bytes (may be the router's)
 * Device pointers; asynchronous on `stream`. With T = 0 the call only
 * zeroes send_counts (when it is given). */
beam_status_t beam_ep_dispatch(const beam_moe_params* p, int n_ranks, const void* x,
                               const int32_t* topk_idx, void* send_x, int32_t* send_expert,
                               int32_t* pair_row, int32_t* send_counts, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Finishes the sublayer on the source rank from the expert outputs returned
 * in send order:
 *   o[t]  = sum_j topk_w[t,j] * recv_y[pair_row[t*top_k+j]]   (FP32, slot order)
 *   out[t] = residual_k >= 2 ? bf16(sqrt((k-1)/k) h_prev[t] + RMSNorm(o[t]) * post_gain / sqrt(k))
 *                            : o[t] (bf16, or fp32 when out_f32)
 *   recv_y [T*top_k,H] fp32; pair_row [T*top_k] int32 (from beam_ep_dispatch);
 *   topk_w [T,top_k] fp32; h_prev [T,H] bf16 (the layer input, with the
 *   residual); post_gain [H] fp32 or NULL; H a multiple of 128, at most 8192. */
beam_status_t beam_ep_combine(int T, int top_k, int H, const float* recv_y,
                              const int32_t* pair_row, const float* topk_w, const void* h_prev,
                              const float* post_gain, float eps, int residual_k, int out_f32,
                              void* out, void* stream);

/* ---- diagnostics (tests and tooling) ---------------------------------- */

/* Byte offsets of the internal buffers inside the forward workspace, in this
 * order: 0 normalised x [T,H] bf16, 1 router partial logits, 2 topk_idx,
 * 3 topk_w, 4 expert counts [E] int32, 5 expert offsets [E+1] int32,
 * 6 row_token [T*top_k] int32, 7 row_weight [T*top_k] fp32, 8 permuted x
 * [T*top_k,H] bf16, 9 SwiGLU activations [T*top_k,I] bf16, 10 the combined
 * expert output o [T,H] fp32 (the down projection's epilogue adds into it),
 * 11 unit counts [4] int32, 12 per-block
 * expert histograms, 13 per-block expert offsets, 14 gate/up work list,
 * 15 down work list, 16 pair -> row map [T*top_k] int32, 17 the router
 * weight split into three BF16 pieces [E, 3H], 18 the router GEMM's work
 * list (tensor-core router only), and with BEAM_FLAG_FP8_EXPERTS or
 * BEAM_FLAG_NVFP4_EXPERTS: 19 scales of the quantised x [rows] fp32 (the
 * quantised x itself occupies entry 8), 20 E4M3 / NVFP4 activation codes,
 * 21 their row scales [rows] fp32; with BEAM_FLAG_NVFP4_EXPERTS also 22 the
 * block scales of x and 23 those of the activations (the SF-group layout
 * with token tiles of 32 or 128 rows -- the GEMM's token tile -- in place
 * of 128-row weight tiles: group (r / tile) * (K / 64) + k / 64, byte
 * (r % 32) * 16 + ((r % tile) / 32) * 4 + (k % 64) / 16); 24 the combine's
 * per-token arrival counters [T] int32, followed by its completion list [T]
 * int32 and two int32 cursors.
 * Row-indexed buffers (6-9, 19-23) hold rows = T*top_k rows, or with NVFP4
 * every expert's rows padded to the token tile (32 or 128). Writes
 * min(n, 25) entries and returns how many it wrote (0 on invalid
 * parameters). */
int beam_moe_workspace_layout(const beam_moe_params* p, size_t* offsets, int n);

/* Launches one block whose single thread waits on a shared-memory barrier
 * that nothing ever completes, with the same bounded wait the GEMM kernels
 * use, giving up after `timeout_ns`. The device error flag then reads
 * BEAM_ERR_TIMEOUT through beam_status(). Used to test the failure path
 * without hanging or faulting the GPU. */
beam_status_t beam_debug_wait_timeout(uint64_t timeout_ns, void* stream);

/* Per-kernel timing. While enabled (on != 0), every kernel launch of this
 * library is bracketed by two CUDA events recorded on its stream. */
void beam_profile_enable(int on);

/* Synchronises the recorded events and returns, per kernel name, the total
 * elapsed milliseconds and the launch count since the last read; then
 * clears the record. `names` receives the names separated by newlines (at
 * most names_len bytes, NUL-terminated); total_ms and launches receive up to
 * max_entries values in the same order. Returns the number of entries. */
int beam_profile_read(char* names, size_t names_len, double* total_ms, int* launches,
                      int max_entries);

#ifdef __cplusplus
}
#endif
#endif /* BEAM_MOE_H_ */
