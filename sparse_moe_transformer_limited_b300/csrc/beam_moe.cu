// Host side of the C ABI declared in include/beam_moe.h: argument checks,
// workspace layout, TMA descriptors and kernel launches. Nothing here
// allocates device memory; all buffers are the caller's.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <utility>
#include <string>
#include <vector>

#include "beam_moe.h"
#include "kernels_attn.cuh"
#include "kernels_combine.cuh"
#include "kernels_ep.cuh"
#include "kernels_gemm.cuh"
#include "kernels_gemm_tm.cuh"
#include "kernels_gemm_wide.cuh"
#include "kernels_gemm_2sm.cuh"
#include "kernels_permute.cuh"
#include "kernels_quant.cuh"
#include "kernels_router.cuh"
#include "kernels_rows.cuh"

namespace {

thread_local std::string t_last_error;

beam_status_t fail(beam_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return s;
}

#define BEAM_CUDA_TRY(expr)                                                              \
  do {                                                                                   \
    cudaError_t e_ = (expr);                                                             \
    if (e_ != cudaSuccess)                                                               \
      return fail(BEAM_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_));        \
  } while (0)

#define BEAM_LAUNCH_CHECK(what)                                                          \
  do {                                                                                   \
    cudaError_t e_ = cudaGetLastError();                                                 \
    if (e_ != cudaSuccess)                                                               \
      return fail(BEAM_ERR_CUDA, "launch of %s failed: %s", what, cudaGetErrorString(e_)); \
  } while (0)

constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per wait

// ------------------------------------------------------------ profiling
// When enabled, every launch is bracketed by two CUDA events recorded on the
// launching stream; beam_profile_read() aggregates their elapsed times.
struct ProfRec {
  const char* name;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof_recs;
std::vector<cudaEvent_t> g_prof_pool;

cudaEvent_t prof_event() {
  if (!g_prof_pool.empty()) {
    cudaEvent_t e = g_prof_pool.back();
    g_prof_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return e;
}

struct ProfScope {
  bool on = false;
  ProfRec rec{};
  cudaStream_t st;
  ProfScope(const char* name, cudaStream_t s) : st(s) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (!g_prof_on) return;
    rec.name = name;
    rec.start = prof_event();
    rec.stop = prof_event();
    if (rec.start && rec.stop && cudaEventRecord(rec.start, st) == cudaSuccess) on = true;
  }
  ~ProfScope() {
    if (!on) return;
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (cudaEventRecord(rec.stop, st) == cudaSuccess) g_prof_recs.push_back(rec);
  }
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------ tiles
// Expert-GEMM path, chosen from the mean tokens per expert:
//  few tokens per expert (decode): weights as the M=128 operand, token tiles
//    of 32 (expert_gemm_kernel);
//  many tokens, BF16 / E4M3 experts with H and I multiples of 256: both
//    GEMMs on the wide 2-SM kernel (expert_gemm_wide_kernel);
//  many tokens, NVFP4 experts with H, I % 256 == 0: both GEMMs on the
//    token-major two-CTA kernel (expert_gemm_tm_kernel);
//  otherwise, or with BEAM_FLAG_PREFILL_WEIGHT_MAJOR: weights as M with token
//    tiles of 128 (expert_gemm_kernel).
enum GemmPath { PATH_W32 = 0, PATH_W128 = 1, PATH_TM = 2, PATH_WIDE = 3 };

GemmPath choose_path(const beam_moe_params& p) {
  const long long pairs = static_cast<long long>(p.T) * p.top_k;
  if (pairs <= 24LL * p.E) return PATH_W32;
  if (p.flags & BEAM_FLAG_PREFILL_WEIGHT_MAJOR) return PATH_W128;
  if (p.flags & BEAM_FLAG_NVFP4_EXPERTS)
    return (p.H % 256 == 0 && p.I % 256 == 0) ? PATH_TM : PATH_W128;
  return (p.H % 256 == 0 && p.I % 256 == 0) ? PATH_WIDE : PATH_W128;
}

int path_nt(GemmPath g) { return g == PATH_W32 ? 32 : (g == PATH_W128 ? 128 : 256); }
// Weight rows per unit of the weight-major down GEMM on 32-token tiles.
int w32_down_rows(bool f4) {
  return f4 ? beam::UnitRows<1, 32, beam::KIND_NVFP4>::value : beam::UnitRows<1, 32, beam::KIND_BF16>::value;
}
int path_mt_down(GemmPath g, int H, bool f4) {
  if (g == PATH_WIDE) return (H + 511) / 512;
  if (g == PATH_TM) return H / 256;
  return g == PATH_W32 ? H / w32_down_rows(f4) : H / 128;
}
// Arrivals that complete one token in the fused combine of the down GEMM:
// every (expert of the token, hidden slice, epilogue warp or lane group) adds
// its share once. Weight-major: four warps per unit (of 128 or 256 hidden
// rows); wide: eight warps (64 hidden rows each, 32 in a last half slice) per
// slice of 512 rows; token-major: two warps of 128 hidden columns per
// 256-column tile.
int combine_expected(GemmPath g, int H, int top_k, bool f4) {
  const int per_expert = g == PATH_WIDE ? 8 * ((H + 511) / 512)
                         : (g == PATH_TM ? H / 128 : 4 * path_mt_down(g, H, f4));
  return top_k * per_expert;
}

// Router logits path: the tensor cores (exact three-way BF16 split of the
// FP32 weight, FP32 accumulation) once there are enough tokens to fill the
// GPU, else the FP32 SIMT kernel with K-slices.
bool router_on_tensor_cores(const beam_moe_params& p) { return p.T >= 512 && p.E == 256; }
constexpr int kRouterKSplit = 2;  // K-slices of the tensor-core router GEMM

// K-slices of the router logits GEMM: enough blocks to cover the SMs when T
// is small. Must divide H / 32 and leave at least 64 columns per slice.
int choose_router_ks(const beam_moe_params& p, int num_sms) {
  if (router_on_tensor_cores(p)) return kRouterKSplit;
  // (an empty batch has no tiles; count one so the split is defined)
  const int tiles = std::max(1, ((p.T + beam::RL_BT - 1) / beam::RL_BT) *
                                    ((p.E + beam::RL_BE - 1) / beam::RL_BE));
  const int want = (2 * num_sms + tiles - 1) / tiles;
  const int nk = p.H / 32;
  int best = 1;
  for (int ks = 1; ks <= nk; ++ks)
    if (nk % ks == 0 && ks <= want && (p.H / ks) >= 64) best = ks;
  return best;
}

constexpr int kLayoutEntries = 25;

struct Layout {
  size_t off[kLayoutEntries];
  // rows of the expert-ordered layout: T * top_k, or with NVFP4 experts every
  // expert's rows padded to a multiple of `pad` (the token tile), so each
  // tile starts at a multiple of 32 inside its 128-row block-scale tile
  long long rows;
  int pad;
  size_t total;
  int KS, NB, NT;
  GemmPath path;
  bool f4;          // NVFP4 experts
  long long units_gu_max, units_dn_max;
};

enum {
  L_XN = 0, L_PART, L_IDX, L_W, L_COUNTS, L_OFFS, L_ROWTOK, L_ROWW, L_XPERM, L_ACT, L_OACC,
  L_NUNITS, L_BLKHIST, L_BLKOFF, L_UGU, L_UDN, L_PAIRROW, L_WR3, L_RUNITS,
  L_XSCALE, L_ACTQ, L_ASCALE, L_XSF, L_ASF, L_ARRIVE
};

// Bytes of the router's unit list and count (tensor-core router only).
size_t router_units_bytes(const beam_moe_params& p) {
  return static_cast<size_t>(kRouterKSplit) * ((p.T + 255) / 256) * 16 + 16;
}

// Opt kernel `fn` into `bytes` of dynamic shared memory on the current
// device. The attribute belongs to the (kernel, device) pair, so it is set
// once per pair, under a lock (launches may come from several host threads).
beam_status_t ensure_smem(const void* fn, int bytes) {
  static std::mutex mu;
  static std::set<std::pair<const void*, int>> done;
  int dev = 0;
  BEAM_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(mu);
  if (done.count({fn, dev}) != 0) return BEAM_OK;
  BEAM_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes));
  done.insert({fn, dev});
  return BEAM_OK;
}

int sm_count() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
  } else {
    cudaGetLastError();
  }
  return n;
}

beam_status_t check_params(const beam_moe_params* p) {
  if (p == nullptr) return fail(BEAM_ERR_INVALID_ARG, "params is NULL");
  if (p->T < 0 || p->H <= 0 || p->E <= 0 || p->I <= 0)
    return fail(BEAM_ERR_INVALID_ARG, "T=%d H=%d E=%d I=%d: sizes must be positive", p->T, p->H,
                p->E, p->I);
  if (p->T > (1 << 22)) return fail(BEAM_ERR_UNSUPPORTED, "T=%d exceeds 4194304", p->T);
  if (p->H % 128 || p->I % 128)
    return fail(BEAM_ERR_UNSUPPORTED, "H=%d and I=%d must be multiples of 128", p->H, p->I);
  if (p->H > 8192 || p->I > 65536)
    return fail(BEAM_ERR_UNSUPPORTED, "H must be at most 8192 and I at most 65536");
  if (p->E % 32 || p->E > 256)
    return fail(BEAM_ERR_UNSUPPORTED, "E=%d must be a multiple of 32 and at most 256", p->E);
  if (p->n_group <= 0 || p->E % p->n_group)
    return fail(BEAM_ERR_INVALID_ARG, "n_group=%d must divide E=%d", p->n_group, p->E);
  if (p->topk_group <= 0 || p->topk_group > p->n_group)
    return fail(BEAM_ERR_INVALID_ARG, "topk_group=%d must be in [1, n_group=%d]", p->topk_group,
                p->n_group);
  if (p->topk_group < p->n_group && p->E / p->n_group != 32)
    return fail(BEAM_ERR_UNSUPPORTED, "group size E/n_group=%d: only groups of 32 are implemented",
                p->E / p->n_group);
  const int cand = p->topk_group * (p->E / p->n_group);
  if (p->top_k <= 0 || p->top_k > 32 || p->top_k > cand)
    return fail(BEAM_ERR_INVALID_ARG, "top_k=%d must be in [1, min(32, %d)]", p->top_k, cand);
  if (!(p->routed_scale > 0.f) || !std::isfinite(p->routed_scale))
    return fail(BEAM_ERR_INVALID_ARG, "routed_scale must be positive and finite");
  if (!(p->rms_eps >= 0.f) || !std::isfinite(p->rms_eps))
    return fail(BEAM_ERR_INVALID_ARG, "rms_eps must be >= 0 and finite");
  if (p->residual_k == 1 || p->residual_k < 0)
    return fail(BEAM_ERR_INVALID_ARG, "residual_k=%d: use 0 (none) or k >= 2", p->residual_k);
  if (p->flags & ~(BEAM_FLAG_PRE_NORM | BEAM_FLAG_FP32_OUT | BEAM_FLAG_RETURN_SCORES |
                   BEAM_FLAG_FP8_EXPERTS | BEAM_FLAG_NVFP4_EXPERTS |
                   BEAM_FLAG_PREFILL_WEIGHT_MAJOR))
    return fail(BEAM_ERR_INVALID_ARG, "unknown flag bits 0x%x", p->flags);
  if ((p->flags & BEAM_FLAG_FP8_EXPERTS) && (p->flags & BEAM_FLAG_NVFP4_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_FP8_EXPERTS and BEAM_FLAG_NVFP4_EXPERTS exclude each other");
  if ((p->flags & BEAM_FLAG_NVFP4_EXPERTS) && (p->H % 256 || p->I % 256))
    return fail(BEAM_ERR_UNSUPPORTED, "NVFP4 experts need H=%d and I=%d to be multiples of 256",
                p->H, p->I);
  if ((p->flags & BEAM_FLAG_FP32_OUT) && p->residual_k >= 2)
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_FP32_OUT applies only without the residual step");
  const long long pairs = static_cast<long long>(p->T) * p->top_k;
  if (pairs > (1LL << 26)) return fail(BEAM_ERR_UNSUPPORTED, "T*top_k too large");
  return BEAM_OK;
}

Layout make_layout(const beam_moe_params& p) {
  Layout L{};
  const int nsm = sm_count();
  L.KS = choose_router_ks(p, nsm);
  L.NB = (p.T + beam::PERM_TPB - 1) / beam::PERM_TPB;
  L.path = choose_path(p);
  L.NT = path_nt(L.path);
  const long long R = static_cast<long long>(p.T) * p.top_k;
  const bool f4 = (p.flags & BEAM_FLAG_NVFP4_EXPERTS) != 0;
  L.f4 = f4;
  L.pad = f4 ? (L.path == PATH_W32 ? 32 : 128) : 1;
  L.rows = f4 ? (R + (L.pad - 1) * std::min<long long>(p.E, R) + 127) / 128 * 128 : R;
  const long long Rr = L.rows;
  const long long tiles = (R + L.NT - 1) / L.NT + p.E;
  if (L.path == PATH_WIDE) {
    // at most ceil(n / 256) token groups per expert, one unit per group and
    // weight slice
    const long long groups = (R + 255) / 256 + p.E;
    L.units_gu_max = groups * (p.I / 256);
    L.units_dn_max = groups * ((p.H + 511) / 512);
  } else if (L.path == PATH_TM) {
    // cluster units (two int4 each): at most MT per 256-row group plus MT/2+1
    // tail units per expert
    const long long groups = (R + 255) / 256 + p.E;
    L.units_gu_max = 2 * (groups * (p.I / 128) + static_cast<long long>(p.E) * (p.I / 256 + 1));
    L.units_dn_max = 2 * (groups * (p.H / 256) + static_cast<long long>(p.E) * (p.H / 512 + 1));
  } else {
    L.units_gu_max = tiles * (p.I / 128);
    L.units_dn_max = tiles * path_mt_down(L.path, p.H, f4);
  }
  size_t sz[kLayoutEntries];
  sz[L_XN] = (p.flags & BEAM_FLAG_PRE_NORM) ? static_cast<size_t>(p.T) * p.H * 2 : 0;
  sz[L_PART] = static_cast<size_t>(L.KS) * p.T * p.E * 4;
  sz[L_IDX] = static_cast<size_t>(R) * 4;
  sz[L_W] = static_cast<size_t>(R) * 4;
  sz[L_COUNTS] = static_cast<size_t>(p.E) * 4;
  sz[L_OFFS] = static_cast<size_t>(p.E + 1) * 4;
  sz[L_ROWTOK] = static_cast<size_t>(Rr) * 4;
  sz[L_ROWW] = static_cast<size_t>(Rr) * 4;
  sz[L_XPERM] = static_cast<size_t>(Rr) * p.H * 2;
  sz[L_ACT] = static_cast<size_t>(Rr) * p.I * 2;
  sz[L_OACC] = static_cast<size_t>(p.T) * p.H * 4;
  sz[L_NUNITS] = 16;
  sz[L_BLKHIST] = static_cast<size_t>(L.NB) * p.E * 4;
  sz[L_BLKOFF] = static_cast<size_t>(L.NB) * p.E * 4;
  sz[L_UGU] = static_cast<size_t>(L.units_gu_max) * 16;
  sz[L_UDN] = static_cast<size_t>(L.units_dn_max) * 16;
  sz[L_PAIRROW] = static_cast<size_t>(R) * 4;
  sz[L_WR3] = router_on_tensor_cores(p) ? static_cast<size_t>(p.E) * 3 * p.H * 2 : 0;
  sz[L_RUNITS] = router_on_tensor_cores(p) ? router_units_bytes(p) : 0;
  const bool f8 = (p.flags & BEAM_FLAG_FP8_EXPERTS) != 0;
  sz[L_XSCALE] = (f8 || f4) ? static_cast<size_t>(Rr) * 4 : 0;
  sz[L_ACTQ] = f8 ? static_cast<size_t>(Rr) * p.I : (f4 ? static_cast<size_t>(Rr) * p.I / 2 : 0);
  sz[L_ASCALE] = (f8 || f4) ? static_cast<size_t>(Rr) * 4 : 0;
  // token block scales: 512-byte groups per (token tile of L.pad rows, K = 64 step)
  sz[L_XSF] = f4 ? static_cast<size_t>(Rr / L.pad) * (p.H / 64) * 512 : 0;
  sz[L_ASF] = f4 ? static_cast<size_t>(Rr / L.pad) * (p.I / 64) * 512 : 0;
  sz[L_ARRIVE] = static_cast<size_t>(p.T) * 8 + 8;   // counters, completion list, cursors
  size_t cur = 0;
  for (int i = 0; i < kLayoutEntries; ++i) {
    L.off[i] = cur;
    cur = align_up(cur + sz[i], 1024);
  }
  L.total = cur;
  return L;
}

// ------------------------------------------------------------- TMA maps
typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                      const cuuint32_t*, CUtensorMapInterleave,
                                      CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);

PFN_encodeTiled_t encode_fn() {
  static PFN_encodeTiled_t fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled_t>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

// Row-major matrix [rows, cols] of bf16 (f8 = false) or one-byte E4M3 codes
// (f8 = true) -> TMA map with a box of one 128-byte row segment (64 bf16 or
// 128 codes) x box_rows rows and the 128-byte swizzle.
beam_status_t make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                       uint32_t box_rows, bool f8 = false) {
  PFN_encodeTiled_t fn = encode_fn();
  if (fn == nullptr) return fail(BEAM_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (f8 ? 1 : 2)};
  cuuint32_t box[2] = {f8 ? 128u : 64u, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                  const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(BEAM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %llux%llu matrix",
                static_cast<int>(r), static_cast<unsigned long long>(rows),
                static_cast<unsigned long long>(cols));
  return BEAM_OK;
}

// --------------------------------------------------------- GEMM launches
template <int MODE, int NT, int STAGES, int KIND>
beam_status_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                          const beam::GemmArgs& args, cudaStream_t st) {
  using C = beam::GemmCfg<MODE, NT, STAGES, KIND>;
  auto kern = beam::expert_gemm_kernel<MODE, NT, STAGES, KIND>;
  beam_status_t sa = ensure_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (sa != BEAM_OK) return sa;
  ProfScope ps(MODE == 0 ? "expert_gemm_gateup_swiglu" : "expert_gemm_down", st);
  kern<<<sm_count(), 192, C::SMEM_BYTES, st>>>(a0, a1, b, args);
  BEAM_LAUNCH_CHECK(MODE == 0 ? "expert_gemm_kernel<gate/up>" : "expert_gemm_kernel<down>");
  return BEAM_OK;
}

template <bool F8>
beam_status_t launch_gemm_pair(const CUtensorMap& a0, const CUtensorMap& tok, const CUtensorMap& tok64,
                               const beam::PairArgs& args, cudaStream_t st, const char* prof_name) {
  using C = beam::PairCfg;
  auto kern = beam::expert_gemm_pair_kernel<F8>;
  beam_status_t sa = ensure_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (sa != BEAM_OK) return sa;
  const int grid = (sm_count() / 2) * 2;
  ProfScope ps(prof_name, st);
  kern<<<grid, 192, C::SMEM_BYTES, st>>>(a0, tok, tok64, args);
  BEAM_LAUNCH_CHECK("expert_gemm_pair_kernel");
  return BEAM_OK;
}

template <int MODE, int KIND>
beam_status_t launch_gemm_tm(const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap& tok,
                             const beam::TmArgs& args, cudaStream_t st) {
  using C = beam::TmCfg<KIND>;
  auto kern = beam::expert_gemm_tm_kernel<MODE, KIND>;
  beam_status_t sa = ensure_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (sa != BEAM_OK) return sa;
  const int grid = (sm_count() / 2) * 2;
  ProfScope ps(MODE == 0 ? "expert_gemm_gateup_swiglu" : "expert_gemm_down", st);
  kern<<<grid, beam::TM_THREADS, C::SMEM_BYTES, st>>>(w0, w1, tok, args);
  BEAM_LAUNCH_CHECK(MODE == 0 ? "expert_gemm_tm_kernel<gate/up>" : "expert_gemm_tm_kernel<down>");
  return BEAM_OK;
}

template <int MODE, bool F8>
beam_status_t launch_gemm_wide(const CUtensorMap& w0, const CUtensorMap& w1, const CUtensorMap (&tok)[4],
                               const beam::WideArgs& args, cudaStream_t st) {
  using C = beam::WideCfg<MODE>;
  auto kern = beam::expert_gemm_wide_kernel<MODE, F8>;
  beam_status_t sa = ensure_smem(reinterpret_cast<const void*>(kern), C::SMEM_BYTES);
  if (sa != BEAM_OK) return sa;
  const int grid = (sm_count() / 2) * 2;
  ProfScope ps(MODE == 0 ? "expert_gemm_gateup_swiglu" : "expert_gemm_down", st);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(w0, w1, tok[0], tok[1], tok[2], tok[3], args);
  BEAM_LAUNCH_CHECK(MODE == 0 ? "expert_gemm_wide_kernel<gate/up>" : "expert_gemm_wide_kernel<down>");
  return BEAM_OK;
}

beam_status_t launch_router(const beam_moe_params& p, const Layout& L, const void* x_in,
                            const float* w_router, const float* bias, const float* pre_gain,
                            int32_t* idx, float* w, float* scores,
                            uint8_t* ws, cudaStream_t st) {
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(x_in);
  if (p.flags & BEAM_FLAG_PRE_NORM) {
    __nv_bfloat16* xn = reinterpret_cast<__nv_bfloat16*>(ws + L.off[L_XN]);
    ProfScope ps("prenorm", st);
    beam::prenorm_kernel<<<(p.T + 7) / 8, 256, 0, st>>>(x, pre_gain, xn, p.T, p.H, p.rms_eps);
    BEAM_LAUNCH_CHECK("prenorm_kernel");
    x = xn;
  }
  float* part = reinterpret_cast<float*>(ws + L.off[L_PART]);
  if (router_on_tensor_cores(p)) {
    // logits [T, E] = [x, x, x] . [W1 | W2 | W3]^T on the tensor cores: the
    // 2-SM pair kernel with the 256 experts as M, tokens as N, K split in
    // kRouterKSplit slices (summed by the select kernel)
    __nv_bfloat16* w3 = reinterpret_cast<__nv_bfloat16*>(ws + L.off[L_WR3]);
    int4* runits = reinterpret_cast<int4*>(ws + L.off[L_RUNITS]);
    int* rcount = reinterpret_cast<int*>(ws + L.off[L_RUNITS] + router_units_bytes(p) - 16);
    {
      ProfScope ps("router_split", st);
      beam::router_split_kernel<<<2 * sm_count(), 256, 0, st>>>(w_router, p.E, p.H, w3, p.T,
                                                                kRouterKSplit, runits, rcount);
    }
    BEAM_LAUNCH_CHECK("router_split_kernel");
    CUtensorMap m_w, m_x, m_x64;
    beam_status_t s;
    if ((s = make_map(&m_w, w3, static_cast<uint64_t>(p.E), static_cast<uint64_t>(3) * p.H,
                      128)) != BEAM_OK)
      return s;
    if ((s = make_map(&m_x, x, static_cast<uint64_t>(p.T), p.H, 16)) != BEAM_OK) return s;
    if ((s = make_map(&m_x64, x, static_cast<uint64_t>(p.T), p.H, 64)) != BEAM_OK) return s;
    beam::PairArgs ra{};
    ra.units = runits;
    ra.n_units = rcount;
    ra.k_blocks = 3 * p.H / 64 / kRouterKSplit;
    ra.w_rows_per_expert = 0;
    ra.y = part;
    ra.out_ld = p.E;
    ra.k_split = kRouterKSplit;
    ra.b_k_wrap = p.H / 64;
    ra.y_split = static_cast<size_t>(p.T) * p.E;
    ra.timeout_ns = kWaitTimeoutNs;
    if ((s = launch_gemm_pair<false>(m_w, m_x, m_x64, ra, st, "router_logits_tc")) != BEAM_OK)
      return s;
  } else {
    dim3 g1((p.T + beam::RL_BT - 1) / beam::RL_BT, (p.E + beam::RL_BE - 1) / beam::RL_BE, L.KS);
    {
      ProfScope ps("router_logits", st);
      beam::router_logits_kernel<<<g1, 256, 0, st>>>(x, w_router, part, p.T, p.H, p.E,
                                                     p.H / L.KS);
    }
    BEAM_LAUNCH_CHECK("router_logits_kernel");
  }
  const int tpb = p.T <= 512 ? 1 : beam::SEL_TOKENS;
  const int nb = (p.T + tpb - 1) / tpb;
  ProfScope ps("router_select", st);
#define BEAM_SEL(NI)                                                                          \
  case NI:                                                                                    \
    beam::router_select_kernel<NI><<<nb, 256, 0, st>>>(part, L.KS, bias, p.T, p.E, p.n_group, \
                                                      p.topk_group, p.top_k, p.routed_scale, \
                                                      idx, w, scores, tpb);                   \
    break;
  switch (p.E / 32) {
    BEAM_SEL(1) BEAM_SEL(2) BEAM_SEL(3) BEAM_SEL(4) BEAM_SEL(5) BEAM_SEL(6) BEAM_SEL(7)
    BEAM_SEL(8)
    default:
      return fail(BEAM_ERR_UNSUPPORTED, "E=%d", p.E);
  }
#undef BEAM_SEL
  BEAM_LAUNCH_CHECK("router_select_kernel");
  return BEAM_OK;
}

// The expert weights of one call: BF16 matrices; E4M3 codes with one FP32
// scale per output row; or NVFP4 codes with block scales (SF groups) and one
// FP32 scale per expert matrix.
struct ExpertWeights {
  const void* gate;
  const void* up;
  const void* down;
  const float* s_gate;  // E4M3: per row; NVFP4: per expert
  const float* s_up;
  const float* s_down;
  const void* sf_gate;  // NVFP4 block scales
  const void* sf_up;
  const void* sf_down;
  int kind;             // beam::KIND_*
};

// Quantised activations of the E4M3 / NVFP4 paths (workspace buffers).
struct QuantBufs {
  const float* xscale;   // per-row scale of the quantised x
  const uint8_t* xsf;    // NVFP4 block scales of x
  uint8_t* aq;           // codes of the SwiGLU output
  float* ascale;         // its per-row scale
  uint8_t* asf;          // NVFP4 block scales
  const int* row_valid;  // NVFP4: row_token (< 0 on padding rows)
  const int* rows_dev;   // NVFP4: device count of rows (offsets[E])
};

// Steps 3-5: gate/up GEMM + SwiGLU into act (bf16), then the down GEMM whose
// epilogue adds the router-weighted expert outputs into each token's FP32
// accumulator and finalises every completed token (post-norm and residual,
// or the output). E4M3 / NVFP4: the expert-ordered x (xop) and the weights
// are quantised; act is quantised per row (into q.aq) before the down GEMM.
template <int KIND>
beam_status_t launch_expert_gemms(const beam_moe_params& prm, const Layout& L,
                                  const ExpertWeights& w, const void* xop, const QuantBufs& q,
                                  __nv_bfloat16* act, const beam::CombineArgs& comb, int4* ugu,
                                  int4* udn, int* nunits, long long R, cudaStream_t st) {
  constexpr bool F8 = KIND == beam::KIND_E4M3;
  constexpr bool F4 = KIND == beam::KIND_NVFP4;
  beam_status_t s = BEAM_OK;
  const int H = prm.H, E = prm.E, I = prm.I;
  const int KB = beam::KBlock<KIND>::ELEMS;
  if (F4 && L.path == PATH_WIDE)
    return fail(BEAM_ERR_UNSUPPORTED, "NVFP4 experts run on the weight-major or token-major kernels");
  const bool bytes = F8 || F4;     // TMA maps over one-byte elements (codes)
  const int hc = F4 ? H / 2 : H;   // row length of the code matrices, in map elements
  const int ic = F4 ? I / 2 : I;
  // operand of the down GEMM: the bf16 act, or its codes
  const void* aop = (F8 || F4) ? static_cast<const void*>(q.aq) : static_cast<const void*>(act);

  // SwiGLU output -> per-row codes and scales (between the two GEMMs)
  auto quant_act = [&]() -> beam_status_t {
    if (!F8 && !F4) return BEAM_OK;
    ProfScope ps("quant_act", st);
    if (F8)
      beam::quant_rows_e4m3_kernel<<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(
          act, nullptr, R, I, q.aq, q.ascale);
    else
      beam::quant_rows_nvfp4_kernel<<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(
          act, nullptr, q.row_valid, R, q.rows_dev, I, 1, nullptr, q.aq, q.asf, q.ascale, L.pad);
    BEAM_LAUNCH_CHECK("quant_rows_*_kernel<act>");
    return BEAM_OK;
  };

  if (L.path == PATH_WIDE) {
    // weights: 128-row boxes; tokens: 64/32/16/8-row boxes
    CUtensorMap m_g, m_u, m_d, m_x[4], m_a[4];
    if ((s = make_map(&m_g, w.gate, static_cast<uint64_t>(E) * I, H, 128, F8)) != BEAM_OK) return s;
    if ((s = make_map(&m_u, w.up, static_cast<uint64_t>(E) * I, H, 128, F8)) != BEAM_OK) return s;
    if ((s = make_map(&m_d, w.down, static_cast<uint64_t>(E) * H, I, 128, F8)) != BEAM_OK) return s;
    const uint32_t boxes[4] = {64, 32, 16, 8};
    for (int j = 0; j < 4; ++j) {
      if ((s = make_map(&m_x[j], xop, R, H, boxes[j], F8)) != BEAM_OK) return s;
      if ((s = make_map(&m_a[j], aop, R, I, boxes[j], F8)) != BEAM_OK) return s;
    }
    beam::WideArgs wa{};
    wa.units = ugu;
    wa.n_units = nunits + 0;
    wa.k_blocks = H / KB;
    wa.w_rows_per_expert = I;
    wa.act = act;
    wa.act_ld = I;
    wa.timeout_ns = kWaitTimeoutNs;
    wa.row_scale = q.xscale;
    wa.w_scale0 = w.s_gate;
    wa.w_scale1 = w.s_up;
    beam::WideArgs wd = wa;
    wd.units = udn;
    wd.n_units = nunits + 1;
    wd.k_blocks = I / KB;
    wd.w_rows_per_expert = H;
    wd.act = nullptr;
    wd.row_scale = nullptr;  // the activation row scales are in the combine coefficient
    wd.w_scale0 = w.s_down;
    wd.w_scale1 = nullptr;
    wd.comb = comb;
    if ((s = launch_gemm_wide<0, F8>(m_g, m_u, m_x, wa, st)) != BEAM_OK) return s;
    if ((s = quant_act()) != BEAM_OK) return s;
    if ((s = launch_gemm_wide<1, F8>(m_d, m_d, m_a, wd, st)) != BEAM_OK) return s;
    return BEAM_OK;
  }

  const uint32_t tok_box = L.path == PATH_TM ? 128 : 16;
  CUtensorMap m_g, m_u, m_d, m_x, m_a;
  if ((s = make_map(&m_g, w.gate, static_cast<uint64_t>(E) * I, hc, 128, bytes)) != BEAM_OK) return s;
  if ((s = make_map(&m_u, w.up, static_cast<uint64_t>(E) * I, hc, 128, bytes)) != BEAM_OK) return s;
  if ((s = make_map(&m_d, w.down, static_cast<uint64_t>(E) * H, ic, 128, bytes)) != BEAM_OK) return s;
  if ((s = make_map(&m_x, xop, R, hc, tok_box, bytes)) != BEAM_OK) return s;
  if ((s = make_map(&m_a, aop, R, ic, tok_box, bytes)) != BEAM_OK) return s;

  if (L.path == PATH_TM) {
    beam::TmArgs ta{};
    ta.units = ugu;
    ta.n_units = nunits + 0;
    ta.k_blocks = H / KB;
    ta.w_rows_per_expert = I;
    ta.out = act;
    ta.out_ld = I;
    ta.timeout_ns = kWaitTimeoutNs;
    ta.row_scale = q.xscale;
    ta.w_scale0 = w.s_gate;
    ta.w_scale1 = w.s_up;
    ta.a_sf = q.xsf;
    ta.w_sf0 = static_cast<const uint8_t*>(w.sf_gate);
    ta.w_sf1 = static_cast<const uint8_t*>(w.sf_up);
    beam::TmArgs td = ta;
    td.units = udn;
    td.n_units = nunits + 1;
    td.k_blocks = I / KB;
    td.w_rows_per_expert = H;
    td.out = nullptr;
    td.out_ld = H;
    td.row_scale = nullptr;  // the activation row scales are in the combine coefficient
    td.w_scale0 = w.s_down;
    td.w_scale1 = nullptr;
    td.a_sf = q.asf;
    td.w_sf0 = static_cast<const uint8_t*>(w.sf_down);
    td.w_sf1 = nullptr;
    td.comb = comb;
    if ((s = launch_gemm_tm<0, KIND>(m_g, m_u, m_x, ta, st)) != BEAM_OK) return s;
    if ((s = quant_act()) != BEAM_OK) return s;
    if ((s = launch_gemm_tm<1, KIND>(m_d, m_d, m_a, td, st)) != BEAM_OK) return s;
    return BEAM_OK;
  }

  beam::GemmArgs ga{};
  ga.units = ugu;  // token tiles, shared by both GEMMs
  ga.n_units = nunits + 0;
  ga.m_tiles = I / 128;
  ga.k_blocks = H / KB;
  ga.a_rows_per_expert = I;
  ga.out = act;
  ga.out_ld = I;
  ga.timeout_ns = kWaitTimeoutNs;
  ga.row_scale = q.xscale;
  ga.w_scale0 = w.s_gate;
  ga.w_scale1 = w.s_up;
  ga.a_sf0 = static_cast<const uint8_t*>(w.sf_gate);
  ga.a_sf1 = static_cast<const uint8_t*>(w.sf_up);
  ga.b_sf = q.xsf;
  beam::GemmArgs gd = ga;
  gd.n_units = nunits + 1;
  gd.k_blocks = I / KB;
  gd.a_rows_per_expert = H;
  gd.out = nullptr;
  gd.out_ld = H;
  gd.row_scale = nullptr;  // the activation row scales are in the combine coefficient
  gd.w_scale0 = w.s_down;
  gd.w_scale1 = nullptr;
  gd.a_sf0 = static_cast<const uint8_t*>(w.sf_down);
  gd.a_sf1 = nullptr;
  gd.b_sf = q.asf;
  gd.comb = comb;
  // stage counts: NVFP4 stages also carry the K-block's block scales
  // (the NVFP4 down GEMM on 32-token tiles loads two 128-row weight tiles
  // per stage)
  constexpr int S_GU32 = F4 ? 5 : 6, S_DN32 = F4 ? 5 : 10;
  if (L.path == PATH_W32) {
    gd.m_tiles = H / beam::UnitRows<1, 32, KIND>::value;
    if ((s = launch_gemm<0, 32, S_GU32, KIND>(m_g, m_u, m_x, ga, st)) != BEAM_OK) return s;
    if ((s = quant_act()) != BEAM_OK) return s;
    if ((s = launch_gemm<1, 32, S_DN32, KIND>(m_d, m_d, m_a, gd, st)) != BEAM_OK) return s;
  } else {
    gd.m_tiles = H / beam::UnitRows<1, 128, KIND>::value;
    if ((s = launch_gemm<0, 128, 4, KIND>(m_g, m_u, m_x, ga, st)) != BEAM_OK) return s;
    if ((s = quant_act()) != BEAM_OK) return s;
    if ((s = launch_gemm<1, 128, 6, KIND>(m_d, m_d, m_a, gd, st)) != BEAM_OK) return s;
  }
  return BEAM_OK;
}

// Steps 2-5 of the sublayer, given the routing (idx, wts): permutation and
// work lists, the expert GEMMs, then the weighted combine with post-norm and
// residual. With dense = true there is one expert that every token uses with
// weight 1 (the dense SwiGLU MLP): the permutation is the identity, set up by
// dense_setup_kernel, and the GEMMs read x in place.
beam_status_t run_experts(const beam_moe_params& prm, const Layout& L, const void* x_in,
                          const __nv_bfloat16* x, const int32_t* idx, float* wts,
                          const ExpertWeights& w, const float* post_gain, void* out, uint8_t* ws,
                          cudaStream_t st, bool dense) {
  const beam_moe_params* p = &prm;
  beam_status_t s = BEAM_OK;
  const int T = p->T, H = p->H, E = p->E, I = p->I, K = p->top_k;
  const long long R = static_cast<long long>(T) * K;
  // 2. permutation, work lists and the expert-ordered copy of x
  int* blk_hist = reinterpret_cast<int*>(ws + L.off[L_BLKHIST]);
  int* blk_off = reinterpret_cast<int*>(ws + L.off[L_BLKOFF]);
  int* counts = reinterpret_cast<int*>(ws + L.off[L_COUNTS]);
  int* offs = reinterpret_cast<int*>(ws + L.off[L_OFFS]);
  int* row_tok = reinterpret_cast<int*>(ws + L.off[L_ROWTOK]);
  float* row_w = reinterpret_cast<float*>(ws + L.off[L_ROWW]);
  int* pair_row = reinterpret_cast<int*>(ws + L.off[L_PAIRROW]);
  __nv_bfloat16* xperm = reinterpret_cast<__nv_bfloat16*>(ws + L.off[L_XPERM]);
  __nv_bfloat16* act = reinterpret_cast<__nv_bfloat16*>(ws + L.off[L_ACT]);
  float* oacc = reinterpret_cast<float*>(ws + L.off[L_OACC]);
  int* arrive = reinterpret_cast<int*>(ws + L.off[L_ARRIVE]);
  int4* ugu = reinterpret_cast<int4*>(ws + L.off[L_UGU]);
  int4* udn = reinterpret_cast<int4*>(ws + L.off[L_UDN]);
  int* nunits = reinterpret_cast<int*>(ws + L.off[L_NUNITS]);
  // E4M3 / NVFP4 paths: x codes (in the permuted-x region), the activations'
  // codes, their scales
  const bool quant = w.kind != beam::KIND_BF16;
  const bool f4 = w.kind == beam::KIND_NVFP4;
  QuantBufs qb{};
  qb.xscale = quant ? reinterpret_cast<float*>(ws + L.off[L_XSCALE]) : nullptr;
  qb.xsf = f4 ? ws + L.off[L_XSF] : nullptr;
  qb.aq = quant ? ws + L.off[L_ACTQ] : nullptr;
  qb.ascale = quant ? reinterpret_cast<float*>(ws + L.off[L_ASCALE]) : nullptr;
  qb.asf = f4 ? ws + L.off[L_ASF] : nullptr;
  qb.row_valid = row_tok;
  qb.rows_dev = offs + E;
  // rows of the expert-ordered layout (NVFP4: padded, bounded by L.rows)
  const long long Rl = f4 ? L.rows : R;

  const int NB = dense ? 1 : L.NB;
  // one permutation block and a token-tile work list (decode): histogram,
  // scan and scatter in one launch
  const bool small = !dense && L.NB == 1 && (L.path == PATH_W32 || L.path == PATH_W128);
  if (small) {
    ProfScope ps("expert_permute", st);
    beam::expert_permute_small_kernel<<<1, 256, 0, st>>>(
        idx, wts, T, K, E, counts, offs, ugu, nunits, L.NT, I / 128, path_mt_down(L.path, H, L.f4),
        L.pad, pair_row, row_tok, row_w);
  } else if (dense) {
    ProfScope ps("dense_setup", st);
    beam::dense_setup_kernel<<<(T + 255) / 256, 256, 0, st>>>(T, blk_hist, pair_row, row_tok,
                                                              row_w, wts);
  } else {
    ProfScope ps("expert_hist", st);
    beam::expert_block_hist_kernel<<<L.NB, beam::PERM_THREADS, 0, st>>>(idx, T, K, E, blk_hist);
  }
  BEAM_LAUNCH_CHECK("expert_block_hist_kernel");
  if (!small) {
    ProfScope ps("expert_scan_units", st);
    if (L.path == PATH_WIDE)
      beam::expert_scan_units_prefill_kernel<beam::LIST_PAIR, beam::LIST_PAIR>
          <<<1, 256, 0, st>>>(blk_hist, NB, E, blk_off, counts, offs, ugu, udn, nunits, I / 256,
                              (H + 511) / 512);
    else if (L.path == PATH_TM)
      beam::expert_scan_units_prefill_kernel<beam::LIST_TM, beam::LIST_TM>
          <<<1, 256, 0, st>>>(blk_hist, NB, E, blk_off, counts, offs, ugu, udn, nunits, I / 128,
                              H / 256, L.pad, row_tok);
    else
      beam::expert_scan_units_kernel<<<1, 256, 0, st>>>(blk_hist, NB, E, blk_off, counts, offs,
                                                        ugu, nunits, L.NT, I / 128,
                                                        path_mt_down(L.path, H, L.f4), L.pad, row_tok);
  }
  BEAM_LAUNCH_CHECK("expert_scan_units_kernel");
  if (quant) {
    // quantise x per token, gathered into expert order (identity when dense)
    if (!dense && !small) {
      ProfScope ps("expert_scatter", st);
      beam::expert_scatter_kernel<<<L.NB, beam::PERM_THREADS, 0, st>>>(
          idx, wts, T, K, E, blk_off, pair_row, row_tok, row_w);
    }
    BEAM_LAUNCH_CHECK("expert_scatter_kernel");
    {
      ProfScope ps("quant_x", st);
      if (f4)
        beam::quant_rows_nvfp4_kernel<<<static_cast<unsigned>((Rl + 7) / 8), 256, 0, st>>>(
            x, dense ? nullptr : row_tok, row_tok, Rl, offs + E, H, 1, nullptr,
            ws + L.off[L_XPERM], ws + L.off[L_XSF], const_cast<float*>(qb.xscale), L.pad);
      else
        beam::quant_rows_e4m3_kernel<<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(
            x, dense ? nullptr : row_tok, R, H, ws + L.off[L_XPERM], const_cast<float*>(qb.xscale));
    }
    BEAM_LAUNCH_CHECK("quant_rows_*_kernel<x>");
  } else if (dense) {
    xperm = const_cast<__nv_bfloat16*>(x);  // identity permutation: read x in place
  } else {
    if (!small) {
      ProfScope ps("expert_scatter", st);
      beam::expert_scatter_kernel<<<L.NB, beam::PERM_THREADS, 0, st>>>(
          idx, wts, T, K, E, blk_off, pair_row, row_tok, row_w);
    }
    BEAM_LAUNCH_CHECK("expert_scatter_kernel");
    {
      ProfScope ps("gather_rows", st);
      beam::gather_rows_kernel<<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(
          x, row_tok, static_cast<int>(R), H, xperm);
    }
    BEAM_LAUNCH_CHECK("gather_rows_kernel");
  }

  // 3. gate/up GEMM + SwiGLU -> act, 4. down GEMM with the fused combine,
  // 5. post-norm + scaled residual (or the output) of every completed token
  const int resid = p->residual_k >= 2;
  const float kf = static_cast<float>(resid ? p->residual_k : 2);
  beam::CombineArgs cb{};
  cb.acc = oacc;
  cb.count = arrive;
  cb.done = arrive + T;
  cb.cursor = arrive + 2 * static_cast<size_t>(T);
  cb.T = T;
  cb.expected = combine_expected(L.path, H, K, L.f4);
  // weight-major kernels (few tokens): one grid-wide completion count
  // instead of per-token arrivals
  cb.grid_done = (L.path == PATH_W32 || L.path == PATH_W128) ? 1 : 0;
  cb.row_token = row_tok;
  cb.row_weight = row_w;
  cb.row_scale = quant ? qb.ascale : nullptr;
  cb.h_prev = static_cast<const __nv_bfloat16*>(x_in);
  cb.gain = post_gain;
  cb.out = out;
  cb.H = H;
  cb.eps = p->rms_eps;
  cb.a = resid ? std::sqrt((kf - 1.f) / kf) : 0.f;
  cb.b = resid ? 1.f / std::sqrt(kf) : 1.f;
  cb.resid = resid;
  cb.out_f32 = (p->flags & BEAM_FLAG_FP32_OUT) != 0;
  {
    ProfScope ps("clear_acc", st);
    const size_t n4 = static_cast<size_t>(T) * H / 4;
    const unsigned blocks = static_cast<unsigned>(
        std::min<size_t>((n4 + 255) / 256, static_cast<size_t>(2 * sm_count())));
    beam::clear_acc_kernel<<<blocks, 256, 0, st>>>(reinterpret_cast<float4*>(oacc), n4, cb.count,
                                                   cb.done, cb.cursor, T);
  }
  BEAM_LAUNCH_CHECK("clear_acc_kernel");
  if (w.kind == beam::KIND_NVFP4)
    s = launch_expert_gemms<beam::KIND_NVFP4>(*p, L, w, xperm, qb, act, cb, ugu, udn, nunits, Rl, st);
  else if (w.kind == beam::KIND_E4M3)
    s = launch_expert_gemms<beam::KIND_E4M3>(*p, L, w, xperm, qb, act, cb, ugu, udn, nunits, R, st);
  else
    s = launch_expert_gemms<beam::KIND_BF16>(*p, L, w, xperm, qb, act, cb, ugu, udn, nunits, R, st);
  if (s != BEAM_OK) return s;
  return BEAM_OK;
}

}  // namespace

extern "C" {

const char* beam_last_error_string(void) { return t_last_error.c_str(); }

size_t beam_moe_workspace_size(const beam_moe_params* p) {
  if (check_params(p) != BEAM_OK) return 0;
  return make_layout(*p).total;
}

int beam_moe_workspace_layout(const beam_moe_params* p, size_t* offsets, int n) {
  if (check_params(p) != BEAM_OK || offsets == nullptr || n <= 0) return 0;
  const Layout L = make_layout(*p);
  const int m = n < kLayoutEntries ? n : kLayoutEntries;
  for (int i = 0; i < m; ++i) offsets[i] = L.off[i];
  return m;
}

beam_status_t beam_moe_route(const beam_moe_params* p, const void* x, const float* w_router,
                             const float* logit_bias, const float* pre_gain, int32_t* topk_idx,
                             float* topk_w, float* scores, void* workspace,
                             size_t workspace_bytes, void* stream) {
  beam_status_t s = check_params(p);
  if (s != BEAM_OK) return s;
  if (p->T == 0) return BEAM_OK;
  if (!x || !w_router || !topk_idx || !topk_w || !workspace)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if ((p->flags & BEAM_FLAG_RETURN_SCORES) && !scores)
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_RETURN_SCORES needs a scores buffer");
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(workspace) ||
      (pre_gain && !aligned16(pre_gain)))
    return fail(BEAM_ERR_INVALID_ARG, "x, w_router, pre_gain and workspace must be 16-byte aligned");
  const Layout L = make_layout(*p);
  if (workspace_bytes < L.total)
    return fail(BEAM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, L.total);
  return launch_router(*p, L, x, w_router, logit_bias, pre_gain, topk_idx, topk_w,
                       (p->flags & BEAM_FLAG_RETURN_SCORES) ? scores : nullptr,
                       static_cast<uint8_t*>(workspace), static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// Checks shared by the BF16 and E4M3 forward entry points, then steps 1-5.
beam_status_t moe_forward_impl(const beam_moe_params* p, const void* x_in, const float* w_router,
                               const float* logit_bias, const ExpertWeights& w,
                               const float* pre_gain, const float* post_gain, void* out,
                               int32_t* topk_idx, float* topk_w, void* workspace,
                               size_t workspace_bytes, void* stream) {
  beam_status_t s = check_params(p);
  if (s != BEAM_OK) return s;
  if (w.kind == beam::KIND_E4M3 && !(p->flags & BEAM_FLAG_FP8_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG,
                "the E4M3 path needs BEAM_FLAG_FP8_EXPERTS in flags (and a workspace sized with it)");
  if (w.kind == beam::KIND_NVFP4 && !(p->flags & BEAM_FLAG_NVFP4_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG,
                "the NVFP4 path needs BEAM_FLAG_NVFP4_EXPERTS in flags (and a workspace sized with it)");
  if (w.kind != beam::KIND_NVFP4 && (p->flags & BEAM_FLAG_NVFP4_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_NVFP4_EXPERTS is for the NVFP4 entry points");
  if (p->T == 0) return BEAM_OK;
  if (!x_in || !w_router || !w.gate || !w.up || !w.down || !out || !workspace)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (w.kind != beam::KIND_BF16 && (!w.s_gate || !w.s_up || !w.s_down))
    return fail(BEAM_ERR_INVALID_ARG, "the quantised weights need their scales");
  if (w.kind == beam::KIND_NVFP4 && (!w.sf_gate || !w.sf_up || !w.sf_down))
    return fail(BEAM_ERR_INVALID_ARG, "the NVFP4 weights need their block scales");
  const void* ptrs[] = {x_in, w_router, w.gate, w.up, w.down, out, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(BEAM_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", q);
  if (w.kind != beam::KIND_BF16 && (!aligned16(w.s_gate) || !aligned16(w.s_up) || !aligned16(w.s_down)))
    return fail(BEAM_ERR_INVALID_ARG, "weight scales must be 16-byte aligned");
  if (w.kind == beam::KIND_NVFP4 && (!aligned16(w.sf_gate) || !aligned16(w.sf_up) || !aligned16(w.sf_down)))
    return fail(BEAM_ERR_INVALID_ARG, "block scales must be 16-byte aligned");
  if ((pre_gain && !aligned16(pre_gain)) || (post_gain && !aligned16(post_gain)))
    return fail(BEAM_ERR_INVALID_ARG, "gains must be 16-byte aligned");
  if (out == x_in) return fail(BEAM_ERR_INVALID_ARG, "out must not alias x_in");
  const Layout L = make_layout(*p);
  if (workspace_bytes < L.total)
    return fail(BEAM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, L.total);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* idx = topk_idx ? topk_idx : reinterpret_cast<int32_t*>(ws + L.off[L_IDX]);
  float* wts = topk_w ? topk_w : reinterpret_cast<float*>(ws + L.off[L_W]);

  // 1. pre-norm (optional) + router
  s = launch_router(*p, L, x_in, w_router, logit_bias, pre_gain, idx, wts, nullptr, ws, st);
  if (s != BEAM_OK) return s;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(x_in);
  if (p->flags & BEAM_FLAG_PRE_NORM) x = reinterpret_cast<const __nv_bfloat16*>(ws + L.off[L_XN]);

  // 2-5. permutation, expert GEMMs, combine and the residual
  return run_experts(*p, L, x_in, x, idx, wts, w, post_gain, out, ws, st, false);
}

}  // namespace

extern "C" {

beam_status_t beam_moe_forward(const beam_moe_params* p, const void* x_in, const float* w_router,
                               const float* logit_bias, const void* w_gate, const void* w_up,
                               const void* w_down, const float* pre_gain, const float* post_gain,
                               void* out, int32_t* topk_idx, float* topk_w, void* workspace,
                               size_t workspace_bytes, void* stream) {
  const ExpertWeights w{w_gate, w_up, w_down, nullptr, nullptr, nullptr,
                        nullptr, nullptr, nullptr, beam::KIND_BF16};
  return moe_forward_impl(p, x_in, w_router, logit_bias, w, pre_gain, post_gain, out, topk_idx,
                          topk_w, workspace, workspace_bytes, stream);
}

beam_status_t beam_moe_forward_fp8(const beam_moe_params* p, const void* x_in,
                                   const float* w_router, const float* logit_bias,
                                   const void* wq_gate, const float* ws_gate, const void* wq_up,
                                   const float* ws_up, const void* wq_down, const float* ws_down,
                                   const float* pre_gain, const float* post_gain, void* out,
                                   int32_t* topk_idx, float* topk_w, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  const ExpertWeights w{wq_gate, wq_up, wq_down, ws_gate, ws_up, ws_down,
                        nullptr, nullptr, nullptr, beam::KIND_E4M3};
  return moe_forward_impl(p, x_in, w_router, logit_bias, w, pre_gain, post_gain, out, topk_idx,
                          topk_w, workspace, workspace_bytes, stream);
}

beam_status_t beam_moe_forward_nvfp4(const beam_moe_params* p, const void* x_in,
                                     const float* w_router, const float* logit_bias,
                                     const void* wq_gate, const void* wsf_gate, const float* wg_gate,
                                     const void* wq_up, const void* wsf_up, const float* wg_up,
                                     const void* wq_down, const void* wsf_down, const float* wg_down,
                                     const float* pre_gain, const float* post_gain, void* out,
                                     int32_t* topk_idx, float* topk_w, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  const ExpertWeights w{wq_gate, wq_up, wq_down, wg_gate, wg_up, wg_down,
                        wsf_gate, wsf_up, wsf_down, beam::KIND_NVFP4};
  return moe_forward_impl(p, x_in, w_router, logit_bias, w, pre_gain, post_gain, out, topk_idx,
                          topk_w, workspace, workspace_bytes, stream);
}

beam_status_t beam_quantize_nvfp4(const void* src, long long rows, int K, int rows_per_group,
                                  void* codes, void* block_scales, float* group_scales,
                                  void* stream) {
  if (rows < 0 || rows % 128 || K <= 0 || K % 64 || rows_per_group <= 0 ||
      (rows > 0 && rows % rows_per_group))
    return fail(BEAM_ERR_INVALID_ARG,
                "rows=%lld K=%d rows_per_group=%d: rows a multiple of 128 and of rows_per_group, "
                "K a positive multiple of 64", rows, K, rows_per_group);
  if (rows > (1LL << 34)) return fail(BEAM_ERR_UNSUPPORTED, "rows=%lld is too large", rows);
  if (rows == 0) return BEAM_OK;
  if (!src || !codes || !block_scales || !group_scales)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(src) || !aligned16(codes) || !aligned16(block_scales) || !aligned16(group_scales))
    return fail(BEAM_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long groups = rows / rows_per_group;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(src);
  unsigned* gmax = reinterpret_cast<unsigned*>(group_scales);
  ProfScope ps("quant_nvfp4", st);
  // group maxima (as float bits, in the output array), quantise, then g
  BEAM_CUDA_TRY(cudaMemsetAsync(gmax, 0, static_cast<size_t>(groups) * 4, st));
  beam::group_amax_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(x, rows, K,
                                                                                rows_per_group, gmax);
  BEAM_LAUNCH_CHECK("group_amax_kernel");
  beam::quant_rows_nvfp4_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      x, nullptr, nullptr, rows, nullptr, K, rows_per_group, gmax,
      static_cast<uint8_t*>(codes), static_cast<uint8_t*>(block_scales), nullptr, 128);
  BEAM_LAUNCH_CHECK("quant_rows_nvfp4_kernel");
  beam::nvfp4_group_scale_kernel<<<static_cast<unsigned>((groups + 255) / 256), 256, 0, st>>>(
      group_scales, groups);
  BEAM_LAUNCH_CHECK("nvfp4_group_scale_kernel");
  return BEAM_OK;
}

beam_status_t beam_quantize_e4m3_rows(const void* src, long long rows, int K, void* q,
                                      float* scale, void* stream) {
  if (rows < 0 || K <= 0 || K % 16)
    return fail(BEAM_ERR_INVALID_ARG, "rows=%lld K=%d: rows >= 0 and K a positive multiple of 16",
                rows, K);
  if (rows > (1LL << 34)) return fail(BEAM_ERR_UNSUPPORTED, "rows=%lld is too large", rows);
  if (rows == 0) return BEAM_OK;
  if (!src || !q || !scale) return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(src) || !aligned16(q) || !aligned16(scale))
    return fail(BEAM_ERR_INVALID_ARG, "src, q and scale must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  ProfScope ps("quant_rows", st);
  beam::quant_rows_e4m3_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(src), nullptr, rows, K, static_cast<uint8_t*>(q), scale);
  BEAM_LAUNCH_CHECK("quant_rows_e4m3_kernel");
  return BEAM_OK;
}

// ------------------------------------------------------------- dense MLP
namespace {

beam_status_t check_dense(const beam_dense_params* d) {
  if (d == nullptr) return fail(BEAM_ERR_INVALID_ARG, "params is NULL");
  if (d->T < 0 || d->H <= 0 || d->I <= 0)
    return fail(BEAM_ERR_INVALID_ARG, "T=%d H=%d I=%d: sizes must be positive", d->T, d->H, d->I);
  if (d->T > (1 << 22)) return fail(BEAM_ERR_UNSUPPORTED, "T=%d exceeds 4194304", d->T);
  if (d->H % 128 || d->I % 128)
    return fail(BEAM_ERR_UNSUPPORTED, "H=%d and I=%d must be multiples of 128", d->H, d->I);
  if (d->H > 8192 || d->I > 65536)
    return fail(BEAM_ERR_UNSUPPORTED, "H must be at most 8192 and I at most 65536");
  if (!(d->rms_eps >= 0.f) || !std::isfinite(d->rms_eps))
    return fail(BEAM_ERR_INVALID_ARG, "rms_eps must be >= 0 and finite");
  if (d->residual_k == 1 || d->residual_k < 0)
    return fail(BEAM_ERR_INVALID_ARG, "residual_k=%d: use 0 (none) or k >= 2", d->residual_k);
  if (d->flags & ~(BEAM_FLAG_PRE_NORM | BEAM_FLAG_FP32_OUT | BEAM_FLAG_FP8_EXPERTS |
                   BEAM_FLAG_NVFP4_EXPERTS | BEAM_FLAG_PREFILL_WEIGHT_MAJOR))
    return fail(BEAM_ERR_INVALID_ARG, "unknown flag bits 0x%x", d->flags);
  if ((d->flags & BEAM_FLAG_FP8_EXPERTS) && (d->flags & BEAM_FLAG_NVFP4_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_FP8_EXPERTS and BEAM_FLAG_NVFP4_EXPERTS exclude each other");
  if ((d->flags & BEAM_FLAG_NVFP4_EXPERTS) && (d->H % 256 || d->I % 256))
    return fail(BEAM_ERR_UNSUPPORTED, "NVFP4 weights need H=%d and I=%d to be multiples of 256",
                d->H, d->I);
  if ((d->flags & BEAM_FLAG_FP32_OUT) && d->residual_k >= 2)
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_FP32_OUT applies only without the residual step");
  return BEAM_OK;
}

// The dense MLP runs as a one-expert sublayer: E = 1, top_k = 1, weight 1.
beam_moe_params dense_as_moe(const beam_dense_params& d) {
  beam_moe_params m{};
  m.T = d.T;
  m.H = d.H;
  m.E = 1;
  m.I = d.I;
  m.n_group = 1;
  m.topk_group = 1;
  m.top_k = 1;
  m.routed_scale = 1.f;
  m.rms_eps = d.rms_eps;
  m.residual_k = d.residual_k;
  m.flags = d.flags;
  return m;
}

}  // namespace

size_t beam_dense_workspace_size(const beam_dense_params* d) {
  if (check_dense(d) != BEAM_OK) return 0;
  return make_layout(dense_as_moe(*d)).total;
}

int beam_dense_workspace_layout(const beam_dense_params* d, size_t* offsets, int n) {
  if (check_dense(d) != BEAM_OK || offsets == nullptr || n <= 0) return 0;
  const Layout L = make_layout(dense_as_moe(*d));
  const int m = n < kLayoutEntries ? n : kLayoutEntries;
  for (int i = 0; i < m; ++i) offsets[i] = L.off[i];
  return m;
}

}  // extern "C"

namespace {

beam_status_t dense_forward_impl(const beam_dense_params* d, const void* x_in,
                                 const ExpertWeights& w, const float* pre_gain,
                                 const float* post_gain, void* out, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  beam_status_t s = check_dense(d);
  if (s != BEAM_OK) return s;
  if (w.kind == beam::KIND_E4M3 && !(d->flags & BEAM_FLAG_FP8_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG,
                "the E4M3 path needs BEAM_FLAG_FP8_EXPERTS in flags (and a workspace sized with it)");
  if (w.kind == beam::KIND_NVFP4 && !(d->flags & BEAM_FLAG_NVFP4_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG,
                "the NVFP4 path needs BEAM_FLAG_NVFP4_EXPERTS in flags (and a workspace sized with it)");
  if (w.kind != beam::KIND_NVFP4 && (d->flags & BEAM_FLAG_NVFP4_EXPERTS))
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_NVFP4_EXPERTS is for the NVFP4 entry points");
  if (d->T == 0) return BEAM_OK;
  if (!x_in || !w.gate || !w.up || !w.down || !out || !workspace)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (w.kind != beam::KIND_BF16 && (!w.s_gate || !w.s_up || !w.s_down))
    return fail(BEAM_ERR_INVALID_ARG, "the quantised weights need their scales");
  if (w.kind == beam::KIND_NVFP4 && (!w.sf_gate || !w.sf_up || !w.sf_down))
    return fail(BEAM_ERR_INVALID_ARG, "the NVFP4 weights need their block scales");
  const void* ptrs[] = {x_in, w.gate, w.up, w.down, out, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(BEAM_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", q);
  if (w.kind != beam::KIND_BF16 && (!aligned16(w.s_gate) || !aligned16(w.s_up) || !aligned16(w.s_down)))
    return fail(BEAM_ERR_INVALID_ARG, "weight scales must be 16-byte aligned");
  if (w.kind == beam::KIND_NVFP4 && (!aligned16(w.sf_gate) || !aligned16(w.sf_up) || !aligned16(w.sf_down)))
    return fail(BEAM_ERR_INVALID_ARG, "block scales must be 16-byte aligned");
  if ((pre_gain && !aligned16(pre_gain)) || (post_gain && !aligned16(post_gain)))
    return fail(BEAM_ERR_INVALID_ARG, "gains must be 16-byte aligned");
  if (out == x_in) return fail(BEAM_ERR_INVALID_ARG, "out must not alias x_in");
  const beam_moe_params mp = dense_as_moe(*d);
  const Layout L = make_layout(mp);
  if (workspace_bytes < L.total)
    return fail(BEAM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, L.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(x_in);
  if (d->flags & BEAM_FLAG_PRE_NORM) {
    __nv_bfloat16* xn = reinterpret_cast<__nv_bfloat16*>(ws + L.off[L_XN]);
    {
      ProfScope ps("prenorm", st);
      beam::prenorm_kernel<<<(d->T + 7) / 8, 256, 0, st>>>(x, pre_gain, xn, d->T, d->H,
                                                           d->rms_eps);
    }
    BEAM_LAUNCH_CHECK("prenorm_kernel");
    x = xn;
  }
  float* wts = reinterpret_cast<float*>(ws + L.off[L_W]);
  return run_experts(mp, L, x_in, x, nullptr, wts, w, post_gain, out, ws, st, true);
}

}  // namespace

extern "C" {

beam_status_t beam_dense_mlp_forward(const beam_dense_params* d, const void* x_in,
                                     const void* w_gate, const void* w_up, const void* w_down,
                                     const float* pre_gain, const float* post_gain, void* out,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  const ExpertWeights w{w_gate, w_up, w_down, nullptr, nullptr, nullptr,
                        nullptr, nullptr, nullptr, beam::KIND_BF16};
  return dense_forward_impl(d, x_in, w, pre_gain, post_gain, out, workspace, workspace_bytes,
                            stream);
}

beam_status_t beam_dense_mlp_forward_fp8(const beam_dense_params* d, const void* x_in,
                                         const void* wq_gate, const float* ws_gate,
                                         const void* wq_up, const float* ws_up,
                                         const void* wq_down, const float* ws_down,
                                         const float* pre_gain, const float* post_gain,
                                         void* out, void* workspace, size_t workspace_bytes,
                                         void* stream) {
  const ExpertWeights w{wq_gate, wq_up, wq_down, ws_gate, ws_up, ws_down,
                        nullptr, nullptr, nullptr, beam::KIND_E4M3};
  return dense_forward_impl(d, x_in, w, pre_gain, post_gain, out, workspace, workspace_bytes,
                            stream);
}

beam_status_t beam_dense_mlp_forward_nvfp4(const beam_dense_params* d, const void* x_in,
                                           const void* wq_gate, const void* wsf_gate,
                                           const float* wg_gate, const void* wq_up,
                                           const void* wsf_up, const float* wg_up,
                                           const void* wq_down, const void* wsf_down,
                                           const float* wg_down, const float* pre_gain,
                                           const float* post_gain, void* out, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  const ExpertWeights w{wq_gate, wq_up, wq_down, wg_gate, wg_up, wg_down,
                        wsf_gate, wsf_up, wsf_down, beam::KIND_NVFP4};
  return dense_forward_impl(d, x_in, w, pre_gain, post_gain, out, workspace, workspace_bytes,
                            stream);
}

beam_status_t beam_residual_step(const void* h_prev, const void* sub_out, int T, int H, int k,
                                 const float* post_gain, float eps, int apply_norm,
                                 int sub_out_is_fp32, void* h_out, void* stream) {
  if (T < 0 || H <= 0 || H % 8) return fail(BEAM_ERR_INVALID_ARG, "T=%d H=%d (H %% 8 == 0)", T, H);
  if (k < 2) return fail(BEAM_ERR_INVALID_ARG, "k=%d: the residual step needs k >= 2", k);
  if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(BEAM_ERR_INVALID_ARG, "eps must be >= 0");
  if (T == 0) return BEAM_OK;
  if (!h_prev || !sub_out || !h_out) return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(h_prev) || !aligned16(sub_out) || !aligned16(h_out) ||
      (post_gain && !aligned16(post_gain)))
    return fail(BEAM_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  if (h_out == sub_out) return fail(BEAM_ERR_INVALID_ARG, "h_out must not alias sub_out");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const double a = std::sqrt((static_cast<double>(k) - 1.0) / k), b = 1.0 / std::sqrt(static_cast<double>(k));
  ProfScope ps("residual_step", st);
  if (sub_out_is_fp32)
    beam::finalize_rows_kernel<float><<<(T + 7) / 8, 256, 0, st>>>(
        static_cast<const float*>(sub_out), static_cast<const __nv_bfloat16*>(h_prev), post_gain,
        static_cast<__nv_bfloat16*>(h_out), T, H, eps, static_cast<float>(a),
        static_cast<float>(b), 1, apply_norm ? 1 : 0);
  else
    beam::finalize_rows_kernel<__nv_bfloat16><<<(T + 7) / 8, 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(sub_out), static_cast<const __nv_bfloat16*>(h_prev),
        post_gain, static_cast<__nv_bfloat16*>(h_out), T, H, eps, static_cast<float>(a),
        static_cast<float>(b), 1, apply_norm ? 1 : 0);
  BEAM_LAUNCH_CHECK("finalize_rows_kernel");
  return BEAM_OK;
}

beam_status_t beam_status(void* stream) {
  BEAM_CUDA_TRY(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int v = 0;
  BEAM_CUDA_TRY(cudaMemcpyFromSymbol(&v, beam::g_beam_err, sizeof(int)));
  if (v == 0) return BEAM_OK;
  const int zero = 0;
  BEAM_CUDA_TRY(cudaMemcpyToSymbol(beam::g_beam_err, &zero, sizeof(int)));
  if (v & beam::DEV_ERR_ALIGN)
    return fail(BEAM_ERR_DEVICE_FLAG, "a device-side copy address was misaligned and skipped (flag 0x%x)", v);
  if (v & beam::DEV_ERR_TIMEOUT) return fail(BEAM_ERR_TIMEOUT, "a device-side wait timed out (flag 0x%x)", v);
  if (v & beam::DEV_ERR_INDEX)
    return fail(BEAM_ERR_DEVICE_FLAG,
                "a given expert index was outside [0, E); its pair was dropped (flag 0x%x)", v);
  return fail(BEAM_ERR_DEVICE_FLAG, "device error flag 0x%x", v);
}

void beam_profile_enable(int on) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  g_prof_on = on != 0;
}

int beam_profile_read(char* names, size_t names_len, double* total_ms, int* launches,
                      int max_entries) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> g(g_prof_mu);
    recs.swap(g_prof_recs);
  }
  std::map<std::string, std::pair<double, int>> agg;
  for (const ProfRec& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.stop) == cudaSuccess &&
        cudaEventElapsedTime(&ms, r.start, r.stop) == cudaSuccess) {
      auto& a = agg[r.name];
      a.first += ms;
      a.second += 1;
    } else {
      cudaGetLastError();
    }
  }
  {
    std::lock_guard<std::mutex> g(g_prof_mu);
    for (const ProfRec& r : recs) {
      g_prof_pool.push_back(r.start);
      g_prof_pool.push_back(r.stop);
    }
  }
  int n = 0;
  size_t used = 0;
  if (names && names_len) names[0] = 0;
  for (const auto& kv : agg) {
    if (n >= max_entries) break;
    const size_t need = kv.first.size() + 1;
    if (names == nullptr || used + need >= names_len) break;
    std::memcpy(names + used, kv.first.c_str(), kv.first.size());
    names[used + kv.first.size()] = '\n';
    used += need;
    names[used] = 0;
    if (total_ms) total_ms[n] = kv.second.first;
    if (launches) launches[n] = kv.second.second;
    ++n;
  }
  return n;
}

beam_status_t beam_debug_wait_timeout(uint64_t timeout_ns, void* stream) {
  beam::debug_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(timeout_ns);
  BEAM_LAUNCH_CHECK("debug_wait_kernel");
  return BEAM_OK;
}

}  // extern "C"

// ===========================================================================
// Attention sublayer (beam_attention_forward).
// ===========================================================================
namespace {

enum { A_XN = 0, A_PROJ, A_Q, A_K, A_VT, A_GATE, A_ATT, A_Y, A_U1, A_U2, A_NU, kAttnEntries };

struct AttnLayout {
  size_t off[kAttnEntries];
  size_t total;
  int Tp, N1, MT1, MT2, groups;
};

beam_status_t check_attn(const beam_attn_params* p) {
  if (p == nullptr) return fail(BEAM_ERR_INVALID_ARG, "params is NULL");
  if (p->T < 0 || p->H <= 0 || p->n_q <= 0 || p->n_kv <= 0)
    return fail(BEAM_ERR_INVALID_ARG, "T=%d H=%d n_q=%d n_kv=%d", p->T, p->H, p->n_q, p->n_kv);
  if (p->T > (1 << 20)) return fail(BEAM_ERR_UNSUPPORTED, "T=%d exceeds 1048576", p->T);
  if (p->head_dim != beam::ATT_D) return fail(BEAM_ERR_UNSUPPORTED, "head_dim must be 128");
  if (p->H % 256 || p->H > 8192) return fail(BEAM_ERR_UNSUPPORTED, "H=%d: a multiple of 256, at most 8192", p->H);
  if (p->n_q % p->n_kv || (p->n_q + p->n_kv) % 2 || p->n_q > 128)
    return fail(BEAM_ERR_UNSUPPORTED, "n_q=%d, n_kv=%d: n_q a multiple of n_kv, n_q + n_kv even, n_q <= 128",
                p->n_q, p->n_kv);
  if (p->window < 0) return fail(BEAM_ERR_INVALID_ARG, "window=%d must be >= 0", p->window);
  if (!(p->rope_theta > 0.f) || !std::isfinite(p->rope_theta))
    return fail(BEAM_ERR_INVALID_ARG, "rope_theta must be positive");
  if (!(p->rms_eps >= 0.f) || !std::isfinite(p->rms_eps)) return fail(BEAM_ERR_INVALID_ARG, "rms_eps");
  if (p->residual_k == 1 || p->residual_k < 0)
    return fail(BEAM_ERR_INVALID_ARG, "residual_k=%d: use 0 (none) or k >= 2", p->residual_k);
  if (p->flags & ~(BEAM_FLAG_PRE_NORM | BEAM_FLAG_FP32_OUT))
    return fail(BEAM_ERR_INVALID_ARG, "unknown flag bits 0x%x", p->flags);
  if ((p->flags & BEAM_FLAG_FP32_OUT) && p->residual_k >= 2)
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_FP32_OUT applies only without the residual step");
  return BEAM_OK;
}

AttnLayout attn_layout(const beam_attn_params& p) {
  AttnLayout L{};
  const size_t T = static_cast<size_t>(p.T);
  L.Tp = (p.T + beam::ATT_BQ - 1) / beam::ATT_BQ * beam::ATT_BQ;
  L.N1 = (2 * p.n_q + 2 * p.n_kv) * beam::ATT_D;
  L.MT1 = L.N1 / 256;
  L.MT2 = p.H / 256;
  L.groups = (p.T + 255) / 256;
  const size_t dq = static_cast<size_t>(p.n_q) * beam::ATT_D;
  size_t sz[kAttnEntries];
  sz[A_XN] = (p.flags & BEAM_FLAG_PRE_NORM) ? T * p.H * 2 : 0;
  sz[A_PROJ] = T * L.N1 * 4;
  sz[A_Q] = static_cast<size_t>(p.n_q) * L.Tp * beam::ATT_D * 2;
  sz[A_K] = static_cast<size_t>(p.n_kv) * L.Tp * beam::ATT_D * 2;
  sz[A_VT] = static_cast<size_t>(p.n_kv) * beam::ATT_D * L.Tp * 2;
  // RoPE (cos, sin) table of the sliding-window layers (the gate logits are
  // read from A_PROJ by the flash epilogue)
  sz[A_GATE] = p.window > 0 ? T * (beam::ATT_D / 2) * sizeof(float2) : 0;
  sz[A_ATT] = T * dq * 2;
  sz[A_Y] = T * p.H * 4;
  sz[A_U1] = static_cast<size_t>(L.MT1) * L.groups * 16;
  sz[A_U2] = static_cast<size_t>(L.MT2) * L.groups * 16;
  sz[A_NU] = 16;
  size_t cur = 0;
  for (int i = 0; i < kAttnEntries; ++i) {
    L.off[i] = cur;
    cur = align_up(cur + sz[i], 1024);
  }
  L.total = cur;
  return L;
}

// y [n, N] (FP32) = x [n, K] W [N, K]^T on the 2-SM pair kernel (one expert).
beam_status_t dense_linear(const void* x, const void* w, int n, int N, int K, float* y,
                           const int4* units, const int* n_units, cudaStream_t st,
                           const char* prof_name) {
  beam_status_t s;
  CUtensorMap m_w, m_x, m_x64;
  if ((s = make_map(&m_w, w, static_cast<uint64_t>(N), K, 128)) != BEAM_OK) return s;
  if ((s = make_map(&m_x, x, static_cast<uint64_t>(n), K, 16)) != BEAM_OK) return s;
  if ((s = make_map(&m_x64, x, static_cast<uint64_t>(n), K, 64)) != BEAM_OK) return s;
  beam::PairArgs a{};
  a.units = units;
  a.n_units = n_units;
  a.k_blocks = K / 64;
  a.w_rows_per_expert = N;
  a.y = y;
  a.out_ld = N;
  a.timeout_ns = kWaitTimeoutNs;
  return launch_gemm_pair<false>(m_w, m_x, m_x64, a, st, prof_name);
}

}  // namespace

extern "C" size_t beam_attention_workspace_size(const beam_attn_params* p) {
  if (check_attn(p) != BEAM_OK) return 0;
  return attn_layout(*p).total;
}

extern "C" int beam_attention_workspace_layout(const beam_attn_params* p, size_t* offsets, int n) {
  if (check_attn(p) != BEAM_OK || offsets == nullptr || n <= 0) return 0;
  const AttnLayout L = attn_layout(*p);
  const int m = n < kAttnEntries ? n : kAttnEntries;
  for (int i = 0; i < m; ++i) offsets[i] = L.off[i];
  return m;
}

extern "C" beam_status_t beam_attention_forward(const beam_attn_params* p, const void* h_in,
                                                const void* w_qkvg, const void* w_o,
                                                const float* q_gain, const float* k_gain,
                                                const float* pre_gain, const float* post_gain,
                                                void* out, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  beam_status_t s = check_attn(p);
  if (s != BEAM_OK) return s;
  if (p->T == 0) return BEAM_OK;
  if (!h_in || !w_qkvg || !w_o || !out || !workspace)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  const void* ptrs[] = {h_in, w_qkvg, w_o, out, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(BEAM_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", q);
  const void* opt[] = {q_gain, k_gain, pre_gain, post_gain};
  for (const void* q : opt)
    if (q && !aligned16(q)) return fail(BEAM_ERR_INVALID_ARG, "gains must be 16-byte aligned");
  if (out == h_in) return fail(BEAM_ERR_INVALID_ARG, "out must not alias h_in");
  const AttnLayout L = attn_layout(*p);
  if (workspace_bytes < L.total)
    return fail(BEAM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, L.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int T = p->T, H = p->H, nq = p->n_q, nkv = p->n_kv;
  const int dq = nq * beam::ATT_D;

  // 1. pre-norm
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(h_in);
  if (p->flags & BEAM_FLAG_PRE_NORM) {
    __nv_bfloat16* xn = reinterpret_cast<__nv_bfloat16*>(ws + L.off[A_XN]);
    {
      ProfScope ps("prenorm", st);
      beam::prenorm_kernel<<<(T + 7) / 8, 256, 0, st>>>(x, pre_gain, xn, T, H, p->rms_eps);
    }
    BEAM_LAUNCH_CHECK("prenorm_kernel");
    x = xn;
  }
  // 2. work lists of the two dense GEMMs, then the fused Q/K/V/gate projection
  int4* u1 = reinterpret_cast<int4*>(ws + L.off[A_U1]);
  int4* u2 = reinterpret_cast<int4*>(ws + L.off[A_U2]);
  int* nu = reinterpret_cast<int*>(ws + L.off[A_NU]);
  beam::linear_units_kernel<<<4, 256, 0, st>>>(T, L.MT1, u1, nu + 0);
  beam::linear_units_kernel<<<4, 256, 0, st>>>(T, L.MT2, u2, nu + 1);
  BEAM_LAUNCH_CHECK("linear_units_kernel");
  float* proj = reinterpret_cast<float*>(ws + L.off[A_PROJ]);
  if ((s = dense_linear(x, w_qkvg, T, L.N1, H, proj, u1, nu + 0, st, "attn_qkvg_proj")) != BEAM_OK)
    return s;
  // 3. QK-norm, RoPE / query scale, V transposed, gate; V^T padding keys zeroed
  __nv_bfloat16* q = reinterpret_cast<__nv_bfloat16*>(ws + L.off[A_Q]);
  __nv_bfloat16* k = reinterpret_cast<__nv_bfloat16*>(ws + L.off[A_K]);
  __nv_bfloat16* vt = reinterpret_cast<__nv_bfloat16*>(ws + L.off[A_VT]);
  const float* gate = proj + static_cast<size_t>(nq + 2 * nkv) * beam::ATT_D;  // gate logits
  if (L.Tp > T)
    BEAM_CUDA_TRY(cudaMemset2DAsync(vt + T, static_cast<size_t>(L.Tp) * 2, 0,
                                    static_cast<size_t>(L.Tp - T) * 2,
                                    static_cast<size_t>(nkv) * beam::ATT_D, st));
  {
    ProfScope ps("attn_prep", st);
    float2* rope_cs = reinterpret_cast<float2*>(ws + L.off[A_GATE]);
    if (p->window > 0) {
      const int n = T * (beam::ATT_D / 2);
      beam::rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(T, p->rope_theta, rope_cs);
    }
    dim3 grid(T, (nq + nkv + 7) / 8);   // query and key heads
    beam::attn_prep_kernel<<<grid, 256, 0, st>>>(proj, T, L.Tp, nq, nkv, q_gain, k_gain,
                                                 p->rms_eps, p->window, rope_cs, q, k, vt);
    beam::attn_vt_kernel<<<dim3((T + 31) / 32, (nkv + 3) / 4), 128, 0, st>>>(proj, T, L.Tp, nq,
                                                                             nkv, vt);
  }
  BEAM_LAUNCH_CHECK("attn_prep_kernel");
  // 4. attention, gated, BF16
  __nv_bfloat16* att = reinterpret_cast<__nv_bfloat16*>(ws + L.off[A_ATT]);
  {
    CUtensorMap m_q, m_k, m_vt;
    if ((s = make_map(&m_q, q, static_cast<uint64_t>(nq) * L.Tp, beam::ATT_D, 128)) != BEAM_OK) return s;
    if ((s = make_map(&m_k, k, static_cast<uint64_t>(nkv) * L.Tp, beam::ATT_D, 128)) != BEAM_OK) return s;
    if ((s = make_map(&m_vt, vt, static_cast<uint64_t>(nkv) * beam::ATT_D, L.Tp, 128)) != BEAM_OK) return s;
    beam::AttnArgs aa{};
    aa.T = T;
    aa.Tp = L.Tp;
    aa.nq = nq;
    aa.nkv = nkv;
    aa.window = p->window;
    aa.n_qt = L.Tp / beam::ATT_BQ;
    aa.n_items = aa.n_qt * nq;
    aa.scale = 1.0f / std::sqrt(static_cast<float>(beam::ATT_D));
    aa.gate = gate;
    aa.gate_ld = (2 * nq + 2 * nkv) * beam::ATT_D;
    aa.out = att;
    aa.timeout_ns = kWaitTimeoutNs;
    if ((s = ensure_smem(reinterpret_cast<const void*>(beam::flash_attn_kernel),
                         beam::AttnCfg::SMEM_BYTES)) != BEAM_OK)
      return s;
    ProfScope ps("flash_attn", st);
    // persistent: one CTA per SM over the (query tile, head) items
    const int grid = std::min(aa.n_items, sm_count());
    beam::flash_attn_kernel<<<grid, beam::ATT_THREADS, beam::AttnCfg::SMEM_BYTES, st>>>(
        m_q, m_k, m_vt, aa);
  }
  BEAM_LAUNCH_CHECK("flash_attn_kernel");
  // 5. output projection (FP32; straight into `out` with BEAM_FLAG_FP32_OUT)
  const bool resid = p->residual_k >= 2;
  float* y = (p->flags & BEAM_FLAG_FP32_OUT) ? static_cast<float*>(out)
                                             : reinterpret_cast<float*>(ws + L.off[A_Y]);
  if ((s = dense_linear(att, w_o, T, H, dq, y, u2, nu + 1, st, "attn_out_proj")) != BEAM_OK) return s;
  // 6. post-norm + scaled residual, or the BF16 output
  if (!(p->flags & BEAM_FLAG_FP32_OUT)) {
    const float kf = static_cast<float>(resid ? p->residual_k : 2);
    const float a = resid ? std::sqrt((kf - 1.f) / kf) : 0.f;
    const float b = resid ? 1.f / std::sqrt(kf) : 1.f;
    ProfScope ps("attn_finalize", st);
    beam::finalize_rows_kernel<float><<<(T + 7) / 8, 256, 0, st>>>(
        y, static_cast<const __nv_bfloat16*>(h_in), post_gain, static_cast<__nv_bfloat16*>(out), T,
        H, p->rms_eps, a, b, resid ? 1 : 0, resid ? 1 : 0);
    BEAM_LAUNCH_CHECK("finalize_rows_kernel");
  }
  return BEAM_OK;
}

// ===========================================================================
// Allocation-free router (beam_moe_route_static).
//
// Its scratch -- the router's partial logits and, with BEAM_FLAG_PRE_NORM,
// the normalised x -- lives in this file-scope device array of
// BEAM_ROUTE_STATIC_SCRATCH_BYTES bytes. Every device that loads the library
// holds the array until the process exits. Host code must not pass the
// array's name to a kernel (on the host it names a stand-in, not device
// memory): the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and passed to the kernels.
// ===========================================================================
static __device__ __align__(256) unsigned char g_route_static_scratch[BEAM_ROUTE_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_route_static_mu;
void* g_route_static_addr[kMaxDevices] = {};
unsigned long long g_route_static_ctx[kMaxDevices] = {};

// Unique ID of the context current on this thread (driver entry points found
// at run time, as for the tensor-map encoder); false when none is current or
// the driver lacks the calls.
bool current_context_id(unsigned long long* id) {
  typedef CUresult (*PFN_ctxGetCurrent_t)(CUcontext*);
  typedef CUresult (*PFN_ctxGetId_t)(CUcontext, unsigned long long*);
  static PFN_ctxGetCurrent_t get_current = nullptr;
  static PFN_ctxGetId_t get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p1 = nullptr;
    void* p2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p1, 12000, cudaEnableDefault, &q1) ==
            cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &p2, 12000, cudaEnableDefault, &q2) ==
            cudaSuccess &&
        q2 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<PFN_ctxGetCurrent_t>(p1);
      get_id = reinterpret_cast<PFN_ctxGetId_t>(p2);
    } else {
      cudaGetLastError();
    }
  });
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the static scratch on the current device. It is looked
// up with cudaGetSymbolAddress (with the device current) on the first call
// for the device and again whenever the device's context has changed since
// (a cudaDeviceReset destroys the context the cached address belonged to);
// otherwise the cached address is used.
beam_status_t route_static_scratch(void** addr) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(BEAM_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return fail(BEAM_ERR_UNSUPPORTED, "device ordinal %d is beyond %d", dev, kMaxDevices);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> g(g_route_static_mu);
  if (!have_id || g_route_static_addr[dev] == nullptr || g_route_static_ctx[dev] != id) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_route_static_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(BEAM_ERR_CUDA, "cudaGetSymbolAddress of the router scratch failed: %s",
                  cudaGetErrorString(e));
    // the lookup made the device's primary context current if none was
    unsigned long long id2 = 0;
    g_route_static_addr[dev] = ptr;
    g_route_static_ctx[dev] = current_context_id(&id2) ? id2 : 0;
  }
  *addr = g_route_static_addr[dev];
  return BEAM_OK;
}

}  // namespace

extern "C" beam_status_t beam_moe_route_static(const beam_moe_params* p, const void* x,
                                               const float* w_router, const float* logit_bias,
                                               const float* pre_gain, int32_t* topk_idx,
                                               float* topk_w, float* scores, void* stream) {
  beam_status_t s = check_params(p);
  if (s != BEAM_OK) return s;
  if (p->T == 0) return BEAM_OK;
  if (!x || !w_router || !topk_idx || !topk_w)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if ((p->flags & BEAM_FLAG_RETURN_SCORES) && !scores)
    return fail(BEAM_ERR_INVALID_ARG, "BEAM_FLAG_RETURN_SCORES needs a scores buffer");
  if (!aligned16(x) || !aligned16(w_router) || (pre_gain && !aligned16(pre_gain)))
    return fail(BEAM_ERR_INVALID_ARG, "x, w_router and pre_gain must be 16-byte aligned");
  // Same K-slicing as beam_moe_route, so both entry points give identical results.
  Layout L{};
  L.KS = choose_router_ks(*p, sm_count());
  const size_t part = align_up(static_cast<size_t>(L.KS) * p->T * p->E * 4, 256);
  const size_t xn = align_up(
      (p->flags & BEAM_FLAG_PRE_NORM) ? static_cast<size_t>(p->T) * p->H * 2 : 0, 256);
  const size_t wr3 =
      router_on_tensor_cores(*p) ? static_cast<size_t>(p->E) * 3 * p->H * 2 : 0;
  const size_t ru = router_on_tensor_cores(*p) ? align_up(router_units_bytes(*p), 256) : 0;
  if (part + xn + wr3 + ru > BEAM_ROUTE_STATIC_SCRATCH_BYTES)
    return fail(BEAM_ERR_UNSUPPORTED,
                "T=%d needs %zu bytes of router scratch; the static scratch holds %zu bytes "
                "(use beam_moe_route with a workspace for this size)",
                p->T, part + xn + wr3 + ru, static_cast<size_t>(BEAM_ROUTE_STATIC_SCRATCH_BYTES));
  void* base = nullptr;
  if ((s = route_static_scratch(&base)) != BEAM_OK) return s;
  L.off[L_PART] = 0;
  L.off[L_XN] = part;
  L.off[L_WR3] = part + xn;
  L.off[L_RUNITS] = part + xn + wr3;
  return launch_router(*p, L, x, w_router, logit_bias, pre_gain, topk_idx, topk_w,
                       (p->flags & BEAM_FLAG_RETURN_SCORES) ? scores : nullptr,
                       static_cast<uint8_t*>(base), static_cast<cudaStream_t>(stream));
}

// ===========================================================================
// Expert parallelism: the sublayer split by expert across ranks (routed
// forward on the expert owners, dispatch and combine on the token owners).
// ===========================================================================
extern "C" beam_status_t beam_moe_forward_routed(const beam_moe_params* p, const void* x_in,
                                                 const int32_t* topk_idx, const float* topk_w,
                                                 const void* w_gate, const void* w_up,
                                                 const void* w_down, const float* pre_gain,
                                                 const float* post_gain, void* out, void* workspace,
                                                 size_t workspace_bytes, void* stream) {
  beam_status_t s = check_params(p);
  if (s != BEAM_OK) return s;
  if (p->flags & (BEAM_FLAG_FP8_EXPERTS | BEAM_FLAG_NVFP4_EXPERTS))
    return fail(BEAM_ERR_UNSUPPORTED, "beam_moe_forward_routed takes BF16 experts");
  if (p->T == 0) return BEAM_OK;
  if (!x_in || !topk_idx || !topk_w || !w_gate || !w_up || !w_down || !out || !workspace)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  const void* ptrs[] = {x_in, topk_idx, topk_w, w_gate, w_up, w_down, out, workspace};
  for (const void* q : ptrs)
    if (!aligned16(q)) return fail(BEAM_ERR_INVALID_ARG, "pointer %p is not 16-byte aligned", q);
  if ((pre_gain && !aligned16(pre_gain)) || (post_gain && !aligned16(post_gain)))
    return fail(BEAM_ERR_INVALID_ARG, "gains must be 16-byte aligned");
  if (out == x_in) return fail(BEAM_ERR_INVALID_ARG, "out must not alias x_in");
  const Layout L = make_layout(*p);
  if (workspace_bytes < L.total)
    return fail(BEAM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, L.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* idx = reinterpret_cast<int32_t*>(ws + L.off[L_IDX]);
  float* wts = reinterpret_cast<float*>(ws + L.off[L_W]);
  const long long n = static_cast<long long>(p->T) * p->top_k;
  {
    ProfScope ps("routed_copy", st);
    beam::routed_copy_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
        topk_idx, topk_w, n, p->E, idx, wts);
  }
  BEAM_LAUNCH_CHECK("routed_copy_kernel");
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(x_in);
  if (p->flags & BEAM_FLAG_PRE_NORM) {
    __nv_bfloat16* xn = reinterpret_cast<__nv_bfloat16*>(ws + L.off[L_XN]);
    {
      ProfScope ps("prenorm", st);
      beam::prenorm_kernel<<<(p->T + 7) / 8, 256, 0, st>>>(x, pre_gain, xn, p->T, p->H, p->rms_eps);
    }
    BEAM_LAUNCH_CHECK("prenorm_kernel");
    x = xn;
  }
  ExpertWeights w{};
  w.gate = w_gate;
  w.up = w_up;
  w.down = w_down;
  w.kind = beam::KIND_BF16;
  return run_experts(*p, L, x_in, x, idx, wts, w, post_gain, out, ws, st, false);
}

extern "C" beam_status_t beam_ep_dispatch(const beam_moe_params* p, int n_ranks, const void* x,
                                          const int32_t* topk_idx, void* send_x,
                                          int32_t* send_expert, int32_t* pair_row,
                                          int32_t* send_counts, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  beam_status_t s = check_params(p);
  if (s != BEAM_OK) return s;
  if (n_ranks <= 0 || p->E % n_ranks)
    return fail(BEAM_ERR_INVALID_ARG, "n_ranks=%d must divide E=%d", n_ranks, p->E);
  if (p->T == 0) {
    // a rank without tokens sends no rows to every rank
    if (send_counts != nullptr)
      BEAM_CUDA_TRY(cudaMemsetAsync(send_counts, 0, static_cast<size_t>(n_ranks) * sizeof(int32_t),
                                    static_cast<cudaStream_t>(stream)));
    return BEAM_OK;
  }
  if (!x || !topk_idx || !send_x || !send_expert || !pair_row || !send_counts || !workspace)
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(x) || !aligned16(send_x) || !aligned16(workspace))
    return fail(BEAM_ERR_INVALID_ARG, "x, send_x and the workspace must be 16-byte aligned");
  const Layout L = make_layout(*p);
  if (workspace_bytes < L.total)
    return fail(BEAM_ERR_WORKSPACE, "workspace of %zu bytes is smaller than the %zu needed",
                workspace_bytes, L.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const long long R = static_cast<long long>(p->T) * p->top_k;
  int32_t* idx = reinterpret_cast<int32_t*>(ws + L.off[L_IDX]);
  float* wts = reinterpret_cast<float*>(ws + L.off[L_W]);
  int* blk_hist = reinterpret_cast<int*>(ws + L.off[L_BLKHIST]);
  int* blk_off = reinterpret_cast<int*>(ws + L.off[L_BLKOFF]);
  int* counts = reinterpret_cast<int*>(ws + L.off[L_COUNTS]);
  int* offs = reinterpret_cast<int*>(ws + L.off[L_OFFS]);
  int* row_tok = reinterpret_cast<int*>(ws + L.off[L_ROWTOK]);
  float* row_w = reinterpret_cast<float*>(ws + L.off[L_ROWW]);
  int4* ugu = reinterpret_cast<int4*>(ws + L.off[L_UGU]);
  int* nunits = reinterpret_cast<int*>(ws + L.off[L_NUNITS]);
  // the caller's routing, range-checked (weights are not needed here)
  {
    ProfScope ps("routed_copy", st);
    beam::routed_copy_kernel<<<static_cast<unsigned>((R + 255) / 256), 256, 0, st>>>(
        topk_idx, wts, R, p->E, idx, wts);
  }
  BEAM_LAUNCH_CHECK("routed_copy_kernel");
  {
    ProfScope ps("expert_hist", st);
    beam::expert_block_hist_kernel<<<L.NB, beam::PERM_THREADS, 0, st>>>(idx, p->T, p->top_k,
                                                                        p->E, blk_hist);
  }
  BEAM_LAUNCH_CHECK("expert_block_hist_kernel");
  {
    ProfScope ps("expert_scan_units", st);
    beam::expert_scan_units_kernel<<<1, 256, 0, st>>>(blk_hist, L.NB, p->E, blk_off, counts, offs,
                                                      ugu, nunits, L.NT, p->I / 128,
                                                      path_mt_down(L.path, p->H, L.f4), 1, row_tok);
  }
  BEAM_LAUNCH_CHECK("expert_scan_units_kernel");
  {
    ProfScope ps("expert_scatter", st);
    beam::expert_scatter_kernel<<<L.NB, beam::PERM_THREADS, 0, st>>>(
        idx, wts, p->T, p->top_k, p->E, blk_off, pair_row, row_tok, row_w);
  }
  BEAM_LAUNCH_CHECK("expert_scatter_kernel");
  {
    ProfScope ps("gather_rows", st);
    beam::gather_rows_kernel<<<static_cast<unsigned>((R + 7) / 8), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(x), row_tok, static_cast<int>(R), p->H,
        static_cast<__nv_bfloat16*>(send_x));
  }
  BEAM_LAUNCH_CHECK("gather_rows_kernel");
  {
    ProfScope ps("ep_meta", st);
    beam::ep_meta_kernel<<<static_cast<unsigned>((R + 255) / 256), 256, 0, st>>>(
        offs, p->E, n_ranks, R, send_expert, send_counts);
  }
  BEAM_LAUNCH_CHECK("ep_meta_kernel");
  return BEAM_OK;
}

extern "C" beam_status_t beam_ep_combine(int T, int top_k, int H, const float* recv_y,
                                         const int32_t* pair_row, const float* topk_w,
                                         const void* h_prev, const float* post_gain, float eps,
                                         int residual_k, int out_f32, void* out, void* stream) {
  if (T < 0 || H <= 0 || top_k <= 0 || top_k > 32)
    return fail(BEAM_ERR_INVALID_ARG, "T=%d H=%d top_k=%d out of range", T, H, top_k);
  if (H % 128 || H > 8192) return fail(BEAM_ERR_UNSUPPORTED, "H=%d must be a multiple of 128, at most 8192", H);
  if (residual_k == 1 || residual_k < 0)
    return fail(BEAM_ERR_INVALID_ARG, "residual_k=%d: use 0 (none) or k >= 2", residual_k);
  if (out_f32 && residual_k >= 2)
    return fail(BEAM_ERR_INVALID_ARG, "an FP32 output applies only without the residual step");
  if (T == 0) return BEAM_OK;
  if (!recv_y || !pair_row || !topk_w || !out || (residual_k >= 2 && !h_prev))
    return fail(BEAM_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(recv_y) || !aligned16(out) || (h_prev && !aligned16(h_prev)) ||
      (post_gain && !aligned16(post_gain)))
    return fail(BEAM_ERR_INVALID_ARG, "recv_y, out, h_prev and post_gain must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int resid = residual_k >= 2;
  const float kf = static_cast<float>(resid ? residual_k : 2);
  const float a = resid ? std::sqrt((kf - 1.f) / kf) : 0.f;
  const float b = resid ? 1.f / std::sqrt(kf) : 1.f;
  ProfScope ps("ep_combine", st);
  if (out_f32)
    beam::ep_combine_kernel<true><<<T, beam::EP_COMBINE_THREADS, 0, st>>>(
        recv_y, pair_row, topk_w, top_k, static_cast<const __nv_bfloat16*>(h_prev), post_gain,
        out, H, eps, a, b, resid);
  else
    beam::ep_combine_kernel<false><<<T, beam::EP_COMBINE_THREADS, 0, st>>>(
        recv_y, pair_row, topk_w, top_k, static_cast<const __nv_bfloat16*>(h_prev), post_gain,
        out, H, eps, a, b, resid);
  BEAM_LAUNCH_CHECK("ep_combine_kernel");
  return BEAM_OK;
}
