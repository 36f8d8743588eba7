// api.cu -- the extern "C" entry points of libgmlp.so declared in
// include/gmlp.h: host-side argument checks (a status before any launch,
// replacing the silent unfused fallback and its warning described in PR #3631
// "Add NVTE_CUTEDSL_FUSED_GROUPED_MLP_WARN_FALLBACK", Changes), workspace
// carving and the launch sequence of each call.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "internal.h"

namespace gmlp {

int quant_read_clear_status();
int gemm_read_clear_status();
int peak_read_clear_status();
int wgrad_read_clear_status();

namespace {

thread_local char g_last_error[512] = "";

gmlp_status fail(gmlp_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return st;
}

gmlp_status cuda_fail(cudaError_t e, const char* where) {
  return fail(GMLP_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// y, dx and the activation input are written or read in 32-byte vectors
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31) == 0; }

size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

// Largest feature count (K, N, weight rows / cols) a call accepts: far past
// any model's hidden or ffn size, and small enough that every per-row count
// the kernels keep in 32 bits (16-byte chunks, scale blocks, TMA coordinates)
// cannot overflow.
constexpr int64_t kMaxFeatures = int64_t(1) << 20;

gmlp_status check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  static int cached[64] = {};  // 0 unknown, 1 ok, 2 bad
  if (dev < 64 && cached[dev] == 1) return GMLP_OK;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3)
    return fail(GMLP_ERR_UNSUPPORTED_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                major, minor);
  if (dev < 64) cached[dev] = 1;
  return GMLP_OK;
}

gmlp_status check_groups(int32_t G, int64_t M, const int64_t* split_sizes) {
  if (G < 1 || G > kMaxGroups) return fail(GMLP_ERR_INVALID_DIMS, "G = %d outside [1, %d]", G, kMaxGroups);
  if (M < 0 || M > (int64_t)0x7FFFFFFF) return fail(GMLP_ERR_INVALID_DIMS, "M = %lld outside [0, 2^31)", (long long)M);
  if (!split_sizes) return fail(GMLP_ERR_INVALID_ARG, "split_sizes is NULL");
  if ((reinterpret_cast<uintptr_t>(split_sizes) & 7) != 0)
    return fail(GMLP_ERR_INVALID_ARG, "split_sizes is not 8-byte aligned");
  return GMLP_OK;
}

#define GMLP_TRY(expr)                 \
  do {                                 \
    gmlp_status st_ = (expr);          \
    if (st_ != GMLP_OK) return st_;    \
  } while (0)

#define GMLP_CUDA(expr, where)                         \
  do {                                                 \
    cudaError_t e_ = (expr);                           \
    if (e_ != cudaSuccess) return cuda_fail(e_, where); \
  } while (0)

size_t tiled_bytes(int64_t M, int32_t G, int64_t nscale) {
  return (size_t)((M + 127) / 128 + G) * 128 * (size_t)nscale;
}

struct FwdLayout {
  size_t x_codes, x_scales, f_codes, f_scales, f_bf16, amax, total;
};

FwdLayout fwd_layout(int64_t M, int64_t K, int64_t N, int32_t G, int fmt) {
  FwdLayout L{};
  size_t cur = 0;
  auto take = [&](size_t b) {
    size_t o = cur;
    cur += align256(b);
    return o;
  };
  const int blk = fmt == GMLP_MXFP8 ? 32 : 16;
  const int cdiv = fmt == GMLP_MXFP8 ? 1 : 2;
  L.x_codes = take((size_t)M * K / cdiv);
  L.x_scales = take(tiled_bytes(M, G, K / blk));
  L.f_codes = take((size_t)M * N / cdiv);
  L.f_scales = take(tiled_bytes(M, G, N / blk));
  if (fmt == GMLP_NVFP4) {
    L.f_bf16 = take((size_t)M * N * 2);
    L.amax = take((size_t)3 * G * sizeof(float));
  }
  L.total = cur;
  return L;
}

struct BwdLayout {
  size_t dy_codes, dy_scales, g_codes, g_scales, total;
};

// backward workspace: dy (MXFP8 rowwise, GEMM_TILED scales) and fc1_dy (same)
BwdLayout bwd_layout(int64_t M, int64_t K, int64_t N1, int32_t G) {
  BwdLayout L{};
  size_t cur = 0;
  auto take = [&](size_t b) {
    size_t o = cur;
    cur += align256(b);
    return o;
  };
  L.dy_codes = take((size_t)M * K);
  L.dy_scales = take(tiled_bytes(M, G, K / 32));
  L.g_codes = take((size_t)M * N1);
  L.g_scales = take(tiled_bytes(M, G, N1 / 32));
  L.total = cur;
  return L;
}

// weight-gradient workspace: four columnwise MXFP8 operands ([C][T] codes and
// their GEMM_TILED scales) with T = 128 x (chunk capacity of M tokens in G groups)
struct WgradLayout {
  int64_t T;
  size_t dy_c, dy_s, f_c, f_s, g_c, g_s, x_c, x_s, total;
};

WgradLayout wgrad_layout(int64_t M, int64_t K, int64_t N, int64_t N1, int32_t G) {
  WgradLayout L{};
  L.T = gmlp_colwise_tokens(M, G);
  size_t cur = 0;
  auto take = [&](size_t b) {
    size_t o = cur;
    cur += align256(b);
    return o;
  };
  L.dy_c = take((size_t)K * L.T);
  L.dy_s = take((size_t)K * L.T / 32);
  L.f_c = take((size_t)N * L.T);
  L.f_s = take((size_t)N * L.T / 32);
  L.g_c = take((size_t)N1 * L.T);
  L.g_s = take((size_t)N1 * L.T / 32);
  L.x_c = take((size_t)K * L.T);
  L.x_s = take((size_t)K * L.T / 32);
  L.total = cur;
  return L;
}

gmlp_status check_recipe(const gmlp_recipe* r) {
  if (!r) return fail(GMLP_ERR_INVALID_ARG, "recipe is NULL");
  if (r->format != GMLP_MXFP8 && r->format != GMLP_NVFP4)
    return fail(GMLP_ERR_UNSUPPORTED_RECIPE, "recipe format %d is neither MXFP8 nor NVFP4", r->format);
  if (r->scale_layout != GMLP_SCALES_COMPACT && r->scale_layout != GMLP_SCALES_GEMM_TILED)
    return fail(GMLP_ERR_INVALID_ARG, "scale_layout %d unknown", r->scale_layout);
  return GMLP_OK;
}

gmlp_status check_qtensor(const gmlp_qtensor* t, const char* what) {
  if (!t) return GMLP_OK;
  if (!t->codes || !t->scales) return fail(GMLP_ERR_INVALID_ARG, "%s codes/scales NULL", what);
  if (!aligned16(t->codes) || !aligned16(t->scales))
    return fail(GMLP_ERR_INVALID_ARG, "%s codes/scales not 16-byte aligned", what);
  return GMLP_OK;
}

}  // namespace

// Error text for entry points defined in other files of the library.
gmlp_status set_last_error(gmlp_status st, const char* msg) { return fail(st, "%s", msg); }

int num_sms() {
  static int cached[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && cached[dev]) return cached[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev < 64) cached[dev] = n;
  return n;
}

}  // namespace gmlp

using namespace gmlp;

// Weight quantisation of G experts, either stacked (Wp[0] -> [G][rows][cols])
// or one pointer per expert (discrete: Wp[g] -> [rows][cols]); the outputs
// are the same stacked codes, GEMM_TILED scales (expert g's tiles from g *
// rows / 128) and per-expert amax / global scale.
static gmlp_status prepare_weights_impl(const uint16_t* const* Wp, bool discrete, int32_t G, int64_t rows,
                                        int64_t cols, int32_t swiglu_interleave, int32_t format, uint8_t* codes,
                                        uint8_t* scales, float* global_scale, float* amax, cudaStream_t s) {
  if (G < 1 || G > kMaxGroups) return fail(GMLP_ERR_INVALID_DIMS, "G = %d outside [1, %d]", G, kMaxGroups);
  if (format != GMLP_MXFP8 && format != GMLP_NVFP4) return fail(GMLP_ERR_UNSUPPORTED_RECIPE, "format %d", format);
  if (rows <= 0 || rows % 128 || rows > kMaxFeatures || (int64_t)G * rows > 0x7FFFFFFF)
    return fail(GMLP_ERR_INVALID_DIMS, "rows = %lld must be a positive multiple of 128, at most 2^20", (long long)rows);
  const int64_t cmod = format == GMLP_MXFP8 ? 128 : 256;
  if (cols <= 0 || cols % cmod || cols > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "cols = %lld must be a positive multiple of %lld, at most 2^20", (long long)cols,
                (long long)cmod);
  if (swiglu_interleave && rows % 64) return fail(GMLP_ERR_INVALID_DIMS, "SwiGLU interleave needs rows %% 64 == 0");
  const int n_src = discrete ? G : 1;
  for (int i = 0; i < n_src; ++i)
    if (!Wp[i] || !aligned16(Wp[i])) return fail(GMLP_ERR_INVALID_ARG, "weight %d NULL or not 16-byte aligned", i);
  if (!codes || !scales || !aligned16(codes) || !aligned16(scales))
    return fail(GMLP_ERR_INVALID_ARG, "codes/scales NULL or not 16-byte aligned");
  if (format == GMLP_NVFP4 && (!global_scale || !amax))
    return fail(GMLP_ERR_INVALID_ARG, "NVFP4 weights need global_scale and amax buffers");
  GMLP_TRY(check_device());
  const int64_t code_bytes = rows * cols / (format == GMLP_MXFP8 ? 1 : 2);           // per expert
  const int64_t scale_bytes = rows / 128 * (cols / (format == GMLP_MXFP8 ? 32 : 16) / 4) * 512;
  const int calls = discrete ? G : 1;
  const int32_t Gc = discrete ? 1 : G;
  for (int i = 0; i < calls; ++i) {
    GroupSrc gs{nullptr, (int32_t)rows, Gc, (int64_t)Gc * rows};
    RowQuantArgs a{};
    a.x = Wp[i];
    a.M = (int64_t)Gc * rows;
    a.K = cols;
    a.grp = gs;
    a.format = format;
    a.tiled = 1;
    a.codes = codes + i * code_bytes;
    a.scales = scales + i * scale_bytes;
    a.swiglu_interleave = swiglu_interleave != 0;
    if (format == GMLP_NVFP4) {
      GMLP_CUDA(launch_group_amax(Wp[i], a.M, cols, gs, amax + i, s), "group_amax launch");
      a.amax = amax + i;
      a.S_out = global_scale + i;
    }
    GMLP_CUDA(launch_row_quant(a, s), "row_quant launch");
  }
  return GMLP_OK;
}

extern "C" {

const char* gmlp_last_error(void) { return g_last_error; }

const char* gmlp_version(void) { return "gmlp 0.1 (sm_103a)"; }

size_t gmlp_tiled_scales_bytes(int64_t M, int32_t G, int64_t nscale) {
  if (M < 0 || G < 0 || nscale < 0) return 0;
  return tiled_bytes(M, G, nscale);
}

gmlp_status gmlp_group_hadamard_amax(const uint16_t* x, int64_t M, int64_t K, const int64_t* split_sizes,
                                     int32_t G, uint32_t rht_sign_mask, float* amax_pre, float* amax_post,
                                     gmlp_stream stream) {
  g_last_error[0] = 0;
  GMLP_TRY(check_groups(G, M, split_sizes));
  if (K <= 0 || K % 128 || K > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "K = %lld must be a positive multiple of 128, at most 2^20", (long long)K);
  if ((M > 0 && !x) || !amax_pre || !amax_post) return fail(GMLP_ERR_INVALID_ARG, "NULL pointer argument");
  if (!aligned16(x) || !aligned16(amax_pre) || !aligned16(amax_post))
    return fail(GMLP_ERR_INVALID_ARG, "pointer not 16-byte aligned");
  GMLP_TRY(check_device());
  GroupSrc gs{split_sizes, 0, G, M};
  GMLP_CUDA(launch_hadamard_amax(x, M, K, gs, rht_sign_mask, amax_pre, amax_post, (cudaStream_t)stream),
            "hadamard_amax launch");
  return GMLP_OK;
}

// An NVFP4 amax pass followed by a row cast of the same x: both on the cast's
// grid, the amax pass reading the last ~80 MB of its warps' shares with an L2
// evict-last policy, the cast (reverse = 1) sweeping its shares backwards
// into them.
static float nvfp4_amax_keep(int64_t M, int64_t K) {
  const double x_bytes = 2.0 * (double)M * (double)K;
  return x_bytes > 0 ? (float)std::min(1.0, 80e6 / x_bytes) : 0.0f;
}

static gmlp_status quantize_with_amax_impl(const uint16_t* x, int64_t M, int64_t K, const int64_t* split_sizes,
                                           int32_t G, const gmlp_recipe* r, const float* amax_pre,
                                           const float* amax_post, const gmlp_qtensor* row_out,
                                           const gmlp_qtensor* col_out, cudaStream_t s) {
  GroupSrc gs{split_sizes, 0, G, M};
  if (r->format == GMLP_MXFP8) {
    if (row_out) {
      RowQuantArgs a{};
      a.x = x;
      a.M = M;
      a.K = K;
      a.grp = gs;
      a.format = GMLP_MXFP8;
      a.tiled = r->scale_layout == GMLP_SCALES_GEMM_TILED;
      a.codes = row_out->codes;
      a.scales = row_out->scales;
      GMLP_CUDA(launch_row_quant(a, s), "row_quant launch");
    }
    if (col_out) {
      ColqArgs q{};
      q.src = x;
      q.ld = K;
      q.C = K;
      q.grp = gs;
      q.T = gmlp_colwise_tokens(M, G);
      q.codes = col_out->codes;
      q.scales = col_out->scales;
      q.mode = COLQ_PLAIN;
      GMLP_CUDA(launch_colq(q, s), "columnwise MXFP8 launch");
    }
    return GMLP_OK;
  }
  if (col_out) {
    ColQuantArgs c{};
    c.x = x;
    c.M = M;
    c.K = K;
    c.grp = gs;
    c.use_rht = r->use_rht != 0;
    c.mask = r->rht_sign_mask & 0xFFFFu;
    c.amax_row = amax_pre;
    c.amax_col = r->use_rht ? amax_post : amax_pre;
    c.row_codes = row_out ? row_out->codes : nullptr;
    c.row_scales = row_out ? row_out->scales : nullptr;
    c.row_tiled = r->scale_layout == GMLP_SCALES_GEMM_TILED;
    c.col_codes = col_out->codes;
    c.col_scales = col_out->scales;
    GMLP_CUDA(launch_col_quant(c, s), "col_quant launch");
    return GMLP_OK;
  }
  RowQuantArgs a{};
  a.x = x;
  a.M = M;
  a.K = K;
  a.grp = gs;
  a.format = GMLP_NVFP4;
  a.tiled = r->scale_layout == GMLP_SCALES_GEMM_TILED;
  a.codes = row_out->codes;
  a.scales = row_out->scales;
  a.amax = amax_pre;
  a.reverse = 1;  // pairs with gmlp_group_quantize's amax pass (any order is correct)
  GMLP_CUDA(launch_row_quant(a, s), "row_quant launch");
  return GMLP_OK;
}

static gmlp_status check_quant_args(const uint16_t* x, int64_t M, int64_t K, const int64_t* split_sizes, int32_t G,
                                    const gmlp_recipe* recipe, const gmlp_qtensor* row_out,
                                    const gmlp_qtensor* col_out) {
  GMLP_TRY(check_groups(G, M, split_sizes));
  GMLP_TRY(check_recipe(recipe));
  if (K <= 0 || K % 128 || K > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "K = %lld must be a positive multiple of 128, at most 2^20", (long long)K);
  if (M > 0 && !x) return fail(GMLP_ERR_INVALID_ARG, "x is NULL");
  if (!aligned16(x)) return fail(GMLP_ERR_INVALID_ARG, "x not 16-byte aligned");
  if (!row_out && !col_out) return fail(GMLP_ERR_INVALID_ARG, "neither row_out nor col_out given");
  if (recipe->format == GMLP_MXFP8 && col_out && (!aligned32(col_out->codes) || !aligned32(col_out->scales)))
    return fail(GMLP_ERR_INVALID_ARG, "columnwise MXFP8 codes / scales not 32-byte aligned");
  GMLP_TRY(check_qtensor(row_out, "row_out"));
  GMLP_TRY(check_qtensor(col_out, "col_out"));
  return GMLP_OK;
}

gmlp_status gmlp_group_quantize_with_amax(const uint16_t* x, int64_t M, int64_t K, const int64_t* split_sizes,
                                          int32_t G, const gmlp_recipe* recipe, const float* amax_pre,
                                          const float* amax_post, const gmlp_qtensor* row_out,
                                          const gmlp_qtensor* col_out, gmlp_stream stream) {
  g_last_error[0] = 0;
  GMLP_TRY(check_quant_args(x, M, K, split_sizes, G, recipe, row_out, col_out));
  if (recipe->format == GMLP_NVFP4) {
    if (!amax_pre) return fail(GMLP_ERR_INVALID_ARG, "NVFP4 needs amax_pre");
    if (col_out && recipe->use_rht && !amax_post) return fail(GMLP_ERR_INVALID_ARG, "RHT columnwise needs amax_post");
  }
  GMLP_TRY(check_device());
  return quantize_with_amax_impl(x, M, K, split_sizes, G, recipe, amax_pre, amax_post, row_out, col_out,
                                 (cudaStream_t)stream);
}

gmlp_status gmlp_group_quantize(const uint16_t* x, int64_t M, int64_t K, const int64_t* split_sizes, int32_t G,
                                const gmlp_recipe* recipe, const gmlp_qtensor* row_out,
                                const gmlp_qtensor* col_out, float* amax_pre, float* amax_post,
                                gmlp_stream stream) {
  g_last_error[0] = 0;
  GMLP_TRY(check_quant_args(x, M, K, split_sizes, G, recipe, row_out, col_out));
  const bool hadamard = recipe->format == GMLP_NVFP4 && col_out && recipe->use_rht;
  if (recipe->format == GMLP_NVFP4) {
    if (!amax_pre || (hadamard && !amax_post))
      return fail(GMLP_ERR_INVALID_ARG, "NVFP4 needs amax_pre (and amax_post for the RHT columnwise output)");
    if (!aligned16(amax_pre) || !aligned16(amax_post)) return fail(GMLP_ERR_INVALID_ARG, "amax not 16-byte aligned");
  }
  GMLP_TRY(check_device());
  cudaStream_t s = (cudaStream_t)stream;
  GroupSrc gs{split_sizes, 0, G, M};
  if (hadamard) {
    GMLP_CUDA(launch_hadamard_amax(x, M, K, gs, recipe->rht_sign_mask, amax_pre, amax_post, s), "hadamard_amax launch");
  } else if (recipe->format == GMLP_NVFP4) {
    const int grid = row_quant_grid(GMLP_NVFP4, recipe->scale_layout == GMLP_SCALES_GEMM_TILED, M);
    GMLP_CUDA(launch_group_amax(x, M, K, gs, amax_pre, s, grid, nvfp4_amax_keep(M, K)), "group_amax launch");
  }
  return quantize_with_amax_impl(x, M, K, split_sizes, G, recipe, amax_pre, amax_post, row_out, col_out, s);
}

gmlp_status gmlp_prepare_weights(const uint16_t* W, int32_t G, int64_t rows, int64_t cols, int32_t swiglu_interleave,
                                 int32_t format, uint8_t* codes, uint8_t* scales, float* global_scale, float* amax,
                                 gmlp_stream stream) {
  g_last_error[0] = 0;
  return prepare_weights_impl(&W, false, G, rows, cols, swiglu_interleave, format, codes, scales, global_scale, amax,
                              (cudaStream_t)stream);
}

gmlp_status gmlp_prepare_weights_discrete(const uint16_t* const* W_experts, int32_t G, int64_t rows, int64_t cols,
                                          int32_t swiglu_interleave, int32_t format, uint8_t* codes, uint8_t* scales,
                                          float* global_scale, float* amax, gmlp_stream stream) {
  g_last_error[0] = 0;
  if (!W_experts) return fail(GMLP_ERR_INVALID_ARG, "W_experts NULL");
  return prepare_weights_impl(W_experts, true, G, rows, cols, swiglu_interleave, format, codes, scales, global_scale,
                              amax, (cudaStream_t)stream);
}

size_t gmlp_forward_workspace_size(int64_t M, int64_t K, int64_t N, int32_t G, int32_t act,
                                   const gmlp_recipe* recipe) {
  (void)act;
  if (!recipe || M < 0 || K <= 0 || N <= 0 || G < 1) return 0;
  return fwd_layout(M, K, N, G, recipe->format).total;
}

gmlp_status gmlp_forward(const uint16_t* x, int64_t M, int64_t K, int64_t N, const int64_t* split_sizes, int32_t G,
                         const gmlp_qweight* W1, const gmlp_qweight* W2, const float* probs, int32_t act,
                         const gmlp_recipe* recipe, uint16_t* y, const gmlp_fwd_aux* aux, void* workspace,
                         size_t workspace_bytes, gmlp_stream stream) {
  g_last_error[0] = 0;
  GMLP_TRY(check_groups(G, M, split_sizes));
  GMLP_TRY(check_recipe(recipe));
  if (act != GMLP_ACT_SWIGLU && act != GMLP_ACT_SRELU && act != GMLP_ACT_TANH_SRELU)
    return fail(GMLP_ERR_INVALID_ARG, "act = %d unknown", act);
  if (act == GMLP_ACT_TANH_SRELU && !(aux && aux->tanh_clamp_scale > 0.0f && std::isfinite(aux->tanh_clamp_scale)))
    return fail(GMLP_ERR_INVALID_ARG, "tanh-SReLU needs aux->tanh_clamp_scale > 0 and finite");
  const int fmt = recipe->format;
  const int64_t n1 = act == GMLP_ACT_SWIGLU ? 2 * N : N;
  if (K <= 0 || K % 256 || K > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "K = %lld must be a positive multiple of 256, at most 2^20", (long long)K);
  if (N <= 0 || n1 % 256 || N % (fmt == GMLP_NVFP4 ? 256 : 128) || N > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "N = %lld: need fc1 width %% 256 == 0 and N %% %d == 0", (long long)N,
                fmt == GMLP_NVFP4 ? 256 : 128);
  if (!W1 || !W2) return fail(GMLP_ERR_INVALID_ARG, "W1 / W2 NULL");
  if (W1->G != G || W2->G != G) return fail(GMLP_ERR_INVALID_DIMS, "weights have %d / %d experts, G = %d", W1->G, W2->G, G);
  if (W1->format != fmt || W2->format != fmt)
    return fail(GMLP_ERR_UNSUPPORTED_RECIPE, "weight formats differ from the recipe's");
  if (W1->rows != n1 || W1->cols != K)
    return fail(GMLP_ERR_INVALID_DIMS, "W1 is [%lld x %lld], expected [%lld x %lld]", (long long)W1->rows,
                (long long)W1->cols, (long long)n1, (long long)K);
  if (W2->rows != K || W2->cols != N)
    return fail(GMLP_ERR_INVALID_DIMS, "W2 is [%lld x %lld], expected [%lld x %lld]", (long long)W2->rows,
                (long long)W2->cols, (long long)K, (long long)N);
  if ((W1->swiglu_interleaved != 0) != (act == GMLP_ACT_SWIGLU) || W2->swiglu_interleaved)
    return fail(GMLP_ERR_INVALID_ARG, "W1 must be SwiGLU-interleaved exactly for SwiGLU; W2 never");
  for (const gmlp_qweight* W : {W1, W2})
    if (!(W->scale_layout == 0 || W->scale_layout == GMLP_SCALES_GEMM_TILED ||
          (W->scale_layout == GMLP_SCALES_GEMM_TILED_X4 && fmt == GMLP_NVFP4)))
      return fail(GMLP_ERR_INVALID_ARG, "weight scale_layout %d: GEMM_TILED, or GEMM_TILED_X4 for NVFP4",
                  W->scale_layout);
  const bool x4_1 = W1->scale_layout == GMLP_SCALES_GEMM_TILED_X4, x4_2 = W2->scale_layout == GMLP_SCALES_GEMM_TILED_X4;
  if (!W1->codes || !W1->scales || !W2->codes || !W2->scales || !aligned16(W1->codes) || !aligned16(W1->scales) ||
      !aligned16(W2->codes) || !aligned16(W2->scales))
    return fail(GMLP_ERR_INVALID_ARG, "weight codes/scales NULL or not 16-byte aligned");
  if (!aligned16(W1->bias) || !aligned16(W2->bias)) return fail(GMLP_ERR_INVALID_ARG, "weight bias not 16-byte aligned");
  if (fmt == GMLP_NVFP4 && (!W1->global_scale || !W2->global_scale))
    return fail(GMLP_ERR_INVALID_ARG, "NVFP4 weights need global_scale");
  if ((M > 0 && (!x || !y)) || !aligned16(x) || !aligned32(y))
    return fail(GMLP_ERR_INVALID_ARG, "x / y NULL, or x not 16-byte or y not 32-byte aligned");
  if (probs && (reinterpret_cast<uintptr_t>(probs) & 3)) return fail(GMLP_ERR_INVALID_ARG, "probs misaligned");
  const FwdLayout L = fwd_layout(M, K, N, G, fmt);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace))
    return fail(GMLP_ERR_WORKSPACE, "workspace %zu bytes, need %zu (16-byte aligned)", workspace_bytes, L.total);
  if (aux && aux->n_stage_events > 0 && !aux->stage_events) return fail(GMLP_ERR_INVALID_ARG, "stage_events NULL");
  if (aux && (aux->fc2x_col_codes || aux->fc2x_col_scales)) {
    if (fmt != GMLP_NVFP4) return fail(GMLP_ERR_INVALID_ARG, "columnwise fc2_x output is an NVFP4 output");
    if (!aux->fc2x_col_codes || !aux->fc2x_col_scales || !aligned16(aux->fc2x_col_codes) ||
        !aligned16(aux->fc2x_col_scales))
      return fail(GMLP_ERR_INVALID_ARG, "fc2x_col_codes / fc2x_col_scales: both, 16-byte aligned");
  }
  if (aux && !aligned32(aux->fc1_pre_act)) return fail(GMLP_ERR_INVALID_ARG, "fc1_pre_act not 32-byte aligned");
  if (aux && aux->gemm_mode == 2 && (aux->fc1_pre_act || W1->bias || W2->bias))
    return fail(GMLP_ERR_INVALID_ARG, "gemm_mode 2 (CTA pairs) takes no biases and saves no activation input");
  if (aux && aux->gemm_mode != 0 && aux->gemm_mode != 2)
    return fail(GMLP_ERR_INVALID_ARG, "gemm_mode %d is neither 0 nor 2", aux->gemm_mode);
  GMLP_TRY(check_device());

  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* x_codes = ws + L.x_codes;
  uint8_t* x_scales = ws + L.x_scales;
  uint8_t* f_codes = (aux && aux->fc2x_codes) ? aux->fc2x_codes : ws + L.f_codes;
  uint8_t* f_scales = (aux && aux->fc2x_scales) ? aux->fc2x_scales : ws + L.f_scales;
  if (!aligned16(f_codes) || !aligned16(f_scales)) return fail(GMLP_ERR_INVALID_ARG, "aux fc2x buffers misaligned");
  GroupSrc gs{split_sizes, 0, G, M};
  int ev = 0;
  auto mark = [&]() -> gmlp_status {
    if (aux && ev < aux->n_stage_events) {
      cudaError_t e = cudaEventRecord((cudaEvent_t)aux->stage_events[ev], s);
      if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    }
    ++ev;
    return GMLP_OK;
  };

  const int epi1 = act == GMLP_ACT_SWIGLU ? EPI_FC1_SWIGLU : act == GMLP_ACT_SRELU ? EPI_FC1_SRELU : EPI_FC1_TANH_SRELU;
  const float tanh_c = act == GMLP_ACT_TANH_SRELU ? aux->tanh_clamp_scale : 0.0f;
  if (fmt == GMLP_MXFP8) {
    RowQuantArgs q{};
    q.x = x;
    q.M = M;
    q.K = K;
    q.grp = gs;
    q.format = GMLP_MXFP8;
    q.tiled = 1;
    q.codes = x_codes;
    q.scales = x_scales;
    GMLP_CUDA(launch_row_quant(q, s), "x quantise launch");
    GMLP_TRY(mark());
    GemmArgs g1{};
    g1.format = GMLP_MXFP8;
    g1.epi = epi1;
    g1.a_codes = x_codes;
    g1.a_scales = x_scales;
    g1.b_codes = W1->codes;
    g1.b_scales = W1->scales;
    g1.bias = W1->bias;
    g1.M = M;
    g1.kbytes = K;
    g1.n_out = n1;
    g1.grp = gs;
    g1.probs = probs;
    g1.tanh_c = tanh_c;
    g1.pre_act_out = aux ? aux->fc1_pre_act : nullptr;
    g1.out_codes = f_codes;
    g1.out_scales = f_scales;
    g1.n_cols_out = N;
    g1.pair = (aux && aux->gemm_mode == 2) ? 2 : 1;
    g1.pdl = 1;
    GMLP_CUDA(launch_gemm(g1, s), "fc1 launch");
    GMLP_TRY(mark());
    GemmArgs g2{};
    g2.format = GMLP_MXFP8;
    g2.epi = EPI_FC2;
    g2.a_codes = f_codes;
    g2.a_scales = f_scales;
    g2.b_codes = W2->codes;
    g2.b_scales = W2->scales;
    g2.bias = W2->bias;
    g2.M = M;
    g2.kbytes = N;
    g2.n_out = K;
    g2.grp = gs;
    g2.out_bf16 = y;
    g2.n_cols_out = K;
    g2.pair = (aux && aux->gemm_mode == 2) ? 2 : 1;
    g2.pdl = 1;
    GMLP_CUDA(launch_gemm(g2, s), "fc2 launch");
    GMLP_TRY(mark());
    return GMLP_OK;
  }

  // NVFP4
  float* amax_ws = reinterpret_cast<float*>(ws + L.amax);
  float* x_amax = amax_ws;
  float* f_pre = (aux && aux->fc2x_amax_pre) ? aux->fc2x_amax_pre : amax_ws + G;
  float* f_post = (aux && aux->fc2x_amax_post) ? aux->fc2x_amax_post : amax_ws + 2 * G;
  uint16_t* f_bf16 = (aux && aux->fc2x_bf16) ? aux->fc2x_bf16 : reinterpret_cast<uint16_t*>(ws + L.f_bf16);
  if (!aligned16(f_bf16)) return fail(GMLP_ERR_INVALID_ARG, "aux fc2x_bf16 misaligned");
  // the amax pass on the x cast's grid (nvfp4_amax_keep)
  GMLP_CUDA(launch_group_amax(x, M, K, gs, x_amax, s, row_quant_grid(GMLP_NVFP4, 1, M), nvfp4_amax_keep(M, K)),
            "x amax launch");
  GMLP_TRY(mark());
  {
    RowQuantArgs q{};
    q.x = x;
    q.M = M;
    q.K = K;
    q.grp = gs;
    q.format = GMLP_NVFP4;
    q.tiled = 1;
    q.codes = x_codes;
    q.scales = x_scales;
    q.amax = x_amax;
    q.zero_ptr = f_pre;   // fc1's epilogue max-accumulates into these
    q.zero_count = G;
    q.zero_ptr2 = f_post;
    q.zero_count2 = G;
    q.pdl = 1;
    q.reverse = 1;
    GMLP_CUDA(launch_row_quant(q, s), "x quantise launch");
  }
  GMLP_TRY(mark());
  GemmArgs g1{};
  g1.format = GMLP_NVFP4;
  g1.epi = epi1;
  g1.a_codes = x_codes;
  g1.a_scales = x_scales;
  g1.b_codes = W1->codes;
  g1.b_scales = W1->scales;
  g1.bias = W1->bias;
  g1.M = M;
  g1.kbytes = K / 2;
  g1.n_out = n1;
  g1.grp = gs;
  g1.a_amax = x_amax;
  g1.b_S = W1->global_scale;
  g1.b_x4 = x4_1;
  g1.probs = probs;
  g1.tanh_c = tanh_c;
  g1.pre_act_out = aux ? aux->fc1_pre_act : nullptr;
  g1.out_bf16 = f_bf16;
  g1.amax_pre = f_pre;
  // the post-RHT amax comes from the fc1 epilogue only when the columnwise
  // cast below needs it up front; otherwise the rowwise cast of fc2_x takes it
  // in its own pass over the tensor
  const bool colwise = aux && aux->fc2x_col_codes;
  g1.amax_post = colwise ? f_post : nullptr;
  g1.rht_mask = recipe->rht_sign_mask & 0xFFFFu;
  g1.n_cols_out = N;
    g1.pair = (aux && aux->gemm_mode == 2) ? 2 : 1;
    g1.pdl = 1;
  GMLP_CUDA(launch_gemm(g1, s), "fc1 launch");
  GMLP_TRY(mark());
  if (colwise) {
    // rowwise (fc2's operand) and columnwise (RHT) NVFP4 of fc2_x in one pass,
    // both from the amaxes the fc1 epilogue produced
    ColQuantArgs c{};
    c.x = f_bf16;
    c.M = M;
    c.K = N;
    c.grp = gs;
    c.use_rht = recipe->use_rht != 0;
    c.mask = recipe->rht_sign_mask & 0xFFFFu;
    c.amax_row = f_pre;
    c.amax_col = recipe->use_rht ? f_post : f_pre;
    c.row_codes = f_codes;
    c.row_scales = f_scales;
    c.row_tiled = 1;
    c.col_codes = aux->fc2x_col_codes;
    c.col_scales = aux->fc2x_col_scales;
    GMLP_CUDA(launch_col_quant(c, s), "fc2_x row + column quantise launch");
  } else if (aux && aux->fc2x_amax_post) {
    // rowwise NVFP4 of fc2_x (fc2's operand) and its post-RHT amax in one pass
    ColQuantArgs c{};
    c.x = f_bf16;
    c.M = M;
    c.K = N;
    c.grp = gs;
    c.use_rht = 1;
    c.mask = recipe->rht_sign_mask & 0xFFFFu;
    c.amax_row = f_pre;
    c.row_codes = f_codes;
    c.row_scales = f_scales;
    c.row_tiled = 1;
    c.amax_post_out = f_post;
    GMLP_CUDA(launch_col_quant(c, s), "fc2_x quantise + post-RHT amax launch");
  } else {
    RowQuantArgs q{};
    q.x = f_bf16;
    q.M = M;
    q.K = N;
    q.grp = gs;
    q.format = GMLP_NVFP4;
    q.tiled = 1;
    q.codes = f_codes;
    q.scales = f_scales;
    q.amax = f_pre;
    q.pdl = 1;
    GMLP_CUDA(launch_row_quant(q, s), "fc2_x quantise launch");
  }
  GMLP_TRY(mark());
  GemmArgs g2{};
  g2.format = GMLP_NVFP4;
  g2.epi = EPI_FC2;
  g2.a_codes = f_codes;
  g2.a_scales = f_scales;
  g2.b_codes = W2->codes;
  g2.b_scales = W2->scales;
  g2.bias = W2->bias;
  g2.M = M;
  g2.kbytes = N / 2;
  g2.n_out = K;
  g2.grp = gs;
  g2.a_amax = f_pre;
  g2.b_S = W2->global_scale;
  g2.b_x4 = x4_2;
  g2.out_bf16 = y;
  g2.n_cols_out = K;
    g2.pair = (aux && aux->gemm_mode == 2) ? 2 : 1;
    g2.pdl = 1;
  GMLP_CUDA(launch_gemm(g2, s), "fc2 launch");
  GMLP_TRY(mark());
  return GMLP_OK;
}

gmlp_status gmlp_fc2x_recompute(const uint16_t* pre_act, const float* probs, int64_t M, int64_t N, int32_t act,
                                float tanh_clamp_scale, uint16_t* fc2x, gmlp_stream stream) {
  g_last_error[0] = 0;
  if (act != GMLP_ACT_SWIGLU && act != GMLP_ACT_SRELU && act != GMLP_ACT_TANH_SRELU)
    return fail(GMLP_ERR_INVALID_ARG, "act = %d unknown", act);
  if (act == GMLP_ACT_TANH_SRELU && !(tanh_clamp_scale > 0.0f && std::isfinite(tanh_clamp_scale)))
    return fail(GMLP_ERR_INVALID_ARG, "tanh-SReLU needs tanh_clamp_scale > 0 and finite");
  if (M < 0 || M > (int64_t)0x7FFFFFFF) return fail(GMLP_ERR_INVALID_DIMS, "M = %lld outside [0, 2^31)", (long long)M);
  if (N <= 0 || N % 16 || N > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "N = %lld must be a positive multiple of 16, at most 2^20", (long long)N);
  if ((M > 0 && (!pre_act || !fc2x)) || !aligned32(pre_act) || !aligned32(fc2x))
    return fail(GMLP_ERR_INVALID_ARG, "pre_act / fc2x NULL or not 32-byte aligned");
  if (probs && (reinterpret_cast<uintptr_t>(probs) & 3)) return fail(GMLP_ERR_INVALID_ARG, "probs misaligned");
  GMLP_TRY(check_device());
  GMLP_CUDA(launch_fc2x_recompute(pre_act, probs, M, N, act, tanh_clamp_scale, fc2x, (cudaStream_t)stream),
            "fc2_x recompute launch");
  return GMLP_OK;
}

gmlp_status gmlp_selftest_bounded_wait(uint64_t limit_ns, gmlp_stream stream) {
  g_last_error[0] = 0;
  if (limit_ns < 1000 || limit_ns > 2000000000ull)
    return fail(GMLP_ERR_INVALID_ARG, "limit_ns %llu outside [1 us, 2 s]", (unsigned long long)limit_ns);
  GMLP_TRY(check_device());
  GMLP_CUDA(launch_selftest_wait(limit_ns, (cudaStream_t)stream), "selftest launch");
  return GMLP_OK;
}

size_t gmlp_backward_workspace_size(int64_t M, int64_t K, int64_t N, int32_t G, int32_t act) {
  if (M < 0 || K <= 0 || N <= 0 || G < 1) return 0;
  return bwd_layout(M, K, act == GMLP_ACT_SWIGLU ? 2 * N : N, G).total;
}

gmlp_status gmlp_backward_dgrad(const uint16_t* dy, int64_t M, int64_t K, int64_t N, const int64_t* split_sizes,
                                int32_t G, const gmlp_qweight* W2t, const gmlp_qweight* W1t,
                                const uint16_t* pre_act, const float* probs, int32_t act, const gmlp_recipe* recipe,
                                uint16_t* dx, float* dprob, uint8_t* fc1_dy_codes, uint8_t* fc1_dy_scales,
                                uint16_t* fc1_dy_bf16, void* workspace, size_t workspace_bytes,
                                gmlp_event* stage_events,
                                int32_t n_stage_events, gmlp_stream stream) {
  g_last_error[0] = 0;
  GMLP_TRY(check_groups(G, M, split_sizes));
  GMLP_TRY(check_recipe(recipe));
  if (recipe->format != GMLP_MXFP8)
    return fail(GMLP_ERR_UNSUPPORTED_RECIPE, "the backward dgrad path is MXFP8 (as the pages' backward)");
  if (act != GMLP_ACT_SWIGLU && act != GMLP_ACT_SRELU)
    return fail(GMLP_ERR_INVALID_ARG, "backward act = %d: SwiGLU or SReLU", act);
  const int64_t N1 = act == GMLP_ACT_SWIGLU ? 2 * N : N;
  if (K <= 0 || K % 256 || N <= 0 || N % 256 || K > kMaxFeatures || N > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "K = %lld, N = %lld: both positive multiples of 256, at most 2^20", (long long)K,
                (long long)N);
  if (!W2t || !W1t || W2t->G != G || W1t->G != G || W2t->format != GMLP_MXFP8 || W1t->format != GMLP_MXFP8)
    return fail(GMLP_ERR_INVALID_ARG, "W2t / W1t: MXFP8 weights of G experts");
  if (W2t->rows != N || W2t->cols != K || W1t->rows != K || W1t->cols != N1)
    return fail(GMLP_ERR_INVALID_DIMS, "W2t must be [N x K] and W1t [K x N1] per expert (the transposed weights)");
  if (W2t->swiglu_interleaved || W1t->swiglu_interleaved || W2t->bias || W1t->bias)
    return fail(GMLP_ERR_INVALID_ARG, "transposed weights carry no interleave and no bias");
  if (!W2t->codes || !W2t->scales || !W1t->codes || !W1t->scales || !aligned16(W2t->codes) ||
      !aligned16(W2t->scales) || !aligned16(W1t->codes) || !aligned16(W1t->scales))
    return fail(GMLP_ERR_INVALID_ARG, "weight codes/scales NULL or not 16-byte aligned");
  if ((M > 0 && (!dy || !dx || !pre_act)) || !aligned16(dy) || !aligned32(dx) || !aligned32(pre_act))
    return fail(GMLP_ERR_INVALID_ARG, "dy / dx / pre_act NULL, or dy not 16-byte or dx / pre_act not 32-byte aligned");
  if ((fc1_dy_codes == nullptr) != (fc1_dy_scales == nullptr) || !aligned16(fc1_dy_codes) ||
      !aligned16(fc1_dy_scales))
    return fail(GMLP_ERR_INVALID_ARG, "fc1_dy_codes / fc1_dy_scales: both or neither, 16-byte aligned");
  if (probs && (reinterpret_cast<uintptr_t>(probs) & 3)) return fail(GMLP_ERR_INVALID_ARG, "probs misaligned");
  if (!aligned32(fc1_dy_bf16)) return fail(GMLP_ERR_INVALID_ARG, "fc1_dy_bf16 not 32-byte aligned");
  if (n_stage_events < 0 || n_stage_events > 3 || (n_stage_events > 0 && !stage_events))
    return fail(GMLP_ERR_INVALID_ARG, "n_stage_events = %d: 0..3, stage_events non-NULL", n_stage_events);
  const BwdLayout L = bwd_layout(M, K, N1, G);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace))
    return fail(GMLP_ERR_WORKSPACE, "workspace %zu bytes, need %zu (16-byte aligned)", workspace_bytes, L.total);
  GMLP_TRY(check_device());
  if (M == 0) return GMLP_OK;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* dy_codes = ws + L.dy_codes;
  uint8_t* dy_scales = ws + L.dy_scales;
  uint8_t* g_codes = fc1_dy_codes ? fc1_dy_codes : ws + L.g_codes;
  uint8_t* g_scales = fc1_dy_scales ? fc1_dy_scales : ws + L.g_scales;
  GroupSrc gs{split_sizes, 0, G, M};
  auto stage_done = [&](int i) -> gmlp_status {
    if (i < n_stage_events) GMLP_CUDA(cudaEventRecord((cudaEvent_t)stage_events[i], s), "stage event record");
    return GMLP_OK;
  };
  {
    RowQuantArgs q{};
    q.x = dy;
    q.M = M;
    q.K = K;
    q.grp = gs;
    q.format = GMLP_MXFP8;
    q.tiled = 1;
    q.codes = dy_codes;
    q.scales = dy_scales;
    q.zero_ptr = dprob;  // the dGLU epilogue adds into it
    q.zero_count = dprob ? M : 0;
    GMLP_CUDA(launch_row_quant(q, s), "dy quantise launch");
  }
  GMLP_TRY(stage_done(0));
  GemmArgs g1{};  // FC2 dGLU: dfc2x = dy W2 per expert, then dGLU x prob -> fc1_dy (MXFP8), dprob
  g1.format = GMLP_MXFP8;
  g1.epi = act == GMLP_ACT_SWIGLU ? EPI_DGLU_SWIGLU : EPI_DSRELU;
  g1.a_codes = dy_codes;
  g1.a_scales = dy_scales;
  g1.b_codes = W2t->codes;
  g1.b_scales = W2t->scales;
  g1.M = M;
  g1.kbytes = K;
  g1.n_out = N;
  g1.grp = gs;
  g1.probs = probs;
  g1.act_in = pre_act;
  g1.dprob = dprob;
  g1.out_codes = g_codes;
  g1.out_scales = g_scales;
  g1.out_bf16 = fc1_dy_bf16;
  g1.n_cols_out = N1;
  g1.pair = 1;
  g1.pdl = 1;
  GMLP_CUDA(launch_gemm(g1, s), "dGLU launch");
  GMLP_TRY(stage_done(1));
  GemmArgs g2{};  // FC1 dgrad: dx = fc1_dy W1 per expert
  g2.format = GMLP_MXFP8;
  g2.epi = EPI_FC2;
  g2.a_codes = g_codes;
  g2.a_scales = g_scales;
  g2.b_codes = W1t->codes;
  g2.b_scales = W1t->scales;
  g2.M = M;
  g2.kbytes = N1;
  g2.n_out = K;
  g2.grp = gs;
  g2.out_bf16 = dx;
  g2.n_cols_out = K;
  g2.pair = 1;
  g2.pdl = 1;
  GMLP_CUDA(launch_gemm(g2, s), "fc1 dgrad launch");
  GMLP_TRY(stage_done(2));
  return GMLP_OK;
}

int64_t gmlp_colwise_tokens(int64_t M, int32_t G) {
  if (M < 0 || G < 1) return 0;
  return 128 * ((M + 127) / 128 + G);
}

int64_t gmlp_query_layout(int32_t kind, const int64_t* split_sizes_host, int32_t G, int64_t ncols, int64_t row,
                          int64_t col) {
  if (G < 1 || !split_sizes_host || ncols <= 0 || row < 0 || col < 0 || col >= ncols) return -1;
  // find row's group: its first row and the number of 128-row tiles before it
  int64_t off = 0, tiles = 0, M = 0;
  int32_t g = -1;
  for (int32_t h = 0; h < G; ++h) {
    const int64_t m = split_sizes_host[h];
    if (m < 0) return -1;
    if (g < 0 && row < M + m) {
      g = h;
      off = M;
    }
    if (g < 0) tiles += (m + 127) / 128;
    M += m;
  }
  if (g < 0) return -1;  // row >= M
  const int64_t lr = row - off;
  const int64_t tile = tiles + lr / 128, rr = lr % 128;
  switch (kind) {
    case GMLP_LAYOUT_TILED_SCALE:
      if (ncols % 4) return -1;
      return (tile * (ncols / 4) + col / 4) * 512 + (rr % 32) * 16 + (rr / 32) * 4 + col % 4;
    case GMLP_LAYOUT_COLWISE_CODE:
      return (tile * ncols + col) * 128 + rr;
    case GMLP_LAYOUT_COLWISE_SCALE: {
      if (ncols % 128) return -1;
      const int64_t chunks = gmlp_colwise_tokens(M, G) / 128, i = col % 128;
      return ((col / 128) * chunks + tile) * 512 + (i % 32) * 16 + (i / 32) * 4 + rr / 32;
    }
    default:
      return -1;
  }
}

size_t gmlp_backward_wgrad_workspace_size(int64_t M, int64_t K, int64_t N, int32_t G, int32_t act) {
  if (M < 0 || K <= 0 || N <= 0 || G < 1) return 0;
  return wgrad_layout(M, K, N, act == GMLP_ACT_SWIGLU ? 2 * N : N, G).total;
}

gmlp_status gmlp_backward_wgrad(const uint16_t* x, const uint16_t* dy, const uint16_t* pre_act, const float* probs,
                                const uint16_t* fc1_dy, int64_t M, int64_t K, int64_t N, const int64_t* split_sizes,
                                int32_t G, int32_t act, float* dW1, float* dW2, float* dbias1, float* dbias2,
                                int32_t accumulate, void* workspace, size_t workspace_bytes, gmlp_event* stage_events,
                                int32_t n_stage_events, gmlp_stream stream) {
  g_last_error[0] = 0;
  GMLP_TRY(check_groups(G, M, split_sizes));
  if (act != GMLP_ACT_SWIGLU && act != GMLP_ACT_SRELU)
    return fail(GMLP_ERR_INVALID_ARG, "wgrad act = %d: SwiGLU or SReLU", act);
  if (n_stage_events < 0 || n_stage_events > 6 || (n_stage_events > 0 && !stage_events))
    return fail(GMLP_ERR_INVALID_ARG, "n_stage_events = %d: 0..6, stage_events non-NULL", n_stage_events);
  if (accumulate != 0 && accumulate != 1) return fail(GMLP_ERR_INVALID_ARG, "accumulate = %d: 0 or 1", accumulate);
  const int64_t N1 = act == GMLP_ACT_SWIGLU ? 2 * N : N;
  if (K <= 0 || K % 256 || N <= 0 || N % 256 || K > kMaxFeatures || N > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "K = %lld, N = %lld: both positive multiples of 256, at most 2^20", (long long)K,
                (long long)N);
  const bool want1 = dW1 || dbias1, want2 = dW2 || dbias2;
  if (M > 0 && ((want2 && !dy) || (dW2 && !pre_act) || (want1 && !fc1_dy) || (dW1 && !x)))
    return fail(GMLP_ERR_INVALID_ARG, "an input a requested gradient needs is NULL");
  if (!aligned16(x) || !aligned16(dy) || !aligned16(fc1_dy) || !aligned32(pre_act))
    return fail(GMLP_ERR_INVALID_ARG, "x / dy / fc1_dy not 16-byte or pre_act not 32-byte aligned");
  if (!aligned32(dW1) || !aligned32(dW2) || (reinterpret_cast<uintptr_t>(dbias1) & 3) ||
      (reinterpret_cast<uintptr_t>(dbias2) & 3))
    return fail(GMLP_ERR_INVALID_ARG, "dW1 / dW2 not 32-byte or dbias1 / dbias2 not 4-byte aligned");
  if (probs && (reinterpret_cast<uintptr_t>(probs) & 3)) return fail(GMLP_ERR_INVALID_ARG, "probs misaligned");
  const WgradLayout L = wgrad_layout(M, K, N, N1, G);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace))
    return fail(GMLP_ERR_WORKSPACE, "workspace %zu bytes, need %zu (16-byte aligned)", workspace_bytes, L.total);
  GMLP_TRY(check_device());
  cudaStream_t s = (cudaStream_t)stream;
  if (!accumulate) {
    // an empty batch still has (zero) gradients; the kernels overwrite the rest
    if (M == 0 && dW1) GMLP_CUDA(cudaMemsetAsync(dW1, 0, sizeof(float) * G * N1 * K, s), "dW1 memset");
    if (M == 0 && dW2) GMLP_CUDA(cudaMemsetAsync(dW2, 0, sizeof(float) * G * K * N, s), "dW2 memset");
    if (dbias1) GMLP_CUDA(cudaMemsetAsync(dbias1, 0, sizeof(float) * G * N1, s), "dbias1 memset");
    if (dbias2) GMLP_CUDA(cudaMemsetAsync(dbias2, 0, sizeof(float) * G * K, s), "dbias2 memset");
  }
  if (M == 0) return GMLP_OK;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const GroupSrc gs{split_sizes, 0, G, M};
  int n_ev = 0;  // stage events go out in launch order
  auto stage_done = [&]() -> gmlp_status {
    if (n_ev < n_stage_events) GMLP_CUDA(cudaEventRecord((cudaEvent_t)stage_events[n_ev], s), "stage event record");
    ++n_ev;
    return GMLP_OK;
  };
  auto colq = [&](const uint16_t* src, int64_t ld, int64_t C, int mode, size_t c_off, size_t s_off,
                  float* colsum) -> gmlp_status {
    ColqArgs q{};
    q.src = src;
    q.ld = ld;
    q.C = C;
    q.up_off = N;
    q.probs = probs;
    q.grp = gs;
    q.T = L.T;
    q.codes = ws + c_off;
    q.scales = ws + s_off;
    q.colsum = colsum;
    q.mode = mode;
    GMLP_CUDA(launch_colq(q, s), "columnwise quantise launch");
    return stage_done();
  };
  auto wgrad = [&](size_t ac, size_t as, size_t bc, size_t bs, int64_t RA, int64_t RB, float* out) -> gmlp_status {
    WgradArgs w{};
    w.a_codes = ws + ac;
    w.a_scales = ws + as;
    w.b_codes = ws + bc;
    w.b_scales = ws + bs;
    w.RA = RA;
    w.RB = RB;
    w.T = L.T;
    w.grp = gs;
    w.out = out;
    w.accumulate = accumulate;
    GMLP_CUDA(launch_wgrad(w, s), "wgrad launch");
    return stage_done();
  };
  if (want2) {  // FC2: dW2_g = dy_g^T fc2_x_g over the group's tokens, dbias2 = token sums of dy
    GMLP_TRY(colq(dy, K, K, COLQ_PLAIN, L.dy_c, L.dy_s, dbias2));
    if (dW2) {
      GMLP_TRY(colq(pre_act, N1, N, act == GMLP_ACT_SWIGLU ? COLQ_SWIGLU : COLQ_SRELU, L.f_c, L.f_s, nullptr));
      GMLP_TRY(wgrad(L.dy_c, L.dy_s, L.f_c, L.f_s, K, N, dW2));
    }
  }
  if (want1) {  // FC1: dW1_g = fc1_dy_g^T x_g, dbias1 = token sums of fc1_dy
    GMLP_TRY(colq(fc1_dy, N1, N1, COLQ_PLAIN, L.g_c, L.g_s, dbias1));
    if (dW1) {
      GMLP_TRY(colq(x, K, K, COLQ_PLAIN, L.x_c, L.x_s, nullptr));
      GMLP_TRY(wgrad(L.g_c, L.g_s, L.x_c, L.x_s, N1, K, dW1));
    }
  }
  return GMLP_OK;
}

gmlp_status gmlp_replicate_weight_scales(const uint8_t* tiled, int32_t G, int64_t rows, int64_t cols, uint8_t* out,
                                         gmlp_stream stream) {
  g_last_error[0] = 0;
  if (!tiled || !out || !aligned16(tiled) || !aligned16(out))
    return fail(GMLP_ERR_INVALID_ARG, "tiled / out NULL or not 16-byte aligned");
  if (G < 1 || G > kMaxGroups || rows <= 0 || cols <= 0 || rows % 256 || cols % 256 || rows > kMaxFeatures ||
      cols > kMaxFeatures)
    return fail(GMLP_ERR_INVALID_DIMS, "G = %d, rows = %lld, cols = %lld: need 1 <= G <= %d, rows and cols %% 256 == 0",
                G, (long long)rows, (long long)cols, kMaxGroups);
  GMLP_TRY(check_device());
  GMLP_CUDA(launch_replicate_scales(tiled, (int64_t)G * rows / 256, cols / 64, out, (cudaStream_t)stream),
            "replicate launch");
  return GMLP_OK;
}

gmlp_status gmlp_mma_peak(int32_t format, int32_t scale_copy, int64_t iters, int32_t ctas, gmlp_stream stream) {
  g_last_error[0] = 0;
  if (format != GMLP_MXFP8 && format != GMLP_NVFP4) return fail(GMLP_ERR_INVALID_ARG, "format %d", format);
  if (scale_copy < 0 || scale_copy > 3 || (scale_copy == 2 && format != GMLP_NVFP4))
    return fail(GMLP_ERR_INVALID_ARG, "scale_copy %d (0, 1, 3, or 2 for NVFP4)", scale_copy);
  if (iters < 1 || iters > (int64_t(1) << 24))
    return fail(GMLP_ERR_INVALID_ARG, "iters %lld outside [1, 2^24]", (long long)iters);
  GMLP_TRY(check_device());
  const int n = ctas > 0 ? ctas : num_sms();
  if (n > 65535) return fail(GMLP_ERR_INVALID_ARG, "ctas %d", n);
  GMLP_CUDA(launch_mma_peak(format, scale_copy, iters, n, (cudaStream_t)stream), "mma peak launch");
  return GMLP_OK;
}

gmlp_status gmlp_check_device_status(gmlp_stream stream) {
  g_last_error[0] = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  const int a = quant_read_clear_status();
  const int b = gemm_read_clear_status();
  const int c = peak_read_clear_status();
  const int d = wgrad_read_clear_status();
  const int code = a ? a : (b ? b : (c ? c : d));
  if (code < 0) return fail(GMLP_ERR_CUDA, "reading the device status word failed");
  if (code == GMLP_ERR_DEVICE_TIMEOUT) return fail(GMLP_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait");
  if (code == GMLP_ERR_DEVICE_BOUNDS)
    return fail(GMLP_ERR_DEVICE_BOUNDS, "split_sizes negative or summing past M");
  if (code) return fail((gmlp_status)code, "device status %d", code);
  return GMLP_OK;
}

}  // extern "C"
