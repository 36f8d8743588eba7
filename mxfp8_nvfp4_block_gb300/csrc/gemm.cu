// gemm.cu -- persistent grouped GEMM on block-scaled tcgen05 tensor cores with
// the fused fc1 epilogue (activation x prob, then MXFP8 requantisation or
// bf16 + NVFP4 amaxes) and the fc2 bf16 epilogue.
//
// Method: PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8" (sequence
// diagram: the FC1 GLU kernel takes the MXFP8 a_tensor, the b_tensor weights
// and prob_tensor and writes the MXFP8 activation with its row scales; the
// FC2 kernel writes the output) and PR #3837 "Reduce NVFP4 quantization work
// for the fused GroupedMLP fc2 input with activation recompute" (the
// Hadamard-fused fc1 kernel returns fc2_x and its pre-RHT and post-RHT amax;
// the sign mask enters the post-RHT amax; the accumulator is rounded through
// the bf16 C type before the activation).
//
// Design (GB300, one CTA per SM, 576 threads):
//   warp 0    TMA producer: A tile 128 x 128 B, B tile 256 x 128 B (128-byte
//             swizzle) and the tile's scale blocks (bulk copies) per stage,
//             4 stages, one mbarrier pair per stage;
//   warp 1    TMEM owner and MMA issuer: per stage the scale blocks go to TMEM
//             (tcgen05.cp 32x128b.warpx4), then 4 MMAs (M=128, N=256, K=32
//             FP8 / K=64 FP4) accumulate into 256 TMEM columns;
//   warps 2-17 epilogue: each drains its 32 lanes x 64 columns into
//             registers, frees the accumulator at once (so the next tile's
//             mainloop overlaps the epilogue math), then computes and stores.
// Tiles: (expert g, 128-row tile of g's tokens, 256-column output tile),
// ordered expert-major and handed out round-robin to the persistent CTAs;
// within an expert the order keeps the smaller operand resident in L2
// (decode_tile).
#include <cudaTypedefs.h>

#include <cstring>

#include "device.cuh"

namespace gmlp {

namespace {

constexpr int kEpiWarps = 16;
constexpr int kBM = 128, kBN = 256, kBKBytes = 128;
constexpr int kATileBytes = kBM * kBKBytes;  // 16 KB
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kTmemCols = 512;

// Per-format, per-shape constants.  PAIR = 1: one CTA computes a 128 x 256
// tile with cta_group::1 MMAs.  PAIR = 2: a CTA pair (cluster of 2) computes a
// 256 x 256 tile with cta_group::2 MMAs; each CTA loads its own 128 A rows and
// one 128-row half of the B tile, so each SM takes in a third fewer bytes.
//
// X4 (NVFP4): the B scales come replicated four times (weight layout
// GEMM_TILED_X4), so one 128x256b copy places the scales of both 128-row
// halves of the B tile for one MMA, replacing two 32x128b.warpx4 copies; each
// copy instruction costs about the same tensor-pipe time whatever its size
// (40-60 cycles), and NVFP4 needs 12 of the small ones per stage.  A
// single-CTA stage is then 66 KB (3 stages fit); a CTA-pair stage, with half
// the B tile, 50 KB (4).
template <int FMT, int PAIR, bool X4 = false>
struct Cfg {
  // bytes of scale factors per 128 rows per stage: MXFP8 4 scales/row (one
  // 512-byte block), NVFP4 16 scales/row (four blocks)
  static constexpr int kSfBytes = FMT == GMLP_MXFP8 ? 512 : 2048;
  static constexpr int kSfBBytes = X4 ? 8 * kSfBytes : 2 * kSfBytes;  // B scales per stage (both halves)
  static constexpr int kBRows = kBN / PAIR;                   // B rows held per CTA
  static constexpr int kBTileBytes = kBRows * kBKBytes;
  static constexpr int kStageBytes = kATileBytes + kBTileBytes + kSfBytes + kSfBBytes;
  static constexpr int kStages = X4 ? (PAIR == 1 ? 3 : 4) : PAIR == 1 ? 4 : (FMT == GMLP_MXFP8 ? 6 : 5);
  static constexpr uint32_t kSfCols = FMT == GMLP_MXFP8 ? 16 : 48;  // TMEM columns per stage
  static constexpr uint32_t kSfbOff = FMT == GMLP_MXFP8 ? 4 : 16;   // SFB after SFA within a stage
  static constexpr size_t kSmem = (size_t)kStages * kStageBytes;
  static constexpr int kTileRows = kBM * PAIR;
  // SST (NVFP4, GEMM_TILED weight scales, single CTA): no scale-factor copies;
  // four scale-writer warps (after the 2 control and 16 epilogue warps) store
  // each stage's scales into TMEM with tcgen05.st (12 small copies per stage
  // otherwise)
  static constexpr bool kSST = FMT == GMLP_NVFP4 && !X4 && PAIR == 1;
  static constexpr int kEpiWarp0 = 2;  // first epilogue warp
  static constexpr int kScaleWarp0 = kEpiWarp0 + kEpiWarps;
  static constexpr int kThreads = 32 * (kScaleWarp0 + (kSST ? 4 : 0));
};

// Instruction descriptor (tcgen05 block-scaled kinds): A/B formats in bits
// 7..9 / 10..12 (MXFP8: E4M3 = 0; NVFP4 kind: E2M1 = 1), K-major A and B,
// N >> 3 in bits 17..22, scale type in bit 23 (UE8M0 = 1, UE4M3 = 0),
// M >> 4 in bits 24..28, scale-factor byte selectors in bits 4..5 (B) and
// 29..30 (A).
template <int FMT, int MROWS>
__device__ __forceinline__ uint32_t idesc_for(int k) {
  if (FMT == GMLP_MXFP8)
    return (uint32_t(kBN >> 3) << 17) | (1u << 23) | (uint32_t(MROWS >> 4) << 24) | (uint32_t(k) << 4) |
           (uint32_t(k) << 29);
  return (1u << 7) | (1u << 10) | (uint32_t(kBN >> 3) << 17) | (uint32_t(MROWS >> 4) << 24);
}

struct Tile {
  int g, mt, nt;
};

// Tile w of the expert-major work list.  Within an expert the tiles that run
// at the same time (consecutive w, dealt round-robin to the CTAs) share one
// operand and stream the other, which must then stay in L2 until the expert is
// done: the expert's weight rows (n-tile fastest) when it has more tokens than
// weight rows, else its tokens (m-tile fastest).
template <int TILE_ROWS>
__device__ __forceinline__ Tile decode_tile(const int* off, const int* ip, int G, int w, int64_t n_out, int n_tiles) {
  int lo = 0, hi = G - 1;  // largest g with ip[g] <= w
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ip[mid] <= w) lo = mid; else hi = mid - 1;
  }
  Tile t;
  t.g = lo;
  const int m = off[lo + 1] - off[lo];
  const int local = w - ip[lo];
  if (m > n_out) {
    t.mt = local / n_tiles;
    t.nt = local - t.mt * n_tiles;
  } else {
    const int mtiles = (m + TILE_ROWS - 1) / TILE_ROWS;
    t.nt = local / mtiles;
    t.mt = local - t.nt * mtiles;
  }
  return t;
}

__device__ __forceinline__ float bf16_half(uint32_t w, int hi) {
  return bf16_bits_to_float(hi ? (w >> 16) : (w & 0xFFFFu));
}

// Two floats as a packed bf16 pair (round to nearest even; lo in the low half),
// in one paired conversion.
__device__ __forceinline__ uint32_t pack2_bf16_rn(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Max |f| over n values as a balanced tree (short dependency chains).
template <int n>
__device__ __forceinline__ float tree_amax(const float* f) {
  float m[n / 2];
#pragma unroll
  for (int i = 0; i < n / 2; ++i) m[i] = fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1]));
#pragma unroll
  for (int w = n / 4; w >= 1; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return m[0];
}

// MXFP8 quantisation of 32 consecutive values f (bf16-exact FP32) into 8
// code words; returns the scale exponent.
__device__ __forceinline__ int mx_block(const float* f, uint32_t* words) {
  const int e = mxfp8_exponent(tree_amax<32>(f));
  const float mul = exp2_neg(e);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    words[i] = e4m3x2(__fmul_rn(f[4 * i], mul), __fmul_rn(f[4 * i + 1], mul)) |
               (e4m3x2(__fmul_rn(f[4 * i + 2], mul), __fmul_rn(f[4 * i + 3], mul)) << 16);
  return e;
}

// ------------------------------------------------------------------ epilogues


// One epilogue thread owns one accumulator row (TMEM lane 32q + lane) and a
// 64-column slice of the 256-column tile.
constexpr int kSliceCols = 64;

// silu'(g) = s (1 + g (1 - s)), s = sigmoid(g)
__device__ __forceinline__ float dsilu(float g, float sg) { return sg * (1.0f + g * (1.0f - sg)); }

// Backward "dGLU" epilogue (MXFP8): acc holds dfc2x for this thread's row and
// 64 fc2_x columns n0..n0+63; d = bf16(dfc2x) (the C dtype).  With the
// forward's activation input h (SwiGLU: gate g at column n, up u at N + n):
//   SwiGLU: a = silu(g) u; dg = d prob u silu'(g); du = d prob silu(g)
//   SReLU:  a = max(h,0)^2; dh = d prob 2 max(h,0)
// fc1_dy = bf16(dg | du | dh) quantised to MXFP8 in 1x32 blocks (codes
// [M][N1], scales GEMM_TILED for the fc1 dgrad), and dprob[row] += sum d a.
// The accumulator is read as bf16 pairs and released at once; each 32-column
// half then yields the gate and up fc1_dy blocks (bf16 pairs in registers) in
// one pass, and both are quantised.
// The dGLU values of two adjacent columns, all operands bf16 pairs (d =
// bf16(dfc2x), g / u the activation input; SReLU: g = h): w0 = fc1_dy of the
// gate (or of h), w1 = fc1_dy of the up columns (SwiGLU), both rounded to bf16
// once, in the packing; dsum += d * a per column, in column order.
template <int EPI>
__device__ __forceinline__ void dglu_pair(uint32_t dp, uint32_t gp, uint32_t up, float prob, uint32_t& w0,
                                          uint32_t& w1, float& dsum) {
  float v0[2], v1[2];
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const float d = bf16_half(dp, kk), g = bf16_half(gp, kk);
    const float da = d * prob;
    if (EPI == EPI_DGLU_SWIGLU) {
      const float u = bf16_half(up, kk);
      const float sg = __fdividef(1.0f, 1.0f + __expf(fminf(-g, 80.0f)));
      const float silu = g * sg;
      dsum += d * (silu * u);
      v0[kk] = da * u * dsilu(g, sg);
      v1[kk] = da * silu;
    } else {
      const float r = fmaxf(g, 0.0f);
      dsum += d * (r * r);
      v0[kk] = da * 2.0f * r;
      v1[kk] = 0.0f;
    }
  }
  w0 = pack2_bf16_rn(v0[0], v0[1]);
  w1 = EPI == EPI_DGLU_SWIGLU ? pack2_bf16_rn(v1[0], v1[1]) : 0u;
}

__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// max(|a|, |b|) of packed bf16 pairs (sign bits are the xor of the inputs').
__device__ __forceinline__ uint32_t bmax_abs2_g(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// MXFP8 block of 32 bf16 values held as 16 packed pairs: scale exponent from
// the bf16 block max, 32 E4M3 codes (element 0 in the low byte) to dst.
__device__ __forceinline__ int mx_block_packed(const uint32_t* w, uint8_t* dst) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m = bmax_abs2_g(m, w[i]);
  m = bmax_abs2_g(m, __byte_perm(m, 0, 0x1032)) & 0x7fffu;
  const int e = mxfp8_exponent(__uint_as_float(m << 16));
  const float mul = exp2_neg(e);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t w0 = w[8 * h + 2 * j], w1 = w[8 * h + 2 * j + 1];
      o[j] = e4m3x2(__fmul_rn(bf16_half(w0, 0), mul), __fmul_rn(bf16_half(w0, 1), mul)) |
             (e4m3x2(__fmul_rn(bf16_half(w1, 0), mul), __fmul_rn(bf16_half(w1, 1), mul)) << 16);
    }
    *reinterpret_cast<uint4*>(dst + 16 * h) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  return e;
}

// One 32-column block b of the dGLU epilogue: d16 = bf16(dfc2x) of columns
// n0 + 32 b .. + 31 of this thread's row as packed pairs; returns sum d * act
// over them.
template <int EPI>
__device__ __forceinline__ float dglu_block(const GemmArgs& a, const uint32_t* d16, const Tile& t, const int* tb,
                                            int lr, int64_t grow, int q, int lane, int slice, float prob, int b) {
  constexpr bool kGlu = EPI == EPI_DGLU_SWIGLU;
  const int n0 = t.nt * kBN + slice * kSliceCols + 32 * b;
  const int64_t N1 = a.n_cols_out;
  const int64_t N = kGlu ? N1 / 2 : N1;
  const uint16_t* hrow = a.act_in + grow * N1;
  uint8_t* crow = a.out_codes + grow * N1;
  const int nscale = (int)(N1 / 32);
  const int64_t sbase = (int64_t)(tb[t.g] + (lr >> 7)) * (nscale >> 2) * 512 + lane * 16 + q * 4;
  float dsum = 0.0f;
  // fc1_dy values (bf16, packed pairs) of the gate half (or h) and of the up half;
  // one pass over the accumulator so each of its values dies once it is used
  uint32_t ow0[16], ow1[kGlu ? 16 : 1];
#pragma unroll
  for (int c = 0; c < 32; c += 16) {
    // one whole 32-byte sector per load (each is read once: no L1 allocation)
    uint32_t gw[8], uw[8];
    ld_global_nc_v8(hrow + n0 + c, gw);
    if (kGlu) ld_global_nc_v8(hrow + N + n0 + c, uw);
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
      uint32_t w0, w1;
      dglu_pair<EPI>(d16[(c + k) >> 1], gw[k >> 1], kGlu ? uw[k >> 1] : 0u, prob, w0, w1, dsum);
      ow0[(c + k) >> 1] = w0;
      if (kGlu) ow1[((c + k) >> 1) & (kGlu ? 15 : 0)] = w1;
    }
  }
  constexpr int kOuts = kGlu ? 2 : 1;  // fc1_dy outputs per fc2_x column (gate and up, or h)
#pragma unroll
  for (int o = 0; o < kOuts; ++o) {
    const int64_t col = (o == 0 ? 0 : N) + n0;
    if (a.out_bf16) {  // fc1_dy in bf16 as well (the weight gradient's operand)
      uint16_t* brow = a.out_bf16 + grow * N1 + col;
      st_global_v8(brow, o == 0 ? ow0 : ow1);
      st_global_v8(brow + 16, (o == 0 ? ow0 : ow1) + 8);
    }
    const int e = mx_block_packed(o == 0 ? ow0 : ow1, crow + col);
    const int kidx = (int)(col / 32);
    a.out_scales[sbase + (int64_t)(kidx >> 2) * 512 + (kidx & 3)] = (uint8_t)(e + 127);
  }
  return dsum;
}

// A thread's 64 bf16 outputs (its row's 128-byte run of the slice) as four
// 32-byte units u[k].  quad_transpose swaps units inside each quad of lanes
// (a 4 x 4 transpose in two xor-shuffle rounds) so that afterwards slot s of
// lane 4g + r holds unit r of the quad's row 4g + s; store_quad_rows then
// writes slot s of the four lanes as one whole 128-byte run, so each warp
// store instruction covers 8 complete runs instead of one 32-byte piece of
// 32 rows.  Used by the scale-writer (SST) kernels, whose bf16 outputs it
// speeds up (NVFP4 fc2 164 -> 140 us); the other kernels measured slower
// with it (MXFP8 fc2 on the 64-expert workload 0.76 -> 0.82 ms) and keep
// row-per-lane stores.
__device__ __forceinline__ void quad_transpose(uint32_t (&u)[4][8], int lane) {
  const bool odd = lane & 1, upper = lane & 2;
#pragma unroll
  for (int p = 0; p < 2; ++p)
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      // after this round slot 2p + j holds unit 2p + (r & 1) of quad row (r & ~1) + j
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? u[2 * p][w] : u[2 * p + 1][w], 1);
      if (odd)
        u[2 * p][w] = recv;
      else
        u[2 * p + 1][w] = recv;
    }
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint32_t recv = __shfl_xor_sync(0xffffffffu, upper ? u[j][w] : u[2 + j][w], 2);
      if (upper)
        u[j][w] = recv;
      else
        u[2 + j][w] = recv;
    }
}

// Stores the transposed units: rows row0 + 4 (lane / 4) + s (s = 0..3) of a
// [rows x ld] bf16 matrix at column col0, rows at or past `limit` skipped.
__device__ __forceinline__ void store_quad_rows(uint16_t* out, int64_t ld, int64_t row0, int limit_rel, int rel0,
                                                int64_t col0, const uint32_t (&u)[4][8], int lane) {
  const int rq = 4 * (lane >> 2);
#pragma unroll
  for (int s = 0; s < 4; ++s)
    if (rel0 + rq + s < limit_rel) st_global_v8(out + (row0 + rq + s) * ld + col0 + 16 * (lane & 3), u[s]);
}

template <int FMT, int EPI, bool XT, bool QT>
__device__ __forceinline__ void epilogue(const GemmArgs& a, float* acc, const Tile& t, const int* off,
                                         const int* tb, const float* atab, int row_base, int q, int lane, int slice,
                                         float prob) {
  const int row = 32 * q + lane;
  const int m_g = off[t.g + 1] - off[t.g];
  const int lr = row_base + row;  // row within the group
  const bool valid = lr < m_g;
  const int64_t grow = (int64_t)off[t.g] + lr;
  float alpha = 1.0f;
  if (FMT == GMLP_NVFP4) alpha = atab[t.g];  // 1 / (S_a S_b), per group, computed once per CTA
  if (XT && a.bias) {
    // per-expert bias, added to the FP32 accumulator before any rounding; the
    // slice's two 32-column runs map to logical rows b0 and b1 of the bias
    // (SwiGLU: its gate and up rows under the 32-row interleave)
    const uint16_t* bg = a.bias + (int64_t)t.g * a.n_out;
    int b0, b1;
    if (EPI == EPI_FC1_SWIGLU) {
      const int c = t.nt * (kBN / 64) + slice;
      b0 = 32 * c;
      b1 = (int)(a.n_out / 2) + 32 * c;
    } else {
      b0 = t.nt * kBN + slice * kSliceCols;
      b1 = b0 + 32;
    }
#pragma unroll
    for (int j = 0; j < kSliceCols; j += 8) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(bg + (j < 32 ? b0 + j : b1 + (j - 32))));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 8; ++k)
        acc[j + k] = __fadd_rn(__fmul_rn(acc[j + k], alpha),
                               bf16_bits_to_float((k & 1) ? (w[k >> 1] >> 16) : (w[k >> 1] & 0xFFFFu)));
    }
    alpha = 1.0f;
  }

  if (EPI == EPI_FC2 && QT) {
    uint32_t u[4][8];
    const f32x2 alpha2 = pk2(alpha, alpha);
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const f32x2 v = mul2(pk2(acc[16 * j + 2 * k], acc[16 * j + 2 * k + 1]), alpha2);
        u[j][k] = pack2_bf16_rn(lo2(v), hi2(v));
      }
    quad_transpose(u, lane);
    // warp rows 32 q .. 32 q + 31 of the tile; this lane's quad stores rows 4 (lane / 4) + s
    store_quad_rows(a.out_bf16, a.n_cols_out, (int64_t)off[t.g] + row_base + 32 * q, m_g, row_base + 32 * q,
                    (int64_t)t.nt * kBN + slice * kSliceCols, u, lane);
    return;
  }
  if (EPI == EPI_FC2) {
    if (!valid) return;
    uint16_t* yrow = a.out_bf16 + grow * a.n_cols_out + (int64_t)t.nt * kBN + slice * kSliceCols;
#pragma unroll
    for (int j = 0; j < kSliceCols; j += 16) {
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = pack2_bf16_rn(acc[j + 2 * k] * alpha, acc[j + 2 * k + 1] * alpha);
      st_global_v8(yrow + j, o);
    }
    return;
  }

  constexpr int kOut = EPI == EPI_FC1_SWIGLU ? 32 : 64;  // fc2_x values this thread produces
  const int64_t oc0 = (int64_t)t.nt * (kBN / (EPI == EPI_FC1_SWIGLU ? 2 : 1)) + slice * kOut;
  if (XT && a.pre_act_out && valid) {
    // the activation input h = bf16(acc * alpha) in logical column order (the
    // backward's saved tensor): SwiGLU gate columns oc0.., up columns N + oc0..
    uint16_t* hrow = a.pre_act_out + grow * a.n_out;
#pragma unroll
    for (int j = 0; j < 64; j += 16) {
      uint32_t o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] = pack2_bf16_rn(acc[j + 2 * k] * alpha, acc[j + 2 * k + 1] * alpha);
      const int64_t col = EPI == EPI_FC1_SWIGLU ? (j < 32 ? oc0 + j : a.n_cols_out + oc0 + (j - 32)) : oc0 + j;
      st_global_v8(hrow + col, o);
    }
  }
  // fc2_x = bf16(act(bf16(acc * alpha)) * prob), in place in acc[0..kOut)
  if (EPI == EPI_FC1_SWIGLU) {
    // a 64-column slice holds 32 gate then 32 up columns of the same 32 outputs
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = fc2x_swiglu(round_bf16(acc[i] * alpha), round_bf16(acc[32 + i] * alpha), prob);
  } else if (EPI == EPI_FC1_TANH_SRELU) {
    // soft clamp of the squared ReLU at c: c * tanh(h^2 / c)
    const float c = a.tanh_c, inv_c = __frcp_rn(a.tanh_c);
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = fc2x_tanh_srelu(round_bf16(acc[i] * alpha), prob, c, inv_c);
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) acc[i] = fc2x_srelu(round_bf16(acc[i] * alpha), prob);
  }

  if (FMT == GMLP_MXFP8) {
    constexpr int kBlocks = kOut / 32;
    uint32_t sbytes = 0;
#pragma unroll
    for (int b = 0; b < kBlocks; ++b) {
      uint32_t words[8];
      const int e = mx_block(acc + 32 * b, words);
      sbytes |= uint32_t(e + 127) << (8 * b);
      if (valid) st_global_v8(a.out_codes + grow * a.n_cols_out + oc0 + 32 * b, words);
    }
    if (valid) {
      const int nscale = (int)(a.n_cols_out / 32);
      const int kidx = (int)(oc0 / 32);
      const int64_t blk = (int64_t)(tb[t.g] + (lr >> 7)) * (nscale >> 2) + (kidx >> 2);
      uint8_t* dst = a.out_scales + blk * 512 + lane * 16 + q * 4 + (kidx & 3);
      if (kBlocks == 1)
        *dst = (uint8_t)sbytes;
      else
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)sbytes;
    }
  } else {
    // NVFP4: store bf16 fc2_x; per-group max |fc2_x| and post-RHT amax over
    // 16-row column chunks (lanes 0-15 and 16-31 each hold one chunk; rows
    // past the group end count as zero).
    float pre = 0.0f, post = 0.0f;
    const bool want_post = a.amax_post != nullptr;  // else the fc2_x cast takes it
    const bool neg = (a.rht_mask >> (lane & 15)) & 1u;
#pragma unroll
    for (int c = 0; c < kOut; ++c) {
      float v = valid ? acc[c] : 0.0f;
      pre = fmaxf(pre, fabsf(v));
      if (want_post) {
        if (neg) v = -v;
#pragma unroll
        for (int h = 1; h < 16; h <<= 1) {
          const float p = __shfl_xor_sync(0xffffffffu, v, h);
          v = (lane & h) ? (p - v) : (v + p);
        }
        post = fmaxf(post, fabsf(v));
      }
    }
    if (QT && kOut == 64) {
      uint32_t u[4][8];
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int k = 0; k < 8; ++k) u[j][k] = pack2_bf16_rn(acc[16 * j + 2 * k], acc[16 * j + 2 * k + 1]);
      quad_transpose(u, lane);
      store_quad_rows(a.out_bf16, a.n_cols_out, (int64_t)off[t.g] + row_base + 32 * q, m_g, row_base + 32 * q, oc0, u,
                      lane);
    } else if (valid) {
      uint16_t* dst = a.out_bf16 + grow * a.n_cols_out + oc0;
#pragma unroll
      for (int j = 0; j < kOut; j += 16) {
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = pack2_bf16_rn(acc[j + 2 * k], acc[j + 2 * k + 1]);
        st_global_v8(dst + j, o);
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      pre = fmaxf(pre, __shfl_xor_sync(0xffffffffu, pre, d));
      post = fmaxf(post, __shfl_xor_sync(0xffffffffu, post, d));
    }
    if (lane == 0) {
      atomicMax(reinterpret_cast<int*>(a.amax_pre + t.g), __float_as_int(pre));
      if (want_post) atomicMax(reinterpret_cast<int*>(a.amax_post + t.g), __float_as_int(post * 0.25f));
    }
  }
}


// ------------------------------------------------------------------ CTA-pair helpers

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Tensor load into this CTA's shared memory that completes its bytes on the
// pair leader's mbarrier (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* smem_dst, const void* tmap, int32_t x, int32_t y,
                                                 uint32_t bar_cluster, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(bar_cluster), "l"(policy)
      : "memory");
}

template <int PAIR>
__device__ __forceinline__ void tmem_alloc_g(uint32_t* slot) {
  if (PAIR == 1) {
    tmem_alloc(slot, kTmemCols);
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int PAIR>
__device__ __forceinline__ void tmem_dealloc_g(uint32_t taddr) {
  if (PAIR == 1)
    tmem_dealloc(taddr, kTmemCols);
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols) : "memory");
}

// Arrive on `bar` (same offset in both CTAs of a pair) when this thread's
// tcgen05 operations complete.
template <int PAIR>
__device__ __forceinline__ void tc_commit_g(uint64_t* bar) {
  if (PAIR == 1)
    tc_commit(bar);
  else
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

template <int PAIR>
__device__ __forceinline__ void tc_cp_g(uint32_t taddr, uint64_t sdesc) {
  if (PAIR == 1)
    tc_cp_32x128b_x4(taddr, sdesc);
  else
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 128 rows x 32 bytes of shared memory into TMEM lanes 0..127, columns taddr ..
// taddr + 7 (a CTA pair: each CTA from its own shared memory into its own TMEM).
template <int PAIR>
__device__ __forceinline__ void tc_cp_wide_g(uint32_t taddr, uint64_t sdesc) {
  if (PAIR == 1)
    tc_cp_128x256b(taddr, sdesc);
  else
    asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

template <int FMT, int PAIR>
__device__ __forceinline__ void tc_mma_g(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
  if (PAIR == 1) {
    if (FMT == GMLP_MXFP8)
      tc_mma_mxf8(d, adesc, bdesc, idesc, sfa, sfb, accumulate);
    else
      tc_mma_nvf4(d, adesc, bdesc, idesc, sfa, sfb, accumulate);
  } else if (FMT == GMLP_MXFP8) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
            d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
            d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
  }
}

// ------------------------------------------------------------------ kernel

template <int FMT, int EPI, int PAIR, bool X4, bool XT>
__global__ void __launch_bounds__(Cfg<FMT, PAIR, X4>::kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                const GemmArgs a) {
  using C = Cfg<FMT, PAIR, X4>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * kATileBytes;
  uint8_t* sSFA = sB + S * C::kBTileBytes;
  uint8_t* sSFB = sSFA + S * C::kSfBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + S * C::kSfBBytes);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint64_t* sfready = drain + 1;  // SST: one per stage, the four scale writers arrive
  uint64_t* sfull = sfready + S;  // SST: the stage's scale bytes have landed (A / B on full)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sfull + S);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* bad = reinterpret_cast<int*>(tslot + 2);
  int* off = reinterpret_cast<int*>(tslot + 4);
  int* tb = off + kMaxGroups + 1;
  int* ip = tb + kMaxGroups + 1;
  float* atab = reinterpret_cast<float*>(ip + kMaxGroups + 1);  // NVFP4: per-group 1 / (S_a S_b)

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int G = a.grp.G;
  const int n_tiles = (int)(a.n_out / kBN);
  const int KB = (int)(a.kbytes / kBKBytes);
  const uint32_t crank = PAIR == 2 ? cluster_ctarank() : 0;
  const int rank = (int)(crank & 1);          // position in the pair
  const uint32_t leader = crank & ~1u;        // cluster rank of the pair leader
  const int unit = blockIdx.x / PAIR, n_units = gridDim.x / PAIR;

  if (warp == 0) {
    // group tables: row offsets, 128-row tile bases, tile-work prefix
    long long c0 = 0, c1 = 0, c2 = 0;
    int b = 0;
    for (int base = 0; base < G; base += 32) {
      const int g = base + lane;
      long long m = 0;
      if (g < G) {
        m = a.grp.splits ? (long long)a.grp.splits[g] : (long long)a.grp.uniform_m;
        if (m < 0 || m > a.grp.M) {
          b = 1;
          m = 0;
        }
      }
      const long long v0 = m, v1 = (m + kBM - 1) / kBM, v2 = (m + C::kTileRows - 1) / C::kTileRows * n_tiles;
      long long i0 = v0, i1 = v1, i2 = v2;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const long long t0 = __shfl_up_sync(0xffffffffu, i0, d), t1 = __shfl_up_sync(0xffffffffu, i1, d),
                        t2 = __shfl_up_sync(0xffffffffu, i2, d);
        if (lane >= d) {
          i0 += t0;
          i1 += t1;
          i2 += t2;
        }
      }
      if (g < G) {
        off[g] = (int)(c0 + i0 - v0);
        tb[g] = (int)(c1 + i1 - v1);
        ip[g] = (int)(c2 + i2 - v2);
      }
      c0 += __shfl_sync(0xffffffffu, i0, 31);
      c1 += __shfl_sync(0xffffffffu, i1, 31);
      c2 += __shfl_sync(0xffffffffu, i2, 31);
      if (c0 > a.grp.M) b = 1;
    }
    b = __any_sync(0xffffffffu, b);
    if (lane == 0) {
      off[G] = (int)c0;
      tb[G] = (int)c1;
      ip[G] = (int)c2;
      *bad = b;
      if (b && blockIdx.x == 0) report_device_error(GMLP_ERR_DEVICE_BOUNDS);
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      if (PAIR == 2) {
        prefetch_tmap(&tmSFA);
        prefetch_tmap(&tmSFB);
      }
    }
  } else if (warp == 1) {
    tmem_alloc_g<PAIR>(tslot);
  } else if (threadIdx.x == 64) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kEpiWarps * PAIR);
    mbar_init(drain, 1);
    if (C::kSST)
      for (int s = 0; s < S; ++s) {
        mbar_init(&sfready[s], 4);
        mbar_init(&sfull[s], 1);
      }
    *abort_flag = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR == 2) cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after();
  griddep_wait();                 // the previous kernel's outputs (A operand, amaxes) are complete
  griddep_launch_dependents();
  if (FMT == GMLP_NVFP4) {
    // the epilogue's alpha per group: the amaxes come from the previous kernels
    for (int g = threadIdx.x; g < G; g += blockDim.x)
      atab[g] = __fdiv_rn(1.0f, __fmul_rn(nvfp4_global_scale(a.a_amax[g]), a.b_S[g]));
    __syncthreads();
  }
  const uint32_t tbase = *tslot;
  const int total = *bad ? 0 : ip[G];

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs of a pair load their own halves)
    const uint64_t pol_a = policy_evict_normal();
    const uint64_t pol_b = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    constexpr uint32_t kTx = (uint32_t)C::kStageBytes * PAIR;
    constexpr int kSfRows = C::kSfBytes / 256;  // SF tensor-map rows per 128-row block
    for (int w = unit; w < total && !*abort_flag; w += n_units) {
      const Tile t = decode_tile<C::kTileRows>(off, ip, G, w, a.n_out, n_tiles);
      const int row0 = t.mt * C::kTileRows + kBM * rank;  // first row of this CTA within the group
      const int rowA = off[t.g] + row0;
      const int64_t tileA = tb[t.g] + (row0 >> 7);
      const int64_t rowB0 = (int64_t)t.g * a.n_out + (int64_t)t.nt * kBN;
      const int64_t tileB = rowB0 / 128;
      const int32_t rowB = (int32_t)(rowB0 + rank * C::kBRows);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) break;
        uint8_t* sfb = sSFB + stage * C::kSfBBytes;
        if (C::kSST) {
          // the scale bytes first, on their own barrier: the scale writers
          // place them in TMEM while the A / B tiles are still arriving
          mbar_arrive_expect_tx(&sfull[stage], (uint32_t)(C::kSfBytes + C::kSfBBytes));
          mbar_arrive_expect_tx(&full[stage], (uint32_t)(kATileBytes + C::kBTileBytes));
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          bulk_load(sSFA + stage * C::kSfBytes, a.a_scales + (tileA * KB + kb) * C::kSfBytes, C::kSfBytes,
                    &sfull[stage]);
          bulk_load(sfb, a.b_scales + (tileB * KB + kb) * C::kSfBytes, C::kSfBytes, &sfull[stage]);
          bulk_load(sfb + C::kSfBytes, a.b_scales + ((tileB + 1) * KB + kb) * C::kSfBytes, C::kSfBytes,
                    &sfull[stage]);
          tma_load_2d(sA + stage * kATileBytes, &tmA, kb * kBKBytes, rowA, &full[stage], pol_a);
          tma_load_2d(sB + stage * C::kBTileBytes, &tmB, kb * kBKBytes, rowB, &full[stage], pol_b);
        } else if (PAIR == 1) {
          mbar_arrive_expect_tx(&full[stage], kTx);
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          tma_load_2d(sA + stage * kATileBytes, &tmA, kb * kBKBytes, rowA, &full[stage], pol_a);
          tma_load_2d(sB + stage * C::kBTileBytes, &tmB, kb * kBKBytes, rowB, &full[stage], pol_b);
          bulk_load(sSFA + stage * C::kSfBytes, a.a_scales + (tileA * KB + kb) * C::kSfBytes, C::kSfBytes,
                    &full[stage]);
          if (X4) {
            bulk_load(sfb, a.b_scales + ((tileB >> 1) * KB + kb) * C::kSfBBytes, C::kSfBBytes, &full[stage]);
          } else {
            bulk_load(sfb, a.b_scales + (tileB * KB + kb) * C::kSfBytes, C::kSfBytes, &full[stage]);
            bulk_load(sfb + C::kSfBytes, a.b_scales + ((tileB + 1) * KB + kb) * C::kSfBytes, C::kSfBytes,
                      &full[stage]);
          }
        } else {
          const uint32_t bar = mapa_shared(smem_u32(&full[stage]), leader);
          if (rank == 0) {
            mbar_arrive_expect_tx(&full[stage], kTx);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          }
          tma_load_2d_pair(sA + stage * kATileBytes, &tmA, kb * kBKBytes, rowA, bar, pol_a);
          tma_load_2d_pair(sB + stage * C::kBTileBytes, &tmB, kb * kBKBytes, rowB, bar, pol_b);
          tma_load_2d_pair(sSFA + stage * C::kSfBytes, &tmSFA, 0, (int32_t)((tileA * KB + kb) * kSfRows), bar,
                           pol_a);
          if (X4) {  // the stage's 16 KB GEMM_TILED_X4 block of the B tile pair, whole in each CTA
            tma_load_2d_pair(sfb, &tmSFB, 0, (int32_t)(((tileB >> 1) * KB + kb) * (C::kSfBBytes / 256)), bar,
                             pol_b);
          } else {
            tma_load_2d_pair(sfb, &tmSFB, 0, (int32_t)((tileB * KB + kb) * kSfRows), bar, pol_b);
            tma_load_2d_pair(sfb + C::kSfBytes, &tmSFB, 0, (int32_t)(((tileB + 1) * KB + kb) * kSfRows), bar,
                             pol_b);
          }
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // every copy signalled on this CTA's barriers must land before it exits
    for (int s = 0; s < S; ++s)
      if (armed & (1u << s)) {
        mbar_wait_drain(&full[s], (armed_parity >> s) & 1u);
        if (C::kSST) mbar_wait_drain(&sfull[s], (armed_parity >> s) & 1u);
      }
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (the pair leader issues for both CTAs)
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    const uint32_t sf_base = tbase + kAccCols;
    for (int w = unit; w < total && !*abort_flag; w += n_units) {
      if (!mbar_wait(tempty, acc_phase ^ 1, abort_flag)) break;
      tc_fence_after();
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag) ||
            (C::kSST && !mbar_wait(&sfready[stage], phase, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = sf_base + stage * C::kSfCols;
        const uint32_t sfb_t = sfa_t + C::kSfbOff;
        const uint32_t sA_addr = smem_u32(sA + stage * kATileBytes);
        const uint32_t sB_addr = smem_u32(sB + stage * C::kBTileBytes);
        const uint32_t sfa_addr = smem_u32(sSFA + stage * C::kSfBytes);
        const uint32_t sfb_addr = smem_u32(sSFB + stage * C::kSfBBytes);
        if (FMT == GMLP_MXFP8) {
          tc_cp_g<PAIR>(sfa_t, smem_desc(sfa_addr, 0, 128, 0));
          tc_cp_g<PAIR>(sfb_t, smem_desc(sfb_addr, 0, 128, 0));
          tc_cp_g<PAIR>(sfb_t + 4, smem_desc(sfb_addr + 512, 0, 128, 0));
        } else if (C::kSST) {
          // the scale writers have placed this stage's scales
        } else if (X4) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc_cp_g<PAIR>(sfa_t + 4 * k, smem_desc(sfa_addr + 512 * k, 0, 128, 0));
            // [4 x half-0 block | 4 x half-1 block]: 128 rows x 32 bytes, the two
            // 16-byte column halves 2048 bytes apart, 8-row groups 128 apart
            tc_cp_wide_g<PAIR>(sfb_t + 8 * k, smem_desc(sfb_addr + 4096 * k, 2048, 128, 0));
          }
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            tc_cp_g<PAIR>(sfa_t + 4 * k, smem_desc(sfa_addr + 512 * k, 0, 128, 0));
            tc_cp_g<PAIR>(sfb_t + 8 * k, smem_desc(sfb_addr + 512 * k, 0, 128, 0));
            tc_cp_g<PAIR>(sfb_t + 8 * k + 4, smem_desc(sfb_addr + 2048 + 512 * k, 0, 128, 0));
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = smem_desc(sA_addr + 32 * k, 16, 1024, 2);
          const uint64_t bd = smem_desc(sB_addr + 32 * k, 16, 1024, 2);
          const uint32_t accumulate = (kb > 0 || k > 0) ? 1u : 0u;
          if (FMT == GMLP_MXFP8)
            tc_mma_g<FMT, PAIR>(tbase, ad, bd, idesc_for<FMT, kBM * PAIR>(k), sfa_t, sfb_t, accumulate);
          else
            tc_mma_g<FMT, PAIR>(tbase, ad, bd, idesc_for<FMT, kBM * PAIR>(k), sfa_t + 4 * k, sfb_t + 8 * k,
                                accumulate);
        }
        tc_commit_g<PAIR>(&empty[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      tc_commit_g<PAIR>(tfull);
      acc_phase ^= 1;
    }
    // all MMAs and copies this thread issued complete before TMEM is freed
    tc_commit_g<PAIR>(drain);
    mbar_wait_drain(drain, 0);
  } else if (C::kSST && warp >= C::kScaleWarp0) {
    // ---------------- scale writers: warp w stores each stage's SFA / SFB into
    // TMEM lanes 32 * (w % 4) .. + 31, in the layout the 32x128b.warpx4 copies
    // would produce, as soon as the stage's scale bytes have landed (sfull,
    // ahead of the A / B tiles), and signals the issuer; the stage's shared
    // memory is not refilled before the issuer's commit, which follows the signal
    const uint32_t lane_base = uint32_t(32 * (warp & 3)) << 16;
    const uint32_t sf_base = tbase + kAccCols;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int w = unit; ok && w < total && !*abort_flag; w += n_units) {
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(&sfull[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        const uint32_t sfa_t = sf_base + stage * C::kSfCols;
        const uint8_t* sfa = sSFA + stage * C::kSfBytes;
        write_stage_scales<FMT>(lane_base, sfa_t, sfa_t + C::kSfbOff, sfa, sSFB + stage * C::kSfBBytes, lane);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp >= C::kEpiWarp0) {
    // ---------------- epilogue: 16 warps; warp w reads TMEM lanes 32 * (w % 4)
    // and the 64-column slice (w - kEpiWarp0) / 4 of this CTA's 128 accumulator rows
    const int q = warp & 3;
    const int slice = (warp - C::kEpiWarp0) >> 2;
    const uint32_t tempty_addr = PAIR == 2 ? mapa_shared(smem_u32(tempty), leader) : 0;
    uint32_t acc_phase = 0;
    for (int w = unit; w < total && !*abort_flag; w += n_units) {
      const Tile t = decode_tile<C::kTileRows>(off, ip, G, w, a.n_out, n_tiles);
      const int row_base = t.mt * C::kTileRows + kBM * rank;
      float prob = 1.0f;
      if (EPI != EPI_FC2 && a.probs) {
        const int lr = row_base + 32 * q + lane;
        if (lr < off[t.g + 1] - off[t.g]) prob = __ldg(a.probs + off[t.g] + lr);
      }
      if (EPI == EPI_DGLU_SWIGLU || EPI == EPI_DSRELU) {
        // start this row's activation-input lines (gate and up) on their way to
        // L2 while the tile's MMAs run
        const int lr = row_base + 32 * q + lane;
        if (lr < off[t.g + 1] - off[t.g]) {
          const int64_t N1 = a.n_cols_out;
          const uint16_t* hp = a.act_in + ((int64_t)off[t.g] + lr) * N1 + t.nt * kBN + slice * kSliceCols;
          prefetch_l2(hp);
          if (EPI == EPI_DGLU_SWIGLU) prefetch_l2(hp + N1 / 2);
        }
      }
      if (!mbar_wait(tfull, acc_phase, abort_flag)) break;
      tc_fence_after();
      const uint32_t taddr = tbase + (uint32_t(32 * q) << 16) + uint32_t(slice * kSliceCols);
      if (EPI == EPI_DGLU_SWIGLU || EPI == EPI_DSRELU) {
        // backward dGLU: the accumulator is read as bf16 pairs (the epilogue's
        // first rounding) and released before any of the math
        const int lr = row_base + 32 * q + lane;
        const bool valid = lr < off[t.g + 1] - off[t.g];
        const int64_t grow = (int64_t)off[t.g] + lr;
        uint32_t d16[32];  // bf16(dfc2x) of the 64 columns, packed pairs
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float acc32[32];
          tmem_ld32(taddr + 32 * h, acc32);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) d16[16 * h + i] = pack2_bf16_rn(acc32[2 * i], acc32[2 * i + 1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty);
        acc_phase ^= 1;
        if (valid) {
          float dsum = dglu_block<EPI>(a, d16, t, tb, lr, grow, q, lane, slice, prob, 0);
          dsum += dglu_block<EPI>(a, d16 + 16, t, tb, lr, grow, q, lane, slice, prob, 1);
          if (a.dprob) atomicAdd(a.dprob + grow, dsum);
        }
        continue;
      }
      float acc[kSliceCols];
      tmem_ld32(taddr, acc);
      tmem_ld32(taddr + 32, acc + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR == 1)
          mbar_arrive(tempty);
        else
          mbar_arrive_cluster(tempty_addr);
      }
      acc_phase ^= 1;
      epilogue<FMT, EPI, XT, C::kSST>(a, acc, t, off, tb, atab, row_base, q, lane, slice, prob);
    }
  }
  __syncthreads();
  if (PAIR == 2) cluster_sync();  // neither CTA leaves while its peer may still signal it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_g<PAIR>(tbase);
  }
}

// ------------------------------------------------------------------ host side

template <int FMT, int EPI, int PAIR, bool X4 = false, bool XT = false>
cudaError_t launch_t(const GemmArgs& a, cudaStream_t s) {
  using C = Cfg<FMT, PAIR, X4>;
  const size_t smem = C::kSmem + 1024 + 256 + 3 * (kMaxGroups + 1) * sizeof(int) +
                      (FMT == GMLP_NVFP4 ? (kMaxGroups + 1) * sizeof(float) : 0);
  auto kern = gemm_kernel<FMT, EPI, PAIR, X4, XT>;
  static bool attr_set[64] = {};
  static int max_units[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR == 2 ? 1 : 0;
  if (!attr_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int units = num_sms() / PAIR;
    if (PAIR == 2) {
      cfg.gridDim = dim3(2 * units);
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      if (clusters < units) units = clusters;
    }
    max_units[dev & 63] = units;
    attr_set[dev & 63] = true;
  }
  const int nscale = (int)(FMT == GMLP_MXFP8 ? a.kbytes / 32 : a.kbytes / 8);
  const int64_t sfa_bytes = ((a.M + 127) / 128 + a.grp.G) * 128LL * nscale;
  const int64_t sfb_bytes = (int64_t)a.grp.G * a.n_out * nscale * (X4 ? 4 : 1);
  CUtensorMap ta, tbm, tsa, tsb;
  if (!make_tmap(&ta, a.a_codes, a.kbytes, a.M, kBKBytes, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tbm, a.b_codes, a.kbytes, (int64_t)a.grp.G * a.n_out, kBKBytes, C::kBRows,
                 CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tsa, a.a_scales, 256, sfa_bytes / 256, 256, C::kSfBytes / 256, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !make_tmap(&tsb, a.b_scales, 256, sfb_bytes / 256, 256, (X4 ? C::kSfBBytes : C::kSfBytes) / 256,
                 CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const int64_t max_tiles = ((a.M + C::kTileRows - 1) / C::kTileRows + a.grp.G) * (a.n_out / kBN);
  int64_t units = max_units[dev & 63];
  if (max_tiles < units) units = max_tiles;
  if (units < 1) units = 1;
  cfg.gridDim = dim3((unsigned)(units * PAIR));
  if (PAIR == 2) {
    cfg.numAttrs = a.pdl ? 2 : 1;
  } else if (a.pdl) {
    cfg.attrs = attr + 1;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, ta, tbm, tsa, tsb, a);
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

bool make_tmap(CUtensorMap* m, const void* base, int64_t row_bytes, int64_t rows, int box_bytes, int box_rows,
               CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_u16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int box_cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int gemm_read_clear_status() { return read_clear_status(); }

// Single-CTA tiles unless the caller asks for CTA pairs.  Biases and the
// saved activation input (XT) have their own single-CTA instantiations, so the
// plain kernels keep their registers.
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.M == 0) return cudaSuccess;
  const bool pair = a.pair == 2;
  const bool xt = a.bias || a.pre_act_out;
  if (xt && pair) return cudaErrorInvalidConfiguration;  // rejected by the API before
#define GMLP_ONE(F, E, X4) \
  return xt ? launch_t<F, E, 1, X4, true>(a, s) : launch_t<F, E, 1, X4, false>(a, s)
#define GMLP_LAUNCH(F, E)                                        \
  if (pair) return launch_t<F, E, 2, false, false>(a, s);        \
  GMLP_ONE(F, E, false)
#define GMLP_X4(F, E)                                    \
  if (pair) return launch_t<F, E, 2, true, false>(a, s); \
  GMLP_ONE(F, E, true)
  if (a.format == GMLP_MXFP8) {
    if (a.epi == EPI_FC1_SWIGLU) { GMLP_LAUNCH(GMLP_MXFP8, EPI_FC1_SWIGLU); }
    if (a.epi == EPI_FC1_SRELU) { GMLP_LAUNCH(GMLP_MXFP8, EPI_FC1_SRELU); }
    if (a.epi == EPI_FC1_TANH_SRELU) { GMLP_LAUNCH(GMLP_MXFP8, EPI_FC1_TANH_SRELU); }
    if (a.epi == EPI_DGLU_SWIGLU) return launch_t<GMLP_MXFP8, EPI_DGLU_SWIGLU, 1>(a, s);
    if (a.epi == EPI_DSRELU) return launch_t<GMLP_MXFP8, EPI_DSRELU, 1>(a, s);
    GMLP_LAUNCH(GMLP_MXFP8, EPI_FC2);
  }
  if (a.b_x4) {  // replicated B scales
    if (a.epi == EPI_FC1_SWIGLU) { GMLP_X4(GMLP_NVFP4, EPI_FC1_SWIGLU); }
    if (a.epi == EPI_FC1_SRELU) { GMLP_X4(GMLP_NVFP4, EPI_FC1_SRELU); }
    if (a.epi == EPI_FC1_TANH_SRELU) { GMLP_X4(GMLP_NVFP4, EPI_FC1_TANH_SRELU); }
    GMLP_X4(GMLP_NVFP4, EPI_FC2);
  }
  if (a.epi == EPI_FC1_SWIGLU) { GMLP_LAUNCH(GMLP_NVFP4, EPI_FC1_SWIGLU); }
  if (a.epi == EPI_FC1_SRELU) { GMLP_LAUNCH(GMLP_NVFP4, EPI_FC1_SRELU); }
  if (a.epi == EPI_FC1_TANH_SRELU) { GMLP_LAUNCH(GMLP_NVFP4, EPI_FC1_TANH_SRELU); }
  GMLP_LAUNCH(GMLP_NVFP4, EPI_FC2);
#undef GMLP_X4
#undef GMLP_LAUNCH
#undef GMLP_ONE
}

}  // namespace gmlp
