// quant.cu -- the group quantisers: rowwise MXFP8 / NVFP4 casts, per-group
// amax, the group Hadamard-amax pass and the fused row + column (RHT) NVFP4
// cast.  All are memory-bound streaming kernels: 128-bit loads that bypass L1,
// warp-shuffle block reductions, and the 16-point Hadamard in registers.
//
// Method: PR #3837 "Reduce NVFP4 quantization work for the fused GroupedMLP
// fc2 input with activation recompute" (Description and Changes: the group
// quantize of the fc2 input, nvfp4_group_hadamard_amax, quantize-with-amax,
// the RHT sign mask in the post-RHT amax); PR #2769 "GEMM + Swiglu fused
// Grouped MLP for MXFP8" (MXFP8 operands with GEMM-swizzled scales).
#include "device.cuh"

namespace gmlp {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Per-group tables built from split_sizes at the start of every kernel.
struct SmemGroups {
  int off[kMaxGroups + 1];  // first row of each group
  int tb[kMaxGroups + 1];   // first 128-row tile of each group (GEMM_TILED scales)
  int up[kMaxGroups + 1];   // first work unit (unit_rows-row block x 256-column slab)
  int mp[kMaxGroups + 1];   // prefix of the 16-row padded group sizes
  int bad;
};

// Warp 0 scans the G split sizes (32 at a time); everything is validated
// against M.  Negative sizes or a total above M set GMLP_ERR_DEVICE_BOUNDS and
// t.bad, and the kernel does nothing.
__device__ void build_group_tables(const GroupSrc& gs, int slabs, SmemGroups& t, int unit_rows = 16) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    long long c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    int bad = 0;
    for (int base = 0; base < gs.G; base += 32) {
      const int g = base + lane;
      long long m = 0;
      if (g < gs.G) {
        m = gs.splits ? (long long)gs.splits[g] : (long long)gs.uniform_m;
        if (m < 0 || m > gs.M) {
          bad = 1;
          m = 0;
        }
      }
      const long long ch = (m + 15) >> 4;
      long long v0 = m, v1 = (m + 127) >> 7, v2 = (m + unit_rows - 1) / unit_rows * slabs, v3 = ch * 16;
      long long i0 = v0, i1 = v1, i2 = v2, i3 = v3;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        long long t0 = __shfl_up_sync(0xffffffffu, i0, d), t1 = __shfl_up_sync(0xffffffffu, i1, d);
        long long t2 = __shfl_up_sync(0xffffffffu, i2, d), t3 = __shfl_up_sync(0xffffffffu, i3, d);
        if (lane >= d) {
          i0 += t0;
          i1 += t1;
          i2 += t2;
          i3 += t3;
        }
      }
      if (g < gs.G) {
        t.off[g] = (int)(c0 + i0 - v0);
        t.tb[g] = (int)(c1 + i1 - v1);
        t.up[g] = (int)(c2 + i2 - v2);
        t.mp[g] = (int)(c3 + i3 - v3);
      }
      c0 += __shfl_sync(0xffffffffu, i0, 31);
      c1 += __shfl_sync(0xffffffffu, i1, 31);
      c2 += __shfl_sync(0xffffffffu, i2, 31);
      c3 += __shfl_sync(0xffffffffu, i3, 31);
      if (c0 > gs.M) bad = 1;
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      t.off[gs.G] = (int)c0;
      t.tb[gs.G] = (int)c1;
      t.up[gs.G] = (int)c2;
      t.mp[gs.G] = (int)c3;
      t.bad = bad;
      if (bad && blockIdx.x == 0) report_device_error(GMLP_ERR_DEVICE_BOUNDS);
    }
  }
  __syncthreads();
}

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// ld_stream with an L2 cache policy (createpolicy)
__device__ __forceinline__ uint4 ld_stream_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

__device__ __forceinline__ void atomic_max_nonneg(float* p, float v) {
  atomicMax(reinterpret_cast<int*>(p), __float_as_int(v));
}

// Group containing row r, searching forward from g.
__device__ __forceinline__ int find_group(const SmemGroups& t, int G, int64_t r) {
  int lo = 0, hi = G - 1;  // largest g with off[g] <= r
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (t.off[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int find_unit_group(const SmemGroups& t, int G, int64_t u) {
  int lo = 0, hi = G - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (t.up[mid] <= u) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------------ rowwise cast

// NVFP4 encode factor for block scale byte c under global scale S:
// fp32(S / E4M3(c)), saturated at FLT_MAX as S is (0 for c = 0).
__device__ __forceinline__ float nvfp4_enc(float S, uint32_t c) {
  return (c == 0 || c == 127) ? 0.0f : fminf(__fdiv_rn(S, e4m3_to_float(c)), 3.402823466e38f);
}

// Eight FP32 values (already multiplied by the encode factor) -> four E2M1
// code bytes packed into one word, element 0 in the low nibble.
__device__ __forceinline__ uint32_t e2m1_pack8(const float* p) {
  uint32_t w;
  asm("{\n .reg .b8 q0, q1, q2, q3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n"
      " mov.b32 %0, {q0, q1, q2, q3};\n}"
      : "=r"(w)
      : "f"(p[0]), "f"(p[1]), "f"(p[2]), "f"(p[3]), "f"(p[4]), "f"(p[5]), "f"(p[6]), "f"(p[7]));
  return w;
}


// max(|a|, |b|) on packed bf16 pairs (sign bits set to the xor of the inputs'
// signs; a NaN operand yields the other one).
__device__ __forceinline__ uint32_t bmax_abs2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Max |x| over the 8 bf16 values of v as a bf16 bit pattern (0..0x7f80):
// NaN values are ignored and a chunk of eight NaNs gives 0, as a chain of
// fmaxf starting from 0 would.
__device__ __forceinline__ uint32_t amax8_bits(const uint4& v) {
  uint32_t m = bmax_abs2(bmax_abs2(v.x, v.y), bmax_abs2(v.z, v.w));
  m = bmax_abs2(m, __byte_perm(m, 0, 0x1032)) & 0x7fffu;
  return m > 0x7f80u ? 0u : m;
}

// The larger of the two bf16 magnitudes in a packed max (as amax8_bits).
__device__ __forceinline__ uint32_t amax_pair_bits(uint32_t m) {
  m = bmax_abs2(m, __byte_perm(m, 0, 0x1032)) & 0x7fffu;
  return m > 0x7f80u ? 0u : m;
}

// Four FP32 values -> four E4M3 bytes (element 0 in the low byte).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n mov.b32 %0, {lo, hi};\n}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// The 8 bf16 values of v (element 2i in the low half of word i) as four
// packed FP32 pairs multiplied by m: exact bf16 -> FP32 widening, then one
// IEEE round-to-nearest-even product per element.
__device__ __forceinline__ void scale8(const uint4& v, float m, float* q) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  const f32x2 m2 = pk2(m, m);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const f32x2 p = mul2(pk2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u)), m2);
    q[2 * i] = lo2(p);
    q[2 * i + 1] = hi2(p);
  }
}

// Bytes of lanes l, l+s, l+2s, l+3s packed into one word (valid in lanes
// whose l+3s stays inside the warp).
__device__ __forceinline__ uint32_t gather4_bytes(uint32_t byte, int s) {
  const uint32_t pair = byte | (__shfl_down_sync(0xffffffffu, byte, s) << 8);
  return pair | (__shfl_down_sync(0xffffffffu, pair, 2 * s) << 16);
}

// Work every launch of the row quantiser does first: the zeroing requests
// (spread over the grid) and the per-group global scales (block 0).
__device__ __forceinline__ void row_quant_setup(const RowQuantArgs& a, int nthreads) {
  const int64_t first = (int64_t)blockIdx.x * nthreads + threadIdx.x, step = (int64_t)gridDim.x * nthreads;
  if (a.zero_ptr)
    for (int64_t i = first; i < a.zero_count; i += step) a.zero_ptr[i] = 0.0f;
  if (a.zero_ptr2)
    for (int64_t i = first; i < a.zero_count2; i += step) a.zero_ptr2[i] = 0.0f;
  if (blockIdx.x != 0) return;
  if (a.S_out)
    for (int g = threadIdx.x; g < a.grp.G; g += nthreads) a.S_out[g] = nvfp4_global_scale(a.amax[g]);
}

// E4M3 scale byte of an NVFP4 block whose max |x| is the bf16 value with bits
// m (0..0x7f80), under global scale S: E4M3(fp32(fp32(b / 6) * S)).  The
// quotient fp32(b / 6) comes from q1 = fp32(b * fp32(1/6)) and one residual
// correction fp32(fma(fma(-6, q1, b), fp32(1/6), q1)); for every finite bf16
// b this equals the IEEE quotient (checked exhaustively over all 2^15
// magnitudes), and b = inf keeps inf.
__device__ __forceinline__ uint32_t nvfp4_block_sf_bf16(uint32_t m, float S) {
  const float b = __uint_as_float(m << 16);
  const float r6 = __uint_as_float(0x3e2aaaabu);  // fp32(1/6)
  const float q1 = __fmul_rn(b, r6);
  const float q = m >= 0x7f80u ? b : __fmaf_rn(__fmaf_rn(-6.0f, q1, b), r6, q1);
  return e4m3x2(__fmul_rn(q, S), 0.0f) & 0xFF;
}

// One pass of the row quantiser: lane l takes chunks c0+l, c0+l+32, ...,
// c0+l+96 of the row (FULL: all inside the row, no per-lane checks).  MXFP8
// blocks (32 elements) span 4 lanes, NVFP4 blocks (16) span 2; four
// consecutive blocks' scale bytes go out as one word from lanes 0/16 (MXFP8)
// or 0/8/16/24 (NVFP4).
template <int FMT, bool TILED, bool FULL>
__device__ __forceinline__ void row_pass(const uint4* xr, uint8_t* crow, uint8_t* srow, int c0, int cpr, int lane,
                                         float S, const float* enc) {
  constexpr int U = 4;
  uint4 v[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int c = c0 + 32 * u + lane;
    v[u] = (FULL || c < cpr) ? ld_stream(xr + c) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int c = c0 + 32 * u + lane;
    const bool active = FULL || c < cpr;
    uint32_t m = amax8_bits(v[u]);
    if (FMT == GMLP_MXFP8) {
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const int e = max((int)(m >> 7) - 135, -127);  // floor(log2 amax) - 8 from the bf16 exponent
      float q[8];
      scale8(v[u], exp2_neg(e), q);
      const uint32_t word = gather4_bytes((uint32_t)(e + 127), 4);
      if (active) {
        *reinterpret_cast<uint2*>(crow + c * 8) =
            make_uint2(e4m3x4(q[0], q[1], q[2], q[3]), e4m3x4(q[4], q[5], q[6], q[7]));
        if ((lane & 15) == 0) *reinterpret_cast<uint32_t*>(srow + (TILED ? (c >> 4) * 512 : (c >> 2))) = word;
      }
    } else {
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      const uint32_t sf = nvfp4_block_sf_bf16(m, S);
      float q[8];
      scale8(v[u], enc[sf], q);
      const uint32_t word = gather4_bytes(sf, 2);
      if (active) {
        *reinterpret_cast<uint32_t*>(crow + c * 4) = e2m1_pack8(q);
        if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(srow + (TILED ? (c >> 3) * 512 : (c >> 1))) = word;
      }
    }
  }
}

// Row quantiser.  The rows are cut into passes of 128 16-byte chunks (the last
// pass of a row may be shorter); warp w takes an equal contiguous share of
// the passes and sets up each row it touches once.  NVFP4 encode factors
// S / E4M3(sf) come from a per-warp table of the current group.
template <int FMT, bool TILED>
__global__ void __launch_bounds__(kThreads, FMT == GMLP_MXFP8 ? 4 : 5) row_quant_kernel(RowQuantArgs a) {
  __shared__ SmemGroups t;
  __shared__ float enc_tab[FMT == GMLP_NVFP4 ? kWarps : 1][128];
  build_group_tables(a.grp, 1, t);
  griddep_wait();
  griddep_launch_dependents();
  if (t.bad) return;
  row_quant_setup(a, kThreads);
  const int G = a.grp.G;
  const int64_t K = a.K;
  const int cpr = (int)(K / 8);            // 16-byte chunks per row
  const int ppr = (cpr + 127) / 128;       // passes per row
  const int nscale = (int)(FMT == GMLP_MXFP8 ? K / 32 : K / 16);
  const int lane = threadIdx.x & 31, wib = threadIdx.x / 32;
  const int64_t rows = t.off[G];
  const int64_t warps = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + wib;
  const int64_t P = rows * ppr;
  const int64_t p0 = P * w / warps, p1 = P * (w + 1) / warps;
  if (p0 >= p1) return;
  float* enc = enc_tab[FMT == GMLP_NVFP4 ? wib : 0];
  // the share's passes in order, or (a.reverse) last pass first: after an
  // amax pass on the same grid that kept each share's last rows in L2
  const int d = a.reverse ? -1 : 1;
  const int64_t pf = a.reverse ? p1 - 1 : p0;
  int r = (int)(pf / ppr), j = (int)(pf - (int64_t)r * ppr);  // first row and pass within it
  int64_t left = p1 - p0;                                     // passes still to do
  int g = find_group(t, G, r);
  int g_tab = -1;
  float S = 0.0f;
  for (; left > 0; r += d, j = a.reverse ? ppr - 1 : 0) {
    int n = (int)min(left, (int64_t)(a.reverse ? j + 1 : ppr - j));
    left -= n;
    while (t.off[g + 1] <= r) ++g;
    while (t.off[g] > r) --g;
    int64_t src = r;
    if (a.swiglu_interleave) {
      const int pr = r - t.off[g];
      const int half = (t.off[g + 1] - t.off[g]) >> 1;
      const int c = pr >> 6, i = pr & 63;
      src = t.off[g] + (i < 32 ? 32 * c + i : half + 32 * c + (i - 32));
    }
    if (FMT == GMLP_NVFP4 && g != g_tab) {
      S = nvfp4_global_scale(a.amax[g]);
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) enc[lane + 32 * i] = nvfp4_enc(S, (uint32_t)(lane + 32 * i));
      __syncwarp();
      g_tab = g;
    }
    // scale-word address of the row: tiled (128-row tile, 512-byte blocks of
    // 4 scales x 128 rows) or compact [rows][nscale]
    uint8_t* srow;
    if (TILED) {
      const int lr = r - t.off[g];
      const int rr = lr & 127;
      srow = a.scales + (int64_t)(t.tb[g] + (lr >> 7)) * (nscale >> 2) * 512 + (rr & 31) * 16 + (rr >> 5) * 4;
    } else {
      srow = a.scales + (int64_t)r * nscale;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + src * K);
    uint8_t* crow = a.codes + (int64_t)r * (FMT == GMLP_MXFP8 ? K : K / 2);
    for (; n > 0; --n, j += d) {
      const int c0 = j * 128;
      if (c0 + 128 <= cpr)
        row_pass<FMT, TILED, true>(xr, crow, srow, c0, cpr, lane, S, enc);
      else
        row_pass<FMT, TILED, false>(xr, crow, srow, c0, cpr, lane, S, enc);
    }
  }
}

// ------------------------------------------------------------------ group amax

// Per-group max |x|.  Work units are 256 16-byte chunks of one row (eight per
// lane, all loads issued before the max), so the warps' shares stay even when
// there are only a few rows per warp; warp w takes a contiguous range of units.
// (5 blocks per SM: it runs on the NVFP4 row cast's grid)
__global__ void __launch_bounds__(kThreads, 5) group_amax_kernel(const uint16_t* x, int64_t K, GroupSrc grp,
                                                                 float* amax, float keep) {
  __shared__ SmemGroups t;
  build_group_tables(grp, 1, t);
  griddep_wait();
  griddep_launch_dependents();
  if (t.bad) return;
  const int G = grp.G;
  const int nch = (int)(K / 8);
  constexpr int U = 8;
  const int upr = (nch + 32 * U - 1) / (32 * U);  // units per row
  const int lane = threadIdx.x & 31;
  const int64_t rows = t.off[G];
  const int64_t warps = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int64_t units = rows * upr;
  const int64_t u0 = units * w / warps, u1 = units * (w + 1) / warps;
  if (u0 >= u1) return;
  int64_t r = u0 / upr;
  int part = (int)(u0 - r * upr);
  int g = find_group(t, G, r);
  // the share's last `keep` fraction is read with an L2 evict-last policy, so
  // a row cast on the same grid sweeping its share backwards finds it in L2
  const int64_t u_keep = u1 - (int64_t)(keep * (float)(u1 - u0));
  const uint64_t pol_keep = policy_evict_last(), pol_rest = policy_evict_normal();
  uint32_t m = 0;  // running max |x| as bf16 bits (non-negative, so integer order is value order)
  for (int64_t u = u0; u < u1; ++u) {
    if (t.off[g + 1] <= r) {
      const float mf = warp_max(__uint_as_float(m << 16));
      if (lane == 0) atomic_max_nonneg(amax + g, mf);
      m = 0;
      while (t.off[g + 1] <= r) ++g;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * K);
    const int c0 = part * 32 * U;
    const uint64_t pol = u >= u_keep ? pol_keep : pol_rest;
    uint4 v[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int c = c0 + 32 * k + lane;
      v[k] = c < nch ? ld_stream_hint(xr + c, pol) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < U; ++k) m = max(m, amax8_bits(v[k]));
    if (++part == upr) {
      part = 0;
      ++r;
    }
  }
  const float mf = warp_max(__uint_as_float(m << 16));
  if (lane == 0) atomic_max_nonneg(amax + g, mf);
}

// ------------------------------------------------------------------ Hadamard helpers

// Work units: (group, 256-column slab, 16-row chunk), chunk fastest.  Each
// warp loads its unit's 16 rows x 8 columns per lane (rows past the group end
// are zero).
struct Unit {
  int g, j, nvalid;
  int64_t row0;
  int64_t col0;
  bool active;
};

__device__ __forceinline__ Unit decode_unit(const SmemGroups& t, int g, int64_t u, int64_t K, int lane) {
  Unit r;
  r.g = g;
  const int m = t.off[g + 1] - t.off[g];
  const int nchunks = (m + 15) >> 4;
  const int64_t local = u - t.up[g];
  const int slab = (int)(local / nchunks);
  r.j = (int)(local % nchunks);
  r.nvalid = min(16, m - 16 * r.j);
  r.row0 = t.off[g] + 16LL * r.j;
  r.col0 = (int64_t)slab * 256 + lane * 8;
  r.active = r.col0 < K;
  return r;
}

__device__ __forceinline__ void load_unit(const uint16_t* x, int64_t K, const Unit& un, uint4* v) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    v[i] = (un.active && i < un.nvalid) ? ld_stream(x + (un.row0 + i) * K + un.col0) : make_uint4(0, 0, 0, 0);
}

// ------------------------------------------------------------------ group Hadamard-amax

// The 16-point FWHT (stages h = 1, 2, 4, 8 mapping (w[i], w[i+h]), (i & h) ==
// 0, to (w[i] + w[i+h], w[i] - w[i+h])) on two columns at once in packed FP32
// pairs: the first three stages, then the last.
__device__ __forceinline__ void fwht16x2_first3(f32x2* w) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (!(i & h)) {
        const f32x2 p = w[i], q = w[i + h];
        w[i] = add2(p, q);
        w[i + h] = sub2(p, q);
      }
}

__device__ __forceinline__ void fwht16x2_last(f32x2* w) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const f32x2 p = w[i], q = w[i + 8];
    w[i] = add2(p, q);
    w[i + 8] = sub2(p, q);
  }
}

// a * b + c on 32-bit integers (modulo 2^32).
__device__ __forceinline__ uint32_t umad(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("mad.lo.u32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// The sign mask as FP32 sign bits per row (0x80000000 for a negated row).
struct RowSigns {
  uint32_t s[16];
};

// amax_pre: max |x| on the raw bf16 words (packed max of magnitudes); amax_post:
// per lane, two columns at a time in packed FP32 pairs, the sign folded into
// the widening, the first three FWHT stages, and max |y| over the last stage's
// outputs (p + q, p - q) taken as fp32(|p| + |q|), which equals it; x 1/4 at
// the end.
__global__ void __launch_bounds__(kThreads, 2) hadamard_amax_kernel(const uint16_t* x, int64_t K, GroupSrc grp,
                                                                 const RowSigns sg, float* amax_pre,
                                                                 float* amax_post) {
  __shared__ SmemGroups t;
  const int slabs = (int)((K + 255) / 256);
  build_group_tables(grp, slabs, t);
  griddep_wait();
  griddep_launch_dependents();
  if (t.bad) return;
  const int G = grp.G;
  const int lane = threadIdx.x & 31;
  const int64_t units = t.up[G];
  const int64_t warps = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int64_t upw = (units + warps - 1) / warps;
  const int64_t u0 = w * upw, u1 = min(units, u0 + upw);
  if (u0 >= u1) return;
  int g = find_unit_group(t, G, u0);
  uint32_t pre_bits = 0;  // packed bf16 magnitudes
  float post = 0.0f;
  for (int64_t u = u0; u < u1; ++u) {
    if (t.up[g + 1] <= u) {
      float pre = bf16_bits_to_float(amax_pair_bits(pre_bits));
      pre = warp_max(pre);
      post = warp_max(post);
      if (lane == 0) {
        atomic_max_nonneg(amax_pre + g, pre);
        atomic_max_nonneg(amax_post + g, post * 0.25f);
      }
      pre_bits = 0;
      post = 0.0f;
      while (t.up[g + 1] <= u) ++g;
    }
    const Unit un = decode_unit(t, g, u, K, lane);
    uint4 v[16];
    load_unit(x, K, un, v);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {  // columns 2cc, 2cc + 1 of the lane's eight
      f32x2 y[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t wd = cc == 0 ? v[i].x : cc == 1 ? v[i].y : cc == 2 ? v[i].z : v[i].w;
        pre_bits = bmax_abs2(pre_bits, wd);
        y[i] = pk2(__uint_as_float(umad(wd, 65536u, sg.s[i])), __uint_as_float((wd & 0xFFFF0000u) ^ sg.s[i]));
      }
      fwht16x2_first3(y);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        post = fmaxf(post, fabsf(lo2(y[i])) + fabsf(lo2(y[i + 8])));
        post = fmaxf(post, fabsf(hi2(y[i])) + fabsf(hi2(y[i + 8])));
      }
    }
  }
  float pre = bf16_bits_to_float(amax_pair_bits(pre_bits));
  pre = warp_max(pre);
  post = warp_max(post);
  if (lane == 0) {
    atomic_max_nonneg(amax_pre + g, pre);
    atomic_max_nonneg(amax_post + g, post * 0.25f);
  }
}

// ------------------------------------------------------------------ row + column NVFP4 cast

// One warp's post-RHT amax of a group: the lanes' max |y| before the quarter,
// then x 1/4 (exact), max-accumulated into the group's word.
__device__ __forceinline__ void flush_post(float* dst, float& post, int lane) {
  const float m = warp_max(post);
  if (lane == 0) atomic_max_nonneg(dst, m * 0.25f);
  post = 0.0f;
}

// Max |x| over the 16 bf16 values of two vectors, as amax8_bits does for 8.
__device__ __forceinline__ uint32_t amax16_bits(const uint4& v, const uint4& u) {
  uint32_t m = bmax_abs2(bmax_abs2(bmax_abs2(v.x, v.y), bmax_abs2(v.z, v.w)),
                         bmax_abs2(bmax_abs2(u.x, u.y), bmax_abs2(u.z, u.w)));
  m = bmax_abs2(m, __byte_perm(m, 0, 0x1032)) & 0x7fffu;
  return m > 0x7f80u ? 0u : m;
}

// fp32(b / 6) for an FP32 block max b: the product with fp32(1/6) and one
// residual correction equals the IEEE quotient for every b in [2^-125,
// FLT_MAX] (checked exhaustively on the CPU); tiny, infinite or NaN b take the
// IEEE division.
__device__ __forceinline__ bool div6_fast_ok(float b) {
  return b >= __uint_as_float(0x01000000u) && b <= 3.402823466e38f;
}
__device__ __forceinline__ float div6_fast(float b) {
  const float r6 = __uint_as_float(0x3e2aaaabu);  // fp32(1/6)
  const float q1 = __fmul_rn(b, r6);
  return __fmaf_rn(__fmaf_rn(-6.0f, q1, b), r6, q1);
}
__device__ __noinline__ float div6_ieee(float b) { return __fdiv_rn(b, 6.0f); }

// Row + column NVFP4 cast on 64-row x 128-column tiles of one group, fed by
// TMA.  Warp 8 is the producer: it streams the block's tiles (a contiguous
// range, 64-row blocks fastest, so consecutive tiles continue each column's
// columnwise run) into two shared-memory buffers, one mbarrier pair each.
// Warps 0-7 compute, each on its own part of the tile, with no block-wide
// barrier:
//   rowwise (ROW): rows 8w .. 8w+7, four at a time; lane l casts the 16-column
//     block l % 8 of row 8w + l / 8 (+ 4): block max, scale, eight code bytes;
//     four adjacent lanes make one 32-bit scale word;
//   columnwise: columns 16w .. 16w+15 in packed FP32 pairs; lane l takes pair
//     l % 8 in the 16-row chunk l / 8: sign mask and 16-point FWHT (RHT),
//     x 1/4, block scale, codes.  Rows past the group's end count as zero.
//     The warp stages its columns' codes and scales for the tile (4 chunks,
//     32 + 4 bytes per column) and writes each column's run with four adjacent
//     lanes, so global stores go out in 32-byte runs.
// 128-column tiles at two blocks per SM measured faster than 256-column ones
// (more tiles in flight per SM for the same shared memory).
constexpr int kRcRows = 64, kRcCols = 128, kRcWarps = 8, kRcBufs = 2, kRcBlocksPerSM = 2;
constexpr int kRcThreads = (kRcWarps + 1) * 32;
constexpr int kRcTileBytes = kRcRows * kRcCols * 2;
constexpr int kRcColStride = 40;  // staged codes per column: 4 chunks x 8 bytes + 8 bytes of bank padding
constexpr int kRcRowLanes = kRcCols / 16;              // rowwise: lanes per row (one 16-column block each)
constexpr int kRcRowsPerPass = 32 / kRcRowLanes;       // rows a warp casts per pass
constexpr int kRcPairs = kRcCols / 2 / kRcWarps;       // columnwise: column pairs per warp
constexpr int kRcChunkLanes = 32 / kRcPairs;           // lanes sharing a pair, one 16-row chunk each
constexpr int kRcColsPerWarp = 2 * kRcPairs;
static_assert(kRcRowsPerPass * (8 / kRcRowsPerPass) == 8 && kRcChunkLanes <= 4 && 4 % kRcChunkLanes == 0, "tile");

struct RcShared {
  uint16_t tile[kRcBufs][kRcRows * kRcCols];
  uint8_t ccode[kRcWarps][kRcColsPerWarp * kRcColStride];
  uint8_t cscale[kRcWarps][kRcColsPerWarp * 4];
  float enc[kRcWarps][2][128];  // per warp: row and column encode factors of its current group
  uint64_t full[kRcBufs];
  uint64_t empty[kRcBufs];
  int abort_flag;
};

// Walks a contiguous range of tiles in order (group, slab, 64-row block),
// block fastest, without a division per tile.
struct RcWalk {
  int g, slab, blk, nblk, nvalid;

  __device__ __forceinline__ void start(const SmemGroups& t, int G, int64_t u) {
    g = find_unit_group(t, G, u);
    const int m = t.off[g + 1] - t.off[g];
    nblk = (m + kRcRows - 1) / kRcRows;
    const int local = (int)(u - t.up[g]);
    slab = local / nblk;
    blk = local - slab * nblk;
    nvalid = min(kRcRows, m - kRcRows * blk);
  }

  // the next tile (called only while one remains)
  __device__ __forceinline__ void next(const SmemGroups& t, int slabs) {
    if (++blk == nblk) {
      blk = 0;
      if (++slab == slabs) {
        slab = 0;
        do ++g; while (t.off[g + 1] == t.off[g]);  // skip empty groups
        nblk = (t.off[g + 1] - t.off[g] + kRcRows - 1) / kRcRows;
      }
    }
    nvalid = min(kRcRows, t.off[g + 1] - t.off[g] - kRcRows * blk);
  }
};

// COLQ = false (with ROW, RHT, TILED): no columnwise codes; the column phase
// only takes the post-RHT amax of the 16-row chunks (per warp, then one
// atomicMax per group and warp), the fused amax the columnwise cast of the
// same tensor would use.  With nothing to stage it fits 72 registers and runs
// three blocks per SM (measured 3% faster than two on nv_srelu's fc2_x).
template <bool ROW, bool RHT, bool TILED, bool COLQ>
__global__ void __launch_bounds__(kRcThreads, COLQ ? kRcBlocksPerSM : 3)
    rowcol_quant_kernel(const __grid_constant__ CUtensorMap tmx, const ColQuantArgs a) {
  __shared__ SmemGroups t;
  extern __shared__ uint8_t rc_raw[];
  RcShared& sm = *reinterpret_cast<RcShared*>((reinterpret_cast<uintptr_t>(rc_raw) + 127) & ~uintptr_t(127));
  const int64_t K = a.K;
  const int slabs = (int)((K + kRcCols - 1) / kRcCols);
  if (threadIdx.x == 0) {
    for (int b = 0; b < kRcBufs; ++b) {
      mbar_init(&sm.full[b], 1);
      mbar_init(&sm.empty[b], kRcWarps);
    }
    sm.abort_flag = 0;
    fence_barrier_init();
  }
  build_group_tables(a.grp, slabs, t, kRcRows);  // ends with a block barrier
  griddep_wait();
  griddep_launch_dependents();
  if (t.bad) return;
  const int G = a.grp.G;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t T = t.up[G];
  const int64_t u0 = T * blockIdx.x / gridDim.x, u1 = T * (blockIdx.x + 1) / gridDim.x;
  volatile int* abort_flag = &sm.abort_flag;

  if (warp == kRcWarps) {
    // ---------------- producer
    if (lane == 0 && u0 < u1) {
      prefetch_tmap(&tmx);
      uint32_t armed = 0;
      RcWalk tl;
      tl.start(t, G, u0);
      int64_t it = 0;
      const uint64_t pol = policy_evict_first();
      for (int64_t u = u0; u < u1; ++u, ++it) {
        const int b = (int)(it & 1);
        const uint32_t ph = (uint32_t)(it >> 1) & 1u;
        if (it > 0) tl.next(t, slabs);
        if (it >= kRcBufs && !mbar_wait(&sm.empty[b], ph ^ 1u, abort_flag)) break;
        mbar_arrive_expect_tx(&sm.full[b], kRcTileBytes);
        armed |= 1u << b;
        tma_load_2d(sm.tile[b], &tmx, tl.slab * kRcCols, t.off[tl.g] + kRcRows * tl.blk, &sm.full[b], pol);
      }
      // the last loads of each buffer land before the block exits
      for (int b = 0; b < kRcBufs; ++b) {
        if (!(armed & (1u << b))) continue;
        const int64_t last = it - 1 - ((it - 1 - b) & 1);  // last load index into buffer b
        mbar_wait_drain(&sm.full[b], (uint32_t)(last >> 1) & 1u);
      }
    }
    return;
  }

  // ---------------- compute warps
  float* enc_row = sm.enc[warp][0];
  float* enc_col = sm.enc[warp][1];
  uint8_t* cstage = sm.ccode[warp];
  uint8_t* sstage = sm.cscale[warp];
  const int nscale_row = (int)(K / 16);
  int g_tab = -1;
  float S_row = 0.0f, S_col = 0.0f;
  float post_acc = 0.0f;  // !COLQ: this lane's max |y| (before the quarter) in the current group
  uint32_t sg[16];  // the sign mask as FP32 sign bits per row, kept in registers
#pragma unroll
  for (int i = 0; i < 16; ++i) sg[i] = RHT ? a.sgn[i] : 0u;
  RcWalk tl;
  if (u0 < u1) tl.start(t, G, u0);
  int64_t it = 0;
  for (int64_t u = u0; u < u1; ++u, ++it) {
    const int b = (int)(it & 1);
    const uint32_t ph = (uint32_t)(it >> 1) & 1u;
    if (it > 0) tl.next(t, slabs);
    if (tl.g != g_tab) {
      if (!COLQ && g_tab >= 0) flush_post(a.amax_post_out + g_tab, post_acc, lane);
      S_row = ROW ? nvfp4_global_scale(a.amax_row[tl.g]) : 0.0f;
      S_col = COLQ ? nvfp4_global_scale(a.amax_col[tl.g]) : 0.0f;
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (ROW) enc_row[lane + 32 * i] = nvfp4_enc(S_row, (uint32_t)(lane + 32 * i));
        if (COLQ) enc_col[lane + 32 * i] = nvfp4_enc(S_col, (uint32_t)(lane + 32 * i));
      }
      __syncwarp();
      g_tab = tl.g;
    }
    const int64_t row0 = (int64_t)t.off[tl.g] + kRcRows * tl.blk;
    const int64_t col0 = (int64_t)tl.slab * kRcCols;
    const int nch = (tl.nvalid + 15) >> 4;
    if (!mbar_wait(&sm.full[b], ph, abort_flag)) break;
    const uint16_t* tile = sm.tile[b];

    if (ROW) {
      // lane l: block l % kRcRowLanes (16 columns) of rows 8w + kRcRowsPerPass k + l / kRcRowLanes
      const int bl = lane % kRcRowLanes;
      const int64_t gcol = col0 + 16 * bl;
      const bool active = gcol < K;
      const int kblk = (int)(gcol >> 4);
      const int r0 = 8 * warp + lane / kRcRowLanes;  // this lane's first row, then every kRcRowsPerPass
      uint8_t* cptr = a.row_codes + (row0 + r0) * (K / 2) + (gcol >> 1);
      // the scale word of row r: a 64-row tile is one half (64 (blk & 1) ..) of a
      // 128-row scale tile, so the tile is fixed and row r sits at (r % 32) * 16 + (r / 32) * 4
      uint8_t* sptr;
      if (TILED)
        sptr = a.row_scales + ((int64_t)(t.tb[tl.g] + (tl.blk >> 1)) * (nscale_row >> 2) + (kblk >> 2)) * 512 +
               (tl.blk & 1) * 8;
      else
        sptr = a.row_scales + row0 * nscale_row + kblk;
#pragma unroll
      for (int k = 0; k < 8 / kRcRowsPerPass; ++k) {
        const int r = r0 + kRcRowsPerPass * k;
        if (8 * warp + kRcRowsPerPass * k >= tl.nvalid) break;
        const uint4 v0 = *reinterpret_cast<const uint4*>(tile + r * kRcCols + 16 * bl);
        const uint4 v1 = *reinterpret_cast<const uint4*>(tile + r * kRcCols + 16 * bl + 8);
        const uint32_t sf = nvfp4_block_sf_bf16(amax16_bits(v0, v1), S_row);
        const float enc = enc_row[sf];
        float q0[8], q1[8];
        scale8(v0, enc, q0);
        scale8(v1, enc, q1);
        const uint32_t sw = gather4_bytes(sf, 1);
        if (active && r < tl.nvalid) {
          *reinterpret_cast<uint2*>(cptr + kRcRowsPerPass * k * (K / 2)) = make_uint2(e2m1_pack8(q0), e2m1_pack8(q1));
          if ((lane & 3) == 0)
            *reinterpret_cast<uint32_t*>(sptr + (TILED ? (r & 31) * 16 + (r >> 5) * 4 : (int64_t)r * nscale_row)) = sw;
        }
      }
    }

    // columnwise: pair p of this warp's kRcPairs column pairs, 16-row chunks
    // lane / kRcPairs + kRcChunkLanes q2
    const uint32_t* tile32 = reinterpret_cast<const uint32_t*>(tile);
    const int p = lane % kRcPairs, pr = kRcPairs * warp + p;
#pragma unroll 1
    for (int q2 = 0; q2 < 4 / kRcChunkLanes; ++q2) {
      // every lane runs the item (the warp votes below); a lane whose chunk is
      // past the tile's rows works on zeros and stores nothing
      const int c = lane / kRcPairs + kRcChunkLanes * q2;
      if (kRcChunkLanes * q2 >= nch) break;  // no lane of the warp has a chunk left
      const bool live = c < nch;
      f32x2 y[16];
      uint32_t wv[16];
      const uint32_t* src = tile32 + 16 * c * (kRcCols / 2) + pr;
      if (16 * c + 16 <= tl.nvalid) {
#pragma unroll
        for (int i = 0; i < 16; ++i) wv[i] = src[i * (kRcCols / 2)];
      } else {  // the group's last chunk: rows past its end count as zero
#pragma unroll
        for (int i = 0; i < 16; ++i) wv[i] = 16 * c + i < tl.nvalid ? src[i * (kRcCols / 2)] : 0u;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        // the two bf16 values widened to FP32 with row i's sign from the mask:
        // lo = wd * 2^16 + s (adding 2^31 flips the top bit), hi = (wd & 0xFFFF0000) ^ s
        y[i] = pk2(__uint_as_float(umad(wv[i], 65536u, sg[i])), __uint_as_float((wv[i] & 0xFFFF0000u) ^ sg[i]));
      }
      float b0 = 0.0f, b1 = 0.0f, b0r = 0.0f, b1r = 0.0f;  // b*r: max |y| before the quarter
      if (RHT) {
        fwht16x2_first3(y);
        // max |y| over the last stage's outputs (p + q, p - q) is fp32(|p| + |q|)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          b0 = fmaxf(b0, fabsf(lo2(y[i])) + fabsf(lo2(y[i + 8])));
          b1 = fmaxf(b1, fabsf(hi2(y[i])) + fabsf(hi2(y[i + 8])));
        }
        if (!COLQ) {  // the post-RHT amax only
          post_acc = fmaxf(post_acc, fmaxf(b0, b1));
          continue;
        }
        fwht16x2_last(y);
        b0r = b0;
        b1r = b1;
        b0 = __fmul_rn(b0, 0.25f);  // = max |fp32(y / 4)|: scaling by 1/4 rounds monotonically
        b1 = __fmul_rn(b1, 0.25f);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          b0 = fmaxf(b0, fabsf(lo2(y[i])));
          b1 = fmaxf(b1, fabsf(hi2(y[i])));
        }
      }
      float d0, d1;
      if (__all_sync(0xffffffffu, !live || (div6_fast_ok(b0) && div6_fast_ok(b1)))) {  // the usual case
        d0 = div6_fast(b0);
        d1 = div6_fast(b1);
      } else {
        d0 = div6_fast_ok(b0) ? div6_fast(b0) : div6_ieee(b0);
        d1 = div6_fast_ok(b1) ? div6_fast(b1) : div6_ieee(b1);
      }
      const uint32_t sf0 = e4m3x2(__fmul_rn(d0, S_col), 0.0f) & 0xFF;
      const uint32_t sf1 = e4m3x2(__fmul_rn(d1, S_col), 0.0f) & 0xFF;
      const float e0 = enc_col[sf0], e1 = enc_col[sf1];
      f32x2 enc = pk2(e0, e1);
      if (RHT) {
        // fp32(fp32(y / 4) * enc) == fp32(y * (enc / 4)) whenever y / 4 and enc / 4
        // are exact (no subnormal); elements below 2^-124 in a block whose max
        // is at least 2^-100 quantise to a zero of their sign either way.  So
        // the quarter folds into the encode factor unless a block is that
        // small or enc is below 2^-124.
        const float kTiny = __uint_as_float(0x0d800000u), kEnc = __uint_as_float(0x01800000u);  // 2^-100, 2^-124
        if (__all_sync(0xffffffffu, !live || (b0r >= kTiny && b1r >= kTiny && e0 >= kEnc && e1 >= kEnc))) {
          enc = pk2(__fmul_rn(e0, 0.25f), __fmul_rn(e1, 0.25f));
        } else {  // some lane of the warp has a block below the fold's range: all take the plain path
          const f32x2 quarter = pk2(0.25f, 0.25f);
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = mul2(y[i], quarter);
        }
      }
      float p0[16], p1[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const f32x2 qv = mul2(y[i], enc);
        p0[i] = lo2(qv);
        p1[i] = hi2(qv);
      }
      if (live) {
        *reinterpret_cast<uint2*>(cstage + (2 * p) * kRcColStride + 8 * c) =
            make_uint2(e2m1_pack8(p0), e2m1_pack8(p0 + 8));
        *reinterpret_cast<uint2*>(cstage + (2 * p + 1) * kRcColStride + 8 * c) =
            make_uint2(e2m1_pack8(p1), e2m1_pack8(p1 + 8));
        sstage[(2 * p) * 4 + c] = (uint8_t)sf0;
        sstage[(2 * p + 1) * 4 + c] = (uint8_t)sf1;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[b]);  // this warp is done reading the tile
    if (!COLQ) continue;

    // the warp's columns: each column's chunks of this tile as one run, four lanes per column
    const int64_t mpad = (int64_t)(t.mp[tl.g + 1] - t.mp[tl.g]);
    const int c = lane & 3;
    const int64_t gc0 = col0 + kRcColsPerWarp * warp + (lane >> 2);  // this lane's column in step i: gc0 + 8 i
    uint8_t* cp = a.col_codes + K * (int64_t)t.mp[tl.g] / 2 + gc0 * (mpad / 2) + 8 * (4 * tl.blk + c);
    uint8_t* sp = a.col_scales + K * (int64_t)t.mp[tl.g] / 16 + gc0 * (mpad / 16) + 4 * tl.blk + c;
    if (c < nch) {
#pragma unroll
      for (int i = 0; i < kRcColsPerWarp / 8; ++i) {
        const int cl = 8 * i + (lane >> 2);
        if (gc0 + 8 * i < K) {
          *reinterpret_cast<uint2*>(cp + 8 * i * (mpad / 2)) =
              *reinterpret_cast<const uint2*>(cstage + cl * kRcColStride + 8 * c);
          sp[8 * i * (mpad / 16)] = sstage[cl * 4 + c];
        }
      }
    }
    __syncwarp();  // the staging buffers are free for the next tile
  }
  if (!COLQ && g_tab >= 0) flush_post(a.amax_post_out + g_tab, post_acc, lane);
}

// Persistent grid: as many blocks as fit on the device at once (one wave),
// fewer when there is less work.
template <typename Kern>
int grid_for(Kern kern, int64_t work_warps, size_t smem = 0) {
  static int per_sm_cache[64][32] = {};
  static const void* keys[64][32] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  int per_sm = 0;
  for (int i = 0; i < 32; ++i)
    if (keys[dev & 63][i] == (const void*)kern) per_sm = per_sm_cache[dev & 63][i];
  if (!per_sm) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem) != cudaSuccess || per_sm < 1)
      per_sm = 1;
    for (int i = 0; i < 32; ++i)
      if (!keys[dev & 63][i]) {
        keys[dev & 63][i] = (const void*)kern;
        per_sm_cache[dev & 63][i] = per_sm;
        break;
      }
  }
  const int64_t max_blocks = (int64_t)num_sms() * per_sm;
  int64_t blocks = (work_warps + kWarps - 1) / kWarps;
  if (blocks > max_blocks) blocks = max_blocks;
  return (int)(blocks < 1 ? 1 : blocks);
}

// ------------------------------------------------------------------ fc2_x rebuild

// fc2_x = bf16(act(h) * prob) from the saved activation input h [M][N1]
// (SwiGLU: N1 = 2N, gate columns then up columns; otherwise N1 = N), with the
// fc1 epilogue's own arithmetic (fc2x_* of device.cuh).  One thread makes 16
// outputs of a row per step (32-byte loads and stores), grid-stride.
template <int ACT>
__global__ void __launch_bounds__(kThreads) fc2x_recompute_kernel(const uint16_t* h, const float* probs, int64_t M,
                                                                  int64_t N, float c, uint16_t* out) {
  const int64_t per_row = N / 16, N1 = ACT == GMLP_ACT_SWIGLU ? 2 * N : N;
  const int64_t total = M * per_row;
  const float inv_c = ACT == GMLP_ACT_TANH_SRELU ? __frcp_rn(c) : 0.0f;
  int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const int64_t st_t = stride / per_row, st_c = stride - st_t * per_row;
  int64_t t = i / per_row, ch = i - t * per_row;
  for (; i < total; i += stride) {
    const float p = probs ? __ldg(probs + t) : 1.0f;
    const uint16_t* row = h + t * N1 + ch * 16;
    uint32_t gw[8], uw[8], ow[8];
    ld_global_nc_v8(row, gw);
    if (ACT == GMLP_ACT_SWIGLU) ld_global_nc_v8(row + N, uw);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float g0 = bf16_bits_to_float(gw[k] & 0xFFFFu), g1 = bf16_bits_to_float(gw[k] >> 16);
      float f0, f1;
      if (ACT == GMLP_ACT_SWIGLU) {
        f0 = fc2x_swiglu(g0, bf16_bits_to_float(uw[k] & 0xFFFFu), p);
        f1 = fc2x_swiglu(g1, bf16_bits_to_float(uw[k] >> 16), p);
      } else if (ACT == GMLP_ACT_TANH_SRELU) {
        f0 = fc2x_tanh_srelu(g0, p, c, inv_c);
        f1 = fc2x_tanh_srelu(g1, p, c, inv_c);
      } else {
        f0 = fc2x_srelu(g0, p);
        f1 = fc2x_srelu(g1, p);
      }
      ow[k] = bf16_bits(f0) | (bf16_bits(f1) << 16);
    }
    st_global_v8(out + t * N + ch * 16, ow);
    t += st_t;
    ch += st_c;
    if (ch >= per_row) {
      ch -= per_row;
      ++t;
    }
  }
}

// One warp waits, through the kernels' bounded wait, on an mbarrier that
// nothing arrives at; the wait gives up after limit_ns and reports
// GMLP_ERR_DEVICE_TIMEOUT in the status word.
__global__ void selftest_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, limit_ns);
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(&bar);  // complete the phase before the barrier goes away
}

}  // namespace

// GEMM_TILED -> GEMM_TILED_X4 for NVFP4 weight scales: for 128-row tile pair
// P, stage kb (4 runs) and run k of the stage, the 4096 bytes at
// ((P * KB + kb) * 4 + k) * 4096 hold tile 2P's block (kb, k) four times, then
// tile 2P+1's block four times.  One 16-byte word per thread step.
__global__ void replicate_scales_kernel(const uint8_t* in, int64_t pairs, int64_t runs, uint8_t* out) {
  const int64_t KB = runs / 4;
  const int64_t n16 = pairs * KB * 4 * 4096 / 16;
  for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < n16; o += (int64_t)gridDim.x * blockDim.x) {
    const int64_t ob = o * 16;
    const int64_t blk = ob >> 12;
    const int within = (int)(ob & 4095);
    const int h = within >> 11, i = within & 511;
    const int64_t pk = blk >> 2, k = blk & 3;
    const int64_t kb = pk % KB, P = pk / KB;
    const int64_t src = ((2 * P + h) * runs + 4 * kb + k) * 512 + i;
    reinterpret_cast<uint4*>(out)[o] = *reinterpret_cast<const uint4*>(in + src);
  }
}

cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(limit_ns);
  return cudaGetLastError();
}

int quant_read_clear_status() { return read_clear_status(); }

cudaError_t launch_replicate_scales(const uint8_t* tiled, int64_t pairs, int64_t runs, uint8_t* out, cudaStream_t s) {
  const int64_t n16 = pairs * (runs / 4) * 4 * 4096 / 16;
  if (n16 == 0) return cudaSuccess;
  int64_t grid = (n16 + 255) / 256;
  if (grid > (int64_t)num_sms() * 8) grid = (int64_t)num_sms() * 8;
  replicate_scales_kernel<<<(unsigned)grid, 256, 0, s>>>(tiled, pairs, runs, out);
  return cudaGetLastError();
}

// Launch with programmatic stream serialization when `pdl` is set.
template <typename... Args>
cudaError_t launch_ex(void (*kern)(Args...), int grid, size_t smem, cudaStream_t s, bool pdl, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int FMT, bool TILED>
cudaError_t launch_row_quant_t(const RowQuantArgs& a, cudaStream_t s) {
  auto kern = row_quant_kernel<FMT, TILED>;
  return launch_ex(kern, grid_for(kern, a.M), 0, s, a.pdl != 0, a);
}

cudaError_t launch_row_quant(const RowQuantArgs& a, cudaStream_t s) {
  if (a.format == GMLP_MXFP8)
    return a.tiled ? launch_row_quant_t<GMLP_MXFP8, true>(a, s) : launch_row_quant_t<GMLP_MXFP8, false>(a, s);
  return a.tiled ? launch_row_quant_t<GMLP_NVFP4, true>(a, s) : launch_row_quant_t<GMLP_NVFP4, false>(a, s);
}

int row_quant_grid(int format, int tiled, int64_t M) {
  if (format == GMLP_MXFP8)
    return tiled ? grid_for(row_quant_kernel<GMLP_MXFP8, true>, M) : grid_for(row_quant_kernel<GMLP_MXFP8, false>, M);
  return tiled ? grid_for(row_quant_kernel<GMLP_NVFP4, true>, M) : grid_for(row_quant_kernel<GMLP_NVFP4, false>, M);
}

cudaError_t launch_group_amax(const uint16_t* x, int64_t M, int64_t K, GroupSrc grp, float* amax, cudaStream_t s,
                              int grid, float keep) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * grp.G, s);
  if (e != cudaSuccess) return e;
  if (grid <= 0) grid = grid_for(group_amax_kernel, M);
  group_amax_kernel<<<grid, kThreads, 0, s>>>(x, K, grp, amax, keep);
  return cudaGetLastError();
}

cudaError_t launch_hadamard_amax(const uint16_t* x, int64_t M, int64_t K, GroupSrc grp, uint32_t mask,
                                 float* amax_pre, float* amax_post, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax_pre, 0, sizeof(float) * grp.G, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(amax_post, 0, sizeof(float) * grp.G, s);
  if (e != cudaSuccess) return e;
  const int64_t units = ((M + 15) / 16 + grp.G) * ((K + 255) / 256);
  RowSigns sg;
  for (int i = 0; i < 16; ++i) sg.s[i] = ((mask >> i) & 1u) ? 0x80000000u : 0u;
  hadamard_amax_kernel<<<grid_for(hadamard_amax_kernel, units), kThreads, 0, s>>>(x, K, grp, sg, amax_pre, amax_post);
  return cudaGetLastError();
}

cudaError_t launch_fc2x_recompute(const uint16_t* h, const float* probs, int64_t M, int64_t N, int act, float c,
                                  uint16_t* out, cudaStream_t s) {
  if (M == 0) return cudaSuccess;
  const int64_t work = M * (N / 16);
  if (act == GMLP_ACT_SWIGLU) {
    fc2x_recompute_kernel<GMLP_ACT_SWIGLU>
        <<<grid_for(fc2x_recompute_kernel<GMLP_ACT_SWIGLU>, work / 32), kThreads, 0, s>>>(h, probs, M, N, c, out);
  } else if (act == GMLP_ACT_TANH_SRELU) {
    fc2x_recompute_kernel<GMLP_ACT_TANH_SRELU>
        <<<grid_for(fc2x_recompute_kernel<GMLP_ACT_TANH_SRELU>, work / 32), kThreads, 0, s>>>(h, probs, M, N, c, out);
  } else {
    fc2x_recompute_kernel<GMLP_ACT_SRELU>
        <<<grid_for(fc2x_recompute_kernel<GMLP_ACT_SRELU>, work / 32), kThreads, 0, s>>>(h, probs, M, N, c, out);
  }
  return cudaGetLastError();
}

template <bool ROW, bool RHT, bool TILED, bool COLQ = true>
cudaError_t launch_rowcol_t(const ColQuantArgs& a, cudaStream_t s) {
  auto kern = rowcol_quant_kernel<ROW, RHT, TILED, COLQ>;
  constexpr size_t smem = sizeof(RcShared) + 128;
  static bool attr[64] = {};
  static int per_sm[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kRcThreads, smem);
    if (e != cudaSuccess) return e;
    per_sm[dev & 63] = n < 1 ? 1 : n;
    attr[dev & 63] = true;
  }
  CUtensorMap tmx;
  if (!make_tmap_u16(&tmx, a.x, a.K, a.M, kRcCols, kRcRows)) return cudaErrorInvalidValue;
  const int64_t tiles = ((a.M + kRcRows - 1) / kRcRows + a.grp.G) * ((a.K + kRcCols - 1) / kRcCols);
  int64_t grid = (int64_t)num_sms() * per_sm[dev & 63];
  if (grid > tiles) grid = tiles;
  if (grid < 1) grid = 1;
  kern<<<(unsigned)grid, kRcThreads, smem, s>>>(tmx, a);
  return cudaGetLastError();
}

cudaError_t launch_col_quant(const ColQuantArgs& a0, cudaStream_t s) {
  if (a0.M == 0) return cudaSuccess;
  ColQuantArgs a = a0;
  for (int i = 0; i < 16; ++i) a.sgn[i] = ((a.mask >> i) & 1u) ? 0x80000000u : 0u;
  const bool row = a.row_codes != nullptr;
  if (!a.col_codes) {  // rowwise (GEMM_TILED) + the post-RHT amax only
    if (!row || !a.row_tiled || !a.amax_post_out) return cudaErrorInvalidValue;
    return launch_rowcol_t<true, true, true, false>(a, s);
  }
  if (a.use_rht) {
    if (!row) return launch_rowcol_t<false, true, false>(a, s);
    return a.row_tiled ? launch_rowcol_t<true, true, true>(a, s) : launch_rowcol_t<true, true, false>(a, s);
  }
  if (!row) return launch_rowcol_t<false, false, false>(a, s);
  return a.row_tiled ? launch_rowcol_t<true, false, true>(a, s) : launch_rowcol_t<true, false, false>(a, s);
}

}  // namespace gmlp
