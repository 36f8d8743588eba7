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
  int up[kMaxGroups + 1];   // first work unit (16-row chunk x 256-column slab)
  int mp[kMaxGroups + 1];   // prefix of the 16-row padded group sizes
  int bad;
};

// Warp 0 scans the G split sizes (32 at a time); everything is validated
// against M.  Negative sizes or a total above M set GMLP_ERR_DEVICE_BOUNDS and
// t.bad, and the kernel does nothing.
__device__ void build_group_tables(const GroupSrc& gs, int slabs, SmemGroups& t) {
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
      long long v0 = m, v1 = (m + 127) >> 7, v2 = ch * slabs, v3 = ch * 16;
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

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = bf16_bits_to_float(w[i] & 0xFFFF);
    f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, d));
  return v;
}

__device__ __forceinline__ void atomic_max_nonneg(float* p, float v) {
  atomicMax(reinterpret_cast<int*>(p), __float_as_int(v));
}

// Byte offset of the scale (row r of group g, scale column kidx).
__device__ __forceinline__ int64_t scale_offset(bool tiled, const SmemGroups& t, int g, int64_t r, int kidx,
                                                int nscale) {
  if (!tiled) return r * nscale + kidx;
  const int lr = (int)(r - t.off[g]);
  const int rr = lr & 127;
  const int64_t blk = (int64_t)(t.tb[g] + (lr >> 7)) * (nscale >> 2) + (kidx >> 2);
  return blk * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (kidx & 3);
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

// One warp per row (contiguous row ranges per warp); lane l takes 16-byte
// chunks l, l+32, ... of the row.  MXFP8: 4 lanes per 32-element block;
// NVFP4: 2 lanes per 16-element block.
template <int FMT>
__global__ void __launch_bounds__(kThreads) row_quant_kernel(RowQuantArgs a) {
  __shared__ SmemGroups t;
  build_group_tables(a.grp, 1, t);
  if (t.bad) return;
  const int G = a.grp.G;
  if (blockIdx.x == 0) {
    if (a.zero_ptr)
      for (int i = threadIdx.x; i < a.zero_count; i += kThreads) a.zero_ptr[i] = 0.0f;
    if (a.S_out)
      for (int g = threadIdx.x; g < G; g += kThreads) a.S_out[g] = nvfp4_global_scale(a.amax[g]);
  }
  const int64_t K = a.K;
  const int nch = (int)(K / 8);
  const int nscale = (int)(FMT == GMLP_MXFP8 ? K / 32 : K / 16);
  const int lane = threadIdx.x & 31;
  const int64_t rows = t.off[G];
  const int64_t warps = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int64_t rpw = (rows + warps - 1) / warps;
  const int64_t r0 = w * rpw, r1 = min(rows, r0 + rpw);
  if (r0 >= r1) return;
  int g = find_group(t, G, r0);
  constexpr int U = 4;
  for (int64_t r = r0; r < r1; ++r) {
    while (t.off[g + 1] <= r) ++g;
    int64_t src = r;
    if (a.swiglu_interleave) {
      const int p = (int)(r - t.off[g]);
      const int half = (t.off[g + 1] - t.off[g]) >> 1;
      const int c = p >> 6, i = p & 63;
      src = t.off[g] + (i < 32 ? 32 * c + i : half + 32 * c + (i - 32));
    }
    const uint4* xr = reinterpret_cast<const uint4*>(a.x + src * K);
    float S = 0.0f;
    if (FMT == GMLP_NVFP4) S = nvfp4_global_scale(a.amax[g]);
    for (int c0 = 0; c0 < nch; c0 += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u + lane;
        v[u] = c < nch ? ld_stream(xr + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u + lane;
        float f[8];
        unpack8(v[u], f);
        float am = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
        if (FMT == GMLP_MXFP8) {
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
          const int e = mxfp8_exponent(am);
          const float mul = exp2_neg(e);
          uint32_t w0 = e4m3x2(__fmul_rn(f[0], mul), __fmul_rn(f[1], mul)) |
                        (e4m3x2(__fmul_rn(f[2], mul), __fmul_rn(f[3], mul)) << 16);
          uint32_t w1 = e4m3x2(__fmul_rn(f[4], mul), __fmul_rn(f[5], mul)) |
                        (e4m3x2(__fmul_rn(f[6], mul), __fmul_rn(f[7], mul)) << 16);
          if (c < nch) {
            *reinterpret_cast<uint2*>(a.codes + r * K + (int64_t)c * 8) = make_uint2(w0, w1);
            if ((lane & 3) == 0)
              a.scales[scale_offset(a.tiled, t, g, r, c >> 2, nscale)] = (uint8_t)(e + 127);
          }
        } else {
          am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
          uint32_t sf;
          const float enc = nvfp4_block_encode(am, S, &sf);
          uint32_t word = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            word |= e2m1x2(__fmul_rn(f[2 * i], enc), __fmul_rn(f[2 * i + 1], enc)) << (8 * i);
          if (c < nch) {
            *reinterpret_cast<uint32_t*>(a.codes + r * (K / 2) + (int64_t)c * 4) = word;
            if ((lane & 1) == 0) a.scales[scale_offset(a.tiled, t, g, r, c >> 1, nscale)] = (uint8_t)sf;
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ group amax

__global__ void __launch_bounds__(kThreads) group_amax_kernel(const uint16_t* x, int64_t K, GroupSrc grp,
                                                              float* amax) {
  __shared__ SmemGroups t;
  build_group_tables(grp, 1, t);
  if (t.bad) return;
  const int G = grp.G;
  const int nch = (int)(K / 8);
  const int lane = threadIdx.x & 31;
  const int64_t rows = t.off[G];
  const int64_t warps = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int64_t rpw = (rows + warps - 1) / warps;
  const int64_t r0 = w * rpw, r1 = min(rows, r0 + rpw);
  if (r0 >= r1) return;
  int g = find_group(t, G, r0);
  float m = 0.0f;
  constexpr int U = 4;
  for (int64_t r = r0; r < r1; ++r) {
    if (t.off[g + 1] <= r) {
      m = warp_max(m);
      if (lane == 0) atomic_max_nonneg(amax + g, m);
      m = 0.0f;
      while (t.off[g + 1] <= r) ++g;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(x + r * K);
    for (int c0 = 0; c0 < nch; c0 += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u + lane;
        v[u] = c < nch ? ld_stream(xr + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float f[8];
        unpack8(v[u], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
      }
    }
  }
  m = warp_max(m);
  if (lane == 0) atomic_max_nonneg(amax + g, m);
}

// ------------------------------------------------------------------ Hadamard helpers

// 16-point FWHT in registers: stages h = 1, 2, 4, 8 mapping (w[i], w[i+h]),
// (i & h) == 0, to (w[i] + w[i+h], w[i] - w[i+h]).
__device__ __forceinline__ void fwht16(float* w) {
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (!(i & h)) {
        const float p = w[i], q = w[i + h];
        w[i] = p + q;
        w[i + h] = p - q;
      }
}

// Column cc (0..7) of a lane's 16 x 8 bf16 tile as 16 floats.
__device__ __forceinline__ void column16(const uint4* v, int cc, float* w) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t word = (cc >> 1) == 0 ? v[i].x : (cc >> 1) == 1 ? v[i].y : (cc >> 1) == 2 ? v[i].z : v[i].w;
    w[i] = bf16_bits_to_float((cc & 1) ? (word >> 16) : (word & 0xFFFF));
  }
}

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

__global__ void __launch_bounds__(kThreads) hadamard_amax_kernel(const uint16_t* x, int64_t K, GroupSrc grp,
                                                                 uint32_t mask, float* amax_pre,
                                                                 float* amax_post) {
  __shared__ SmemGroups t;
  const int slabs = (int)((K + 255) / 256);
  build_group_tables(grp, slabs, t);
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
  float pre = 0.0f, post = 0.0f;
  for (int64_t u = u0; u < u1; ++u) {
    if (t.up[g + 1] <= u) {
      pre = warp_max(pre);
      post = warp_max(post);
      if (lane == 0) {
        atomic_max_nonneg(amax_pre + g, pre);
        atomic_max_nonneg(amax_post + g, post * 0.25f);
      }
      pre = post = 0.0f;
      while (t.up[g + 1] <= u) ++g;
    }
    const Unit un = decode_unit(t, g, u, K, lane);
    uint4 v[16];
    load_unit(x, K, un, v);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      float wv[16];
      column16(v, cc, wv);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        pre = fmaxf(pre, fabsf(wv[i]));
        if ((mask >> i) & 1u) wv[i] = -wv[i];
      }
      fwht16(wv);
#pragma unroll
      for (int i = 0; i < 16; ++i) post = fmaxf(post, fabsf(wv[i]));
    }
  }
  pre = warp_max(pre);
  post = warp_max(post);
  if (lane == 0) {
    atomic_max_nonneg(amax_pre + g, pre);
    atomic_max_nonneg(amax_post + g, post * 0.25f);
  }
}

// ------------------------------------------------------------------ row + column NVFP4 cast

__global__ void __launch_bounds__(kThreads) col_quant_kernel(ColQuantArgs a) {
  __shared__ SmemGroups t;
  const int64_t K = a.K;
  const int slabs = (int)((K + 255) / 256);
  build_group_tables(a.grp, slabs, t);
  if (t.bad) return;
  const int G = a.grp.G;
  const int lane = threadIdx.x & 31;
  const int nscale_row = (int)(K / 16);
  const int64_t units = t.up[G];
  const int64_t warps = (int64_t)gridDim.x * kWarps;
  const int64_t w = (int64_t)blockIdx.x * kWarps + threadIdx.x / 32;
  const int64_t upw = (units + warps - 1) / warps;
  const int64_t u0 = w * upw, u1 = min(units, u0 + upw);
  if (u0 >= u1) return;
  int g = find_unit_group(t, G, u0);
  for (int64_t u = u0; u < u1; ++u) {
    while (t.up[g + 1] <= u) ++g;
    const Unit un = decode_unit(t, g, u, K, lane);
    uint4 v[16];
    load_unit(a.x, K, un, v);
    if (a.row_codes) {
      const float S = nvfp4_global_scale(a.amax_row[g]);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (i >= un.nvalid) break;
        float f[8];
        unpack8(v[i], f);
        float am = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) am = fmaxf(am, fabsf(f[k]));
        am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
        uint32_t sf;
        const float enc = nvfp4_block_encode(am, S, &sf);
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          word |= e2m1x2(__fmul_rn(f[2 * k], enc), __fmul_rn(f[2 * k + 1], enc)) << (8 * k);
        if (un.active) {
          const int64_t r = un.row0 + i;
          *reinterpret_cast<uint32_t*>(a.row_codes + r * (K / 2) + un.col0 / 2) = word;
          if ((lane & 1) == 0)
            a.row_scales[scale_offset(a.row_tiled, t, g, r, (int)(un.col0 >> 4), nscale_row)] = (uint8_t)sf;
        }
      }
    }
    if (a.col_codes && un.active) {
      const float S = nvfp4_global_scale(a.amax_col[g]);
      const int64_t mpad = (int64_t)(t.mp[g + 1] - t.mp[g]);
      const int64_t cbase = K * (int64_t)t.mp[g] / 2, sbase = K * (int64_t)t.mp[g] / 16;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        float y[16];
        column16(v, cc, y);
        if (a.use_rht) {
#pragma unroll
          for (int i = 0; i < 16; ++i)
            if ((a.mask >> i) & 1u) y[i] = -y[i];
          fwht16(y);
#pragma unroll
          for (int i = 0; i < 16; ++i) y[i] = y[i] * 0.25f;
        }
        float b = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) b = fmaxf(b, fabsf(y[i]));
        uint32_t sf;
        const float enc = nvfp4_block_encode(b, S, &sf);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          lo |= e2m1x2(__fmul_rn(y[2 * k], enc), __fmul_rn(y[2 * k + 1], enc)) << (8 * k);
          hi |= e2m1x2(__fmul_rn(y[8 + 2 * k], enc), __fmul_rn(y[9 + 2 * k], enc)) << (8 * k);
        }
        const int64_t col = un.col0 + cc;
        *reinterpret_cast<uint2*>(a.col_codes + cbase + col * (mpad / 2) + 8LL * un.j) = make_uint2(lo, hi);
        a.col_scales[sbase + col * (mpad / 16) + un.j] = (uint8_t)sf;
      }
    }
  }
}

int grid_for(int64_t work_warps) {
  const int64_t max_blocks = (int64_t)num_sms() * 8;
  int64_t blocks = (work_warps + kWarps - 1) / kWarps;
  if (blocks > max_blocks) blocks = max_blocks;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

int quant_read_clear_status() { return read_clear_status(); }

cudaError_t launch_row_quant(const RowQuantArgs& a, cudaStream_t s) {
  const int grid = grid_for(a.M);
  if (a.format == GMLP_MXFP8)
    row_quant_kernel<GMLP_MXFP8><<<grid, kThreads, 0, s>>>(a);
  else
    row_quant_kernel<GMLP_NVFP4><<<grid, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_group_amax(const uint16_t* x, int64_t M, int64_t K, GroupSrc grp, float* amax,
                              cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * grp.G, s);
  if (e != cudaSuccess) return e;
  group_amax_kernel<<<grid_for(M), kThreads, 0, s>>>(x, K, grp, amax);
  return cudaGetLastError();
}

cudaError_t launch_hadamard_amax(const uint16_t* x, int64_t M, int64_t K, GroupSrc grp, uint32_t mask,
                                 float* amax_pre, float* amax_post, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax_pre, 0, sizeof(float) * grp.G, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(amax_post, 0, sizeof(float) * grp.G, s);
  if (e != cudaSuccess) return e;
  const int64_t units = ((M + 15) / 16 + grp.G) * ((K + 255) / 256);
  hadamard_amax_kernel<<<grid_for(units), kThreads, 0, s>>>(x, K, grp, mask & 0xFFFFu, amax_pre, amax_post);
  return cudaGetLastError();
}

cudaError_t launch_col_quant(const ColQuantArgs& a, cudaStream_t s) {
  const int64_t units = ((a.M + 15) / 16 + a.grp.G) * ((a.K + 255) / 256);
  col_quant_kernel<<<grid_for(units), kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace gmlp
