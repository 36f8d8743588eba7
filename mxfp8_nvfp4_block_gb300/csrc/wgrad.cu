// wgrad.cu -- the weight-gradient half of the fused grouped-MLP backward
// (MXFP8): columnwise quantisation of the token-major operands, and grouped
// GEMMs whose contraction runs over each expert's tokens.
//
// Method: PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8", sequence
// diagram, backward pass: beside the FC2 dGLU and FC1 dGrad kernels the
// weight gradients come from grouped GEMMs ("wgrad via general_grouped_gemm")
// on columnwise MXFP8 operands (the forward's d_col_tensor, the dGLU's
// columnwise fc1_dy).
//
// Columnwise operand (colq_kernel): group g's m_g tokens are cut into
// 128-token chunks counted from its first token; chunk w of all groups
// (groups in order) becomes the slab [C][128] at w * C * 128 of a chunk-major
// code array [T/128][C][128] (the group's transpose zero-padded to a multiple
// of 128 tokens), with one E8M0 scale per 32 tokens.  A GEMM stage's operand
// tile is then one contiguous block (128 or 256 rows x 128 bytes), where a
// token-contiguous [C][T] matrix would put its rows T bytes apart and halve
// the TMA unit's row rate.  The scales sit in the GEMM_TILED layout of a
// [C]-row operand with T/32 scales per row, so chunk w of column tile r is the
// 512-byte block r * (T / 128) + w, exactly what one GEMM stage loads.
//
// Grouped GEMM (wgrad_kernel; one CTA per SM, 576 threads, as gemm.cu):
// tile (g, 128-row tile of A, 256-row tile of B) accumulates over the group's
// chunks (one 128-token stage each) into 256 TMEM columns; the epilogue writes
// FP32 (or adds into it).  A group with no tokens gets zeros without an MMA.
// Tiles are ordered by their groups' chunk counts, longest first, and dealt to
// the persistent CTAs in alternating directions, so the ragged groups balance.
#include <cudaTypedefs.h>

#include "device.cuh"

namespace gmlp {

namespace {

// ------------------------------------------------------------------ columnwise MXFP8

constexpr int kColThreads = 128;  // one thread per output column of a 128-column tile

// 16-byte global -> shared copy; the bytes past src_bytes (0 or 16) are zeros
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kColThreads) colq_kernel(const ColqArgs a) {
  __shared__ __align__(16) uint16_t tile[128][128];  // [token][column] bf16
  __shared__ int off[kMaxGroups + 1];                // token offsets
  __shared__ int cb[kMaxGroups + 1];                 // chunk bases
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid & 31;
  const int G = a.grp.G;
  if (tid < 32) {
    long long c0 = 0, c1 = 0;
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
      const long long v0 = m, v1 = (m + 127) / 128;
      long long i0 = v0, i1 = v1;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const long long t0 = __shfl_up_sync(0xffffffffu, i0, d), t1 = __shfl_up_sync(0xffffffffu, i1, d);
        if (lane >= d) {
          i0 += t0;
          i1 += t1;
        }
      }
      if (g < G) {
        off[g] = (int)(c0 + i0 - v0);
        cb[g] = (int)(c1 + i1 - v1);
      }
      c0 += __shfl_sync(0xffffffffu, i0, 31);
      c1 += __shfl_sync(0xffffffffu, i1, 31);
      if (c0 > a.grp.M) b = 1;
    }
    b = __any_sync(0xffffffffu, b);
    if (lane == 0) {
      off[G] = (int)c0;
      cb[G] = (int)c1;
      bad = b;
      if (b && blockIdx.x == 0 && blockIdx.y == 0) report_device_error(GMLP_ERR_DEVICE_BOUNDS);
    }
  }
  __syncthreads();
  const int w = blockIdx.x;
  if (bad || w >= cb[G]) return;
  int lo = 0, hi = G - 1;  // the group of chunk w: largest g with cb[g] <= w
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (cb[mid] <= w) lo = mid; else hi = mid - 1;
  }
  const int g = lo;
  const int local = w - cb[g];
  const int valid = min(128, off[g + 1] - off[g] - 128 * local);
  const int64_t t0 = (int64_t)off[g] + 128 * local;
  const int64_t c0 = (int64_t)blockIdx.y * 128;

  // 1. the chunk's 128 tokens x 128 columns as bf16 (zero past the group's end);
  // thread tid moves 16-byte vector vc = tid % 16 of rows tid / 16 + 8 i
  const int vc = tid & 15, r0 = tid >> 4;
  if (MODE == COLQ_PLAIN) {
    // all 16 copies in flight at once; rows past the group's end are zero-filled
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t = r0 + 8 * i;
      const uint16_t* src = a.src + (t0 + (t < valid ? t : 0)) * a.ld + c0 + 8 * vc;
      cp_async16(smem_u32(&tile[t][8 * vc]), src, t < valid ? 16u : 0u);
    }
    cp_async_wait_all();
  } else {
#pragma unroll 1
    for (int i0 = 0; i0 < 16; i0 += 4) {
      uint4 hv[4], uv[4];
      float pv[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int t = r0 + 8 * (i0 + k);
        hv[k] = uv[k] = make_uint4(0, 0, 0, 0);
        pv[k] = 0.0f;
        if (t < valid) {
          const uint16_t* row = a.src + (t0 + t) * a.ld + c0 + 8 * vc;
          hv[k] = __ldg(reinterpret_cast<const uint4*>(row));
          if (MODE == COLQ_SWIGLU) uv[k] = __ldg(reinterpret_cast<const uint4*>(row + a.up_off));
          pv[k] = a.probs ? __ldg(a.probs + t0 + t) : 1.0f;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // fc2_x = bf16(act(h) * prob), the fc1 epilogue's own arithmetic (an
        // invalid row has h = 0, prob = 0: zero)
        const uint32_t hw[4] = {hv[k].x, hv[k].y, hv[k].z, hv[k].w};
        const uint32_t uw[4] = {uv[k].x, uv[k].y, uv[k].z, uv[k].w};
        const float p = pv[k];
        uint32_t ow[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float f0, f1;
          if (MODE == COLQ_SWIGLU) {
            f0 = fc2x_swiglu(bf16_bits_to_float(hw[e] & 0xFFFFu), bf16_bits_to_float(uw[e] & 0xFFFFu), p);
            f1 = fc2x_swiglu(bf16_bits_to_float(hw[e] >> 16), bf16_bits_to_float(uw[e] >> 16), p);
          } else {
            f0 = fc2x_srelu(bf16_bits_to_float(hw[e] & 0xFFFFu), p);
            f1 = fc2x_srelu(bf16_bits_to_float(hw[e] >> 16), p);
          }
          ow[e] = bf16_bits(f0) | (bf16_bits(f1) << 16);
        }
        *reinterpret_cast<uint4*>(&tile[r0 + 8 * (i0 + k)][8 * vc]) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
    }
  }
  __syncthreads();

  // 2. thread c: column c0 + c, four 32-token blocks -> 4 x 32 codes, 4 scales
  const int c = tid;
  uint8_t* crow = a.codes + ((int64_t)w * a.C + c0 + c) * 128;
  uint32_t sc = 0;
  float csum = 0.0f;
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    float v[32], m[16], sm[16];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = bf16_bits_to_float(tile[32 * j + i][c]);
    // block max and (for the bias gradient) block sum as balanced trees: short
    // dependency chains instead of one 32-long chain each
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      m[i] = fmaxf(fabsf(v[i]), fabsf(v[i + 16]));
      sm[i] = v[i] + v[i + 16];
    }
#pragma unroll
    for (int h = 8; h > 0; h >>= 1)
#pragma unroll
      for (int i = 0; i < h; ++i) {
        m[i] = fmaxf(m[i], m[i + h]);
        sm[i] = sm[i] + sm[i + h];
      }
    const float amax = m[0];
    csum += sm[0];
    const int e = mxfp8_exponent(amax);
    const float mul = exp2_neg(e);
    uint32_t wd[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      wd[k] = e4m3x2(v[4 * k] * mul, v[4 * k + 1] * mul) | (e4m3x2(v[4 * k + 2] * mul, v[4 * k + 3] * mul) << 16);
    st_global_v8(crow + 32 * j, wd);
    sc |= (uint32_t)(e + 127) << (8 * j);
  }
  const int64_t blk = (int64_t)blockIdx.y * (a.T / 128) + w;
  *reinterpret_cast<uint32_t*>(a.scales + blk * 512 + (c & 31) * 16 + (c >> 5) * 4) = sc;
  if (a.colsum) atomicAdd(a.colsum + (int64_t)g * a.C + c0 + c, csum);
}

// ------------------------------------------------------------------ grouped wgrad GEMM

constexpr int kWThreads = 576;  // producer, MMA issuer, 16 epilogue warps
constexpr int kWEpiWarps = 16;
constexpr int kWStages = 4;
constexpr int kWATile = 128 * 128;  // 128 rows x 128 tokens (bytes)
constexpr int kWBTile = 256 * 128;
constexpr int kWSfA = 512, kWSfB = 1024;
constexpr int kWStageBytes = kWATile + kWBTile + kWSfA + kWSfB;
constexpr uint32_t kWAccCols = 256;
constexpr uint32_t kWSfCols = 16;  // TMEM scale columns per stage (SFA 4, SFB 8)

// kind::mxf8f6f4, E4M3 x E4M3, UE8M0 scales, M = 128, N = 256, K-major A
// and B, scale byte k of each 32-bit TMEM scale word for the k-th MMA.
__device__ __forceinline__ uint32_t wgrad_idesc(int k) {
  return (uint32_t(256 >> 3) << 17) | (1u << 23) | (uint32_t(128 >> 4) << 24) | (uint32_t(k) << 4) |
         (uint32_t(k) << 29);
}

__device__ __forceinline__ void ld_global_v8(const void* p, uint32_t* w) {
  asm volatile("ld.global.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

__global__ void __launch_bounds__(kWThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const WgradArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kWStages * kWATile;
  uint8_t* sSFA = sB + kWStages * kWBTile;
  uint8_t* sSFB = sSFA + kWStages * kWSfA;
  uint64_t* full = reinterpret_cast<uint64_t*>(sSFB + kWStages * kWSfB);
  uint64_t* empty = full + kWStages;
  uint64_t* tfull = empty + kWStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  int* bad = reinterpret_cast<int*>(tslot + 2);
  int* nkb = reinterpret_cast<int*>(tslot + 4);  // chunks per group
  int* cb = nkb + kMaxGroups + 1;               // chunk bases
  int* ord = cb + kMaxGroups + 1;               // groups, longest first

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  const int G = a.grp.G;
  const int MT = (int)(a.RA / 128), NT = (int)(a.RB / 256);
  const int TPG = MT * NT;
  const int64_t KBT = a.T / 128;

  if (warp == 0) {
    long long c1 = 0, c0 = 0;
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
      const long long v1 = (m + 127) / 128;
      long long i1 = v1, i0 = m;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const long long t1 = __shfl_up_sync(0xffffffffu, i1, d), t0 = __shfl_up_sync(0xffffffffu, i0, d);
        if (lane >= d) {
          i1 += t1;
          i0 += t0;
        }
      }
      if (g < G) {
        nkb[g] = (int)v1;
        cb[g] = (int)(c1 + i1 - v1);
      }
      c1 += __shfl_sync(0xffffffffu, i1, 31);
      c0 += __shfl_sync(0xffffffffu, i0, 31);
      if (c0 > a.grp.M || c1 > KBT) b = 1;
    }
    b = __any_sync(0xffffffffu, b);
    if (lane == 0) {
      cb[G] = (int)c1;
      *bad = b;
      if (b && blockIdx.x == 0) report_device_error(GMLP_ERR_DEVICE_BOUNDS);
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
    }
  } else if (warp == 1) {
    tmem_alloc(tslot, 512);
  } else if (threadIdx.x == 64) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, kWEpiWarps);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // tile order: groups by chunk count, longest first (ties by index)
  for (int g = threadIdx.x; g < G; g += kWThreads) {
    const int v = nkb[g];
    int r = 0;
    for (int h = 0; h < G; ++h) {
      const int u = nkb[h];
      r += (u > v) || (u == v && h < g);
    }
    ord[r] = g;
  }
  __syncthreads();
  const uint32_t tbase = *tslot;
  const int total = *bad ? 0 : G * TPG;
  // round i of the tile list goes left to right when i is even and right to
  // left when odd, so a CTA that drew a long tile draws a short one next
  auto snake_tile = [&](int i) {
    return i * (int)gridDim.x + ((i & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x);
  };

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    const uint64_t pol_a = policy_evict_normal();
    const uint64_t pol_b = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_parity = 0;
    for (int i = 0; i * (int)gridDim.x < total && !*abort_flag; ++i) {
      const int w = snake_tile(i);
      if (w >= total) continue;
      const int g = ord[w / TPG], local = w % TPG;
      const int mt = local % MT, nt = local / MT;
      for (int kb = 0; kb < nkb[g]; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)kWStageBytes);
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
        const int64_t chunk = (int64_t)cb[g] + kb;
        tma_load_2d(sA + stage * kWATile, &tmA, 0, (int32_t)(chunk * a.RA + mt * 128), &full[stage], pol_a);
        tma_load_2d(sB + stage * kWBTile, &tmB, 0, (int32_t)(chunk * a.RB + nt * 256), &full[stage], pol_b);
        bulk_load(sSFA + stage * kWSfA, a.a_scales + ((int64_t)mt * KBT + chunk) * 512, 512, &full[stage]);
        bulk_load(sSFB + stage * kWSfB, a.b_scales + ((int64_t)(2 * nt) * KBT + chunk) * 512, 512, &full[stage]);
        bulk_load(sSFB + stage * kWSfB + 512, a.b_scales + ((int64_t)(2 * nt + 1) * KBT + chunk) * 512, 512,
                  &full[stage]);
        if (++stage == kWStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // every copy signalled on this CTA's barriers lands before it exits
    for (int s = 0; s < kWStages; ++s)
      if (armed & (1u << s)) mbar_wait_drain(&full[s], (armed_parity >> s) & 1u);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    const uint32_t sf_base = tbase + kWAccCols;
    for (int i = 0; i * (int)gridDim.x < total && !*abort_flag; ++i) {
      const int w = snake_tile(i);
      if (w >= total) continue;
      const int g = ord[w / TPG];
      if (!mbar_wait(tempty, acc_phase ^ 1, abort_flag)) break;
      tc_fence_after();
      bool ok = true;
      for (int kb = 0; kb < nkb[g]; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sfa_t = sf_base + stage * kWSfCols;
        const uint32_t sfb_t = sfa_t + 4;
        const uint32_t sA_addr = smem_u32(sA + stage * kWATile);
        const uint32_t sB_addr = smem_u32(sB + stage * kWBTile);
        const uint32_t sfa_addr = smem_u32(sSFA + stage * kWSfA);
        const uint32_t sfb_addr = smem_u32(sSFB + stage * kWSfB);
        tc_cp_32x128b_x4(sfa_t, smem_desc(sfa_addr, 0, 128, 0));
        tc_cp_32x128b_x4(sfb_t, smem_desc(sfb_addr, 0, 128, 0));
        tc_cp_32x128b_x4(sfb_t + 4, smem_desc(sfb_addr + 512, 0, 128, 0));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = smem_desc(sA_addr + 32 * k, 16, 1024, 2);
          const uint64_t bd = smem_desc(sB_addr + 32 * k, 16, 1024, 2);
          tc_mma_mxf8(tbase, ad, bd, wgrad_idesc(k), sfa_t, sfb_t, (kb > 0 || k > 0) ? 1u : 0u);
        }
        tc_commit(&empty[stage]);
        if (++stage == kWStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      tc_commit(tfull);  // with no MMA (empty group) it arrives at once
      acc_phase ^= 1;
    }
    // all MMAs and copies this thread issued complete before TMEM is freed
    tc_commit(drain);
    mbar_wait_drain(drain, 0);
  } else if (warp >= 2) {
    // ---------------- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 and
    // the 64-column slice (w - 2) / 4 of the 256-column accumulator
    const int q = warp & 3;
    const int slice = (warp - 2) >> 2;
    uint32_t acc_phase = 0;
    for (int i = 0; i * (int)gridDim.x < total && !*abort_flag; ++i) {
      const int w = snake_tile(i);
      if (w >= total) continue;
      const int g = ord[w / TPG], local = w % TPG;
      const int mt = local % MT, nt = local / MT;
      if (!mbar_wait(tfull, acc_phase, abort_flag)) break;
      tc_fence_after();
      float acc[64];
      const bool has = nkb[g] > 0;
      if (has) {
        const uint32_t taddr = tbase + (uint32_t(32 * q) << 16) + uint32_t(slice * 64);
        tmem_ld32(taddr, acc);
        tmem_ld32(taddr + 32, acc + 32);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.0f;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      acc_phase ^= 1;
      if (!has && a.accumulate) continue;
      // 4 x 4 transpose of 8-column chunks inside each quad of lanes (two
      // xor-shuffle rounds): afterwards chunk s of each 32-column block of lane
      // 4a + b holds row 4a + s, columns 8b .. 8b + 7, so one store instruction
      // writes whole 128-byte lines (a row per quad) rather than a 32-byte
      // sector per lane and row, a quarter of the L2 write requests.
      const int b = lane & 3;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int m = 1; m <= 2; m <<= 1) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (c & m) continue;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              float& lo = acc[32 * u + 8 * c + e];
              float& hi = acc[32 * u + 8 * (c | m) + e];
              const float recv = __shfl_xor_sync(0xffffffffu, (b & m) ? lo : hi, m);
              if (b & m) lo = recv; else hi = recv;
            }
          }
        }
      }
      const int64_t row0 = (int64_t)g * a.RA + (int64_t)mt * 128 + 32 * q + (lane & ~3);
      float* obase = a.out + row0 * a.RB + (int64_t)nt * 256 + slice * 64 + 8 * b;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          float* op = obase + (int64_t)s4 * a.RB + 32 * u;
          const float* v = acc + 32 * u + 8 * s4;
          uint32_t o[8];
          if (a.accumulate) {
            ld_global_v8(op, o);
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) + v[k]);
          } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) o[k] = __float_as_uint(v[k]);
          }
          st_global_v8(op, o);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

constexpr size_t kWSmem = (size_t)kWStages * kWStageBytes + 1024 + 256 + 3 * (kMaxGroups + 1) * sizeof(int);

}  // namespace

int wgrad_read_clear_status() { return read_clear_status(); }

cudaError_t launch_colq(const ColqArgs& a, cudaStream_t s) {
  if (a.grp.M == 0 || a.C == 0) return cudaSuccess;
  const dim3 grid((unsigned)(a.T / 128), (unsigned)(a.C / 128));
  if (a.mode == COLQ_SWIGLU)
    colq_kernel<COLQ_SWIGLU><<<grid, kColThreads, 0, s>>>(a);
  else if (a.mode == COLQ_SRELU)
    colq_kernel<COLQ_SRELU><<<grid, kColThreads, 0, s>>>(a);
  else
    colq_kernel<COLQ_PLAIN><<<grid, kColThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_wgrad(const WgradArgs& a, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    cudaError_t e = cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kWSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev & 63] = true;
  }
  CUtensorMap ta, tb;
  // chunk-major codes: rows (chunk, operand row) of 128 token bytes
  if (!make_tmap(&ta, a.a_codes, 128, a.T / 128 * a.RA, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap(&tb, a.b_codes, 128, a.T / 128 * a.RB, 128, 256, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const int64_t tiles = (int64_t)a.grp.G * (a.RA / 128) * (a.RB / 256);
  int64_t units = num_sms();
  if (tiles < units) units = tiles;
  if (units < 1) units = 1;
  wgrad_kernel<<<(unsigned)units, kWThreads, kWSmem, s>>>(ta, tb, a);
  return cudaGetLastError();
}

}  // namespace gmlp
