// peak.cu -- tensor-core ceiling of the grouped GEMM's mainloop: the same
// block-scaled tcgen05 instruction mix (per stage: the scale-factor copies to
// TMEM, four M=128 N=256 MMAs, one commit) issued in a loop from shared memory
// that is filled once, so no global memory is read.  The time of one launch
// gives the dense FP8 / FP4 rate this MMA shape reaches at the running clock;
// the GEMM kernels are measured against it.
//
// A stage s reuses the shared-memory buffers and scale columns of stage s - 4,
// so the issuer waits for that stage's commit before overwriting its scales,
// exactly as the GEMM's producer waits on its `empty` barrier (here with an
// infinitely fast producer).  SFCOPY = 0: the scales of all four stages are
// copied once before the loop, which isolates the copy cost; 1: the copies of
// GEMM_TILED weight scales (3 per stage for MXFP8, 12 for NVFP4); 2 (NVFP4):
// those of GEMM_TILED_X4 weight scales (4 SFA copies and 4 128x256b SFB copies
// per stage, all from the stage's first 6 KB of scale bytes); 3: no copies --
// the four warps write each stage's scale factors into their own lane
// quarters of TMEM with tcgen05.st (the layout the 32x128b.warpx4 copies
// produce) while the MMAs of earlier stages run, and signal the issuing
// thread through an mbarrier.
#include "device.cuh"

namespace gmlp {

namespace {

constexpr int kPeakThreads = 128;
constexpr int kStagesP = 4;
constexpr int kATile = 128 * 128;  // 128 rows x 128 bytes
constexpr int kBTile = 256 * 128;  // 256 rows x 128 bytes

template <int FMT>
struct PeakCfg {
  static constexpr int kSfBytes = FMT == GMLP_MXFP8 ? 512 : 2048;  // per 128 rows per stage
  static constexpr int kStageBytes = kATile + kBTile + 3 * kSfBytes;
  static constexpr uint32_t kSfCols = FMT == GMLP_MXFP8 ? 16 : 48;
  static constexpr uint32_t kSfbOff = FMT == GMLP_MXFP8 ? 4 : 16;
  static constexpr size_t kSmem = (size_t)kStagesP * kStageBytes + 1024 + 256 + 64;
};

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

// Operand bytes: random codes (E4M3 with the two NaN codes avoided; any E2M1
// nibbles).  Scale bytes: E8M0 in [2^-7, 2^8] or positive finite UE4M3.
template <int FMT>
__device__ __forceinline__ uint32_t operand_word(uint32_t i) {
  uint32_t w = mix32(i * 0x9e3779b9u + 0x1234567u);
  if (FMT == GMLP_MXFP8) {
    // clear bit 0 of any byte whose low seven bits are all ones (0x7f / 0xff)
    const uint32_t low7 = w & 0x7f7f7f7fu;
    const uint32_t nan = ((low7 + 0x01010101u) & 0x80808080u) >> 7;  // 1 per byte with low7 == 0x7f
    w &= ~nan;
  }
  return w;
}

template <int FMT>
__device__ __forceinline__ uint32_t scale_word(uint32_t i) {
  const uint32_t h = mix32(i + 0xabcdefu);
  return FMT == GMLP_MXFP8 ? (0x78787878u + (h & 0x0f0f0f0fu)) : (0x30303030u + (h & 0x1f1f1f1fu));
}

template <int FMT, int SFCOPY>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int64_t iters) {
  using C = PeakCfg<FMT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStagesP * kATile;
  uint8_t* sSF = sB + kStagesP * kBTile;  // per stage: SFA block(s), then the two SFB halves
  uint64_t* done = reinterpret_cast<uint64_t*>(sSF + kStagesP * 3 * C::kSfBytes);
  uint64_t* retired = done + 1;  // one per stage
  uint64_t* sfready = retired + kStagesP;  // SFCOPY 3: one per stage, 4 warp arrivals
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sfready + kStagesP);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);

  const int warp = threadIdx.x / 32;
  {
    uint32_t* w = reinterpret_cast<uint32_t*>(sA);
    const uint32_t n_ops = (uint32_t)(kStagesP * (kATile + kBTile)) / 4;
    for (uint32_t i = threadIdx.x; i < n_ops; i += kPeakThreads) w[i] = operand_word<FMT>(i);
    uint32_t* s = reinterpret_cast<uint32_t*>(sSF);
    const uint32_t n_sf = (uint32_t)(kStagesP * 3 * C::kSfBytes) / 4;
    for (uint32_t i = threadIdx.x; i < n_sf; i += kPeakThreads) s[i] = scale_word<FMT>(i);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
  } else if (threadIdx.x == 0) {
    mbar_init(done, 1);
    for (int s = 0; s < kStagesP; ++s) {
      mbar_init(&retired[s], 1);
      mbar_init(&sfready[s], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (SFCOPY == 3) {
    // all four warps write scale factors; thread 0 also issues the MMAs
    const uint32_t sf_base = tbase + 256;
    const int lane = threadIdx.x & 31;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    bool ok = true;
    for (int64_t it = 0; it < iters && ok; ++it) {
      const int stage = (int)(it & (kStagesP - 1));
      const uint32_t sfa_t = sf_base + stage * C::kSfCols;
      const uint32_t sfb_t = sfa_t + C::kSfbOff;
      if (it >= kStagesP) {  // the MMAs that read this stage's scale columns have completed
        ok = mbar_wait(&retired[stage], (uint32_t)((it / kStagesP - 1) & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
      }
      const uint8_t* sfa = sSF + stage * 3 * C::kSfBytes;
      write_stage_scales<FMT>(lane_base, sfa_t, sfb_t, sfa, sfa + C::kSfBytes, lane);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfready[stage]);
      if (threadIdx.x == 0) {
        ok = mbar_wait(&sfready[stage], (uint32_t)((it / kStagesP) & 1), abort_flag);
        if (ok) {
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + stage * kATile);
          const uint32_t b_addr = smem_u32(sB + stage * kBTile);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = smem_desc(a_addr + 32 * k, 16, 1024, 2);
            const uint64_t bd = smem_desc(b_addr + 32 * k, 16, 1024, 2);
            const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
            if (FMT == GMLP_MXFP8) {
              const uint32_t idesc = (256u >> 3 << 17) | (1u << 23) | (128u >> 4 << 24) | (uint32_t(k) << 4) |
                                     (uint32_t(k) << 29);
              tc_mma_mxf8(tbase, ad, bd, idesc, sfa_t, sfb_t, acc);
            } else {
              const uint32_t idesc = (1u << 7) | (1u << 10) | (256u >> 3 << 17) | (128u >> 4 << 24);
              tc_mma_nvf4(tbase, ad, bd, idesc, sfa_t + 4 * k, sfb_t + 8 * k, acc);
            }
          }
          tc_commit(&retired[stage]);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0 && !*abort_flag;
    }
    if (threadIdx.x == 0) {
      // every tcgen05 operation issued above completes before TMEM is freed
      tc_commit(done);
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(done, 0))
        if (globaltimer() - t0 > kWaitLimitNs) {
          report_device_error(GMLP_ERR_DEVICE_TIMEOUT);
          break;
        }
    }
  } else if (threadIdx.x == 0) {
    const uint32_t sf_base = tbase + 256;
    auto copy_scales = [&](int stage) {
      const uint32_t sfa_t = sf_base + stage * C::kSfCols;
      const uint32_t sfb_t = sfa_t + C::kSfbOff;
      const uint32_t sfa = smem_u32(sSF + stage * 3 * C::kSfBytes);
      const uint32_t sfb = sfa + C::kSfBytes;
      if (FMT == GMLP_NVFP4 && SFCOPY == 2) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tc_cp_32x128b_x4(sfa_t + 4 * k, smem_desc(sfa + 512 * k, 0, 128, 0));
          tc_cp_128x256b(sfb_t + 8 * k, smem_desc(sfb, 2048, 128, 0));
        }
      } else if (FMT == GMLP_MXFP8) {
        tc_cp_32x128b_x4(sfa_t, smem_desc(sfa, 0, 128, 0));
        tc_cp_32x128b_x4(sfb_t, smem_desc(sfb, 0, 128, 0));
        tc_cp_32x128b_x4(sfb_t + 4, smem_desc(sfb + 512, 0, 128, 0));
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tc_cp_32x128b_x4(sfa_t + 4 * k, smem_desc(sfa + 512 * k, 0, 128, 0));
          tc_cp_32x128b_x4(sfb_t + 8 * k, smem_desc(sfb + 512 * k, 0, 128, 0));
          tc_cp_32x128b_x4(sfb_t + 8 * k + 4, smem_desc(sfb + 2048 + 512 * k, 0, 128, 0));
        }
      }
    };
    if (SFCOPY == 0)
      for (int s = 0; s < kStagesP; ++s) copy_scales(s);
    bool ok = true;
    for (int64_t it = 0; it < iters && ok; ++it) {
      const int stage = (int)(it & (kStagesP - 1));
      if (it >= kStagesP) {
        ok = mbar_wait(&retired[stage], (uint32_t)((it / kStagesP - 1) & 1), abort_flag);
        if (!ok) break;
        tc_fence_after();
      }
      if (SFCOPY != 0) copy_scales(stage);
      const uint32_t sfa_t = sf_base + stage * C::kSfCols;
      const uint32_t sfb_t = sfa_t + C::kSfbOff;
      const uint32_t a_addr = smem_u32(sA + stage * kATile);
      const uint32_t b_addr = smem_u32(sB + stage * kBTile);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint64_t ad = smem_desc(a_addr + 32 * k, 16, 1024, 2);
        const uint64_t bd = smem_desc(b_addr + 32 * k, 16, 1024, 2);
        const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
        if (FMT == GMLP_MXFP8) {
          const uint32_t idesc = (256u >> 3 << 17) | (1u << 23) | (128u >> 4 << 24) | (uint32_t(k) << 4) |
                                 (uint32_t(k) << 29);
          tc_mma_mxf8(tbase, ad, bd, idesc, sfa_t, sfb_t, acc);
        } else {
          const uint32_t idesc = (1u << 7) | (1u << 10) | (256u >> 3 << 17) | (128u >> 4 << 24);
          tc_mma_nvf4(tbase, ad, bd, idesc, sfa_t + 4 * k, sfb_t + 8 * k, acc);
        }
      }
      tc_commit(&retired[stage]);
    }
    // every tcgen05 operation issued above completes before TMEM is freed
    tc_commit(done);
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(done, 0))
      if (globaltimer() - t0 > kWaitLimitNs) {
        report_device_error(GMLP_ERR_DEVICE_TIMEOUT);
        break;
      }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int FMT, int SFCOPY>
cudaError_t launch_peak_t(int64_t iters, int ctas, cudaStream_t s) {
  auto kern = mma_peak_kernel<FMT, SFCOPY>;
  constexpr size_t smem = PeakCfg<FMT>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<ctas, kPeakThreads, smem, s>>>(iters);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_mma_peak(int format, int scale_copy, int64_t iters, int ctas, cudaStream_t s) {
  if (format == GMLP_MXFP8) {
    if (scale_copy == 3) return launch_peak_t<GMLP_MXFP8, 3>(iters, ctas, s);
    return scale_copy ? launch_peak_t<GMLP_MXFP8, 1>(iters, ctas, s) : launch_peak_t<GMLP_MXFP8, 0>(iters, ctas, s);
  }
  if (scale_copy == 3) return launch_peak_t<GMLP_NVFP4, 3>(iters, ctas, s);
  if (scale_copy == 2) return launch_peak_t<GMLP_NVFP4, 2>(iters, ctas, s);
  return scale_copy ? launch_peak_t<GMLP_NVFP4, 1>(iters, ctas, s) : launch_peak_t<GMLP_NVFP4, 0>(iters, ctas, s);
}

int peak_read_clear_status() { return read_clear_status(); }

}  // namespace gmlp
