// device.cuh -- device helpers of the CUDA path: format conversions through the
// hardware cvt instructions, mbarrier / TMA / tcgen05 inline-PTX wrappers, the
// device status word and bounded waits.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace gmlp {

// ----------------------------------------------------------------- status word

// Set once per failure (first writer wins); read and cleared by
// gmlp_check_device_status.  One word per translation unit (no relocatable
// device code), each read through read_clear_status() of its own unit.
static __device__ int g_device_status = 0;

static inline int read_clear_status() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return -1;
  if (cudaMemcpyToSymbol(g_device_status, &z, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

__device__ __forceinline__ void report_device_error(int code) {
  atomicCAS(&g_device_status, 0, code);
}

// ----------------------------------------------------------------- formats

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Round an FP32 value to bf16 (round-to-nearest-even) and return it as FP32.
__device__ __forceinline__ float round_bf16(float f) { return __bfloat162float(__float2bfloat16_rn(f)); }

__device__ __forceinline__ uint32_t bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return (uint32_t)(*reinterpret_cast<uint16_t*>(&h));
}

// Two FP32 values -> two E4M3 bytes (round-to-nearest-even, saturating);
// lo goes to bits 0..7, hi to bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two FP32 values -> two E2M1 nibbles; lo in bits 0..3, hi in bits 4..7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// E4M3 byte -> FP32 (exact).
__device__ __forceinline__ float e4m3_to_float(uint32_t byte) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(byte & 0xFF)));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

// MXFP8 block scale exponent from the block amax (an FP32 holding a bf16
// value or a product of them): floor(log2 amax) - 8 clamped to [-127, 127];
// zero and FP32-subnormal amax (floor(log2) <= -127) give -127.
__device__ __forceinline__ int mxfp8_exponent(float amax) {
  int E = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  int e = E - 135;
  return e < -127 ? -127 : e;
}

// 2^-e for e in [-127, 126] as an exact FP32.
__device__ __forceinline__ float exp2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// NVFP4 global encode scale S = 2688 / amax (FP32, IEEE division); amax 0 -> 1;
// overflow -> FLT_MAX.
__device__ __forceinline__ float nvfp4_global_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  float S = __fdiv_rn(2688.0f, amax);
  return isinf(S) ? 3.402823466e38f : S;
}

// ----------------------------------------------------------------- dependent launch

// Wait until the preceding kernel in the stream (launched before this one with
// programmatic stream serialization) has completed and its writes are visible.
// A kernel launched normally returns at once.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next kernel in the stream begin its prologue.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------- bounded waits

// A wait gives up after this many nanoseconds of %globaltimer; the longest
// legitimate wait in these kernels is far below a millisecond.
constexpr uint64_t kWaitLimitNs = 4000000000ull;

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// reports GMLP_ERR_DEVICE_TIMEOUT) when the time limit passes or *abort is set.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        report_device_error(7 /* GMLP_ERR_DEVICE_TIMEOUT */);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait used only while shutting down after an abort (no new report).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > 500000000ull) return;
}

// ----------------------------------------------------------------- TMA / bulk copies

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ----------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive on an mbarrier when every tcgen05 operation this thread issued so far
// (MMAs and copies) has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Copy one 512-byte block of 32 rows x 16 bytes from shared memory into four
// TMEM columns of lanes 0..31, replicated to all four lane quarters.
__device__ __forceinline__ void tc_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Copy 128 rows x 32 bytes of shared memory into TMEM: row i -> lane i,
// columns taddr .. taddr + 7.
__device__ __forceinline__ void tc_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Block-scaled MMAs, D(tmem) (+)= A(smem) * B(smem)^T with per-block scales in TMEM.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_mma_nvf4(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// 32 consecutive FP32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Packed pairs of FP32 (two columns side by side); each lane of the pair is an
// IEEE round-to-nearest-even operation, identical to the scalar one.
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float lo2(f32x2 v) {
  float a;
  [[maybe_unused]] float b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return a;
}
__device__ __forceinline__ float hi2(f32x2 v) {
  [[maybe_unused]] float a;
  float b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
  return b;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// 16 consecutive 32-bit TMEM columns of this warp's 32 lanes from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Scale factors of one stage from shared memory into this warp's lane quarter
// of TMEM, in the layout the 32x128b.warpx4 copies produce: lane l, column c
// of a 512-byte block's four columns holds the block's 4-byte word 4 l + c.
template <int FMT>
__device__ __forceinline__ void write_stage_scales(uint32_t lane_base, uint32_t sfa_t, uint32_t sfb_t,
                                                   const uint8_t* sfa, const uint8_t* sfb, int lane) {
  uint32_t r[16];
  if (FMT == GMLP_MXFP8) {  // SFA one block (4 columns), SFB two blocks (8 columns): 12 of 16 columns
    const uint4 a = *reinterpret_cast<const uint4*>(sfa + 16 * lane);
    const uint4 b0 = *reinterpret_cast<const uint4*>(sfb + 16 * lane);
    const uint4 b1 = *reinterpret_cast<const uint4*>(sfb + 512 + 16 * lane);
    const uint32_t w[16] = {a.x, a.y, a.z, a.w, b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w, 0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = w[i];
    tmem_st16(lane_base | sfa_t, r);
  } else {  // SFA four blocks (16 columns); SFB per MMA k the two halves' blocks (8 columns), 32 columns
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 a = *reinterpret_cast<const uint4*>(sfa + 512 * k + 16 * lane);
      r[4 * k] = a.x, r[4 * k + 1] = a.y, r[4 * k + 2] = a.z, r[4 * k + 3] = a.w;
    }
    tmem_st16(lane_base | sfa_t, r);
#pragma unroll
    for (int hk = 0; hk < 2; ++hk) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {  // columns 8k .. 8k + 7 for k = 2 hk + j / 2
        const int k = 2 * hk + (j >> 1), h = j & 1;
        const uint4 b = *reinterpret_cast<const uint4*>(sfb + 2048 * h + 512 * k + 16 * lane);
        r[4 * j] = b.x, r[4 * j + 1] = b.y, r[4 * j + 2] = b.z, r[4 * j + 3] = b.w;
      }
      tmem_st16(lane_base | (sfb_t + 16 * hk), r);
    }
  }
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (>> 4), the fixed version bits 46..48 = 0b001, and the
// swizzle mode in bits 61..63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 7) << 61;
  return d;
}

// ----------------------------------------------------------------- global memory

// 32-byte store (one full sector per lane); dst must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* dst, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// 32 bytes from global memory through the read-only path without allocating
// in L1 (p 32-byte aligned).
__device__ __forceinline__ void ld_global_nc_v8(const void* p, uint32_t* w) {
  asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

// ----------------------------------------------------------------- activations

// silu(gate) * up in FP32 with the fast exponential and division (their
// error is far below the bf16 rounding that follows).
__device__ __forceinline__ float silu_times(float gate, float up) {
  return __fdividef(gate, 1.0f + __expf(fminf(-gate, 80.0f))) * up;
}

// fc2_x = bf16(act(h) * prob) from bf16 activation-input values (FP32
// arithmetic).  The fc1 epilogue and every rebuild of fc2_x from the saved
// activation input call these, so the two give the same bits.
//   SwiGLU:     silu(g) * u          (g gate, u up)
//   SReLU:      max(h, 0)^2
//   tanh-SReLU: c * tanh(max(h, 0)^2 / c), with inv_c = 1 / c rounded once
__device__ __forceinline__ float fc2x_swiglu(float g, float u, float prob) { return round_bf16(silu_times(g, u) * prob); }

__device__ __forceinline__ float fc2x_srelu(float h, float prob) {
  const float r = fmaxf(h, 0.0f);
  return round_bf16(r * r * prob);
}

__device__ __forceinline__ float fc2x_tanh_srelu(float h, float prob, float c, float inv_c) {
  const float r = fmaxf(h, 0.0f);
  return round_bf16(c * tanhf(r * r * inv_c) * prob);
}

}  // namespace gmlp
