// internal.h -- declarations shared by the CUDA path's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gmlp.h"

namespace gmlp {

constexpr int kMaxGroups = 512;

// Per-group tables every kernel derives from split_sizes at its start
// (split sizes stay on the device).  When `splits` is null the G groups all
// have `uniform_m` rows (the experts of a stacked weight).
struct GroupSrc {
  const int64_t* splits;
  int32_t uniform_m;
  int32_t G;
  int64_t M;
};

// ---- quantisers (quant.cu) ----

struct RowQuantArgs {
  const uint16_t* x;        // bf16 [M][K] (or weights [G][rows][K])
  int64_t M, K;
  GroupSrc grp;
  int format;               // GMLP_MXFP8 / GMLP_NVFP4
  int tiled;                // scales in GEMM_TILED layout
  uint8_t* codes;
  uint8_t* scales;
  const float* amax;        // NVFP4: per-group amax giving S_g
  float* S_out;             // optional: write S_g for every group
  int swiglu_interleave;    // weights: gate/up 32-row interleave within each group
  float* zero_ptr;          // optional: floats zeroed by the grid before any later kernel (for its atomics)
  int zero_count;
  float* zero_ptr2;         // optional second range
  int zero_count2;
  int pdl;                  // launch as a programmatic dependent of the previous kernel
  int reverse;              // each warp sweeps its share last pass first (after launch_group_amax on
                            // the same grid with keep > 0, whose evict-last reads are still in L2)
};
cudaError_t launch_row_quant(const RowQuantArgs& a, cudaStream_t s);

// the row quantiser's grid for M rows (one wave of its persistent blocks)
int row_quant_grid(int format, int tiled, int64_t M);

// per-group max |x| into amax[G] (zeroed by the launcher).  grid > 0 sets
// the block count; the last `keep` fraction (0..1) of each warp's share is
// read with an L2 evict-last policy (for a row cast on the same grid with
// reverse = 1).
cudaError_t launch_group_amax(const uint16_t* x, int64_t M, int64_t K, GroupSrc grp, float* amax, cudaStream_t s,
                              int grid = 0, float keep = 0.0f);

cudaError_t launch_hadamard_amax(const uint16_t* x, int64_t M, int64_t K, GroupSrc grp, uint32_t mask,
                                 float* amax_pre, float* amax_post, cudaStream_t s);

struct ColQuantArgs {
  const uint16_t* x;
  int64_t M, K;
  GroupSrc grp;
  int use_rht;
  uint32_t mask;
  const float* amax_row;    // S for the rowwise output
  const float* amax_col;    // S for the columnwise output
  uint8_t* row_codes;       // nullable: also write rowwise NVFP4 in the same pass
  uint8_t* row_scales;
  int row_tiled;
  uint8_t* col_codes;       // nullable: then rowwise (GEMM_TILED) + amax_post_out only
  uint8_t* col_scales;
  float* amax_post_out;     // with col_codes null: max-accumulates the post-RHT amax per group (zeroed before)
  uint32_t sgn[16];         // set by the launcher: 0x80000000 (the FP32 sign bit) for the rows the mask negates
};
cudaError_t launch_col_quant(const ColQuantArgs& a, cudaStream_t s);

// fc2_x = bf16(act(h) * prob) from the saved activation input h [M][N1]
cudaError_t launch_fc2x_recompute(const uint16_t* h, const float* probs, int64_t M, int64_t N, int act, float c,
                                  uint16_t* out, cudaStream_t s);

// ---- grouped GEMM (gemm.cu) ----

enum Epilogue : int {
  EPI_FC1_SWIGLU = 0,  // fc1 + SwiGLU (gate/up 32-column interleave) x prob
  EPI_FC1_SRELU = 1,   // fc1 + squared ReLU x prob
  EPI_FC2 = 2,         // fc2: bf16 output
  EPI_FC1_TANH_SRELU = 3,  // fc1 + tanh soft clamp of the squared ReLU x prob
  EPI_DGLU_SWIGLU = 4,     // backward: dfc2x -> dSwiGLU x prob (fc1_dy, MXFP8) and dprob
  EPI_DSRELU = 5,          // backward: dfc2x -> dSReLU x prob (fc1_dy, MXFP8) and dprob
};

struct GemmArgs {
  int format;              // GMLP_MXFP8 / GMLP_NVFP4 (both operands)
  int epi;                 // Epilogue
  const uint8_t* a_codes;  // [M][kbytes]
  const uint8_t* a_scales; // GEMM_TILED, groups of the token split
  const uint8_t* b_codes;  // [G][n_out][kbytes]
  const uint8_t* b_scales; // GEMM_TILED, experts as groups of n_out rows
  int64_t M;
  int64_t kbytes;          // contraction bytes per row (K or K/2)
  int64_t n_out;           // accumulator columns per expert (fc1: 2N or N; fc2: K)
  GroupSrc grp;
  const float* a_amax;     // NVFP4: per-group amax of A (S_a = 2688 / amax)
  const float* b_S;        // NVFP4: per-expert S of B
  const uint16_t* bias;    // optional bf16 [G][n_out], logical row order of B (before any interleave)
  const float* probs;      // fc1: [M] or null
  // MXFP8 fc1 outputs (fc2_x quantised in the epilogue)
  uint8_t* out_codes;      // [M][n_cols_out]
  uint8_t* out_scales;     // GEMM_TILED over the token split
  // NVFP4 fc1 output and fc2 output
  uint16_t* out_bf16;      // [M][n_cols_out]
  uint16_t* pre_act_out;   // optional fc1: bf16 activation input [M][n_out], logical column order
  const uint16_t* act_in;  // backward dGLU: the forward's bf16 activation input [M][n_cols_out]
  float* dprob;            // backward dGLU: [M] d(loss)/d(prob), accumulated with atomicAdd (zeroed before)
  float* amax_pre;         // NVFP4 fc1: [G] (atomicMax, zeroed before)
  float* amax_post;
  uint32_t rht_mask;
  float tanh_c;            // EPI_FC1_TANH_SRELU: soft-clamp scale
  int64_t n_cols_out;      // row length of the output (fc1: N; fc2: K)
  int b_x4;                // NVFP4: b_scales in the replicated GEMM_TILED_X4 layout
  int pair;                // 2: CTA pairs (cta_group::2); otherwise single-CTA tiles
  int pdl;                 // launch as a programmatic dependent of the previous kernel
};
cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s);

// ---- weight gradients (wgrad.cu) ----

// Columnwise MXFP8 of a token-sorted bf16 matrix (or of fc2_x rebuilt from the
// saved activation input): per group, 128-token chunks become [C][128] slabs
// of a chunk-major code array [T/128][C][128] (1x32 blocks along the tokens,
// zero past the group's end), scales GEMM_TILED for a [C]-row operand with
// T/32 per row.
enum ColqMode { COLQ_PLAIN = 0, COLQ_SWIGLU = 1, COLQ_SRELU = 2 };
struct ColqArgs {
  const uint16_t* src;  // [M][ld] bf16 (COLQ_SWIGLU / COLQ_SRELU: the activation input h)
  int64_t ld;           // row stride of src (elements)
  int64_t C;            // output columns (multiple of 128)
  int64_t up_off;       // COLQ_SWIGLU: column of the first up value (N)
  const float* probs;   // COLQ_SWIGLU / COLQ_SRELU: [M] routing probabilities, null = 1
  GroupSrc grp;
  int64_t T;            // 128 x (chunk capacity)
  uint8_t* codes;       // [T / 128][C][128]
  uint8_t* scales;      // (C / 128) x (T / 128) blocks of 512 bytes
  float* colsum;        // [G][C] per-group column sums (accumulated), or null
  int mode;             // ColqMode
};
cudaError_t launch_colq(const ColqArgs& a, cudaStream_t s);

// Per group g: out_g [RA][RB] (FP32) = A_g B_g^T over the group's padded
// tokens, A [RA][T] and B [RB][T] columnwise MXFP8 operands from launch_colq.
struct WgradArgs {
  const uint8_t* a_codes;
  const uint8_t* a_scales;
  const uint8_t* b_codes;
  const uint8_t* b_scales;
  int64_t RA, RB;       // RA % 128 == 0, RB % 256 == 0
  int64_t T;            // as ColqArgs::T
  GroupSrc grp;
  float* out;           // [G][RA][RB], 32-byte aligned
  int accumulate;       // 1: out += result; 0: out = result
};
cudaError_t launch_wgrad(const WgradArgs& a, cudaStream_t s);

int num_sms();

// 2D uint8 tensor map over [rows][row_bytes] with a box of box_rows x
// box_bytes (gemm.cu); false if the driver entry point or the encode fails.
bool make_tmap(CUtensorMap* m, const void* base, int64_t row_bytes, int64_t rows, int box_bytes, int box_rows,
               CUtensorMapSwizzle swz);

// 2D 16-bit tensor map over [rows][cols] (row stride cols * 2 bytes) with a box
// of box_cols x box_rows, no swizzle; out-of-range elements read as zero.
bool make_tmap_u16(CUtensorMap* m, const void* base, int64_t cols, int64_t rows, int box_cols, int box_rows);

cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_mma_peak(int format, int scale_copy, int64_t iters, int ctas, cudaStream_t s);

// NVFP4 weight scales: GEMM_TILED -> GEMM_TILED_X4 (see gmlp_replicate_weight_scales)
cudaError_t launch_replicate_scales(const uint8_t* tiled, int64_t pairs, int64_t runs, uint8_t* out, cudaStream_t s);

gmlp_status set_last_error(gmlp_status st, const char* msg);

}  // namespace gmlp
