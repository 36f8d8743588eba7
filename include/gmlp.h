/*
 * gmlp.h -- C ABI of the fused grouped-MLP forward for mixture-of-experts
 * layers with MXFP8 / NVFP4 block quantisation, for GB300 (sm_103a).
 *
 * Library: libgmlp.so (hand-written CUDA; TMA, tcgen05 block-scaled MMA, TMEM).
 *
 * What it computes (TransformerEngine pull-request pages):
 *   - PR #2769 "GEMM + Swiglu fused Grouped MLP for MXFP8", Greptile summary and
 *     sequence diagram: MXFP8 x (a_tensor) -> FC1 GLU kernel with the stacked
 *     expert weights (b_tensor) and per-token probs (prob_tensor) -> MXFP8
 *     activation (d_tensor, sfd_row_tensor) -> FC2 kernel -> output.
 *   - PR #3837 "Reduce NVFP4 quantization work for the fused GroupedMLP fc2
 *     input with activation recompute", Description, Changes and flowchart:
 *     FC1 + activation -> fc2 input and its (pre-RHT, post-RHT) amax ->
 *     row-wise NVFP4 quantization -> FC2; the group Hadamard-amax pass and the
 *     quantize-with-amax cast as separate calls.
 *   - PR #3631 "Add NVTE_CUTEDSL_FUSED_GROUPED_MLP_WARN_FALLBACK", Changes:
 *     the fusion preconditions; here each unmet one is a status code, and there
 *     is no fallback path.
 *
 * Conventions (all calls):
 *   - Every pointer argument named as device memory is a device pointer owned
 *     by the caller; the library never allocates, frees or keeps it.  Device
 *     pointers must be 16-byte aligned; the bf16 outputs y and dx and the
 *     activation input h (fc1_pre_act, pre_act), which move in 32-byte
 *     vectors, 32-byte aligned.
 *   - Calls are asynchronous on `stream` and never synchronise the host,
 *     except gmlp_check_device_status.  Host structs are read during the call
 *     only.
 *   - bf16 tensors are passed as uint16_t bit patterns, row-major.
 *   - x is token-sorted: the rows of group g are rows off_g .. off_g + m_g - 1
 *     with off_g = m_0 + ... + m_{g-1}; split_sizes (int64, device, [G]) stay on
 *     the device, so M (their sum) is passed from the host.  The sum must equal
 *     M; a negative size or a sum above M is detected on the device and
 *     reported by gmlp_check_device_status as GMLP_ERR_DEVICE_BOUNDS (no
 *     output written past M).
 *   - Feature counts (K, N, weight rows and cols) are at most 2^20 and token
 *     counts M below 2^31; larger values are GMLP_ERR_INVALID_DIMS.
 *   - Host-side argument checks return a status before anything is launched.
 *     No C++ exception crosses the ABI.  gmlp_last_error() describes the last
 *     non-OK status of the calling thread.
 *
 * Formats (fixed by the method statement; the pages give no arithmetic):
 *   MXFP8: E4M3 codes (max 448, no infinity), one E8M0 scale per 1x32 block
 *     along a row: e = floor(log2 amax) - 8 (clamped to [-127,127], amax 0 ->
 *     -127), byte e + 127, codes E4M3(x * 2^-e), round-to-nearest-even,
 *     saturating.
 *   NVFP4: E2M1 codes packed two per byte (even element in the low nibble),
 *     one E4M3 scale per 1x16 block, and an FP32 global scale per group
 *     S = 448*6 / amax (amax 0 -> 1).  Block: t = (b/6)*S in FP32, sf = E4M3(t),
 *     enc = S/sf (0 when sf is 0), codes E2M1(x * enc).  Dequantised value:
 *     code * sf / S.
 *   RHT: y = 1/4 * H16 * diag(s) * v over 16 consecutive ROWS of one column
 *     of one group (chunks start at the group's first row; a short last chunk
 *     is zero-padded), s_i = -1 when bit i of rht_sign_mask is set; FP32.
 *
 * Scale layouts of rowwise outputs ([rows, cols/block] logical):
 *   GMLP_SCALES_COMPACT:    row-major [M][cols/block].
 *   GMLP_SCALES_GEMM_TILED: what the tensor-core MMA reads.  Each group's rows
 *     are cut into 128-row tiles counted from the group's first row (the last
 *     tile padded); group g's tiles are numbered from T_g = sum_{h<g}
 *     ceil(m_h/128).  A tile's scale columns are cut into runs of 4; every
 *     (tile, run) pair is a 512-byte block at byte ((T_g + t) * (cols/block/4)
 *     + run) * 512, and the scale of tile row r, run column j sits at
 *     (r % 32) * 16 + (r / 32) * 4 + j inside it.  Padding rows' bytes are
 *     unspecified.  Buffer size: gmlp_tiled_scales_bytes().  cols/block must be
 *     a multiple of 4.
 * Columnwise NVFP4 output (per group, groups concatenated in order): codes
 *   [cols][Mpad_g/2] and scales [cols][Mpad_g/16], Mpad_g = 16*ceil(m_g/16).
 * Columnwise MXFP8 output (the weight-gradient GEMM operand): chunk-major
 *   codes [T/128][cols][128], T = gmlp_colwise_tokens(M, G) = 128 (ceil(M/128)
 *   + G); group g's tokens, cut into 128-token chunks from its first token,
 *   are chunks c_g .. c_g + ceil(m_g/128) - 1 with c_g = sum_{h<g}
 *   ceil(m_h/128); chunk c holds, for every column i, the 128 codes of its
 *   tokens at byte (c * cols + i) * 128 (zero codes past the group's end;
 *   chunks past the last are not written); one E8M0 scale per 32 tokens, in
 *   the GEMM_TILED form of a
 *   [cols]-row operand with T/32 scales per row: the 512-byte block of column
 *   tile r (128 columns) and chunk c at byte (r * (T/128) + c) * 512, the scale
 *   of column 128 r + i, block j of the chunk at (i % 32) * 16 + (i / 32) * 4 + j.
 *   Scales buffer: cols * T / 32 bytes.
 */
#ifndef GMLP_H_
#define GMLP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GMLP_API __attribute__((visibility("default")))
#else
#define GMLP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
struct CUevent_st;
typedef struct CUstream_st* gmlp_stream; /* a cudaStream_t; NULL = legacy default stream */
typedef struct CUevent_st* gmlp_event;   /* a cudaEvent_t */

typedef enum gmlp_status {
  GMLP_OK = 0,
  GMLP_ERR_INVALID_ARG = 1,        /* NULL or misaligned pointer, bad enum value */
  GMLP_ERR_INVALID_DIMS = 2,       /* a size outside the supported range (see each call) */
  GMLP_ERR_UNSUPPORTED_RECIPE = 3, /* format / option combination this path does not have */
  GMLP_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
  GMLP_ERR_WORKSPACE = 5,          /* workspace NULL or smaller than the size query returns */
  GMLP_ERR_CUDA = 6,               /* a CUDA runtime / driver call failed (see gmlp_last_error) */
  GMLP_ERR_DEVICE_TIMEOUT = 7,     /* a kernel gave up a bounded wait (device status word) */
  GMLP_ERR_DEVICE_BOUNDS = 8       /* split_sizes negative or summing past M (device status word) */
} gmlp_status;

typedef enum gmlp_format { GMLP_MXFP8 = 0, GMLP_NVFP4 = 1 } gmlp_format;
/* GMLP_ACT_TANH_SRELU: the SReLU soft clamp of PR #3837 (Changes, ScaledTanhSReLU
 * with tanh_clamp_scale c); the pages give no formula, the reading here is the
 * soft clamp of the SReLU output at c: c * tanh(max(h,0)^2 / c).  c comes in
 * gmlp_fwd_aux.tanh_clamp_scale. */
typedef enum gmlp_act { GMLP_ACT_SWIGLU = 0, GMLP_ACT_SRELU = 1, GMLP_ACT_TANH_SRELU = 2 } gmlp_act;
typedef enum gmlp_scale_layout {
  GMLP_SCALES_COMPACT = 0,
  GMLP_SCALES_GEMM_TILED = 1,
  GMLP_SCALES_GEMM_TILED_X4 = 2 /* NVFP4 weights only: see gmlp_replicate_weight_scales */
} gmlp_scale_layout;

/* Quantisation recipe (PR #3631 Changes, the recipe preconditions; PR #3837,
 * rht_sign_mask).  MXFP8 always uses E4M3 (E5M2 gradients are not a forward
 * concern); NVFP4 may run with or without the RHT on its columnwise output. */
typedef struct gmlp_recipe {
  int32_t format;         /* gmlp_format */
  int32_t use_rht;        /* NVFP4 columnwise output: apply the 16-point RHT (0/1) */
  uint32_t rht_sign_mask; /* low 16 bits: bit i set negates element i of each chunk */
  int32_t scale_layout;   /* gmlp_scale_layout of rowwise scales */
} gmlp_recipe;

/* A quantised tensor: two caller-owned device buffers. */
typedef struct gmlp_qtensor {
  uint8_t* codes;
  uint8_t* scales;
} gmlp_qtensor;

/* T of the columnwise MXFP8 layout: 128 (ceil(M / 128) + G) (0 if M < 0 or G < 1). */
GMLP_API int64_t gmlp_colwise_tokens(int64_t M, int32_t G);

/* Bytes of a GEMM_TILED scale buffer for M rows in G groups with `nscale`
 * scale columns per row (cols/32 for MXFP8, cols/16 for NVFP4). */
GMLP_API size_t gmlp_tiled_scales_bytes(int64_t M, int32_t G, int64_t nscale);

/* Layout queries (host only: no CUDA call, no device memory, callable without a
 * GPU).  The machine-readable form of the two swizzled layouts described at the
 * top of this file, so that a caller can de-swizzle scales and codes without
 * re-deriving them.  split_sizes_host: host int64 [G], each >= 0; M is their
 * sum.
 *
 * gmlp_query_layout(GMLP_LAYOUT_TILED_SCALE, ...): byte offset, inside a
 *   GEMM_TILED scale buffer with `ncols` scale columns per row (a multiple of
 *   4), of the scale of row `row` (0 <= row < M), scale column `col`.
 * gmlp_query_layout(GMLP_LAYOUT_COLWISE_CODE, ...): byte offset, inside a
 *   columnwise MXFP8 code buffer of an [M, ncols] tensor, of the code of token
 *   `row`, column `col`.
 * gmlp_query_layout(GMLP_LAYOUT_COLWISE_SCALE, ...): byte offset, inside that
 *   tensor's columnwise scale buffer, of the E8M0 scale of the 32-token block
 *   holding token `row`, column `col` (ncols a multiple of 128).
 * Returns -1 for an unknown kind, a NULL split_sizes_host with G > 0, a
 * negative size, or row / col out of range. */
typedef enum gmlp_layout_kind {
  GMLP_LAYOUT_TILED_SCALE = 0,
  GMLP_LAYOUT_COLWISE_CODE = 1,
  GMLP_LAYOUT_COLWISE_SCALE = 2
} gmlp_layout_kind;
GMLP_API int64_t gmlp_query_layout(int32_t kind, const int64_t* split_sizes_host, int32_t G, int64_t ncols,
                                   int64_t row, int64_t col);

/* gmlp_group_hadamard_amax -- nvfp4_group_hadamard_amax (PR #3837, Changes:
 * the binding exposes the group Hadamard-amax pass on its own; the sign-mask
 * fix makes the mask part of the post-RHT amax).  One read-only pass over a
 * token-sorted bf16 x [M, K]:
 *   amax_pre[g]  = max |x| over group g's rows,
 *   amax_post[g] = max |RHT(chunk)| over all columns and 16-row chunks of group g.
 * amax_pre, amax_post: device float [G], overwritten (0 for an empty group).
 * Limits: 1 <= G <= 512, K % 128 == 0, M >= 0 (M == 0 writes zeros). */
GMLP_API gmlp_status gmlp_group_hadamard_amax(const uint16_t* x, int64_t M, int64_t K,
                                     const int64_t* split_sizes, int32_t G,
                                     uint32_t rht_sign_mask, float* amax_pre, float* amax_post,
                                     gmlp_stream stream);

/* gmlp_group_quantize_with_amax -- nvfp4_group_quantize_with_amax (PR #3837,
 * Changes: the backward re-quantisation reuses the forward amaxes, so this call
 * is the cast alone, with the amaxes the caller supplies).
 *   row_out (nullable): rowwise codes [M][K] (MXFP8) / [M][K/2] (NVFP4) and
 *     scales in recipe->scale_layout.  NVFP4 rowwise uses S_g from amax_pre[g].
 *   col_out (nullable, NVFP4 only): columnwise codes/scales (layout above) of
 *     the RHT-transformed chunks with S_g from amax_post[g] when
 *     recipe->use_rht, else of the plain chunks with S_g from amax_pre[g].
 *   amax_pre / amax_post: device float [G] (NVFP4; ignored for MXFP8).
 *   col_out with MXFP8: the columnwise MXFP8 layout above (no amax needed).
 * Limits: 1 <= G <= 512, K % 128 == 0.  At least one of row_out / col_out. */
GMLP_API gmlp_status gmlp_group_quantize_with_amax(const uint16_t* x, int64_t M, int64_t K,
                                          const int64_t* split_sizes, int32_t G,
                                          const gmlp_recipe* recipe, const float* amax_pre,
                                          const float* amax_post, const gmlp_qtensor* row_out,
                                          const gmlp_qtensor* col_out, gmlp_stream stream);

/* gmlp_group_quantize -- the generic group quantize (PR #3837, Description:
 * the fc2-input group quantize, row- and/or column-wise, with the split sizes
 * kept on the device; PR #3631 recipe checks).
 * MXFP8: one pass, amax_pre/amax_post unused (may be NULL).
 * NVFP4: first the per-group amax (the Hadamard-amax pass when col_out and
 * use_rht, else max |x| only), written to amax_pre [G] (and amax_post [G]
 * when that pass runs; amax_post may be NULL otherwise), then the cast as in
 * gmlp_group_quantize_with_amax. */
GMLP_API gmlp_status gmlp_group_quantize(const uint16_t* x, int64_t M, int64_t K,
                                const int64_t* split_sizes, int32_t G, const gmlp_recipe* recipe,
                                const gmlp_qtensor* row_out, const gmlp_qtensor* col_out,
                                float* amax_pre, float* amax_post, gmlp_stream stream);

/* gmlp_prepare_weights_discrete -- as gmlp_prepare_weights, but expert g's
 * bf16 weight [rows][cols] is at W_experts[g] (a host array of G device
 * pointers, each 16-byte aligned; PR #2769 discusses discrete per-expert
 * weights next to the single grouped weight).  The outputs are the same
 * stacked codes, GEMM_TILED scales, amax and global_scale, so the forward
 * reads either alike.  One quantisation launch per expert (plus one amax
 * launch for NVFP4). */
GMLP_API gmlp_status gmlp_prepare_weights_discrete(const uint16_t* const* W_experts, int32_t G, int64_t rows,
                                                   int64_t cols, int32_t swiglu_interleave, int32_t format,
                                                   uint8_t* codes, uint8_t* scales, float* global_scale,
                                                   float* amax, gmlp_stream stream);

/* gmlp_replicate_weight_scales -- GEMM_TILED_X4 copy of NVFP4 weight scales
 * (no counterpart on the pages: a layout for this GEMM).  `tiled` holds the
 * GEMM_TILED scales of G experts of `rows` rows (from gmlp_prepare_weights,
 * cols/16 scale columns, so runs of 4 columns R = cols/64 and stages of 4 runs
 * KB = cols/256).  For tile pair P (tiles 2P, 2P+1 of the stacked experts),
 * stage kb < KB and run k < 4, `out` holds at byte ((P * KB + kb) * 4 + k) *
 * 4096 the 512-byte block (tile 2P, run 4kb+k) four times, then the block
 * (tile 2P+1, run 4kb+k) four times: the image the GEMM copies into tensor
 * memory with one 128-row copy per MMA instead of two.  out: 4 * G * rows *
 * (cols / 16) bytes, device, 16-byte aligned; neither buffer is kept.  Limits: rows % 256 == 0, cols % 256 == 0.
 * gmlp_forward reads it when a weight's scale_layout is GEMM_TILED_X4 (in both
 * GEMM modes). */
GMLP_API gmlp_status gmlp_replicate_weight_scales(const uint8_t* tiled, int32_t G, int64_t rows, int64_t cols,
                                                  uint8_t* out, gmlp_stream stream);

/* Quantised stacked expert weights (PR #2769: single grouped weight, the
 * b_tensor of the FC1 / FC2 kernels).  Produced by gmlp_prepare_weights. */
typedef struct gmlp_qweight {
  const uint8_t* codes;       /* [G][rows][cols] (MXFP8) / [G][rows][cols/2] (NVFP4) */
  const uint8_t* scales;      /* GEMM_TILED, the G experts as G groups of `rows` rows */
  const float* global_scale;  /* NVFP4: [G] per-expert S; NULL for MXFP8 */
  int64_t rows;               /* output features of the GEMM (fc1: 2N or N; fc2: K) */
  int64_t cols;               /* contraction features (fc1: K; fc2: N) */
  int32_t G;
  int32_t format;             /* gmlp_format */
  int32_t swiglu_interleaved; /* 1: rows hold the SwiGLU gate/up interleave below */
  int32_t scale_layout;       /* layout of `scales`: 0 or GMLP_SCALES_GEMM_TILED, or (NVFP4)
                                 GMLP_SCALES_GEMM_TILED_X4 from gmlp_replicate_weight_scales */
  const uint16_t* bias;       /* optional bf16 [G][rows] in logical row order (fc1 SwiGLU: gate rows
                                 [0,N) then up rows [N,2N), whatever the interleave of `codes`); the
                                 GEMM adds it to the FP32 accumulator (after the NVFP4 1/(S_a S_b)
                                 factor) before the bf16 rounding (PR #2769: the FC1 kernel takes a
                                 bias); 16-byte aligned; NULL = none */
} gmlp_qweight;

/* gmlp_prepare_weights -- per-expert quantisation of stacked bf16 weights W
 * [G][rows][cols] along cols (done once per weight version, off the forward's
 * timed path).  NVFP4 uses one global scale per expert from that expert's
 * amax, written to amax [G] and global_scale [G] (device; NULL for MXFP8).
 * swiglu_interleave = 1 (fc1 of SwiGLU, rows = 2N with gate rows [0,N) and up
 * rows [N,2N)) stores the rows in the order the fused epilogue wants: output
 * row p of an expert holds logical row 32c + i (gate) for p = 64c + i and
 * N + 32c + i (up) for p = 64c + 32 + i, i < 32.
 * codes: [G][rows][cols or cols/2]; scales: gmlp_tiled_scales_bytes(G*rows, G,
 * cols/block) bytes.  Limits: rows % 128 == 0, cols % 128 == 0 (NVFP4: % 256),
 * swiglu_interleave needs rows % 64 == 0. */
GMLP_API gmlp_status gmlp_prepare_weights(const uint16_t* W, int32_t G, int64_t rows, int64_t cols,
                                 int32_t swiglu_interleave, int32_t format, uint8_t* codes,
                                 uint8_t* scales, float* global_scale, float* amax,
                                 gmlp_stream stream);

/* Optional extras of gmlp_forward (every field nullable / zero). */
typedef struct gmlp_fwd_aux {
  uint8_t* fc2x_codes;     /* out: fc2 input codes [M][N] (MXFP8) / [M][N/2] (NVFP4) */
  uint8_t* fc2x_scales;    /* out: fc2 input scales, GEMM_TILED */
  uint16_t* fc2x_bf16;     /* out, NVFP4: bf16 fc2_x [M][N] */
  float* fc2x_amax_pre;    /* out, NVFP4: [G] per-group max |fc2_x| */
  float* fc2x_amax_post;   /* out, NVFP4: [G] per-group post-RHT amax of fc2_x */
  gmlp_event* stage_events; /* recorded on `stream` after each kernel of the call */
  int32_t n_stage_events;   /* MXFP8: 3 (x quant, fc1, fc2); NVFP4: 5 (x amax, x quant, fc1, fc2_x quant, fc2) */
  int32_t gemm_mode;        /* 0: one CTA per 128 x 256 tile (default); 2: CTA pairs on 256 x 256 tiles
                               (cta_group::2 MMA, each CTA loading half of the B tile) */
  /* out, NVFP4, optional (both or neither): columnwise NVFP4 of fc2_x, the
   * wgrad operand of a training step that does not recompute fc2_x (PR #3837
   * Changes: columnwise data is requested only when the backward will not
   * rebuild the tensor).  16-row column chunks per group, RHT with the
   * recipe's sign mask when recipe->use_rht, global scale from the fused
   * post-RHT (or, without RHT, pre-RHT) amax; layout as the columnwise output
   * of gmlp_group_quantize_with_amax: per group codes [N][Mpad_g/2] and
   * scales [N][Mpad_g/16], Mpad_g = 16 * ceil(m_g / 16), groups in order.
   * N * (M + 16 * G) / 2 and N * (M + 16 * G) / 16 bytes hold any split.  The
   * same pass writes fc2's rowwise operand. */
  uint8_t* fc2x_col_codes;
  uint8_t* fc2x_col_scales;
  float tanh_clamp_scale;  /* GMLP_ACT_TANH_SRELU: the soft-clamp scale c (> 0, finite); aux is then required */
  /* out, optional: the activation input h = bf16(fc1 accumulator) [M][N1] in
   * logical column order (SwiGLU: gate columns [0,N), up [N,2N)), the tensor
   * the backward's dGLU step reads (PR #2769 sequence diagram: c_tensor,
   * swiglu_in).  32-byte aligned. */
  uint16_t* fc1_pre_act;
} gmlp_fwd_aux;

/* Workspace bytes gmlp_forward needs for these sizes (x and fc2_x codes and
 * scales, per-group amaxes and scales). */
GMLP_API size_t gmlp_forward_workspace_size(int64_t M, int64_t K, int64_t N, int32_t G, int32_t act,
                                   const gmlp_recipe* recipe);

/* gmlp_forward -- the fused grouped-MLP forward (PR #2769 sequence diagram,
 * forward pass; PR #3837 flowchart):
 *   1. x [M,K] bf16 -> rowwise MXFP8 / NVFP4 (per-group amax) codes + scales;
 *   2. fc1 per group g: H = dq(xq_g) dq(W1q_g)^T (FP32 accumulate; NVFP4 times
 *      1/(S_x,g S_w1,g));
 *   3. h = bf16(H); act = SwiGLU (silu(gate)*up), SReLU (max(h,0)^2) or
 *      tanh-SReLU (c * tanh(max(h,0)^2 / c));
 *      fc2_x = bf16(act * probs[t]) (probs NULL = 1);
 *   4. MXFP8: fc2_x is quantised inside the fc1 epilogue and never stored in
 *      bf16.  NVFP4: the epilogue stores bf16 fc2_x and the per-group
 *      (pre-RHT, post-RHT) amax, then fc2_x is cast with that amax;
 *   5. fc2 per group: y_g = bf16(dq(fc2xq_g) dq(W2q_g)^T) [M,K] row-major.
 * W1: rows 2N (SwiGLU, interleaved) or N (SReLU), cols K; W2: rows K, cols N;
 * both with recipe->format.  y: device bf16 [M][K], rows of empty groups and
 * rows past sum(split_sizes) untouched.
 * Limits: 1 <= G <= 512, K % 256 == 0, N % 128 == 0 (SReLU or NVFP4: N % 256
 * == 0), recipe->scale_layout is ignored (the GEMMs read GEMM_TILED).
 * workspace: >= gmlp_forward_workspace_size() bytes of device memory. */
GMLP_API gmlp_status gmlp_forward(const uint16_t* x, int64_t M, int64_t K, int64_t N,
                         const int64_t* split_sizes, int32_t G, const gmlp_qweight* W1,
                         const gmlp_qweight* W2, const float* probs, int32_t act,
                         const gmlp_recipe* recipe, uint16_t* y, const gmlp_fwd_aux* aux,
                         void* workspace, size_t workspace_bytes, gmlp_stream stream);

/* gmlp_forward_noalloc -- gmlp_forward without a caller workspace.  The
 * pages have no counterpart: this is an addition for callers that cannot
 * allocate device memory themselves -- for example code running inside a
 * host framework that owns every device allocation through its own fixed
 * pool, real-time loops that must not pay the implicit device synchronisation
 * of cudaMalloc/cudaFree, or bindings that have no device allocator at all.
 * The scratch is a static device array inside the library, 64 MiB, which
 * every GPU that loads the library keeps reserved until the process exits;
 * sizes whose gmlp_forward_workspace_size() exceeds it are rejected with
 * GMLP_ERR_WORKSPACE before anything is launched.  The call allocates
 * nothing: the caller still provides x, y, the weights and the aux outputs.
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * The address is kept for the life of the process: after cudaDeviceReset (or
 * anything else that destroys the device's primary context) it is stale, so
 * do not call the library on that device again in that process.
 * All calls share the one array and it keeps the previous call's contents
 * (the forward zeroes what it accumulates into), so calls whose work overlaps
 * on the GPU -- on different streams, or from different threads -- race; keep
 * them ordered on one stream.  Arguments, limits and results are those of
 * gmlp_forward. */
GMLP_API gmlp_status gmlp_forward_noalloc(const uint16_t* x, int64_t M, int64_t K, int64_t N,
                                          const int64_t* split_sizes, int32_t G, const gmlp_qweight* W1,
                                          const gmlp_qweight* W2, const float* probs, int32_t act,
                                          const gmlp_recipe* recipe, uint16_t* y, const gmlp_fwd_aux* aux,
                                          gmlp_stream stream);

/* gmlp_fc2x_recompute -- the fc2 input rebuilt from the saved activation
 * input, for a backward that recomputes fc2_x instead of keeping it (PR #3837,
 * Description and Changes: with activation recompute the backward regenerates
 * fc2_x, and the column-wise NVFP4 cast of it reuses the forward's amaxes
 * through gmlp_group_quantize_with_amax; recompute on and off give bitwise
 * equal results).
 *   fc2x[t, n] = bf16(act(h[t, :])[n] * probs[t])  (probs NULL = 1)
 * with exactly the arithmetic of gmlp_forward's fc1 epilogue (step 3 there),
 * so it equals the forward's fc2_x bit for bit.
 * pre_act: device bf16 [M][N1], the forward's gmlp_fwd_aux.fc1_pre_act (N1 =
 * 2N for SwiGLU, gate columns then up columns; N otherwise), 32-byte aligned;
 * probs: device float [M] or NULL; fc2x: device bf16 [M][N] out, 32-byte
 * aligned.  act: SWIGLU, SRELU or TANH_SRELU (tanh_clamp_scale > 0, finite;
 * ignored otherwise).  Limits: N % 16 == 0, N <= 2^20, 0 <= M < 2^31. */
GMLP_API gmlp_status gmlp_fc2x_recompute(const uint16_t* pre_act, const float* probs, int64_t M, int64_t N,
                                         int32_t act, float tanh_clamp_scale, uint16_t* fc2x, gmlp_stream stream);

/* Synchronises `stream`, then reads and clears the device status word the
 * kernels set on a bounded-wait timeout or inconsistent split sizes. */
GMLP_API gmlp_status gmlp_check_device_status(gmlp_stream stream);

/* Workspace bytes gmlp_backward_dgrad needs (dy and fc1_dy codes and scales). */
GMLP_API size_t gmlp_backward_workspace_size(int64_t M, int64_t K, int64_t N, int32_t G, int32_t act);

/* gmlp_backward_dgrad -- the data-gradient half of the fused grouped-MLP
 * backward, MXFP8 (PR #2769 sequence diagram, backward pass: "FC2 dGLU
 * kernel" then "FC1 dGrad kernel"; the weight gradients are not computed):
 *   1. dy [M,K] bf16 -> rowwise MXFP8 (1x32 blocks along K);
 *   2. per expert g: dfc2x = bf16(dq(dy_g) dq(W2t_g)^T) [m_g, N] (W2t = W2^T,
 *      [N][K] per expert, quantised along K);
 *   3. with the forward's activation input h (pre_act, gmlp_fwd_aux.fc1_pre_act)
 *      and prob p: SwiGLU (g = h[:, :N], u = h[:, N:]): dg = dfc2x p u silu'(g),
 *      du = dfc2x p silu(g); SReLU: dh = dfc2x p 2 max(h,0); fc1_dy =
 *      bf16(dg | du) or bf16(dh) [M, N1], quantised to MXFP8 rowwise (codes and
 *      GEMM_TILED scales to fc1_dy_codes / fc1_dy_scales when given; the bf16
 *      values to fc1_dy_bf16 [M, N1] when given, 32-byte aligned: the operand
 *      gmlp_backward_wgrad takes);
 *      dprob[t] = sum_n dfc2x[t,n] act(h)[t,n] (zeroed, then accumulated);
 *   4. dx = bf16(dq(fc1_dy_g) dq(W1t_g)^T) [m_g, K] (W1t = W1^T in logical
 *      gate/up order, [K][N1] per expert, quantised along N1).
 * W2t / W1t come from gmlp_prepare_weights on the transposed bf16 weights
 * (no interleave).  probs NULL = 1; dprob NULL skips it.  act: SWIGLU or SRELU.
 * stage_events (n_stage_events of them, at most 3, NULL when 0) are recorded
 * on `stream` after the dy quantise, the dGLU GEMM and the dgrad GEMM.
 * Limits: K % 256 == 0, N % 256 == 0. */
GMLP_API gmlp_status gmlp_backward_dgrad(const uint16_t* dy, int64_t M, int64_t K, int64_t N,
                                         const int64_t* split_sizes, int32_t G, const gmlp_qweight* W2t,
                                         const gmlp_qweight* W1t, const uint16_t* pre_act, const float* probs,
                                         int32_t act, const gmlp_recipe* recipe, uint16_t* dx, float* dprob,
                                         uint8_t* fc1_dy_codes, uint8_t* fc1_dy_scales, uint16_t* fc1_dy_bf16,
                                         void* workspace, size_t workspace_bytes, gmlp_event* stage_events,
                                         int32_t n_stage_events, gmlp_stream stream);

/* Workspace bytes gmlp_backward_wgrad needs: four columnwise MXFP8 operands
 * of T = 128 (ceil(M / 128) + G) padded tokens (about (2K + N + N1) T bytes). */
GMLP_API size_t gmlp_backward_wgrad_workspace_size(int64_t M, int64_t K, int64_t N, int32_t G, int32_t act);

/* gmlp_backward_wgrad -- the weight-gradient half of the fused grouped-MLP
 * backward, MXFP8 (PR #2769 sequence diagram, backward pass: "wgrad via
 * general_grouped_gemm" beside the dGLU and dGrad kernels, on columnwise
 * MXFP8 operands):
 *   colq(A) = per expert g, A_g^T zero-padded to 128 ceil(m_g / 128) tokens and
 *             quantised to MXFP8 in 1x32 blocks along the tokens (counted from
 *             the expert's first token);
 *   fc2_x   = bf16(act(h) p), rebuilt from pre_act exactly as the forward's
 *             fc1 epilogue computes it;
 *   dW2_g   = dq(colq(dy_g)) dq(colq(fc2_x_g))^T      [K, N]  (FP32, per expert)
 *   dW1_g   = dq(colq(fc1_dy_g)) dq(colq(x_g))^T      [N1, K] (logical gate/up order)
 *   dbias2_g = sum over g's tokens of dy [K];  dbias1_g = sum of fc1_dy [N1].
 * x [M,K] (the forward input), dy [M,K], fc1_dy [M,N1] (gmlp_backward_dgrad's
 * fc1_dy_bf16) bf16, 16-byte aligned; pre_act [M,N1] (gmlp_fwd_aux.fc1_pre_act)
 * 32-byte aligned; probs [M] or NULL (= 1).  Outputs on the device, FP32:
 * dW1 [G][N1][K] and dW2 [G][K][N] (32-byte aligned), dbias1 [G][N1],
 * dbias2 [G][K]; any of them may be NULL (its work is skipped; an input only
 * it needs may then be NULL).  accumulate = 0 overwrites them (an expert with
 * no tokens gets zeros); 1 adds the new gradients into them.  The GEMMs
 * accumulate in FP32 on the tensor cores; the bias sums are FP32 atomics.
 * stage_events (n_stage_events of them, at most 6, NULL when 0) are recorded
 * on `stream` after each launched kernel in order: the dy cast, the fc2_x
 * cast, the dW2 GEMM, the fc1_dy cast, the x cast, the dW1 GEMM (those that
 * the requested outputs need).
 * act: SWIGLU or SRELU.  Limits: K % 256 == 0, N % 256 == 0. */
GMLP_API gmlp_status gmlp_backward_wgrad(const uint16_t* x, const uint16_t* dy, const uint16_t* pre_act,
                                         const float* probs, const uint16_t* fc1_dy, int64_t M, int64_t K, int64_t N,
                                         const int64_t* split_sizes, int32_t G, int32_t act, float* dW1, float* dW2,
                                         float* dbias1, float* dbias2, int32_t accumulate, void* workspace,
                                         size_t workspace_bytes, gmlp_event* stage_events, int32_t n_stage_events,
                                         gmlp_stream stream);

/* Self-test of the device failure path (no counterpart on the pages): one
 * warp waits, through the same bounded mbarrier wait the kernels use, on a
 * barrier nothing arrives at.  After limit_ns (1 us .. 2 s) the wait gives up
 * and sets the device status word, which the next gmlp_check_device_status
 * returns as GMLP_ERR_DEVICE_TIMEOUT; the context stays usable. */
GMLP_API gmlp_status gmlp_selftest_bounded_wait(uint64_t limit_ns, gmlp_stream stream);

/* Tensor-core ceiling of the grouped GEMM's mainloop (a measurement tool; the
 * pages have no counterpart).  Launches `ctas` CTAs (<= 0: one per SM), each
 * issuing `iters` stages (1 .. 2^24) of the GEMM's block-scaled MMA mix from
 * shared memory filled once with random codes: per stage four M=128, N=256
 * MMAs (K = 32 for GMLP_MXFP8, 64 for GMLP_NVFP4) and one commit, preceded by
 * the stage's scale-factor copies to TMEM as in the GEMM: scale_copy 0 none
 * (copied once up front), 1 those for GEMM_TILED weight scales (3 for MXFP8,
 * 12 for NVFP4), 2 (NVFP4 only) those for GEMM_TILED_X4 weight scales (4 + 4),
 * 3 none: the CTA's four warps write each stage's scale factors into their
 * TMEM lane quarters with tcgen05.st while earlier stages' MMAs run.
 * Reads and writes no global memory.
 * One launch performs ctas * iters * 4 * 2 * 128 * 256 * K floating-point
 * operations; time it with events on `stream`.  A stage waits for the MMAs of
 * the stage four back (bounded; a timeout sets the device status word). */
GMLP_API gmlp_status gmlp_mma_peak(int32_t format, int32_t scale_copy, int64_t iters, int32_t ctas,
                                   gmlp_stream stream);

/* Text of the calling thread's last non-OK status ("" if none). */
GMLP_API const char* gmlp_last_error(void);

/* Library version string. */
GMLP_API const char* gmlp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GMLP_H_ */
