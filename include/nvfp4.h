/*
 * nvfp4.h -- C ABI of libnvfp4: the NVFP4 W4A4 linear layer on sm_103a.
 *
 * NVFP4 stores a matrix as 4-bit E2M1 codes, one FP8 E4M3 scale per 16
 * consecutive elements along the contraction axis, and one FP32 per-tensor
 * global scale g = amax / (6*448).  Sources:
 *   - "GLM-5.2-NVFP4" model card, "Quantization recipe" (FP4 weights, FP8
 *     block scales, block size 16);
 *   - "vroomfondel/glm-5.2-reap-504B-v2-W4A4" model card, "How it was
 *     produced" (weight_scale_2 = amax/(6*448), linear block scales, static
 *     per-tensor input_scale for the W4A4 path) and "Kernel choice" (the W4A4
 *     product of two quantized operands, scaled_fp4_mm);
 *   - "Getting GLM-5.2 NVFP4 Post-Training off the ground", sections "Going
 *     deeper", "Why can't we just transpose the one copy?" and "The bottom
 *     line" (1-D blocks along the contraction axis; the transposed operand is
 *     a separate quantization, values packed two per byte and swizzled for the
 *     tensor-core tile), "TN, NT, and what actually binds" (both operands
 *     K-major), TL;DR and "A model no kernel wanted to serve" (frozen NVFP4
 *     base with a bf16 rank-64 LoRA whose delta is added to the base output).
 *
 * Conventions shared by every entry point:
 *   - Every pointer is caller-owned DEVICE memory unless stated otherwise; the
 *     library never allocates.  Scratch space is the caller's `workspace`,
 *     sized with the matching *_workspace_bytes query, 256-byte aligned; its
 *     first 4 bytes (the device status word) must be zero before first use.
 *     Calls that share a workspace must be ordered (same stream).
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; 0 = the
 *     legacy default stream).  A returned NVFP4_OK means the arguments were
 *     valid and the kernels were launched.  Host-side validation happens
 *     before anything is launched; on error nothing is enqueued.
 *   - Kernels never trap.  Every wait inside a kernel is bounded; when a wait
 *     expires the kernel records NVFP4_ERR_TIMEOUT in the first 4 bytes of
 *     the workspace and returns.  nvfp4_read_device_status() reads it.
 *   - Matrices are row-major.  Codes: element 2j of a row in the low nibble,
 *     2j+1 in the high nibble of byte j.  Scales are E4M3 bytes.
 *   - Swizzled scale layout (what the tensor core consumes): rows padded to
 *     128, scale columns (cols/16) padded to 4; scale (r, c) at byte
 *       512*((r/128)*(pad4(cols/16)/4) + c/4) + 16*(r%32) + 4*((r%128)/32) + c%4.
 *     Linear layout: [rows][cols/16].  Pad bytes are written as 0.
 *   - Rounding: every scale operation is one IEEE fp32 operation in the
 *     order q = bamax/(6g), sb = E4M3(q), s_dec = sb*g, s_enc = 1/s_dec,
 *     v = x*s_enc; E4M3 and E2M1 round to nearest even and saturate; a block
 *     whose scale is 0 stores +0 codes; the code's sign is the sign of x.
 */
#ifndef NVFP4_H_
#define NVFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *nvfp4_stream;   /* == cudaStream_t */

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,        /* null pointer, bad enum, non-positive size (an empty
                                       operand: nothing is launched or written) */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 2,  /* size outside what the kernels take */
  NVFP4_ERR_ALIGNMENT = 3,          /* pointer or leading dimension misaligned */
  NVFP4_ERR_WORKSPACE = 4,          /* workspace missing or too small */
  NVFP4_ERR_CUDA = 5,               /* a CUDA runtime call failed */
  NVFP4_ERR_TIMEOUT = 6,            /* a bounded in-kernel wait expired */
  NVFP4_ERR_UNSUPPORTED_DEVICE = 7, /* not an sm_103 device */
  NVFP4_ERR_DEVICE_BOUNDS = 8       /* status word, builds with NVFP4_CHECKED defined only:
                                       a device-side index check failed (caller routing data
                                       out of range, or a broken internal invariant); the
                                       access was skipped.  Other builds skip or clamp such
                                       caller data without recording it. */
} nvfp4_status;

typedef enum { NVFP4_SF_LINEAR = 0, NVFP4_SF_SWIZZLED = 1 } nvfp4_sf_layout;
typedef enum { NVFP4_PACK_ROW = 1, NVFP4_PACK_COL = 2, NVFP4_PACK_BOTH = 3 } nvfp4_pack;
typedef enum { NVFP4_OUT_BF16 = 0, NVFP4_OUT_FP32 = 1 } nvfp4_out_dtype;

/* ------------------------------------------------------------------------ *
 * nvfp4_quantize -- bf16 -> NVFP4, rowwise and/or columnwise packing.
 *
 * Quantizes `batch` matrices src[b] = bf16 [rows][ld] (first `cols` columns
 * used), each with its own global scale.  Row packing (1x16 blocks along
 * cols, the forward operand) writes codes_row[b] = [rows][cols/2] and
 * sf_row[b]; column packing (16x1 blocks along rows: the quantization of the
 * transpose, the operand of the other contraction, made on demand rather than
 * kept as a second copy) writes codes_col[b] = [cols][rows/2] and sf_col[b]
 * ("Why can't we just transpose the one copy?").  Both share the global scale.
 *
 * global_scale_in: NULL = dynamic (g = amax/2688 per matrix, computed on
 *   device); else device float[batch] of static scales (the W4A4 input_scale),
 *   each finite and > 0.
 * global_scale_out: device float[batch], receives the g used (may be NULL
 *   only in static mode).
 * Per-matrix output strides are the packed sizes: nvfp4_codes_bytes(rows,
 *   cols) and nvfp4_sf_bytes(rows, cols, sf_layout) (row packing), the same
 *   with rows and cols swapped for column packing.
 * Requirements: cols % 16 == 0 (row), rows % 16 == 0 (col); ld % 8 == 0 and
 *   src 16-byte aligned; code/scale pointers 16-byte aligned.  rows, cols
 *   <= 2^31 for the row packing alone, < 2^30 when the column packing is asked
 *   for (else NVFP4_ERR_UNSUPPORTED_SHAPE).
 * Workspace: nvfp4_quantize_workspace_bytes(&args).
 * ------------------------------------------------------------------------ */
typedef struct {
  const void *src;               /* bf16 */
  int64_t batch, rows, cols, ld, batch_stride;  /* strides in elements */
  int32_t pack;                  /* nvfp4_pack */
  int32_t sf_layout;             /* nvfp4_sf_layout */
  const float *global_scale_in;  /* NULL = dynamic */
  float *global_scale_out;
  uint8_t *codes_row, *sf_row, *codes_col, *sf_col;
  void *workspace;
  size_t workspace_bytes;
  /* Optional cudaEvent_t pair (may be NULL) recorded on `stream` immediately
   * before and after the packing kernel, for timing it alone. */
  void *prof_begin, *prof_end;
} nvfp4_quant_args;

nvfp4_status nvfp4_quantize(const nvfp4_quant_args *args, nvfp4_stream stream);
size_t nvfp4_quantize_workspace_bytes(const nvfp4_quant_args *args);

/* ------------------------------------------------------------------------ *
 * nvfp4_quantize_noalloc -- nvfp4_quantize for callers that cannot allocate.
 *
 * The pages have no counterpart of this entry point; it serves callers that
 * hold no device allocator at the point of the call -- for example a plugin or
 * custom-op hook that receives only its input and output pointers and must not
 * allocate there (an allocation could synchronize the device or fall outside
 * the host framework's memory accounting), or a statically planned memory
 * layout with no slot for per-call scratch.
 *
 * Same arguments, results and requirements as nvfp4_quantize, except that
 * `workspace` and `workspace_bytes` are ignored (never read or written) and
 * nothing is allocated: the scratch the dynamic global scale needs (one 32-bit
 * word per (matrix, part), min(rows, 512) parts per matrix) lives in a 64 KiB
 * array inside the library (16384 words), present on every GPU that loads the
 * library until the process exits.  Returns NVFP4_ERR_WORKSPACE, before any
 * device work, when batch * min(rows, 512) exceeds 16384 (static global scales
 * need none).  The same array holds this entry point's own device status word
 * (in place of the workspace's first word): an expired in-kernel wait records
 * NVFP4_ERR_TIMEOUT there, and nvfp4_read_device_status(NULL, stream) reads
 * and clears it for the current device.
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  All calls
 * on a device share the array and it keeps the last call's contents (every
 * amax word a call reads is first written by that call, and the status word
 * is cleared only by reading it); calls that overlap on the GPU (different
 * streams, no ordering) race on it.
 * ------------------------------------------------------------------------ */
nvfp4_status nvfp4_quantize_noalloc(const nvfp4_quant_args *args, nvfp4_stream stream);

/* ------------------------------------------------------------------------ *
 * nvfp4_gemm -- D = (g_a*g_b) * sum_k (a_k*sfa)(b_k*sfb)  [+ LoRA]
 *
 * The W4A4 product of "Kernel choice" on tcgen05 block-scaled MMA
 * (kind::mxf4nvf4, one E4M3 scale per 16 elements), fp32 accumulation in
 * tensor memory, both operands K-major ("TN, NT, and what actually binds").
 *   A (activations) [M][K]: either packed (a_codes [M][K/2] + a_sf swizzled +
 *     a_global_scale device scalar), or bf16 a_bf16 [M][lda] quantized inside
 *     the call into the workspace (a_global_scale = static input_scale, or
 *     NULL for the dynamic amax rule); with a_bf16 the decode path for M <= 4
 *     is a CUDA-core GEMV that quantizes X on the fly (static scale only),
 *     and other products of M <= 32 rows without LoRA run with the operands
 *     swapped (the weights as the MMA's 128-row side).  The results are the
 *     same product within the tolerance of the header; which path runs
 *     depends only on M, the scale form and the LoRA.
 *   B (weights) [N][K]: b_codes [N][K/2], b_sf swizzled, b_global_scale.
 *   D [M][ldd] bf16 or fp32, written (not accumulated).
 *   LoRA (lora_a != NULL): D += (alpha/rank) * (X A^T) B^T with X = the bf16
 *     input (lora_x, or a_bf16 when given), A = lora_a bf16 [rank][K] and
 *     B = lora_b bf16 [N][rank] (the Linear-weight layouts), added in the same
 *     pass as an extra bf16 tensor-core step into the fp32 accumulator; X A^T
 *     is formed in fp32 and rounded once to bf16 after scaling.
 * Requirements: K % 32 == 0; rank % 32 == 0, 32 <= rank <= 256; ldd % 8 == 0
 *   (bf16 out) or % 4 (fp32 out); lda % 8 == 0; D and all operands 16-byte
 *   aligned.
 * Workspace: nvfp4_gemm_workspace_bytes(&args).
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t M, N, K;
  const uint8_t *a_codes, *a_sf;
  const float *a_global_scale;
  const void *a_bf16;
  int64_t lda;                   /* elements, for a_bf16 / lora_x */
  const uint8_t *b_codes, *b_sf;
  const float *b_global_scale;
  int32_t out_dtype;             /* nvfp4_out_dtype */
  void *d;
  int64_t ldd;                   /* elements */
  const void *lora_x, *lora_a, *lora_b;
  int32_t rank;
  float alpha;
  void *workspace;
  size_t workspace_bytes;
  /* Optional cudaEvent_t pair recorded around the tensor-core GEMM kernel
   * (or the GEMV kernel on the decode path). */
  void *prof_begin, *prof_end;
} nvfp4_gemm_args;

nvfp4_status nvfp4_gemm(const nvfp4_gemm_args *args, nvfp4_stream stream);
size_t nvfp4_gemm_workspace_bytes(const nvfp4_gemm_args *args);

/* ------------------------------------------------------------------------ *
 * nvfp4_grouped_gemm -- routed MoE experts, one W4A4 GEMM per expert.
 *
 * 256 routed experts with 8 per token ("GLM-5.2-NVFP4" card); a LoRA per
 * expert over the FP4 experts ("A model no kernel wanted to serve").
 * Routing, one of:
 *   expert_ids: device int32 [num_tokens*top_k], pair p = token*top_k + slot
 *     (grouped on the device: rows of expert e contiguous, ordered by p);
 *   offsets_in [E+1] + perm_in [num_tokens*top_k] (device int32, expert_ids
 *     NULL): the grouping already made -- grouped row i holds pair perm_in[i],
 *     rows offsets_in[e] .. offsets_in[e+1]-1 belong to expert e.  Device data
 *     the host cannot check: the kernels clamp counts to [0, P] cumulatively
 *     and treat pair indices outside [0, P) as padding, so inconsistent
 *     routing gives wrong rows, never an access outside the buffers.
 * Activations, one of:
 *   x_bf16 [num_tokens][K]: quantized once with one tensor-wide global scale
 *     (x_global_scale static, or NULL = dynamic amax);
 *   x_codes [num_tokens][K/2] + x_sf linear [num_tokens][K/16] (x_bf16 may
 *     be NULL without LoRA): token rows already quantized with the global
 *     scale x_global_scale (required) -- scaled_fp4_mm's input of "Kernel
 *     choice" on the "vroomfondel/glm-5.2-reap-504B-v2-W4A4" card.  The LoRA
 *     branch still reads the unquantized x_bf16.
 *   Weights of all experts stacked: w_codes [E][N][K/2] and w_sf [E][swizzled
 *     N x K/16], w_global_scale device float[E].
 *   Optional per-expert LoRA: lora_a bf16 [E][rank][K], lora_b bf16 [E][N][rank].
 *   Output d [num_tokens*top_k][N], bf16 or fp32 (out_dtype), in the grouped
 *   order; perm_out[i] = the pair index of grouped row i (required with
 *   expert_ids, optional with perm_in); expert_offsets_out (optional) [E+1].
 * Requirements: N % 256 == 0, K % 32 == 0, E <= 1024, as nvfp4_gemm otherwise;
 *   x_codes, x_sf, offsets_in, perm_in 16-byte aligned.
 * Workspace: nvfp4_grouped_workspace_bytes(&args).
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t num_tokens, top_k, num_experts, N, K;
  const int32_t *expert_ids;
  const void *x_bf16;
  const float *x_global_scale;
  const uint8_t *w_codes, *w_sf;
  const float *w_global_scale;
  const void *lora_a, *lora_b;
  int32_t rank;
  float alpha;
  void *d;
  int32_t *perm_out;
  int32_t *expert_offsets_out;
  void *workspace;
  size_t workspace_bytes;
  /* Optional cudaEvent_t pair recorded around the grouped GEMM kernel. */
  void *prof_begin, *prof_end;
  /* Pre-quantized activations (see above); NULL = quantize x_bf16. */
  const uint8_t *x_codes, *x_sf;
  /* Precomputed routing (see above); NULL = route expert_ids. */
  const int32_t *offsets_in, *perm_in;
  int32_t out_dtype;             /* nvfp4_out_dtype of d (0 = bf16) */
} nvfp4_grouped_args;

nvfp4_status nvfp4_grouped_gemm(const nvfp4_grouped_args *args, nvfp4_stream stream);
size_t nvfp4_grouped_workspace_bytes(const nvfp4_grouped_args *args);

/* ------------------------------------------------------------------------ *
 * nvfp4_lora_epilogue -- the non-fused LoRA path: Y += (alpha/rank) X A^T B^T.
 *
 * The delta applied "in the open" after the base product ("A model no kernel
 * wanted to serve"), in place on y (bf16 or fp32 [M][ldy]).  X bf16 [M][ldx],
 * A bf16 [rank][K], B bf16 [N][rank].  delta_sq_norm_out (optional, device
 * float) receives sum of the squared delta over the output, the quantity that
 * exposed a collapsing adapter on that page.
 * Requirements: as nvfp4_gemm's LoRA branch.
 * Workspace: nvfp4_lora_workspace_bytes(&args).
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t M, N, K;
  const void *x;
  int64_t ldx;
  const void *lora_a, *lora_b;
  int32_t rank;
  float alpha;
  int32_t y_dtype;               /* nvfp4_out_dtype */
  void *y;
  int64_t ldy;
  float *delta_sq_norm_out;
  void *workspace;
  size_t workspace_bytes;
} nvfp4_lora_args;

nvfp4_status nvfp4_lora_epilogue(const nvfp4_lora_args *args, nvfp4_stream stream);
size_t nvfp4_lora_workspace_bytes(const nvfp4_lora_args *args);

/* ------------------------------------------------------------------------ *
 * nvfp4_dequantize -- NVFP4 -> bf16, optionally transposed.
 *
 * The backward of the frozen QLoRA base keeps only the rowwise (forward)
 * packing and rebuilds the weight in bf16, transposed, on the fly
 * ("Getting GLM-5.2 NVFP4 Post-Training off the ground", "Why can't we just
 * transpose the one copy?" and "For a frozen QLoRA base").  Per element, in
 * IEEE fp32 with one rounding per operation:
 *     s_dec = E4M3(sb) * g;   v = E2M1(code) * s_dec;   out = bf16_rn(v)
 * (s_dec is the quantizer's decode scale).  codes [rows][cols/2] with scales
 * in `sf_layout`; transpose = 0 writes out[r][c] (ldo >= cols), 1 writes
 * out[c][r] (ldo >= rows).
 * Requirements: cols % 64 == 0; rows % 2 == 0 when transposed; codes/sf/out
 *   16-byte aligned; ldo % 8 == 0 (ldo % 2 == 0 when transposed).  No workspace.
 * ------------------------------------------------------------------------ */
typedef struct {
  const void *codes, *sf;
  int32_t sf_layout;             /* nvfp4_sf_layout */
  const float *global_scale;     /* device scalar g */
  int64_t rows, cols;            /* of the packed matrix */
  int32_t transpose;
  void *out;                     /* bf16 */
  int64_t ldo;
} nvfp4_dequant_args;

nvfp4_status nvfp4_dequantize(const nvfp4_dequant_args *args, nvfp4_stream stream);

/* ------------------------------------------------------------------------ *
 * nvfp4_dgrad -- input gradient of the frozen linear: dX = dY W.
 *
 * dY bf16 [M][N] (lddy), W the [N][K] base weight, dX [M][K] (lddx), fp32
 * accumulation.  Two ways to serve the backward's contraction over N, the two
 * the page weighs ("Why can't we just transpose the one copy?", "The bottom
 * line"):
 *   NVFP4_DGRAD_DEQUANT_BF16: w_codes/w_sf (the rowwise packing, swizzled
 *     scales) + w_global_scale are dequantized into the workspace as W^T in
 *     bf16 (nvfp4_dequantize's arithmetic), then a bf16 tensor-core GEMM.
 *   NVFP4_DGRAD_FP4_COLPACK: wcol_codes/wcol_sf = the column packing of W
 *     (nvfp4_quantize pack=COL: codes [K][N/2], swizzled scales, blocks of 16
 *     along N) with its global scale w_global_scale; dY is quantized in the
 *     call along N (dynamic amax, or dy_global_scale when given) and the
 *     product is the W4A4 FP4 GEMM (nvfp4_gemm's arithmetic).
 * Requirements: N % 64 == 0 and K % 32 == 0; dy 16-byte aligned, lddy % 8;
 *   dx 16-byte aligned, lddx % 8 (bf16) or % 4 (fp32).
 * Workspace: nvfp4_dgrad_workspace_bytes(&args).
 * ------------------------------------------------------------------------ */
typedef enum { NVFP4_DGRAD_DEQUANT_BF16 = 0, NVFP4_DGRAD_FP4_COLPACK = 1 } nvfp4_dgrad_mode;

typedef struct {
  int64_t M, N, K;
  int32_t mode;                  /* nvfp4_dgrad_mode */
  const void *dy;                /* bf16 [M][lddy] */
  int64_t lddy;
  const void *w_codes, *w_sf;    /* DEQUANT_BF16 */
  const void *wcol_codes, *wcol_sf;   /* FP4_COLPACK */
  const float *w_global_scale;
  const float *dy_global_scale;  /* FP4_COLPACK: NULL = dynamic */
  int32_t out_dtype;             /* nvfp4_out_dtype */
  void *dx;
  int64_t lddx;
  void *workspace;
  size_t workspace_bytes;
  void *prof_begin, *prof_end;   /* optional cudaEvent_t pair around the GEMM */
} nvfp4_dgrad_args;

nvfp4_status nvfp4_dgrad(const nvfp4_dgrad_args *args, nvfp4_stream stream);
size_t nvfp4_dgrad_workspace_bytes(const nvfp4_dgrad_args *args);

/* ------------------------------------------------------------------------ *
 * nvfp4_wgrad -- weight-gradient product on the FP4 datapath: dW = dY^T X.
 *
 * The contraction runs over the M tokens, so both operands need blocks of 16
 * along M: the columnwise packing of the activations and of the output
 * gradient (the layout the weight-gradient GEMM prefers, "Going deeper: why a
 * 4-bit weight needs two copies"; the per-axis blocking of "Why can't we just
 * transpose the one copy?").  dY bf16 [M][N] (lddy) and X bf16 [M][K] (ldx)
 * are quantized in the call (nvfp4_quantize pack=COL: dynamic amax, or the
 * given static scales), then dW [N][K] (lddw) = the W4A4 GEMM of the two
 * column packings (nvfp4_gemm's arithmetic).
 * Requirements: M % 32 == 0, N % 16 == 0, K % 16 == 0; dy, x 16-byte aligned
 *   with lddy, ldx % 8 == 0; dw 16-byte aligned, lddw % 8 (bf16) or % 4 (fp32).
 * Workspace: nvfp4_wgrad_workspace_bytes(&args).
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t M, N, K;
  const void *dy;                /* bf16 [M][lddy] */
  int64_t lddy;
  const void *x;                 /* bf16 [M][ldx] */
  int64_t ldx;
  const float *dy_global_scale;  /* NULL = dynamic */
  const float *x_global_scale;   /* NULL = dynamic */
  int32_t out_dtype;             /* nvfp4_out_dtype */
  void *dw;
  int64_t lddw;
  void *workspace;
  size_t workspace_bytes;
  void *prof_begin, *prof_end;   /* optional cudaEvent_t pair around the GEMM */
} nvfp4_wgrad_args;

nvfp4_status nvfp4_wgrad(const nvfp4_wgrad_args *args, nvfp4_stream stream);
size_t nvfp4_wgrad_workspace_bytes(const nvfp4_wgrad_args *args);

/* ------------------------------------------------------------------------ *
 * nvfp4_moe_down_combine -- routed-expert down-projection and combine.
 *
 * Completes the routed expert FFN after nvfp4_grouped_gemm (256 routed
 * experts, 8 per token: "GLM-5.2-NVFP4" model card; an expert's contribution
 * is weighted by its gate weight: the REAP saliency gate_weight x
 * ||expert_output|| on the "vroomfondel/glm-5.2-reap-504B-v2-W4A4" card):
 *   h      bf16 [P = num_tokens*top_k][K], the (activated) up-projection
 *          output in the expert-grouped order nvfp4_grouped_gemm produced;
 *   D[i]   = W4A4(h_i, W_e) [+ LoRA_e] for grouped row i of expert e, with h
 *          quantized once with one tensor-wide g (dynamic amax, or
 *          h_global_scale), stored as bf16;
 *   y[t]   = sum over slots j = 0..top_k-1, in order, of
 *            route_weights[t][j] * D[row of pair t*top_k + j], fp32 (one
 *            fused multiply-add per slot), rounded once to bf16.
 * perm and expert_offsets are nvfp4_grouped_gemm's perm_out and
 * expert_offsets_out.  W_e: stacked codes [E][N][K/2], swizzled scales over
 * [E*N][K/16], global scales [E]; optional LoRA A [E][rank][K], B [E][N][rank].
 * Requirements: N % 256 == 0, K % 32 == 0; as nvfp4_grouped_gemm otherwise.
 * Workspace: nvfp4_moe_down_workspace_bytes(&args).
 * ------------------------------------------------------------------------ */
typedef struct {
  int64_t num_tokens, top_k, num_experts, N, K;
  const void *h;                 /* bf16 [num_tokens*top_k][K], expert-grouped rows */
  const int32_t *perm;           /* [P]: grouped row -> token*top_k + slot */
  const int32_t *expert_offsets; /* [E+1] */
  const float *route_weights;    /* [num_tokens][top_k] */
  const float *h_global_scale;   /* NULL = dynamic */
  const void *w_codes, *w_sf;
  const float *w_global_scale;   /* [E] */
  const void *lora_a, *lora_b;   /* NULL = no LoRA */
  int32_t rank;
  float alpha;
  void *y;                       /* bf16 [num_tokens][N] */
  void *workspace;
  size_t workspace_bytes;
  void *prof_begin, *prof_end;   /* optional cudaEvent_t pair around the grouped GEMM */
} nvfp4_moe_down_args;

nvfp4_status nvfp4_moe_down_combine(const nvfp4_moe_down_args *args, nvfp4_stream stream);
size_t nvfp4_moe_down_workspace_bytes(const nvfp4_moe_down_args *args);

/* ------------------------------------------------------------------------ *
 * Size queries and status.
 * ------------------------------------------------------------------------ */
/* Bytes of packed codes of a [rows][cols] matrix: rows * cols / 2. */
size_t nvfp4_codes_bytes(int64_t rows, int64_t cols);
/* Bytes of the scales of a [rows][cols] matrix (1x16 blocks along cols). */
size_t nvfp4_sf_bytes(int64_t rows, int64_t cols, int32_t sf_layout);
/* Static text for a status code. */
const char *nvfp4_status_string(nvfp4_status s);
/* Text of the last CUDA runtime error that a library call on the calling
 * host thread met (the cause behind NVFP4_ERR_CUDA); "no error" if none.
 * Library diagnostics only: the pages have no counterpart. */
const char *nvfp4_last_cuda_error(void);
/* Synchronizes `stream`, reads (and clears) the device status word at the
 * start of `workspace` and returns it (NVFP4_OK when no wait expired).
 * workspace = NULL reads the status word of nvfp4_quantize_noalloc on the
 * current device instead. */
nvfp4_status nvfp4_read_device_status(void *workspace, nvfp4_stream stream);
/* Bound, in nanoseconds, of every in-kernel wait launched afterwards by this
 * process (default 2e9).  Returns the previous value.  0 is a test hook: each
 * GEMM kernel, and each packing kernel of nvfp4_quantize(_noalloc), launched
 * afterwards first waits on a barrier that nothing arrives at, so its expiry
 * path (status word NVFP4_ERR_TIMEOUT, drain of its own copies and MMAs, TMEM
 * freed, early return) runs without any hang. */
uint64_t nvfp4_set_wait_timeout_ns(uint64_t ns);
/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t nvfp4_version(void);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H_ */
