// internal.h -- host/device structures shared by the library's translation units.
#pragma once

#include <utility>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// ------------------------------------------------------------- quantization --
struct QuantParams {
  const __nv_bfloat16 *src;
  int64_t rows, cols, ld, bstride;    // per matrix; strides in elements
  int64_t batch;
  const float *g_in;                  // static scales [batch] or null
  float *g_out;                       // receives g [batch] (may be null)
  uint32_t *amax_part;                // [batch][nparts] magnitude bits (dynamic)
  int nparts;
  uint8_t *codes_row, *sf_row, *codes_col, *sf_col;
  int64_t codes_row_bstride, sf_row_bstride, codes_col_bstride, sf_col_bstride;
  int sf_swizzled;
  const int32_t *row_map;             // optional gather: dst row -> src row (<0: skip)
  int64_t dst_rows;                   // rows written by the row packing
  const int32_t *num_mtiles;          // optional (device, batch 1): only rows < 128 x this are in use
  // optional LoRA hand-off: T' = bf16(T * (lora_scale / (g * g_b))) per row
  const float *t_f32;                 // [t_splits][dst_rows][rank], summed in order
  int t_splits;
  __nv_bfloat16 *t_out;               // [dst_rows][rank]
  int rank;
  float lora_scale;
  const float *g_b;
  // in-kernel waits (the staged and tiled packing kernels): budget and status word
  int *status;
  uint64_t timeout_ns;
  int stall_probe;                    // test hook: first wait on a barrier nothing arrives at
};

int amax_parts_for(int64_t rows);
// The quantize path with caller-supplied amax scratch of `words` 32-bit words
// and the device status word its bounded waits write.
nvfp4_status quantize_with_amax_scratch(const nvfp4_quant_args *a, uint32_t *scratch, size_t words,
                                        int *status, cudaStream_t st);
// Device address (current device) of the status word of the workspace-free
// quantize entry point.
nvfp4_status noalloc_status_word(int **out);
cudaError_t launch_amax(const QuantParams &p, cudaStream_t st);
cudaError_t launch_quant_rows(const QuantParams &p, int num_sms, cudaStream_t st);
cudaError_t launch_quant_tiles(const QuantParams &p, int num_sms, cudaStream_t st);
// 3-D tiled map (x = innermost), no swizzle, zero fill out of bounds.
bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, const uint64_t (&dims)[3],
                 const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3]);
// NVFP4 -> bf16 (transpose: out[c][r]).
cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *sf, int sf_swz, const float *g, int64_t rows,
                           int64_t cols, int transpose, __nv_bfloat16 *out, int64_t ldo, int num_sms,
                           cudaStream_t st);
// Token-row codes + linear scales -> expert-grouped rows + swizzled scales.
// src_rows: token rows of the source (index checks); status: device status word.
cudaError_t launch_gather_packed(const uint8_t *codes_src, const uint8_t *sf_src, const int32_t *row_map,
                                 int64_t rows, const int32_t *num_mtiles, int64_t K, uint8_t *codes_dst, uint8_t *sf_dst, int num_sms,
                                 cudaStream_t st, int64_t src_rows, int *status);

// --------------------------------------------------------------------- GEMM --
// One grouped m-tile: expert, first A row (padded grouped order), valid rows,
// first output row (unpadded grouped order).
struct GroupTile {
  int32_t expert, a_row0, valid_rows, out_row0;
};

struct GemmParams {
  int64_t M, N, K;            // N = rows of one expert's B (dense: all of B)
  int num_kt;                 // 256-element K tiles of the FP4 product (0: LoRA only)
  int nk64;                   // 64-element K steps in total: ceil(K/64)
  const uint8_t *a_sf, *b_sf;
  int64_t a_sf_katoms, b_sf_katoms;   // 128x4 atoms per 128-row group
  int64_t b_sf_row_chunks;            // 128-row chunks present in b_sf (all experts)
  const float *g_a;           // scalar
  const float *g_b;           // [experts] (dense: 1)
  void *d;
  int64_t ldd;
  int out_fp32;
  int accumulate_d;           // D += result (the standalone LoRA path)
  float *sqnorm;              // optional sum of squares of the written result
  int lora_steps;             // 64-wide bf16 K steps of the LoRA up-projection
  int tiles_m, tiles_n;
  const GroupTile *gtiles;    // grouped mode: m-tile table
  const int32_t *gnum_mtiles; // grouped mode: number of m-tiles (device)
  int64_t out_rows;           // grouped mode: rows of D (index checks)
  int ksplit;                 // >1: K split into ranges, fp32 partials [ksplit][M][N]
  float *partial;
  int *status;
  uint64_t timeout_ns;
  int stall_probe;            // test hook: first wait on a barrier nothing arrives at
  int store_tma;              // pair kernel, bf16 output: D leaves through GemmMaps::d
  int pair_half_tail;         // pair kernel: a last wave of at most half the pairs runs as 256 x 128 units
};

struct GemmMaps {
  CUtensorMap a, b, t, lb;
  CUtensorMap d;   // pair kernel, bf16 output: D [M][ldd] in 32 x 32 boxes, 64-byte swizzle
  CUtensorMap bh, lbh;   // pair kernel: b and lb with 64-row boxes (the 256 x 128 units)
  bool has_d = false;
  bool has_half = false;
};

cudaError_t launch_gemm_fp4(const GemmParams &p, const GemmMaps &maps, int bn, int num_sms,
                            cudaStream_t st);
// The dense product on CTA pairs (256 x 256 tiles, tcgen05 cta_group::2):
// p.tiles_n = ceil(N / 256); maps.b and maps.lb with 128-row boxes (each CTA
// loads its half of the B tile), maps.bh and maps.lbh (has_half) the same
// with 64-row boxes; no grouped tiles, split-K or accumulation.
cudaError_t launch_gemm_fp4_pair(const GemmParams &p, const GemmMaps &maps, int num_sms, cudaStream_t st);
// The product for M <= 32 activation rows with the operands swapped (weights
// as the MMA's 128-row A side): x = activation codes in 32-row boxes of a
// buffer padded to 128 rows, w = weight codes in 128-row boxes; p.tiles_n =
// ceil(N / 128); split-K partials as k_gemm_fp4's.
cudaError_t launch_gemm_fp4_skinny(const GemmParams &p, const CUtensorMap &x, const CUtensorMap &w, int num_sms,
                                   cudaStream_t st);
// Sums split-K partials in order: D = sum_s partial[s] (bf16 or fp32 out).
cudaError_t launch_splitk_reduce(const GemmParams &p, int num_sms, cudaStream_t st);

// LoRA down-projection: T' = bf16(scale_row * X A^T), X gathered for grouped.
struct LoraDownParams {
  int64_t M, K;
  int rank;
  int num_k64;                // ceil(K/64)
  float lora_scale;           // alpha / rank
  const float *g_a;           // null: T' = bf16(scale * T); else divide by g_a * g_b[e]
  const float *g_b;
  __nv_bfloat16 *t_out;       // [rows][rank]
  int tiles_m;
  const GroupTile *gtiles;
  const int32_t *gnum_mtiles;
  const int32_t *row_map;     // grouped: padded row -> token (gather)
  const __nv_bfloat16 *x;     // grouped: token rows of X, leading dimension K
  int64_t x_rows;             // grouped: token rows of X (index checks)
  uint32_t *amax_part;        // optional: per-CTA max |x| magnitude bits of the X tiles read
  float *t_f32;               // optional: write T in fp32 (unscaled) instead of T'
  int ksplit;                 // with t_f32: K split in ranges, partials [ksplit][M][rank]
  int *status;
  uint64_t timeout_ns;
};

struct LoraDownMaps {
  CUtensorMap x, a;
};

cudaError_t launch_lora_down(const LoraDownParams &p, const LoraDownMaps &maps, int num_sms,
                             cudaStream_t st);

// -------------------------------------------------------------------- GEMV --
struct GemvParams {
  int64_t M, N, K;
  const __nv_bfloat16 *x;
  int64_t ldx;
  const float *g_x;           // static input scale
  const uint8_t *w_codes, *w_sf;
  int64_t w_sf_katoms;
  const float *g_w;
  void *d;
  int64_t ldd;
  int out_fp32;
};
// partial: fp32 [chunks][M][N] scratch when gemv_workspace_bytes() > 0.
cudaError_t launch_gemv_ws(const GemvParams &p, int num_sms, cudaStream_t st, float *partial);
size_t gemv_smem_bytes(int64_t M, int64_t K);
size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K);

// ------------------------------------------------------------------ routing --
struct RouteParams {
  const int32_t *expert_ids;
  int64_t pairs;              // tokens * top_k
  int top_k;
  int num_experts;
  int chunk;                  // pairs per chunk
  int nchunks;
  int32_t *hist;              // [nchunks][E] -> chunk bases after the scan
  int32_t *counts;            // [E]
  int32_t *offsets;           // [E+1]
  int32_t *poffsets;          // [E+1] padded (multiples of 128)
  int32_t *perm;              // [pairs]
  int32_t *row_map;           // [padded_rows_max]
  int64_t padded_rows_max;
  GroupTile *gtiles;          // [max m-tiles]
  int32_t *gnum_mtiles;
  int32_t *offsets_out;       // optional copy of offsets for the caller
  int *status;                // device status word (index checks)
};
cudaError_t launch_route(const RouteParams &p, cudaStream_t st);
// Padded grouped layout (goffsets = the clamped offsets rebuilt, poffsets,
// m-tiles, row_map -> grouped row, or -> token through perm / top_k) of rows
// that arrive already grouped with the given expert offsets.
cudaError_t launch_layout_from_offsets(const int32_t *offsets, int E, int64_t pairs, int64_t padded_rows_max,
                                       int32_t *goffsets, int32_t *poffsets, GroupTile *gtiles,
                                       int32_t *gnum_mtiles, int32_t *row_map, const int32_t *perm, int top_k,
                                       int num_sms, cudaStream_t st, int *status);
// y[t] = sum_j w[t][j] d[inverse perm (t*top_k + j)] (bf16 rows, fp32 sums).
cudaError_t launch_moe_combine(const __nv_bfloat16 *d, const int32_t *perm, int32_t *inv, const float *w,
                               int64_t tokens, int top_k, int64_t N, __nv_bfloat16 *y, int num_sms,
                               cudaStream_t st, int *status);

// ------------------------------------------------------------- tensor maps --
// Encodes a 2-D row-major tensor map; returns false on failure.
bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
                 uint64_t rows, uint64_t row_pitch_bytes, uint32_t box_inner,
                 uint32_t box_rows, CUtensorMapSwizzle sw);

// Raises `func`'s dynamic shared-memory limit on the current device to at
// least `bytes`.  The attribute is one value per device and function for the
// whole process, so the library keeps one record of it per device and
// function under a lock and only ever raises it (to the largest size asked
// for so far): a smaller request from any thread never lowers a limit that a
// concurrent larger launch relies on.
cudaError_t ensure_dynamic_smem(const void *func, size_t bytes);

// Launch with programmatic stream serialization: the kernel may begin (its
// setup) while the previous kernel in the stream drains; every kernel launched
// this way calls griddep_wait() before touching global memory.
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace nvfp4
