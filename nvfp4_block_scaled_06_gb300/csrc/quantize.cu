// quantize.cu -- bf16 -> NVFP4 (E2M1 codes, E4M3 per-16 scales, fp32 global).
//
// Operation order (one IEEE fp32 rounding per step, no contraction):
//   g = amax / 2688            (weight_scale_2 = amax/(6*448): the
//                               "vroomfondel/glm-5.2-reap-504B-v2-W4A4" card,
//                               "How it was produced")
//   q = bamax / (6*g);  sb = E4M3_rn_satfinite(q)
//   s_dec = sb * g;  s_enc = min(1/s_dec, FLT_MAX);  v = x * s_enc
//   code = sign(x) | E2M1_rn_satfinite(|v|);  sb == 0 => all codes +0
// Blocks are 16 consecutive elements along the contraction axis ("GLM-5.2-
// NVFP4" card, "Quantization recipe"); the column packing quantizes the
// transpose from the same bf16 values, with the same g ("Getting GLM-5.2
// NVFP4 Post-Training off the ground", "Why can't we just transpose the one
// copy?").  All kernels here are HBM-bound: one pass over bf16 input, packed
// codes and scales written once.
#include <cfloat>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

// ------------------------------------------------------------------ helpers --

__device__ __forceinline__ int64_t sf_swz_offset(int64_t r, int64_t c, int64_t sf_cols_pad) {
  return 512 * ((r >> 7) * (sf_cols_pad >> 2) + (c >> 2)) + 16 * (r & 31) +
         4 * ((r & 127) >> 5) + (c & 3);
}

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Max over the block; every thread must call it.  `scratch` holds >= 32 words.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t *scratch) {
  v = warp_max_u32(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  const int nw = (blockDim.x + 31) >> 5;
  v = (l < nw) ? scratch[l] : 0u;
  return warp_max_u32(v);
}

// Global scale of matrix b: static, or amax/2688 from the per-part maxima of
// |bf16| bit patterns (for non-NaN bf16, the order of |x| is the order of its
// magnitude bits, so the integer max is the exact amax).
__device__ __forceinline__ float resolve_global_scale(const QuantParams &p, int b,
                                                      uint32_t *scratch) {
  if (p.g_in) return p.g_in[b];
  uint32_t m = 0;
  for (int i = threadIdx.x; i < p.nparts; i += blockDim.x)
    m = max(m, p.amax_part[(int64_t)b * p.nparts + i]);
  m = block_max_u32(m, scratch);
  const float amax = __uint_as_float(m << 16);
  return __fdiv_rn(amax, 2688.0f);
}

struct BlockScale {
  float t6g, g;
  bool gzero;
  const float *senc;   // per-CTA table: senc[c] = min(1 / fl(E4M3(c) * g), FLT_MAX)
};

// Every thread of the block must call this (it fills a shared table of >= 128
// floats and synchronizes).  A block's encode scale depends only on its E4M3
// code, so the reciprocal of each of the 127 possible decode scales is formed
// once per CTA -- with the same IEEE operations as per block -- and looked up.
__device__ __forceinline__ BlockScale make_block_scale(float g, float *tab) {
  BlockScale s;
  s.g = g;
  s.t6g = __fmul_rn(6.0f, g);
  s.gzero = !(g > 0.0f);
  for (int c = threadIdx.x; c < 128; c += blockDim.x)
    tab[c] = fminf(__frcp_rn(__fmul_rn(e4m3_to_f32((uint32_t)c), g)), FLT_MAX);
  __syncthreads();
  s.senc = tab;
  return s;
}

// max of |x| over the two bf16 halves of each word (sign bits cleared; the bf16
// maximum of non-negative values is exact).
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Eight bf16 pairs times one fp32 scale (one IEEE rounding each), encoded as
// 16 E2M1 codes: element 2i in the low nibble of byte i.
__device__ __forceinline__ uint64_t encode16(const uint32_t (&w)[8], float senc) {
  const uint64_t ss = ((uint64_t)__float_as_uint(senc) << 32) | __float_as_uint(senc);
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint64_t x = ((uint64_t)(w[i] & 0xFFFF0000u) << 32) | (uint64_t)(w[i] << 16);
    uint64_t y;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(x), "l"(ss));
    v[2 * i] = __uint_as_float((uint32_t)y);
    v[2 * i + 1] = __uint_as_float((uint32_t)(y >> 32));
  }
  uint32_t out[2];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(out[h])
        : "f"(v[8 * h]), "f"(v[8 * h + 1]), "f"(v[8 * h + 2]), "f"(v[8 * h + 3]),
          "f"(v[8 * h + 4]), "f"(v[8 * h + 5]), "f"(v[8 * h + 6]), "f"(v[8 * h + 7]));
  return (uint64_t)out[0] | ((uint64_t)out[1] << 32);
}

// Four bf16 pairs times one fp32 scale -> 8 E2M1 codes (element 2i in the low
// nibble of byte i of the result).
__device__ __forceinline__ uint32_t encode8(const uint32_t (&w)[4], float senc) {
  const uint64_t ss = ((uint64_t)__float_as_uint(senc) << 32) | __float_as_uint(senc);
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t x = ((uint64_t)(w[i] & 0xFFFF0000u) << 32) | (uint64_t)(w[i] << 16);
    uint64_t y;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(x), "l"(ss));
    v[2 * i] = __uint_as_float((uint32_t)y);
    v[2 * i + 1] = __uint_as_float((uint32_t)(y >> 32));
  }
  uint32_t out;
  asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
      "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// Quantize 16 bf16 values held as 8 words (element 2i in the low half of w[i]).
// Returns the 8 code bytes (element 2i in the low nibble of byte i) and the
// E4M3 scale byte.
__device__ __forceinline__ uint64_t quant16(const uint32_t (&w)[8], const BlockScale &s,
                                            uint32_t &sf_out) {
  uint32_t m2 = w[0] & 0x7FFF7FFFu;
#pragma unroll
  for (int i = 1; i < 8; ++i) m2 = bmax2(m2, w[i] & 0x7FFF7FFFu);
  const uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
  const float bamax = __uint_as_float(mb << 16);
  uint32_t sb = 0;
  if (!s.gzero) sb = cvt_e4m3(__fdiv_rn(bamax, s.t6g));
  sf_out = sb;
  if (sb == 0) return 0ull;
  return encode16(w, s.senc[sb]);
}

template <bool kV8>
__device__ __forceinline__ void load16(const __nv_bfloat16 *src, uint32_t (&w)[8], uint64_t pol) {
  if (kV8) {
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
          "=r"(w[7])
        : "l"(src), "l"(pol));
  } else {
    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(src));
    const uint4 b = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}

// -------------------------------------------------------------------- amax --
// Grid (nparts, batch).  Part i of matrix b reduces rows i, i+nparts, ... and
// writes max |bf16| magnitude bits to amax_part[b*nparts + i].
template <bool kRowPairs>
__global__ void __launch_bounds__(256) k_amax_partial(QuantParams p) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  __shared__ uint32_t scratch[32];
  const int b = blockIdx.y;
  const __nv_bfloat16 *base = p.src + (int64_t)b * p.bstride;
  const int64_t vec_per_row = p.cols / 8;
  uint32_t m2 = 0;
  if (kRowPairs) {
    // one matrix: two rows at a time, up to four 16-byte vectors of each per
    // thread and step, every load of a step issued before its maxima
    // (predicated past the row's end: rows of 6144 elements are 768 vectors,
    // three per thread).  A batch of matrices takes the loop below (its own
    // instance: with the pairs' registers the 32-matrix sweep ran 8% slower):
    // its grid already has enough loads in flight.
    for (int64_t r = blockIdx.x; r < p.rows; r += 2 * (int64_t)gridDim.x) {
      const int64_t r2 = r + gridDim.x;
      const bool two = r2 < p.rows;
      const uint4 *row = reinterpret_cast<const uint4 *>(base + r * p.ld);
      const uint4 *row2 = reinterpret_cast<const uint4 *>(base + (two ? r2 : r) * p.ld);
      for (int64_t v = threadIdx.x; v < vec_per_row; v += 4 * 256) {
        uint4 a[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const bool in = v + u * 256 < vec_per_row;
          a[u] = in ? __ldg(row + v + u * 256) : make_uint4(0, 0, 0, 0);
          a[4 + u] = in && two ? __ldg(row2 + v + u * 256) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          m2 = __vmaxu2(m2, a[u].x & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, a[u].y & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, a[u].z & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, a[u].w & 0x7FFF7FFFu);
        }
      }
    }
  } else {
    for (int64_t r = blockIdx.x; r < p.rows; r += gridDim.x) {
      const uint4 *row = reinterpret_cast<const uint4 *>(base + r * p.ld);
      int64_t v = threadIdx.x;
      for (; v + 3 * 256 < vec_per_row; v += 4 * 256) {
        uint4 a[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) a[u] = __ldg(row + v + u * 256);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          m2 = __vmaxu2(m2, a[u].x & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, a[u].y & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, a[u].z & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, a[u].w & 0x7FFF7FFFu);
        }
      }
      for (; v < vec_per_row; v += 256) {
        const uint4 a = __ldg(row + v);
        m2 = __vmaxu2(m2, a.x & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, a.y & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, a.z & 0x7FFF7FFFu);
        m2 = __vmaxu2(m2, a.w & 0x7FFF7FFFu);
      }
    }
  }
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = block_max_u32(m, scratch);
  if (threadIdx.x == 0) p.amax_part[(int64_t)b * p.nparts + blockIdx.x] = m;
}

// ------------------------------------------------------------- row packing --
// One warp per destination row, one lane per 16-element block.  Grid
// (ctas, batch); rows are striped over the warps of the grid.  Destination row
// r reads source row row_map[r] (gather) or r; row_map < 0 rows are skipped.
// With the swizzled layout, rows up to pad128 and scale columns up to pad4 are
// written (zeros outside the matrix).
template <bool kV8>
__global__ void __launch_bounds__(256) k_quant_rows(QuantParams p) {
  // The wait comes first: a kernel launched after this one starts only once
  // every earlier kernel of the stream has completed, so it may read data
  // that this kernel does not write (the operand-swapped GEMM streams its
  // weights) before its own wait.
  griddep_wait();   // inputs may come from the previous kernel in the stream
  griddep_launch_dependents();
  __shared__ uint32_t scratch[32];
  __shared__ float senc_tab[128];
  const int b = blockIdx.y;
  const float g = resolve_global_scale(p, b, scratch);
  if (blockIdx.x == 0 && threadIdx.x == 0 && p.g_out) p.g_out[b] = g;
  const BlockScale s = make_block_scale(g, senc_tab);

  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t nblk = p.cols / 16;
  const int64_t sfc_pad = (nblk + 3) & ~int64_t(3);
  const int64_t rows_out = p.sf_swizzled ? ((p.dst_rows + 127) & ~int64_t(127)) : p.dst_rows;
  const __nv_bfloat16 *src = p.src + (int64_t)b * p.bstride;
  uint8_t *codes = p.codes_row + (int64_t)b * p.codes_row_bstride;
  uint8_t *sf = p.sf_row + (int64_t)b * p.sf_row_bstride;
  const int64_t row_bytes = p.cols / 2;

  const float t_scale = p.t_f32 ? __fdiv_rn(p.lora_scale, acc_scale_of(g, *p.g_b)) : 0.0f;
  // last use of the source rows: let L2 drop them first
  const uint64_t pol = l2_policy_evict_first();
  // work item = (row, chunk of 128 blocks): short rows keep every warp busy
  const int64_t nch = (sfc_pad + 127) / 128;
  for (int64_t wi = warp; wi < rows_out * nch; wi += nwarps) {
    const int64_t r = wi / nch, ch = wi - r * nch;
    int64_t sr = -1;
    if (r < p.dst_rows) sr = p.row_map ? (int64_t)p.row_map[r] : r;
    if (!NVFP4_GUARD(sr < p.rows, p.status)) sr = -1;
    if (p.row_map && sr < 0) continue;   // unmapped (padding) rows are left untouched
    if (p.t_f32 && r < p.dst_rows && ch == 0) {
      // LoRA hand-off: the down-projection's fp32 row, scaled and rounded once to bf16
      for (int j = lane; j < p.rank; j += 32) {
        float t = p.t_f32[r * p.rank + j];
        for (int k = 1; k < p.t_splits; ++k) t = __fadd_rn(t, p.t_f32[(k * p.dst_rows + r) * p.rank + j]);
        p.t_out[r * p.rank + j] = __float2bfloat16_rn(__fmul_rn(t, t_scale));
      }
    }
    const __nv_bfloat16 *srow = src + sr * p.ld;
    {
      const int64_t blk0 = ch * 128;
      uint32_t w[4][8];
      uint64_t c[4];
      uint32_t sb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t blk = blk0 + u * 32 + lane;
        if (sr >= 0 && blk < nblk) load16<kV8>(srow + blk * 16, w[u], pol);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t blk = blk0 + u * 32 + lane;
        c[u] = 0;
        sb[u] = 0;
        if (sr >= 0 && blk < nblk) c[u] = quant16(w[u], s, sb[u]);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int64_t blk = blk0 + u * 32 + lane;
        if (blk0 + u * 32 >= sfc_pad) break;
        if (sr >= 0 && blk < nblk)
          *reinterpret_cast<uint2 *>(codes + r * row_bytes + blk * 8) =
              make_uint2((uint32_t)c[u], (uint32_t)(c[u] >> 32));
        if (p.sf_swizzled) {
          uint32_t v = sb[u];
          v |= __shfl_down_sync(0xffffffffu, sb[u], 1) << 8;
          v |= __shfl_down_sync(0xffffffffu, sb[u], 2) << 16;
          v |= __shfl_down_sync(0xffffffffu, sb[u], 3) << 24;
          if ((lane & 3) == 0 && blk < sfc_pad)
            *reinterpret_cast<uint32_t *>(sf + sf_swz_offset(r, blk, sfc_pad)) = v;
        } else if (sr >= 0 && blk < nblk) {
          sf[r * nblk + blk] = (uint8_t)sb[u];
        }
      }
    }
  }
}

// ------------------------------------------------------ staged row packing --
// The row packing with the source staged through shared memory by bulk
// copies.  The work is cut into units (matrix, row, K segment of <= 2048
// elements); every warp owns a contiguous run of units and a private ring of
// `slots` shared-memory buffers, and keeps the copies of its next units in
// flight while it packs the current one (~130 KB of reads outstanding per SM
// with few registers).  Units are walked with incremental cursors (no
// integer division per unit).  A lane packs two 16-element blocks per step: 2 x 32
// bytes from shared memory, 2 x 8 code bytes and two scale bytes out.
// Same results, bit for bit, as k_quant_rows (the same per-block operations).
constexpr int kQWarps = 16;
constexpr uint64_t kQDrainNs = 200000000ull;
constexpr int64_t kQSegMax = 2048;
constexpr int kQHeaderBytes = 8704;   // barriers (<= 512 B) + per-warp 128-entry tables

struct StagedCfg {
  int64_t seg = 0;   // elements per unit (multiple of 64), last segment of a row may be shorter
  int nseg = 0, slots = 0;
  size_t smem = 0;
};

StagedCfg staged_cfg(int64_t cols) {
  StagedCfg c;
  c.nseg = (int)((cols + kQSegMax - 1) / kQSegMax);
  const int64_t per = (cols + c.nseg - 1) / c.nseg;
  c.seg = (per + 63) / 64 * 64;
  const int64_t ring = (int64_t)kQWarps * c.seg * 2;
  c.slots = (int)std::min<int64_t>(4, (224 * 1024 - kQHeaderBytes) / ring);
  c.smem = (size_t)kQHeaderBytes + (size_t)c.slots * (size_t)ring;
  return c;
}

// Global scale of matrix b computed by one warp (same operations as
// resolve_global_scale).
__device__ __forceinline__ float warp_global_scale(const QuantParams &p, int64_t b) {
  if (p.g_in) return p.g_in[b];
  uint32_t m = 0;
  for (int i = threadIdx.x & 31; i < p.nparts; i += 32) m = max(m, p.amax_part[b * p.nparts + i]);
  m = warp_max_u32(m);
  return __fdiv_rn(__uint_as_float(m << 16), 2688.0f);
}

// max(|a|, |b|) per bf16 half; the sign bits of the result are not
// meaningful (cleared by the caller).  Exact for finite inputs.
__device__ __forceinline__ uint32_t bmaxabs2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// One 16-element block held as two 16-byte halves: `a` = elements 8h..8h+7,
// `c` = the other half (h = which half `a` is).  Returns the code bytes
// (element 2i in the low nibble of byte i) and the E4M3 scale.
__device__ __forceinline__ uint2 pack_block(const uint4 a, const uint4 c, int h, float t6g, bool gzero,
                                            const float *tab, uint32_t &sb) {
  const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wc[4] = {c.x, c.y, c.z, c.w};
  const uint32_t m2 = bmaxabs2(bmaxabs2(bmaxabs2(wa[0], wa[1]), bmaxabs2(wa[2], wa[3])),
                               bmaxabs2(bmaxabs2(wc[0], wc[1]), bmaxabs2(wc[2], wc[3]))) &
                      0x7FFF7FFFu;
  const uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
  sb = gzero ? 0u : cvt_e4m3(__fdiv_rn(__uint_as_float(mb << 16), t6g));
  uint32_t lo = 0, hi = 0;
  if (sb) {
    const float senc = tab[sb];
    const uint32_t ea = encode8(wa, senc), ec = encode8(wc, senc);
    lo = h ? ec : ea;
    hi = h ? ea : ec;
  }
  return make_uint2(lo, hi);
}

__global__ void __launch_bounds__(kQWarps * 32, 1)
    k_quant_rows_staged(const QuantParams p, int64_t seg, int nseg, int slots) {
  extern __shared__ __align__(128) uint8_t qsm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t slot_bytes = seg * 2;
  uint64_t *full = reinterpret_cast<uint64_t *>(qsm) + warp * slots;
  float *tab = reinterpret_cast<float *>(qsm + 512) + warp * 128;
  const uint32_t ring = smem_u32(qsm + kQHeaderBytes) + (uint32_t)(warp * slots * slot_bytes);
  if (lane == 0) {
    for (int s = 0; s < slots; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  griddep_launch_dependents();
  griddep_wait();   // inputs of this kernel come from the previous one in the stream
  if (p.stall_probe) {
    // test hook: wait on a slot barrier before any copy is armed, so the wait
    // expires and the expiry path (status word, early return) runs
    if (lane == 0 && !mbar_wait(&full[0], 0, p.timeout_ns)) record_timeout(p.status);
    return;
  }

  int64_t rows_out = (p.sf_swizzled && !p.row_map) ? ((p.dst_rows + 127) & ~int64_t(127)) : p.dst_rows;
  // a layout whose used size is known only on the device: split the rows in
  // use evenly (the rest are never read)
  if (p.num_mtiles && p.batch == 1) rows_out = min(rows_out, (int64_t)128 * (int64_t)*p.num_mtiles);
  const int64_t per_b = rows_out * nseg, U = per_b * p.batch;
  const int64_t W = (int64_t)gridDim.x * kQWarps, gw = (int64_t)blockIdx.x * kQWarps + warp;
  // an even split: every warp gets floor(U/W) or ceil(U/W) consecutive units
  const int64_t u_begin = gw * U / W, u_end = (gw + 1) * U / W;
  const int64_t nblk = p.cols / 16, sfc_pad = (nblk + 3) & ~int64_t(3);
  const int64_t row_bytes = p.cols / 2;
  const uint64_t pol = l2_policy_evict_first();   // last use of the source rows

  // unit -> (matrix, row, segment, source row); source row < 0: nothing to copy
  auto source_row = [&](int64_t r) -> int64_t {
    if (r >= p.dst_rows) return -1;
    const int64_t sr = p.row_map ? (int64_t)p.row_map[r] : r;
    return NVFP4_GUARD(sr < p.rows, p.status) ? sr : -1;
  };
  struct Cursor {
    int64_t b, r, sg;
  };
  auto advance = [&](Cursor &c) {
    if (++c.sg == nseg) {
      c.sg = 0;
      if (++c.r == rows_out) {
        c.r = 0;
        ++c.b;
      }
    }
  };
  Cursor cur;   // the unit being packed
  cur.b = u_begin / per_b;
  cur.r = (u_begin % per_b) / nseg;
  cur.sg = u_begin % nseg;
  Cursor icur = cur;          // the next unit to copy (lane 0)
  int64_t inext = u_begin;
  uint32_t armed = 0, parity = 0;   // per slot: copy in flight / phase to wait for
  auto issue = [&](int s) {   // lane 0 only: copy unit `inext` into slot s
    if (inext >= u_end) return;
    const int64_t sr = source_row(icur.r);
    if (sr >= 0) {
      const int64_t c0 = icur.sg * seg, len = seg < p.cols - c0 ? seg : p.cols - c0;
      const uint32_t bar = smem_u32(&full[s]);
      mbar_arrive_expect_tx_u(bar, (uint32_t)(len * 2));
      bulk_load_hint_u(ring + (uint32_t)(s * slot_bytes), p.src + icur.b * p.bstride + sr * p.ld + c0,
                       (uint32_t)(len * 2), bar, pol);
      armed |= 1u << s;
    }
    ++inext;
    advance(icur);
  };
  if (lane == 0)
    for (int s = 0; s < slots; ++s) issue(s);

  int64_t cur_b = -1;
  float g = 0.0f, t6g = 0.0f, t_scale = 0.0f;
  bool gzero = true;
  int s = 0;
  // lanes alternate which 16-byte half of a block they read first, so the
  // eight lanes of each quarter-warp touch eight different bank groups
  const int h = (lane >> 2) & 1;
  for (int64_t u = u_begin; u < u_end; ++u, advance(cur)) {
    const int64_t b = cur.b, r = cur.r, sg = cur.sg;
    if (b != cur_b) {
      // this warp's block-scale table for matrix b
      g = warp_global_scale(p, b);
      t6g = __fmul_rn(6.0f, g);
      gzero = !(g > 0.0f);
      for (int c = lane; c < 128; c += 32)
        tab[c] = fminf(__frcp_rn(__fmul_rn(e4m3_to_f32((uint32_t)c), g)), FLT_MAX);
      if (p.t_f32) t_scale = __fdiv_rn(p.lora_scale, acc_scale_of(g, *p.g_b));
      __syncwarp();
      cur_b = b;
    }
    if (r == 0 && sg == 0 && lane == 0 && p.g_out) p.g_out[b] = g;   // the matrix's first unit
    const int64_t sr = source_row(r);
    const bool skip = p.row_map && sr < 0;   // unmapped (padding) rows are left untouched
    if (!skip) {
      if (sr >= 0) {
        const bool got = mbar_wait_u(smem_u32(&full[s]), (parity >> s) & 1, p.timeout_ns);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) record_timeout(p.status);
          break;
        }
        parity ^= 1u << s;
        if (lane == 0) armed &= ~(1u << s);
      }
      if (p.t_f32 && sg == 0 && r < p.dst_rows) {
        // LoRA hand-off: the down-projection's fp32 row, scaled and rounded once to bf16
        for (int j = lane; j < p.rank; j += 32) {
          float t = p.t_f32[r * p.rank + j];
          for (int k = 1; k < p.t_splits; ++k) t = __fadd_rn(t, p.t_f32[(k * p.dst_rows + r) * p.rank + j]);
          p.t_out[r * p.rank + j] = __float2bfloat16_rn(__fmul_rn(t, t_scale));
        }
      }
      const int64_t c0 = sg * seg, len = seg < p.cols - c0 ? seg : p.cols - c0;
      const int blk0 = (int)(c0 / 16), nb = (int)(len / 16);
      const int nb_sf = (p.sf_swizzled && sg == nseg - 1) ? (int)(sfc_pad - blk0) : nb;
      const bool live = sr >= 0;
      uint2 *codes = reinterpret_cast<uint2 *>(p.codes_row + b * p.codes_row_bstride + r * row_bytes) + blk0;
      // scale addresses: row part once per unit, block part in 32-bit arithmetic
      uint8_t *sfr = p.sf_row + b * p.sf_row_bstride +
                     (p.sf_swizzled ? 512 * ((r >> 7) * (sfc_pad >> 2)) + 16 * (r & 31) + 4 * ((r & 127) >> 5)
                                    : r * nblk);
      const uint32_t sbase = ring + (uint32_t)(s * slot_bytes) + 16 * h;
      const uint32_t other = h ? (uint32_t)-16 : 16u;
      for (int bi = lane; bi < nb_sf; bi += 64) {
        const int bj = bi + 32;
        const bool v0 = live && bi < nb, v1 = live && bj < nb;
        uint4 a0 = make_uint4(0, 0, 0, 0), c0v = a0, a1 = a0, c1v = a0;
        if (v0) {
          a0 = lds128(sbase + 32u * bi);
          c0v = lds128(sbase + 32u * bi + other);
        }
        if (v1) {
          a1 = lds128(sbase + 32u * bj);
          c1v = lds128(sbase + 32u * bj + other);
        }
        uint32_t sb0 = 0, sb1 = 0;
        const uint2 k0 = pack_block(a0, c0v, h, t6g, gzero || !v0, tab, sb0);
        const uint2 k1 = pack_block(a1, c1v, h, t6g, gzero || !v1, tab, sb1);
        if (v0) codes[bi] = k0;
        if (v1) codes[bj] = k1;
        if (p.sf_swizzled) {
          const int x0 = blk0 + bi, x1 = blk0 + bj;
          sfr[512 * (int64_t)(x0 >> 2) + (x0 & 3)] = (uint8_t)sb0;
          if (bj < nb_sf) sfr[512 * (int64_t)(x1 >> 2) + (x1 & 3)] = (uint8_t)sb1;
        } else {
          if (v0) sfr[blk0 + bi] = (uint8_t)sb0;
          if (v1) sfr[blk0 + bj] = (uint8_t)sb1;
        }
      }
    }
    // slot s is free again: start the copy of the unit `slots` ahead
    __syncwarp();
    if (lane == 0) issue(s);
    if (++s == slots) s = 0;
  }
  // copies still in flight (only after a timeout): wait for them before exiting
  if (lane == 0)
    for (int k = 0; k < slots; ++k)
      if (armed & (1u << k)) mbar_wait(&full[k], (parity >> k) & 1, kQDrainNs);
}

// ------------------------------------------------- tiled col (+row) packing --
// A CTA quantizes 64 x 256 tiles of one matrix (grid-stride over tiles).  The
// tiles arrive by TMA (one 3-D box per tile, rows and columns past the matrix
// zero-filled) into two shared-memory buffers, so that the next tile streams
// in while this one is packed.  Every thread ends a tile with 32 contiguous
// bytes of codes per packing (one full sector) and one word of scales:
//   row role: thread t owns row t/4 of the tile and its 64-column quarter t%4,
//     four whole 16-element blocks;
//   column role: lanes 2i and 2i+1 read the column pair (two columns per
//     32-bit word) of their warp's pair index over the upper and lower 32 rows,
//     pack two 16-row blocks of both columns, and swap one column's half, so
//     that each ends with the four blocks of one column.
// Requires rows % 16 == 0 for the column packing.
constexpr int kTR = 64, kTC = 256;
constexpr int kTileBytes = kTR * kTC * 2;
constexpr uint64_t kTileDrainNs = 200000000ull;

// quant16 with the block maximum taken by max.xorsign.abs (same magnitude).
__device__ __forceinline__ uint64_t quant16_abs(const uint32_t (&w)[8], const BlockScale &s, uint32_t &sf_out) {
  const uint32_t m2 = bmaxabs2(bmaxabs2(bmaxabs2(w[0], w[1]), bmaxabs2(w[2], w[3])),
                               bmaxabs2(bmaxabs2(w[4], w[5]), bmaxabs2(w[6], w[7]))) &
                      0x7FFF7FFFu;
  const uint32_t mb = max(m2 & 0xFFFFu, m2 >> 16);
  uint32_t sb = 0;
  if (!s.gzero) sb = cvt_e4m3(__fdiv_rn(__uint_as_float(mb << 16), s.t6g));
  sf_out = sb;
  if (sb == 0) return 0ull;
  return encode16(w, s.senc[sb]);
}

// Stores the codes of blocks 0..nvalid-1 (8 bytes each) at dst: one 32-byte
// store when all four are valid and dst is 32-byte aligned, else smaller ones.
__device__ __forceinline__ void store_blocks4(uint8_t *dst, const uint64_t (&cd)[4], int nvalid) {
  const uint32_t w[8] = {(uint32_t)cd[0], (uint32_t)(cd[0] >> 32), (uint32_t)cd[1], (uint32_t)(cd[1] >> 32),
                         (uint32_t)cd[2], (uint32_t)(cd[2] >> 32), (uint32_t)cd[3], (uint32_t)(cd[3] >> 32)};
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst);
  if (nvalid == 4 && (a & 31) == 0) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                 "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
  } else if (nvalid == 4 && (a & 15) == 0) {
    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nvalid) reinterpret_cast<uint2 *>(dst)[j] = make_uint2(w[2 * j], w[2 * j + 1]);
  }
}

// Destinations of one matrix's packings (row: [rows][cols/2] codes; column:
// [cols][rows/2]) and their scale layouts.
struct TileOut {
  uint8_t *codes_r, *sf_r, *codes_c, *sf_c;
  int32_t rows, cols, nblk_r, sfc_pad_r, nblk_c, sfc_pad_c;
  bool do_row, do_col;
};

__device__ __forceinline__ TileOut tile_out(const QuantParams &p, int64_t b) {
  TileOut o;
  o.rows = (int32_t)p.rows;
  o.cols = (int32_t)p.cols;
  o.do_row = p.codes_row != nullptr;
  o.do_col = p.codes_col != nullptr;
  o.nblk_r = o.cols / 16;
  o.sfc_pad_r = (o.nblk_r + 3) & ~3;
  o.nblk_c = o.rows / 16;
  o.sfc_pad_c = (o.nblk_c + 3) & ~3;
  o.codes_r = o.do_row ? p.codes_row + b * p.codes_row_bstride : nullptr;
  o.sf_r = o.do_row ? p.sf_row + b * p.sf_row_bstride : nullptr;
  o.codes_c = o.do_col ? p.codes_col + b * p.codes_col_bstride : nullptr;
  o.sf_c = o.do_col ? p.sf_col + b * p.sf_col_bstride : nullptr;
  return o;
}

// Both packings of one staged [kTR][kTC] bf16 tile whose first element is
// (r0, c0).  Thread t has the row role (tile row t / 4, 64-column quarter
// t % 4) and the column role (column pair t / 2, 32-row half t % 2).
__device__ __forceinline__ void pack_tile(const QuantParams &p, const BlockScale &s, const uint32_t *tile,
                                          int32_t r0, int32_t c0, const TileOut &o, int t) {
  const int32_t rows = o.rows, cols = o.cols;
  const int rr = t >> 2, qd = t & 3;          // row role: tile row, 64-column quarter
  const int cp = t >> 1, rh = t & 1;          // column role: column pair, 32-row half
  if (o.do_row) {
    const int32_t gr = r0 + rr, gq = c0 + 64 * qd;   // this thread's row and first column
    if (gr < rows) {
      // the 16-byte pairs are read in an order rotated by the quarter, so
      // that the four quarters of a row hit different bank groups: w-block
      // m holds block (m + qd) % 4 of the quarter
      uint32_t w[32];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int c = (k + 2 * qd) & 7;
        const uint4 v = *reinterpret_cast<const uint4 *>(&tile[rr * (kTC / 2) + 32 * qd + 4 * c]);
        w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
      }
      const int nvalid = min(4, (cols - gq) / 16);
      uint64_t cm[4];
      uint32_t sm[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint32_t(&wb)[8] = *reinterpret_cast<const uint32_t(*)[8]>(&w[8 * m]);
        sm[m] = 0;
        cm[m] = ((m + qd) & 3) < nvalid ? quant16_abs(wb, s, sm[m]) : 0ull;
      }
      // back to block order j = 0..3 (w-block (j - qd) % 4)
      uint64_t cd[4];
      uint32_t sbw = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int m0 = (j - qd) & 3;
        cd[j] = m0 == 0 ? cm[0] : m0 == 1 ? cm[1] : m0 == 2 ? cm[2] : cm[3];
        sbw |= (m0 == 0 ? sm[0] : m0 == 1 ? sm[1] : m0 == 2 ? sm[2] : sm[3]) << (8 * j);
      }
      store_blocks4(o.codes_r + (int64_t)gr * (cols / 2) + gq / 2, cd, nvalid);
      const int32_t blk = gq / 16;
      if (p.sf_swizzled) {
        if (blk < o.sfc_pad_r) *reinterpret_cast<uint32_t *>(o.sf_r + sf_swz_offset(gr, blk, o.sfc_pad_r)) = sbw;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nvalid) o.sf_r[(int64_t)gr * o.nblk_r + blk + j] = (uint8_t)(sbw >> (8 * j));
      }
    }
  }
  if (o.do_col) {
    // rows 32*rh .. 32*rh+31 of columns 2cp, 2cp+1: blocks 2rh, 2rh+1 of each
    uint64_t cda[2], cdb[2];
    uint32_t sba[2], sbb[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const int rb = 2 * rh + h2;               // 16-row block of the tile
      uint32_t ca[8], cb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t w0 = tile[(16 * rb + 2 * i) * (kTC / 2) + cp];
        const uint32_t w1 = tile[(16 * rb + 2 * i + 1) * (kTC / 2) + cp];
        ca[i] = __byte_perm(w0, w1, 0x5410);   // column 2cp: rows 2i, 2i+1
        cb[i] = __byte_perm(w0, w1, 0x7632);   // column 2cp+1
      }
      const bool bin = r0 + 16 * rb < rows;
      sba[h2] = sbb[h2] = 0;
      cda[h2] = (bin && c0 + 2 * cp < cols) ? quant16_abs(ca, s, sba[h2]) : 0ull;
      cdb[h2] = (bin && c0 + 2 * cp + 1 < cols) ? quant16_abs(cb, s, sbb[h2]) : 0ull;
    }
    // lane rh = 0 keeps column 2cp and receives its blocks 2, 3; lane rh = 1
    // keeps column 2cp+1 and receives its blocks 0, 1
    uint64_t keep[2], give[2];
    uint32_t skeep[2], sgive[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      keep[h2] = rh ? cdb[h2] : cda[h2];
      give[h2] = rh ? cda[h2] : cdb[h2];
      skeep[h2] = rh ? sbb[h2] : sba[h2];
      sgive[h2] = rh ? sba[h2] : sbb[h2];
    }
    uint64_t got2[2];
    uint32_t sgot[2];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2) {
      const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)give[h2], 1);
      const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(give[h2] >> 32), 1);
      got2[h2] = ((uint64_t)hi << 32) | lo;
      sgot[h2] = __shfl_xor_sync(0xffffffffu, sgive[h2], 1);
    }
    const int32_t oc = c0 + 2 * cp + rh;        // this thread's output row (= input column)
    if (oc < cols) {
      const uint64_t cd[4] = {rh ? got2[0] : keep[0], rh ? got2[1] : keep[1], rh ? keep[0] : got2[0],
                              rh ? keep[1] : got2[1]};
      const uint32_t sbw = (rh ? sgot[0] : skeep[0]) | ((rh ? sgot[1] : skeep[1]) << 8) |
                           ((rh ? skeep[0] : sgot[0]) << 16) | ((rh ? skeep[1] : sgot[1]) << 24);
      const int nvalid = min(4, (rows - r0) / 16);
      store_blocks4(o.codes_c + (int64_t)oc * (rows / 2) + r0 / 2, cd, nvalid);
      const int32_t blk = r0 / 16;              // first of the tile's 4 column blocks
      if (p.sf_swizzled) {
        if (blk < o.sfc_pad_c) *reinterpret_cast<uint32_t *>(o.sf_c + sf_swz_offset(oc, blk, o.sfc_pad_c)) = sbw;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j < nvalid) o.sf_c[(int64_t)oc * o.nblk_c + blk + j] = (uint8_t)(sbw >> (8 * j));
      }
    }
  }
}

__global__ void __launch_bounds__(256) k_quant_tiles(const QuantParams p, const __grid_constant__ CUtensorMap tm) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  extern __shared__ __align__(128) uint8_t qts[];           // two tiles [kTR][kTC] bf16, row-major
  __shared__ uint32_t scratch[32];
  __shared__ float senc_tab[128];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ __align__(8) uint64_t never;   // test hook: a barrier nothing arrives at
  const int b = blockIdx.y;
  const int t = threadIdx.x;
  if (t == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&never, 1);
    fence_barrier_init();
  }
  const float g = resolve_global_scale(p, b, scratch);
  if (blockIdx.x == 0 && t == 0 && p.g_out) p.g_out[b] = g;
  const BlockScale s = make_block_scale(g, senc_tab);   // synchronizes (barrier init visible)
  if (p.stall_probe) {
    // test hook: the expiry path (status word, early return) before any copy is issued
    if (t == 0 && !mbar_wait(&never, 0, p.timeout_ns)) record_timeout(p.status);
    return;
  }

  const int32_t rows = (int32_t)p.rows, cols = (int32_t)p.cols;
  const int32_t tiles_r = (rows + kTR - 1) / kTR, tiles_c = (cols + kTC - 1) / kTC;
  const int32_t ntiles = tiles_r * tiles_c;
  const TileOut o = tile_out(p, b);

  // tile it of this CTA -> buffer it % 2 (thread 0)
  int32_t issued = 0;
  auto issue = [&](int32_t it) {
    const int32_t tix = (int32_t)blockIdx.x + it * (int32_t)gridDim.x;
    if (tix >= ntiles) return;
    const int32_t tr = tix / tiles_c;
    uint64_t *bar = &full[it & 1];
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_3d(qts + (it & 1) * kTileBytes, &tm, bar, (tix - tr * tiles_c) * kTC, tr * kTR, b);
    issued = it + 1;
  };
  if (t == 0) {
    issue(0);
    issue(1);
  }
  for (int32_t it = 0;; ++it) {
    const int32_t tix = (int32_t)blockIdx.x + it * (int32_t)gridDim.x;
    if (tix >= ntiles) break;
    const int buf = it & 1;
    const bool got = mbar_wait(&full[buf], (uint32_t)(it >> 1) & 1u, p.timeout_ns);
    if (__syncthreads_or(!got)) {
      if (t == 0) record_timeout(p.status);
      break;
    }
    const uint32_t *tile = reinterpret_cast<const uint32_t *>(qts + buf * kTileBytes);   // [kTR][kTC/2] words
    const int32_t tr = tix / tiles_c;
    const int32_t r0 = tr * kTR, c0 = (tix - tr * tiles_c) * kTC;
    pack_tile(p, s, tile, r0, c0, o, t);
    __syncthreads();   // every read of this buffer is done
    if (t == 0) issue(it + 2);
  }
  // tiles still in flight (only after a timeout) land before the CTA exits
  if (t == 0)
    for (int32_t it = issued > 2 ? issued - 2 : 0; it < issued; ++it)
      mbar_wait(&full[it & 1], (uint32_t)(it >> 1) & 1u, kTileDrainNs);
}

// ---------------------------------------------------------- grouped gather --
// The expert-grouped, 128-padded A operand of the grouped GEMM from the token
// rows quantized once (one tensor-wide g): destination row r takes the codes
// and scales of token row_map[r]; rows with row_map < 0 (padding) get no
// codes and zero scales.  Scales arrive in the linear [tokens][K/16] layout and
// leave in the swizzled 128x4-atom layout (scale columns past K/16 inside the
// last 4-column group are zero).  One warp per group of four destination rows
// r, r+32, r+64, r+96 of a 128-row group: their scale words share one 16-byte
// slot of every atom, which the warp writes whole; each row's codes are copied
// with up to eight 16-byte loads per lane in flight.
__global__ void __launch_bounds__(256) k_gather_packed(const uint8_t *__restrict__ codes_src,
                                                       const uint8_t *__restrict__ sf_src,
                                                       const int32_t *__restrict__ row_map, int64_t rows,
                                                       const int32_t *__restrict__ num_mtiles, int64_t K,
                                                       uint8_t *__restrict__ codes_dst,
                                                       uint8_t *__restrict__ sf_dst, int64_t src_rows,
                                                       int *status) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t vec_per_row = K / 32;               // 16-byte vectors of codes
  const int64_t nblk = K / 16, sfc_pad = (nblk + 3) & ~int64_t(3), ngrp = sfc_pad >> 2;
  // only the rows of the routed layout (128 x its m-tile count) are read later
  if (num_mtiles) rows = min(rows, (int64_t)128 * (int64_t)*num_mtiles);
  const int64_t quads = ((rows + 127) >> 7) * 32;
  const bool word_sf = (nblk & 3) == 0;             // source scale rows are 4-byte aligned
  for (int64_t qd = warp; qd < quads; qd += nwarps) {
    const int64_t r0 = (qd >> 5) * 128 + (qd & 31);  // rows r0 + 32 i, i = 0..3
    int64_t sr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = r0 + 32 * i;
      sr[i] = r < rows ? (int64_t)row_map[r] : -1;
      if (!NVFP4_GUARD(sr[i] < src_rows, status)) sr[i] = -1;
    }
    // codes of the four rows, eight 16-byte loads per lane in flight
#pragma unroll
    for (int ri = 0; ri < 4; ++ri) {
      if (sr[ri] < 0) continue;
      const uint4 *cs = reinterpret_cast<const uint4 *>(codes_src + sr[ri] * (K / 2));
      uint4 *cd = reinterpret_cast<uint4 *>(codes_dst + (r0 + 32 * ri) * (K / 2));
      for (int64_t i0 = 0; i0 < vec_per_row; i0 += 256) {
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int64_t i = i0 + 32 * j + lane;
          if (i < vec_per_row) v[j] = __ldg(cs + i);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int64_t i = i0 + 32 * j + lane;
          if (i < vec_per_row) cd[i] = v[j];
        }
      }
    }
    // scales: slot 16 * (r0 % 32) of atom (r0 / 128, group) holds the four rows' words
    uint8_t *sd = sf_dst + 512 * ((r0 >> 7) * ngrp) + 16 * (r0 & 31);
    for (int64_t gI = lane; gI < ngrp; gI += 32) {
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[i] = 0;
        if (sr[i] < 0) continue;
        const uint8_t *ss = sf_src + sr[i] * nblk + 4 * gI;
        if (word_sf) {
          w[i] = __ldg(reinterpret_cast<const uint32_t *>(ss));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (4 * gI + j < nblk) w[i] |= (uint32_t)__ldg(ss + j) << (8 * j);
        }
      }
      *reinterpret_cast<uint4 *>(sd + 512 * gI) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

cudaError_t launch_gather_packed(const uint8_t *codes_src, const uint8_t *sf_src, const int32_t *row_map,
                                 int64_t rows, const int32_t *num_mtiles, int64_t K, uint8_t *codes_dst, uint8_t *sf_dst, int num_sms,
                                 cudaStream_t st, int64_t src_rows, int *status) {
  const int64_t quads = ((rows + 127) / 128) * 32;   // one warp per four rows
  const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>((quads + 7) / 8, (int64_t)num_sms * 8));
  return launch_pdl(k_gather_packed, dim3((unsigned)ctas), dim3(256), 0, st, codes_src, sf_src, row_map, rows,
                    num_mtiles, K, codes_dst, sf_dst, src_rows, status);
}

// Zero the swizzled padding of a scale buffer that the tile kernel does not
// reach: rows in [rows, pad128(rows)) of every matrix.  Columns beyond the
// matrix inside a reached row are written by the kernels themselves.
__global__ void k_zero_sf_pad_rows(uint8_t *sf, int64_t bstride, int64_t rows, int64_t sf_cols) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  const int b = blockIdx.y;
  const int64_t sfc_pad = (sf_cols + 3) & ~int64_t(3);
  const int64_t prow = (rows + 127) & ~int64_t(127);
  const int64_t n = (prow - rows) * sfc_pad;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = rows + i / sfc_pad, c = i % sfc_pad;
    sf[(int64_t)b * bstride + sf_swz_offset(r, c, sfc_pad)] = 0;
  }
}

// ---------------------------------------------------------------- launchers --

int amax_parts_for(int64_t rows) { return (int)std::min<int64_t>(rows, 512); }

cudaError_t launch_amax(const QuantParams &p, cudaStream_t st) {
  dim3 grid(p.nparts, (unsigned)p.batch);
  if (p.batch == 1) return launch_pdl(k_amax_partial<true>, grid, dim3(256), 0, st, p);
  return launch_pdl(k_amax_partial<false>, grid, dim3(256), 0, st, p);
}

static cudaError_t launch_quant_rows_staged(const QuantParams &p, int num_sms, cudaStream_t st) {
  const StagedCfg c = staged_cfg(p.cols);
  if (cudaError_t e = ensure_dynamic_smem((const void *)k_quant_rows_staged, c.smem); e != cudaSuccess) return e;
  const int64_t rows_out =
      (p.sf_swizzled && !p.row_map) ? ((p.dst_rows + 127) & ~int64_t(127)) : p.dst_rows;
  const int64_t units = rows_out * c.nseg * p.batch;
  const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>(num_sms, (units + kQWarps - 1) / kQWarps));
  return launch_pdl(k_quant_rows_staged, dim3((unsigned)ctas), dim3(kQWarps * 32), c.smem, st, p, c.seg,
                    c.nseg, c.slots);
}

cudaError_t launch_quant_rows(const QuantParams &p, int num_sms, cudaStream_t st) {
  // bulk copies need 16-byte aligned rows and segments
  const bool staged = ((reinterpret_cast<uintptr_t>(p.src) & 15) == 0) && (p.ld % 8 == 0) &&
                      (p.bstride % 8 == 0) && (p.cols % 16 == 0);
  // a few rows (decode activations) take the plain kernel: the staged ring's
  // set-up would outweigh the work
  const bool tiny = p.dst_rows <= 64 && p.batch == 1 && !p.row_map;
  if (staged && !tiny) return launch_quant_rows_staged(p, num_sms, st);
  const int64_t rows_out = p.sf_swizzled ? ((p.dst_rows + 127) & ~int64_t(127)) : p.dst_rows;
  const int64_t nch = ((p.cols / 16 + 3) / 4 * 4 + 127) / 128;
  int64_t ctas = (rows_out * nch + 7) / 8;      // 8 warps per CTA, one (row, chunk) each per pass
  const int64_t cap = (int64_t)num_sms * 8 / std::max<int64_t>(1, p.batch);
  ctas = std::max<int64_t>(1, std::min<int64_t>(ctas, std::max<int64_t>(cap, 1)));
  dim3 grid((unsigned)ctas, (unsigned)p.batch);
  const bool v8 = ((reinterpret_cast<uintptr_t>(p.src) & 31) == 0) && (p.ld % 16 == 0) &&
                  (p.bstride % 16 == 0);
  if (v8) return launch_pdl(k_quant_rows<true>, grid, dim3(256), 0, st, p);
  return launch_pdl(k_quant_rows<false>, grid, dim3(256), 0, st, p);
}

// The source as [batch][rows][cols] bf16, one kTC x kTR x 1 box per tile.
static bool tiles_map(const QuantParams &p, CUtensorMap *tm) {
  const uint64_t dims[3] = {(uint64_t)p.cols, (uint64_t)p.rows, (uint64_t)p.batch};
  const uint64_t bstride = p.batch > 1 ? (uint64_t)p.bstride : (uint64_t)p.rows * (uint64_t)p.ld;
  const uint64_t strides[2] = {(uint64_t)p.ld * 2, bstride * 2};
  const uint32_t box[3] = {kTC, kTR, 1};
  return make_map_3d(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p.src, dims, strides, box);
}

// Swizzled scales: rows beyond the matrix inside the last 128-row atom.
static cudaError_t zero_pad_rows(const QuantParams &p, cudaStream_t st) {
  if (!p.sf_swizzled) return cudaSuccess;
  if (p.codes_row && (p.rows % 128) != 0) {
    if (cudaError_t e2 = launch_pdl(k_zero_sf_pad_rows, dim3(4, (unsigned)p.batch), dim3(256), 0, st, p.sf_row,
                                    p.sf_row_bstride, p.rows, p.cols / 16);
        e2 != cudaSuccess)
      return e2;
  }
  if (p.codes_col && (p.cols % 128) != 0) {
    if (cudaError_t e2 = launch_pdl(k_zero_sf_pad_rows, dim3(4, (unsigned)p.batch), dim3(256), 0, st, p.sf_col,
                                    p.sf_col_bstride, p.cols, p.rows / 16);
        e2 != cudaSuccess)
      return e2;
  }
  return cudaGetLastError();
}

cudaError_t launch_quant_tiles(const QuantParams &p, int num_sms, cudaStream_t st) {
  CUtensorMap tm;
  if (!tiles_map(p, &tm)) return cudaErrorInvalidValue;
  if (cudaError_t e = ensure_dynamic_smem((const void *)k_quant_tiles, 2 * kTileBytes); e != cudaSuccess) return e;
  const int64_t tiles = ((p.rows + kTR - 1) / kTR) * ((p.cols + kTC - 1) / kTC);
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_quant_tiles, 256, 2 * kTileBytes);
  per_sm = std::max(per_sm, 1);
  // one wave of resident CTAs, shared by the matrices of the batch
  int64_t ctas = std::min<int64_t>(tiles, std::max<int64_t>(1, (int64_t)num_sms * per_sm / std::max<int64_t>(1, p.batch)));
  dim3 grid((unsigned)ctas, (unsigned)p.batch);
  cudaError_t e = launch_pdl(k_quant_tiles, grid, dim3(256), 2 * kTileBytes, st, p, tm);
  if (e != cudaSuccess) return e;
  return zero_pad_rows(p, st);
}

}  // namespace nvfp4
