// route.cu -- group (token, slot) pairs by routed expert for the grouped GEMM.
//
// 256 routed experts, 8 per token ("GLM-5.2-NVFP4" card): the pairs are
// grouped stably by expert id (rows of one expert contiguous, ordered by pair
// index token*top_k + slot).  Three small kernels, no atomics on global memory:
//   hist     per 1024-pair chunk, per-expert counts -> hist[chunk][e]
//   scan     one CTA: counts, offsets, 128-padded offsets, the m-tile table
//            and the padding rows of row_map
//   scatter  per chunk: its base per expert (offset + earlier chunks' counts),
//            then the stable rank of each pair among same-expert pairs (warp
//            match + per-warp counts) -> perm and row_map
// Expert ids outside [0, E) are dropped.
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

constexpr int kRouteChunk = 1024;

__global__ void __launch_bounds__(1024) k_route_hist(const RouteParams p) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  extern __shared__ int32_t sh_hist[];   // [E]
  for (int e = threadIdx.x; e < p.num_experts; e += blockDim.x) sh_hist[e] = 0;
  __syncthreads();
  const int64_t i = (int64_t)blockIdx.x * p.chunk + threadIdx.x;
  if (threadIdx.x < p.chunk && i < p.pairs) {
    const int e = p.expert_ids[i];
    if (NVFP4_NOTE(e >= 0 && e < p.num_experts, p.status)) atomicAdd(&sh_hist[e], 1);   // others are dropped
  }
  __syncthreads();
  for (int e = threadIdx.x; e < p.num_experts; e += blockDim.x)
    p.hist[(int64_t)blockIdx.x * p.num_experts + e] = sh_hist[e];
}

// Exclusive scan of one value per thread over a 1024-thread block.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t *scratch, int32_t &total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[w] = x;
  __syncthreads();
  if (w == 0) {
    int32_t s = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    scratch[32 + lane] = s;     // inclusive warp-sum prefix
  }
  __syncthreads();
  total = scratch[32 + 31];
  const int32_t before = w > 0 ? scratch[32 + w - 1] : 0;
  return before + x - v;
}

// The same scan with every partial sum capped at `cap` (inputs in [0, cap]):
// min(a + b, cap) is associative on such values, so the result is the exact
// prefix sum clamped to cap, and nothing overflows.
__device__ __forceinline__ int32_t block_exclusive_scan_capped(int32_t v, int32_t cap, int32_t *scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = min(x, cap - y) + y;
  }
  __syncthreads();
  if (lane == 31) scratch[w] = x;
  __syncthreads();
  if (w == 0) {
    int32_t s = scratch[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s = min(s, cap - y) + y;
    }
    scratch[32 + lane] = s;
  }
  const int32_t prev = __shfl_up_sync(0xffffffffu, x, 1);
  const int32_t in_warp = lane > 0 ? prev : 0;   // capped exclusive prefix within the warp
  __syncthreads();
  const int32_t before = w > 0 ? scratch[32 + w - 1] : 0;
  return min(in_warp, cap - before) + before;
}

__global__ void __launch_bounds__(1024) k_route_scan(const RouteParams p) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  __shared__ int32_t scratch[64];
  const int e = threadIdx.x;
  const bool act = e < p.num_experts;
  int32_t count = 0;
  // up to 32 chunks: every chunk count of this expert in registers at once,
  // and after the scan each chunk's first grouped position is written back
  // over its count; more chunks: eight loads in flight per step, and the
  // scatter kernel forms the chunk bases itself
  const bool few = p.nchunks <= 32;
  int32_t hv[32];
  if (act && few) {
    // unconditional loads (the last chunk repeated, its value masked): all
    // 32 are in flight together
#pragma unroll
    for (int j = 0; j < 32; ++j) hv[j] = p.hist[(int64_t)min(j, p.nchunks - 1) * p.num_experts + e];
#pragma unroll
    for (int j = 0; j < 32; ++j) hv[j] = j < p.nchunks ? hv[j] : 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) count += hv[j];
  } else if (act) {
    int c = 0;
    for (; c + 8 <= p.nchunks; c += 8) {
      int32_t v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = p.hist[(int64_t)(c + j) * p.num_experts + e];
#pragma unroll
      for (int j = 0; j < 8; ++j) count += v[j];
    }
    for (; c < p.nchunks; ++c) count += p.hist[(int64_t)c * p.num_experts + e];
  }
  const int32_t padded = (count + 127) & ~127;
  const int32_t mt = padded / 128;
  int32_t total, ptotal, mtotal;
  const int32_t off = block_exclusive_scan(count, scratch, total);
  const int32_t poff = block_exclusive_scan(padded, scratch, ptotal);
  const int32_t moff = block_exclusive_scan(mt, scratch, mtotal);
  if (act && few) {
    int32_t b = off;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < p.nchunks) p.hist[(int64_t)j * p.num_experts + e] = b;
      b += hv[j];
    }
  }
  __shared__ int32_t s_cnt[1024], s_off[1024], s_poff[1024], s_moff[1024];
  if (act) {
    p.counts[e] = count;
    p.offsets[e] = off;
    p.poffsets[e] = poff;
    if (p.offsets_out) p.offsets_out[e] = off;
    s_cnt[e] = count;
    s_off[e] = off;
    s_poff[e] = poff;
    s_moff[e] = moff;
  }
  __syncthreads();
  // one warp per expert: its m-tile entries and its padding rows (up to 127)
  // written by the 32 lanes
  {
    const int lane = threadIdx.x & 31;
    for (int x = threadIdx.x >> 5; x < p.num_experts; x += blockDim.x >> 5) {
      const int32_t cnt = s_cnt[x], of = s_off[x], pf = s_poff[x], mo = s_moff[x];
      const int32_t pad = (cnt + 127) & ~127;
      for (int j = lane; j < pad / 128; j += 32) {
        GroupTile g;
        g.expert = x;
        g.a_row0 = pf + 128 * j;
        g.valid_rows = min(128, cnt - 128 * j);
        g.out_row0 = of + 128 * j;
        if (NVFP4_GUARD(mo + j < p.padded_rows_max / 128, p.status)) p.gtiles[mo + j] = g;
      }
      for (int32_t i = cnt + lane; i < pad; i += 32)
        if (NVFP4_GUARD(pf + i < p.padded_rows_max, p.status)) p.row_map[pf + i] = -1;
    }
  }
  if (threadIdx.x == 0) {
    p.offsets[p.num_experts] = total;
    p.poffsets[p.num_experts] = ptotal;
    if (p.offsets_out) p.offsets_out[p.num_experts] = total;
    *p.gnum_mtiles = mtotal;
  }
  // rows past ptotal (= 128 x the m-tile count) are never read: every user of
  // the layout is bounded by the m-tile count
}

__global__ void __launch_bounds__(1024) k_route_scatter(const RouteParams p) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  extern __shared__ int32_t sh_base[];   // [E] first grouped position of this chunk's pairs
  const int E = p.num_experts;
  uint16_t *sh_cnt = reinterpret_cast<uint16_t *>(sh_base + E);   // [32 warps][E]
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) sh_cnt[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    if (p.nchunks <= 32) {
      sh_base[e] = p.hist[(int64_t)blockIdx.x * E + e];   // written by the scan kernel
    } else {
      int32_t b = p.offsets[e];
      for (int c = 0; c < (int)blockIdx.x; ++c) b += p.hist[(int64_t)c * E + e];
      sh_base[e] = b;
    }
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t i = (int64_t)blockIdx.x * p.chunk + threadIdx.x;
  int e = -1;
  if (threadIdx.x < p.chunk && i < p.pairs) {
    e = p.expert_ids[i];
    if (e < 0 || e >= E) e = -1;
  }
  const unsigned same = __match_any_sync(0xffffffffu, e);
  const unsigned lt = (1u << lane) - 1u;
  const int rank_w = __popc(same & lt);
  if (e >= 0 && (same & lt) == 0) sh_cnt[w * E + e] = (uint16_t)__popc(same);
  __syncthreads();
  if (e >= 0) {
    int before = 0;
    for (int v = 0; v < w; ++v) before += sh_cnt[v * E + e];
    const int32_t pos = sh_base[e] + before + rank_w;
    const int64_t prow = (int64_t)p.poffsets[e] + (pos - p.offsets[e]);
    if (NVFP4_GUARD(pos >= 0 && pos < p.pairs && prow >= 0 && prow < p.padded_rows_max, p.status)) {
      p.perm[pos] = (int32_t)i;
      p.row_map[prow] = (int32_t)(i / p.top_k);
    }
  }
}

cudaError_t launch_route(const RouteParams &p, cudaStream_t st) {
  cudaError_t e = launch_pdl(k_route_hist, dim3(p.nchunks), dim3(kRouteChunk), p.num_experts * sizeof(int32_t), st, p);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_route_scan, dim3(1), dim3(1024), 0, st, p);
  if (e != cudaSuccess) return e;
  const size_t sm = (size_t)p.num_experts * sizeof(int32_t) + (size_t)32 * p.num_experts * sizeof(uint16_t);
  if ((e = ensure_dynamic_smem((const void *)k_route_scatter, sm)) != cudaSuccess) return e;
  return launch_pdl(k_route_scatter, dim3(p.nchunks), dim3(kRouteChunk), sm, st, p);
}

// ------------------------------------------- layout from given expert offsets --
// The grouped operand's padded layout when the rows already arrive grouped
// (the down-projection input, in the order of the up-projection's output, or
// a caller's precomputed routing): per expert e, its rows keep their order
// and start at the 128-aligned padded offset.  The offsets are the caller's
// device data, so the counts are clamped to [0, pairs] cumulatively and the
// layout is rebuilt from the clamped counts (goffsets): consistent offsets
// give back the same offsets, inconsistent ones can never index past the
// grouped rows or the padded bound.
__global__ void __launch_bounds__(1024) k_offsets_layout(const int32_t *__restrict__ offsets, int E, int64_t pairs,
                                                         int32_t *goffsets, int32_t *poffsets, GroupTile *gtiles,
                                                         int32_t *gnum_mtiles, int64_t max_tiles, int *status) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  __shared__ int32_t scratch[64];
  const int e = threadIdx.x;
  const bool act = e < E;
  const int64_t diff = act ? (int64_t)offsets[e + 1] - (int64_t)offsets[e] : 0;
  int32_t count = (int32_t)(diff < 0 ? 0 : diff > pairs ? pairs : diff);
  const int32_t before = block_exclusive_scan_capped(count, (int32_t)pairs, scratch);
  count = min(count, (int32_t)pairs - before);
  (void)NVFP4_NOTE(!act || (int64_t)count == diff, status);   // the caller's offsets were clamped
  if (threadIdx.x == 0) (void)NVFP4_NOTE(offsets[0] == 0, status);
  const int32_t padded = (count + 127) & ~127;
  const int32_t mt = padded / 128;
  int32_t ctotal, ptotal, mtotal;
  const int32_t off = block_exclusive_scan(count, scratch, ctotal);
  const int32_t poff = block_exclusive_scan(padded, scratch, ptotal);
  const int32_t moff = block_exclusive_scan(mt, scratch, mtotal);
  if (act) {
    goffsets[e] = off;
    poffsets[e] = poff;
    for (int j = 0; j < mt; ++j) {
      GroupTile g;
      g.expert = e;
      g.a_row0 = poff + 128 * j;
      g.valid_rows = min(128, count - 128 * j);
      g.out_row0 = off + 128 * j;
      if (NVFP4_GUARD(moff + j < max_tiles, status)) gtiles[moff + j] = g;
    }
  }
  if (threadIdx.x == 0) {
    goffsets[E] = ctotal;
    poffsets[E] = ptotal;
    *gnum_mtiles = mtotal;
  }
}

// row_map[r] = the grouped row that padded row r holds, or -1 (padding); with
// perm given, the token of that row's pair instead (perm[row] / top_k; pair
// indices outside [0, pairs) count as padding).
__global__ void k_rowmap_from_offsets(const int32_t *__restrict__ goffsets,
                                      const int32_t *__restrict__ poffsets, int E, int64_t rows,
                                      const int32_t *__restrict__ perm, int top_k, int64_t pairs,
                                      int32_t *row_map, int *status) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    int32_t v = -1;
    if (r < poffsets[E]) {
      int lo = 0, hi = E - 1;            // the last e with poffsets[e] <= r
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (poffsets[mid] <= r) lo = mid;
        else hi = mid - 1;
      }
      const int64_t i = r - poffsets[lo];
      if (i < goffsets[lo + 1] - goffsets[lo]) {
        v = (int32_t)(goffsets[lo] + i);
        if (perm) {
          const int32_t pr = perm[v];
          v = NVFP4_NOTE(pr >= 0 && pr < pairs, status) ? pr / top_k : -1;
        }
      }
    }
    row_map[r] = v;
  }
}

cudaError_t launch_layout_from_offsets(const int32_t *offsets, int E, int64_t pairs, int64_t padded_rows_max,
                                       int32_t *goffsets, int32_t *poffsets, GroupTile *gtiles,
                                       int32_t *gnum_mtiles, int32_t *row_map, const int32_t *perm, int top_k,
                                       int num_sms, cudaStream_t st, int *status) {
  cudaError_t e = launch_pdl(k_offsets_layout, dim3(1), dim3(1024), 0, st, offsets, E, pairs, goffsets, poffsets,
                             gtiles, gnum_mtiles, padded_rows_max / 128, status);
  if (e != cudaSuccess) return e;
  const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>((padded_rows_max + 255) / 256, (int64_t)num_sms * 4));
  return launch_pdl(k_rowmap_from_offsets, dim3((unsigned)ctas), dim3(256), 0, st, (const int32_t *)goffsets,
                    (const int32_t *)poffsets, E, padded_rows_max, perm, top_k, pairs, row_map, status);
}

// ----------------------------------------------------------------- combine --
// y[t][n] = sum over slots j (in order) of w[t][j] * d[g(t, j)][n], fp32
// accumulation (one fused multiply-add per slot), rounded once to bf16, where
// g(t, j) is the grouped row of pair t*top_k + j (the inverse of perm).
// perm is the caller's device data: entries outside [0, pairs) are skipped,
// and inv is first filled with -1 so that a pair no entry names reads nothing.
__global__ void k_invert_perm(const int32_t *__restrict__ perm, int64_t pairs, int32_t *inv, int *status) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pairs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int32_t q = perm[i];
    if (NVFP4_NOTE(q >= 0 && q < pairs, status)) inv[q] = (int32_t)i;
  }
}
__global__ void k_fill_i32(int32_t *p, int64_t n, int32_t v) {
  griddep_launch_dependents();
  griddep_wait();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = v;
}

// A warp takes a token: its slots' row indices and weights are read once, and
// for top_k <= 8 the 16-byte loads of all slots are in flight together before
// the sums (which keep the slot order).
__global__ void __launch_bounds__(256) k_moe_combine(const __nv_bfloat16 *__restrict__ d,
                                                     const int32_t *__restrict__ inv,
                                                     const float *__restrict__ w, int64_t tokens, int top_k,
                                                     int64_t N, __nv_bfloat16 *__restrict__ y, int *status) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  constexpr int kMaxK = 8;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t vecs = N / 8;                       // 16-byte vectors of a row
  for (int64_t t = warp; t < tokens; t += nwarps) {
    if (top_k <= kMaxK) {
      const uint4 *rows[kMaxK];
      float wj[kMaxK];
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        int32_t g = j < top_k ? inv[t * top_k + j] : -1;
        if (!NVFP4_GUARD(g < tokens * top_k, status)) g = -1;
        rows[j] = g >= 0 ? reinterpret_cast<const uint4 *>(d + (int64_t)g * N) : nullptr;
        wj[j] = g >= 0 ? w[t * top_k + j] : 0.0f;
      }
      for (int64_t v = lane; v < vecs; v += 32) {
        uint4 q[kMaxK];
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) q[j] = rows[j] ? __ldg(rows[j] + v) : make_uint4(0, 0, 0, 0);
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
          if (j >= top_k) break;
          const uint32_t qw[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[2 * i] = __fmaf_rn(wj[j], __uint_as_float(qw[i] << 16), acc[2 * i]);
            acc[2 * i + 1] = __fmaf_rn(wj[j], __uint_as_float(qw[i] & 0xFFFF0000u), acc[2 * i + 1]);
          }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
          o[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        reinterpret_cast<uint4 *>(y + t * N)[v] = make_uint4(o[0], o[1], o[2], o[3]);
      }
      continue;
    }
    for (int64_t v = lane; v < vecs; v += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      for (int j = 0; j < top_k; ++j) {
        const int64_t g = inv[t * top_k + j];
        if (g < 0 || !NVFP4_GUARD(g < tokens * top_k, status)) continue;
        const float wv = w[t * top_k + j];
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(d + g * N) + v);
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] = __fmaf_rn(wv, __uint_as_float(qw[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = __fmaf_rn(wv, __uint_as_float(qw[i] & 0xFFFF0000u), acc[2 * i + 1]);
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t *>(&h);
      }
      reinterpret_cast<uint4 *>(y + t * N)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

cudaError_t launch_moe_combine(const __nv_bfloat16 *d, const int32_t *perm, int32_t *inv, const float *w,
                               int64_t tokens, int top_k, int64_t N, __nv_bfloat16 *y, int num_sms,
                               cudaStream_t st, int *status) {
  const int64_t pairs = tokens * top_k;
  const int64_t c1 = std::max<int64_t>(1, std::min<int64_t>((pairs + 255) / 256, (int64_t)num_sms * 4));
  cudaError_t e = launch_pdl(k_fill_i32, dim3((unsigned)c1), dim3(256), 0, st, inv, pairs, (int32_t)-1);
  if (e != cudaSuccess) return e;
  e = launch_pdl(k_invert_perm, dim3((unsigned)c1), dim3(256), 0, st, perm, pairs, inv, status);
  if (e != cudaSuccess) return e;
  const int64_t c2 = std::max<int64_t>(1, std::min<int64_t>((tokens + 7) / 8, (int64_t)num_sms * 8));
  return launch_pdl(k_moe_combine, dim3((unsigned)c2), dim3(256), 0, st, d, (const int32_t *)inv, w, tokens, top_k,
                    N, y, status);
}

}  // namespace nvfp4
