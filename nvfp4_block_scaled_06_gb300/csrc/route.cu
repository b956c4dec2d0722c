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
  extern __shared__ int32_t sh_hist[];   // [E]
  for (int e = threadIdx.x; e < p.num_experts; e += blockDim.x) sh_hist[e] = 0;
  __syncthreads();
  const int64_t i = (int64_t)blockIdx.x * p.chunk + threadIdx.x;
  if (threadIdx.x < p.chunk && i < p.pairs) {
    const int e = p.expert_ids[i];
    if (e >= 0 && e < p.num_experts) atomicAdd(&sh_hist[e], 1);
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

__global__ void __launch_bounds__(1024) k_route_scan(const RouteParams p) {
  __shared__ int32_t scratch[64];
  const int e = threadIdx.x;
  const bool act = e < p.num_experts;
  int32_t count = 0;
  if (act) {
    // eight independent loads in flight per step (the chunk bases are formed
    // by the scatter kernel)
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
  if (act) {
    p.counts[e] = count;
    p.offsets[e] = off;
    p.poffsets[e] = poff;
    if (p.offsets_out) p.offsets_out[e] = off;
    for (int j = 0; j < mt; ++j) {
      GroupTile g;
      g.expert = e;
      g.a_row0 = poff + 128 * j;
      g.valid_rows = min(128, count - 128 * j);
      g.out_row0 = off + 128 * j;
      p.gtiles[moff + j] = g;
    }
    for (int32_t i = count; i < padded; ++i) p.row_map[poff + i] = -1;
  }
  if (threadIdx.x == 0) {
    p.offsets[p.num_experts] = total;
    p.poffsets[p.num_experts] = ptotal;
    if (p.offsets_out) p.offsets_out[p.num_experts] = total;
    *p.gnum_mtiles = mtotal;
  }
  for (int64_t r = ptotal + threadIdx.x; r < p.padded_rows_max; r += blockDim.x) p.row_map[r] = -1;
}

__global__ void __launch_bounds__(1024) k_route_scatter(const RouteParams p) {
  extern __shared__ int32_t sh_base[];   // [E] first grouped position of this chunk's pairs
  const int E = p.num_experts;
  uint16_t *sh_cnt = reinterpret_cast<uint16_t *>(sh_base + E);   // [32 warps][E]
  for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) sh_cnt[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int32_t b = p.offsets[e];
    for (int c = 0; c < (int)blockIdx.x; ++c) b += p.hist[(int64_t)c * E + e];
    sh_base[e] = b;
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
    p.perm[pos] = (int32_t)i;
    p.row_map[p.poffsets[e] + (pos - p.offsets[e])] = (int32_t)(i / p.top_k);
  }
}

cudaError_t launch_route(const RouteParams &p, cudaStream_t st) {
  k_route_hist<<<p.nchunks, kRouteChunk, p.num_experts * sizeof(int32_t), st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_route_scan<<<1, 1024, 0, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t sm = (size_t)p.num_experts * sizeof(int32_t) + (size_t)32 * p.num_experts * sizeof(uint16_t);
  static size_t configured = 48 * 1024;
  if (sm > configured) {
    e = cudaFuncSetAttribute(k_route_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    configured = sm;
  }
  k_route_scatter<<<p.nchunks, kRouteChunk, sm, st>>>(p);
  return cudaGetLastError();
}

}  // namespace nvfp4
