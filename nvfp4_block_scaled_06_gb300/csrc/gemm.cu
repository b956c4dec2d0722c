// gemm.cu -- W4A4 block-scaled FP4 GEMM on tcgen05, with the bf16 LoRA overlay.
//
// D[m, n] = (g_a g_b) * sum_k e2m1(a_mk) sfa(m, k/16) e2m1(b_nk) sfb(n, k/16)
//           + (alpha/r) * sum_j T[m, j] LB[n, j],      T = X A^T (bf16 X)
// The product of two NVFP4 operands with fp32 accumulation ("vroomfondel/
// glm-5.2-reap-504B-v2-W4A4" card, "Kernel choice": scaled_fp4_mm, W4A4),
// both operands K-major with one E4M3 scale per 16 elements along K ("Getting
// GLM-5.2 NVFP4 Post-Training off the ground", "TN, NT, and what actually
// binds" / "The bottom line"), plus the bf16 rank-r LoRA over the frozen FP4
// base (same page, TL;DR and "A model no kernel wanted to serve").
//
// Design (sm_103a): a persistent kernel, one CTA per SM, 192 threads:
//   warp 0      TMA producer: 128x256 FP4 A tile, BNx256 FP4 B tile (128-byte
//               swizzle), their 128x4 scale atoms by bulk copy; a 4-stage ring.
//   warp 1      one thread issues tcgen05.cp (scales -> TMEM) and
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (M=128,
//               N=BN, K=64) into a BN-column fp32 accumulator in TMEM; then,
//               for the LoRA, kind::f16 MMAs of T' (bf16, pre-scaled by
//               (alpha/r)/(g_a g_b)) against LB into the same accumulator.
//   warps 2..5  epilogue: tcgen05.ld -> * g_a g_b -> bf16/fp32 -> global.
// Every mbarrier wait is bounded; on expiry the CTA records a timeout, waits
// for its own copies and MMAs in flight, frees TMEM and exits.
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

constexpr int kBM = 128;
constexpr int kEpiWarps = 8;                       // two per TMEM lane quarter
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;  // producer, MMA, epilogue
constexpr uint64_t kDrainNs = 200000000ull;

template <int BN>
struct GemmCfg {
  static constexpr int kStages = BN >= 256 ? 4 : 6;
  static constexpr int kABytes = kBM * 128;
  static constexpr int kBBytes = BN * 128;
  static constexpr int kSfbChunks = BN >= 128 ? BN / 128 : 1;
  static constexpr int kSfaBytes = 4 * 512;
  static constexpr int kSfbBytes = kSfbChunks * 4 * 512;
  static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSmemBytes = kStages * kStageBytes + kBarBytes + 1024;
  static constexpr int kSfbColsPerK = kSfbChunks * 4;
  static constexpr int kSfColsPerStage = 16 + 4 * kSfbColsPerK;
  static constexpr int kTmemCols = 512;
  static_assert(BN + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct TileInfo {
  int e;
  int valid_rows;
  int64_t a_row0, out_row0, b_row0, n0;
};

// Dense: n-tile major (concurrent CTAs share B tiles; all of A stays in L2).
// Grouped: m-tile major (the 8 n-tiles of one expert's m-tile run together, so
// its gathered A tile is read from L2 and each expert's weights stream once).
template <int BN>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams &p, int t, int nmt) {
  TileInfo ti;
  const int nt = p.gtiles ? t % p.tiles_n : t / nmt;
  const int j = p.gtiles ? t / p.tiles_n : t % nmt;
  ti.n0 = (int64_t)nt * BN;
  if (p.gtiles) {
    const GroupTile g = p.gtiles[j];
    ti.e = g.expert;
    ti.a_row0 = g.a_row0;
    ti.valid_rows = g.valid_rows;
    ti.out_row0 = g.out_row0;
    ti.b_row0 = (int64_t)g.expert * p.N + ti.n0;
  } else {
    ti.e = 0;
    ti.a_row0 = (int64_t)j * kBM;
    ti.valid_rows = (int)(p.M - ti.a_row0 < kBM ? p.M - ti.a_row0 : kBM);
    ti.out_row0 = ti.a_row0;
    ti.b_row0 = ti.n0;
  }
  return ti;
}

// The scale applied to the fp32 accumulator; shared (bit for bit) with the
// LoRA pre-scaling so that (alpha/r)/(g_a g_b) * (g_a g_b) cancels.  A zero
// product means the FP4 operand is all zero codes; 1 keeps the LoRA exact.
__device__ __forceinline__ float acc_scale(const float *g_a, const float *g_b, int e) {
  return acc_scale_of(g_a ? *g_a : 1.0f, g_b ? g_b[e] : 1.0f);
}

__device__ __forceinline__ void signal_abort(volatile int *abort_flag, int *status) {
  *abort_flag = 1;
  record_timeout(status);
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_fp4(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmLB,
               const GemmParams p) {
  using C = GemmCfg<BN>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = base;
  uint8_t *sB = sA + S * C::kABytes;
  uint8_t *sSFA = sB + S * C::kBBytes;
  uint8_t *sSFB = sSFA + S * C::kSfaBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sSFB + S * C::kSfbBytes);
  uint64_t *full = bars, *empty = bars + S;
  uint64_t *acc_full = bars + 2 * S, *acc_empty = acc_full + 1, *drain = acc_full + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  uint64_t *never = acc_full + 4;          // test hook: a barrier nothing arrives at

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kEpiWarps);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.lora_steps) {
      tma_prefetch_desc(&tmT);
      tma_prefetch_desc(&tmLB);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int nmt = p.gtiles ? *p.gnum_mtiles : p.tiles_m;
  const int ksplit = p.ksplit > 1 ? p.ksplit : 1;
  const int num_tiles = nmt * p.tiles_n * ksplit;     // work units: (tile, K range)
  const int kt_per = (p.num_kt + ksplit - 1) / ksplit;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;   // bit s: stage s has an outstanding fill
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_tiles; u += gridDim.x) {
        const TileInfo ti = decode_tile<BN>(p, u / ksplit, nmt);
        const int kt0 = (u % ksplit) * kt_per;
        const int kt1 = min(p.num_kt, kt0 + kt_per);
        for (int kk = kt0; kk < kt1 + p.lora_steps; ++kk) {
          const int kt = kk < kt1 ? kk : p.num_kt + (kk - kt1);   // LoRA steps follow the FP4 range
          if (*abort_flag || !mbar_wait(&empty[stage], phase ^ 1, p.timeout_ns)) {
            signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          if (kt < p.num_kt) {
            const int nk = min(4, p.nk64 - kt * 4);
            int chunks = 0;
            const int64_t chunk0 = ti.b_row0 >> 7;
#pragma unroll
            for (int c = 0; c < C::kSfbChunks; ++c)
              if (chunk0 + c < p.b_sf_row_chunks) chunks = c + 1;
            const uint32_t bytes = C::kABytes + C::kBBytes + nk * 512 + chunks * nk * 512;
            mbar_arrive_expect_tx(&full[stage], bytes);
            tma_load_2d(sA + stage * C::kABytes, &tmA, &full[stage], kt * 128, (int)ti.a_row0);
            tma_load_2d(sB + stage * C::kBBytes, &tmB, &full[stage], kt * 128, (int)ti.b_row0);
            bulk_load(sSFA + stage * C::kSfaBytes,
                      p.a_sf + 512 * ((ti.a_row0 >> 7) * p.a_sf_katoms + kt * 4), nk * 512,
                      &full[stage]);
            for (int c = 0; c < chunks; ++c)
              bulk_load(sSFB + stage * C::kSfbBytes + c * 2048,
                        p.b_sf + 512 * ((chunk0 + c) * p.b_sf_katoms + kt * 4), nk * 512,
                        &full[stage]);
          } else {
            const int ls = kt - p.num_kt;
            mbar_arrive_expect_tx(&full[stage], C::kABytes + C::kBBytes);
            tma_load_2d(sA + stage * C::kABytes, &tmT, &full[stage], ls * 64, (int)ti.a_row0);
            tma_load_2d(sB + stage * C::kBBytes, &tmLB, &full[stage], ls * 64, (int)ti.b_row0);
          }
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every fill this thread started must land before the CTA may exit
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (armed_par >> s) & 1, kDrainNs);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue --
    if (lane == 0) {
      const uint32_t idesc = idesc_nvfp4(kBM, BN);
      const uint32_t idesc_l = idesc_bf16(kBM, BN);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      if (p.stall_probe && !mbar_wait(never, 0, p.timeout_ns)) {
        signal_abort(abort_flag, p.status);   // expected: the expiry path under test
        ok = false;
      }
      for (int u = blockIdx.x; ok && u < num_tiles; u += gridDim.x) {
        const TileInfo ti = decode_tile<BN>(p, u / ksplit, nmt);
        const int kt0 = (u % ksplit) * kt_per;
        const int kt1 = min(p.num_kt, kt0 + kt_per);
        if (*abort_flag || !mbar_wait(acc_empty, acc_phase ^ 1, p.timeout_ns)) {
          signal_abort(abort_flag, p.status);
          break;
        }
        tc_fence_after();
        uint32_t accumulate = 0;
        const uint32_t sfb_lane_col = (uint32_t)((ti.b_row0 & 127) >> 5);
        for (int kk = kt0; kk < kt1 + p.lora_steps; ++kk) {
          const int kt = kk < kt1 ? kk : p.num_kt + (kk - kt1);
          if (*abort_flag || !mbar_wait(&full[stage], phase, p.timeout_ns)) {
            signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_k_sw128(sA + stage * C::kABytes);
          const uint64_t bdesc = sdesc_k_sw128(sB + stage * C::kBBytes);
          if (kt < p.num_kt) {
            const int nk = min(4, p.nk64 - kt * 4);
            const uint32_t sfa_col = tmem + BN + stage * C::kSfColsPerStage;
            const uint32_t sfb_col = sfa_col + 16;
            const int64_t chunk0 = ti.b_row0 >> 7;
            for (int j = 0; j < nk; ++j) {
              tc_cp_32x128b_x4(sfa_col + 4 * j, sdesc_sf_atom(sSFA + stage * C::kSfaBytes + 512 * j));
#pragma unroll
              for (int c = 0; c < C::kSfbChunks; ++c)
                if (chunk0 + c < p.b_sf_row_chunks)
                  tc_cp_32x128b_x4(sfb_col + j * C::kSfbColsPerK + 4 * c,
                                   sdesc_sf_atom(sSFB + stage * C::kSfbBytes + c * 2048 + 512 * j));
            }
            for (int j = 0; j < nk; ++j) {
              tc_mma_nvfp4(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col + 4 * j,
                           sfb_col + j * C::kSfbColsPerK + sfb_lane_col, accumulate);
              accumulate = 1;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tc_mma_bf16(tmem, adesc + 2 * j, bdesc + 2 * j, idesc_l, accumulate);
              accumulate = 1;
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_phase ^= 1;
      }
      // all MMAs and copies issued by this thread complete before TMEM is freed
      tc_commit(drain);
      mbar_wait(drain, 0, kDrainNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    // Warp w reads TMEM lane quarter (w % 4) and half (w - 2) / 4 of the BN
    // columns: all of its accumulator columns are loaded into registers, the
    // accumulator is released to the MMA warp, then the values are scaled,
    // converted and stored while the next tile's MMAs run.
    constexpr int kCh = BN / 64;            // 32-column chunks per thread
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;            // accumulator row owned by this thread
    uint32_t acc_phase = 0;
    float sq = 0.0f;
    for (int u = blockIdx.x; u < num_tiles; u += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(p, u / ksplit, nmt);
      const int ks = u % ksplit;
      // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
      if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(acc_full, acc_phase, p.timeout_ns))) {
        if (lane == 0) signal_abort(abort_flag, p.status);
        break;
      }
      tc_fence_after();
      uint32_t v[kCh][32];
#pragma unroll
      for (int c = 0; c < kCh; ++c)
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (half * kCh + c) * 32, v[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      acc_phase ^= 1;

      const float alpha = p.accumulate_d ? 1.0f : acc_scale(p.g_a, p.g_b, ti.e);
      if (r >= ti.valid_rows) continue;
      const int64_t orow = ti.out_row0 + r;
#pragma unroll
      for (int c = 0; c < kCh; ++c) {
        const int64_t n = ti.n0 + (half * kCh + c) * 32;
        if (n >= p.N) break;
        float f[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) f[i] = __fmul_rn(__uint_as_float(v[c][i]), alpha);
        const bool full_chunk = n + 32 <= p.N;
        const int nvalid = full_chunk ? 32 : (int)(p.N - n);
        if (p.partial) {
          float *dst = p.partial + ((int64_t)ks * p.M + orow) * p.N + n;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < nvalid) dst[i] = f[i];
        } else if (p.out_fp32) {
          float *dst = reinterpret_cast<float *>(p.d) + orow * p.ldd + n;
          if (p.accumulate_d) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) {
                sq += f[i] * f[i];
                dst[i] = dst[i] + f[i];
              }
          } else if (full_chunk) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4 *>(dst + i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
            if (p.sqnorm)
#pragma unroll
              for (int i = 0; i < 32; ++i) sq += f[i] * f[i];
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) {
                dst[i] = f[i];
                sq += f[i] * f[i];
              }
          }
        } else {
          __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.d) + orow * p.ldd + n;
          if (p.accumulate_d) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) {
                sq += f[i] * f[i];
                dst[i] = __float2bfloat16_rn(__fadd_rn(__bfloat162float(dst[i]), f[i]));
              }
          } else if (full_chunk) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
              w[i] = *reinterpret_cast<const uint32_t *>(&h);
            }
#pragma unroll
            for (int i = 0; i < 16; i += 4)
              *reinterpret_cast<uint4 *>(dst + 2 * i) = make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
            if (p.sqnorm)
#pragma unroll
              for (int i = 0; i < 32; ++i) sq += f[i] * f[i];
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < nvalid) {
                dst[i] = __float2bfloat16_rn(f[i]);
                sq += f[i] * f[i];
              }
          }
        }
      }
    }
    if (p.sqnorm) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (lane == 0) atomicAdd(p.sqnorm, sq);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------ LoRA down --
// T'[row, j] = bf16( s_row * sum_k X[src(row), k] A[j, k] ), fp32 accumulation
// in TMEM (kind::f16, M=128, N=rank, K=16 per instruction).  s_row =
// (alpha/r) / (g_a g_b[e]) when the result feeds the FP4 accumulator, alpha/r
// for the standalone path.  Grouped mode gathers X rows with tile::gather4.
constexpr int kLoraStages = 6;
constexpr int kLoraThreads = 192;

__host__ __device__ constexpr int lora_stage_bytes(int rank) { return kBM * 128 + rank * 128; }
__host__ __device__ constexpr int lora_smem_bytes(int rank, int stages) {
  return stages * lora_stage_bytes(rank) + 256 + 1024;
}
__host__ __device__ constexpr int lora_stages_for(int rank) {
  return lora_smem_bytes(rank, kLoraStages) <= 200 * 1024 ? kLoraStages
                                                           : (200 * 1024 - 1280) / lora_stage_bytes(rank);
}
__host__ __device__ constexpr uint32_t tmem_cols_for(int n) {
  return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : 256;
}

__global__ void __launch_bounds__(kLoraThreads, 1)
    k_lora_down(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmA,
                const LoraDownParams p, int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int sbytes = lora_stage_bytes(p.rank);
  uint64_t *bars = reinterpret_cast<uint64_t *>(base + stages * sbytes);
  uint64_t *full = bars, *empty = bars + stages;
  uint64_t *acc_full = bars + 2 * stages, *acc_empty = acc_full + 1, *drain = acc_full + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 3);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  uint32_t *amax_smem = tmem_slot + 2;
  const uint32_t tcols = tmem_cols_for(p.rank);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool scan = p.amax_part != nullptr;   // epilogue warps also scan X for amax
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], scan ? 5 : 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *amax_smem = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int num_tiles = p.gtiles ? *p.gnum_mtiles : p.tiles_m;

  if (warp == 0) {
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_par = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      const int64_t row0 = p.gtiles ? (int64_t)p.gtiles[t].a_row0 : (int64_t)t * kBM;
      const int a_row = p.gtiles ? p.gtiles[t].expert * p.rank : 0;   // this expert's A
      int32_t src[4] = {0, 0, 0, 0};
      if (p.row_map) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int32_t s = p.row_map[row0 + lane * 4 + i];
          src[i] = s < 0 ? 0 : s;
        }
      }
      for (int kt = 0; kt < p.num_k64; ++kt) {
        bool good = true;
        if (lane == 0)
          good = !*abort_flag && mbar_wait(&empty[stage], phase ^ 1, p.timeout_ns);
        good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
        if (!good) {
          if (lane == 0) signal_abort(abort_flag, p.status);
          ok = false;
          break;
        }
        uint8_t *sx = base + stage * sbytes;
        uint8_t *sa = sx + kBM * 128;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], kBM * 128 + p.rank * 128);
          tma_load_2d(sa, &tmA, &full[stage], kt * 64, a_row);
          if (!p.row_map) tma_load_2d(sx, &tmX, &full[stage], kt * 64, (int)row0);
        }
        __syncwarp();
        if (p.row_map)
          tma_gather4(sx + lane * 4 * 128, &tmX, &full[stage], kt * 64, src[0], src[1], src[2],
                      src[3]);
        if (lane == 0) {
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        }
        if (++stage == stages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    if (lane == 0)
      for (int s = 0; s < stages; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (armed_par >> s) & 1, kDrainNs);
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kBM, p.rank);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
        if (*abort_flag || !mbar_wait(acc_empty, acc_phase ^ 1, p.timeout_ns)) {
          signal_abort(abort_flag, p.status);
          break;
        }
        tc_fence_after();
        for (int kt = 0; kt < p.num_k64; ++kt) {
          if (*abort_flag || !mbar_wait(&full[stage], phase, p.timeout_ns)) {
            signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sdesc_k_sw128(base + stage * sbytes);
          const uint64_t bdesc = sdesc_k_sw128(base + stage * sbytes + kBM * 128);
#pragma unroll
          for (int j = 0; j < 4; ++j) tc_mma_bf16(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, (kt | j) != 0);
          tc_commit(&empty[stage]);
          if (++stage == stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_phase ^= 1;
      }
      tc_commit(drain);
      mbar_wait(drain, 0, kDrainNs);
    }
  } else {
    const int q = warp & 3;
    const int r = q * 32 + lane;
    uint32_t acc_phase = 0;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t m2 = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x) {
      int64_t row0;
      int e = 0;
      if (scan) {
        // max |x| over this warp's 32 rows of every X tile, read from shared memory
        for (int kt = 0; kt < p.num_k64; ++kt) {
          if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(&full[stage], phase, p.timeout_ns))) {
            if (lane == 0) signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          const uint4 *row = reinterpret_cast<const uint4 *>(base + stage * sbytes + r * 128);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 v = row[i];
            m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
            m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
            m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
            m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
          if (++stage == stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
      }
      if (p.gtiles) {
        row0 = p.gtiles[t].a_row0;
        e = p.gtiles[t].expert;
      } else {
        row0 = (int64_t)t * kBM;
      }
      if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(acc_full, acc_phase, p.timeout_ns))) {
        if (lane == 0) signal_abort(abort_flag, p.status);
        break;
      }
      tc_fence_after();
      float s = p.lora_scale;
      if (p.g_a) s = __fdiv_rn(p.lora_scale, acc_scale(p.g_a, p.g_b, e));
      const int64_t row = row0 + r;
      const bool row_ok = p.gtiles ? true : row < p.M;
      if (p.t_f32) {
        for (int c = 0; c < p.rank / 32; ++c) {
          uint32_t v[32];
          __syncwarp();
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, v);
          tmem_ld_wait();
          if (c == p.rank / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
          }
          if (!row_ok) continue;
          float4 *dst = reinterpret_cast<float4 *>(p.t_f32 + row * p.rank + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                 __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        }
        acc_phase ^= 1;
        continue;
      }
      for (int c = 0; c < p.rank / 32; ++c) {
        uint32_t v[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + c * 32, v);
        tmem_ld_wait();
        if (c == p.rank / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty);
        }
        if (!row_ok) continue;
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[2 * i]), s),
                                                         __fmul_rn(__uint_as_float(v[2 * i + 1]), s));
          w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        __nv_bfloat16 *dst = p.t_out + row * p.rank + c * 32;
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<uint4 *>(dst + 2 * i) = make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
      }
      acc_phase ^= 1;
    }
    if (scan) {
      uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      if (lane == 0) atomicMax(amax_smem, m);
    }
  }
  __syncthreads();
  if (scan && threadIdx.x == 0) p.amax_part[blockIdx.x] = *amax_smem;
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tcols);
  }
}

// ----------------------------------------------------------- split-K sum --
__global__ void k_splitk_reduce(const GemmParams p) {
  const int64_t total = p.M * p.N;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / p.N, n = i % p.N;
    float s = p.partial[i];
    for (int k = 1; k < p.ksplit; ++k) s = __fadd_rn(s, p.partial[k * total + i]);
    if (p.out_fp32) reinterpret_cast<float *>(p.d)[m * p.ldd + n] = s;
    else reinterpret_cast<__nv_bfloat16 *>(p.d)[m * p.ldd + n] = __float2bfloat16_rn(s);
  }
}

cudaError_t launch_splitk_reduce(const GemmParams &p, int num_sms, cudaStream_t st) {
  const int64_t total = p.M * p.N;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 4));
  k_splitk_reduce<<<grid, 256, 0, st>>>(p);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- launch --

template <int BN>
static cudaError_t launch_bn(const GemmParams &p, const GemmMaps &m, int num_sms, cudaStream_t st) {
  using C = GemmCfg<BN>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_fp4<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  int64_t tiles = (int64_t)p.tiles_n * (p.gtiles ? 0 : p.tiles_m) * std::max(1, p.ksplit);
  int grid = num_sms;
  if (!p.gtiles) grid = (int)std::min<int64_t>(tiles, num_sms);
  if (grid <= 0) return cudaSuccess;
  k_gemm_fp4<BN><<<grid, kGemmThreads, C::kSmemBytes, st>>>(m.a, m.b, m.t, m.lb, p);
  return cudaGetLastError();
}

cudaError_t launch_gemm_fp4(const GemmParams &p, const GemmMaps &m, int bn, int num_sms,
                            cudaStream_t st) {
  switch (bn) {
    case 256: return launch_bn<256>(p, m, num_sms, st);
    case 128: return launch_bn<128>(p, m, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_lora_down(const LoraDownParams &p, const LoraDownMaps &m, int num_sms,
                             cudaStream_t st) {
  const int stages = lora_stages_for(p.rank);
  const int smem = lora_smem_bytes(p.rank, stages);
  static int configured_bytes = 0;
  if (configured_bytes < smem) {
    cudaError_t e = cudaFuncSetAttribute(k_lora_down, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured_bytes = smem;
  }
  int grid = num_sms;
  if (!p.gtiles) grid = std::min(p.tiles_m, num_sms);
  if (grid <= 0) return cudaSuccess;
  k_lora_down<<<grid, kLoraThreads, smem, st>>>(m.x, m.a, p, stages);
  return cudaGetLastError();
}

}  // namespace nvfp4
