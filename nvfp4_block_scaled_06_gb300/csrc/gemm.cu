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
// Design (sm_103a): a persistent kernel, one CTA per SM, 320 threads:
//   warp 0      TMA producer: 128x256 FP4 A tile, BNx256 FP4 B tile (128-byte
//               swizzle), their 128x4 scale atoms by bulk copy; a 4- or 6-stage ring.
//   warp 1      one thread issues tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M=128, N=BN, K=64) into a BN-column fp32 accumulator in TMEM; then,
//               for the LoRA, kind::f16 MMAs of T' (bf16, pre-scaled by
//               (alpha/r)/(g_a g_b)) against LB into the same accumulator.
//   warps 2..5  scales: shared memory -> TMEM with tcgen05.st (one lane quarter each).
//   warps 6..9  epilogue: tcgen05.ld -> * g_a g_b -> bf16/fp32 -> global.
// Every mbarrier wait is bounded; on expiry the CTA records a timeout, waits
// for its own copies and MMAs in flight, frees TMEM and exits.
#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

constexpr int kBM = 128;
constexpr int kSfWarps = 4;                        // scale-factor writers, one per lane quarter
constexpr int kEpiWarps = 4;                       // accumulator drain, one per lane quarter
constexpr int kGemmThreads = 64 + 32 * (kSfWarps + kEpiWarps);
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
    GroupTile g = p.gtiles[j];
    if (!NVFP4_GUARD(g.expert >= 0 && (int64_t)(g.expert + 1) * p.N <= p.b_sf_row_chunks * 128 && g.a_row0 >= 0 &&
                         g.a_row0 + kBM <= p.M && g.valid_rows >= 0 && g.valid_rows <= kBM && g.out_row0 >= 0 &&
                         g.out_row0 + g.valid_rows <= p.out_rows,
                     p.status)) {
      g.expert = 0;       // an in-range tile that stores nothing
      g.a_row0 = 0;
      g.valid_rows = 0;
      g.out_row0 = 0;
    }
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

// Optional wait statistics (compile with -DNVFP4_WAIT_STATS): cycles each role
// spends in waits, summed over CTAs into 64-bit counters at byte 64 of the
// workspace (the status word's reserved block).  Off in normal builds.
#ifdef NVFP4_WAIT_STATS
#define WSTAT_T0() const long long _ws_t0 = clock64()
#define WSTAT_ADD(p, i) \
  atomicAdd(reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>((p).status) + 64) + (i), \
            (unsigned long long)(clock64() - _ws_t0))
#else
#define WSTAT_T0() (void)0
#define WSTAT_ADD(p, i) (void)0
#endif

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
#ifdef NVFP4_WAIT_STATS
  const long long kernel_t0 = clock64();
#endif
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = base;
  uint8_t *sB = sA + S * C::kABytes;
  uint8_t *sSFA = sB + S * C::kBBytes;
  uint8_t *sSFB = sSFA + S * C::kSfaBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sSFB + S * C::kSfbBytes);
  uint64_t *full = bars, *empty = bars + S, *sfready = bars + 2 * S;
  uint64_t *acc_full = bars + 3 * S, *acc_empty = acc_full + 1, *drain = acc_full + 2;
  uint64_t *never = acc_full + 3;          // test hook: a barrier nothing arrives at
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 4);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sfready[s], kSfWarps);
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
  griddep_launch_dependents();
  griddep_wait();   // inputs of this kernel come from the previous one in the stream

  const int nmt = p.gtiles ? *p.gnum_mtiles : p.tiles_m;
  const int ksplit = p.ksplit > 1 ? p.ksplit : 1;
  const int num_tiles = nmt * p.tiles_n * ksplit;     // work units: (tile, K range)
  const int kt_per = (p.num_kt + ksplit - 1) / ksplit;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      // Every per-stage address is a precomputed base plus a constant: this
      // single thread issues ~6 operations per 256-wide K step.
      const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
      const uint32_t sfa_base = smem_u32(sSFA), sfb_base = smem_u32(sSFB);
      const uint32_t full_base = smem_u32(full), empty_base = smem_u32(empty);
      const int last_nk = p.nk64 - (p.num_kt - 1) * 4;    // K steps of the last K tile
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_par = 0;   // bit s: stage s has an outstanding fill
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_tiles; u += gridDim.x) {
        const TileInfo ti = decode_tile<BN>(p, u / ksplit, nmt);
        const int kt0 = (u % ksplit) * kt_per;
        const int kt1 = min(p.num_kt, kt0 + kt_per);
        const int64_t chunk0 = ti.b_row0 >> 7;
        int chunks = 0;
#pragma unroll
        for (int c = 0; c < C::kSfbChunks; ++c)
          if (chunk0 + c < p.b_sf_row_chunks) chunks = c + 1;
        const int a_row = (int)ti.a_row0, b_row = (int)ti.b_row0;
        const uint8_t *sfa_src = p.a_sf + 512 * ((ti.a_row0 >> 7) * p.a_sf_katoms + (int64_t)kt0 * 4);
        const uint8_t *sfb_src = p.b_sf + 512 * (chunk0 * p.b_sf_katoms + (int64_t)kt0 * 4);
        const int64_t sfb_chunk_stride = 512 * p.b_sf_katoms;
        const int nsteps = (kt1 - kt0) + p.lora_steps;
        for (int i = 0; i < nsteps; ++i) {
          const int kt = kt0 + i;
          const uint32_t fb = full_base + 8 * stage;
          WSTAT_T0();
          const bool got = !*abort_flag && mbar_wait_u(empty_base + 8 * stage, phase ^ 1, p.timeout_ns);
          WSTAT_ADD(p, 0);
          if (!got) {
            signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          const uint32_t a_dst = a_base + stage * C::kABytes, b_dst = b_base + stage * C::kBBytes;
          if (kt < kt1) {
            const int nk = kt == p.num_kt - 1 ? last_nk : 4;
            const uint32_t sfb = nk * 512;
            mbar_arrive_expect_tx_u(fb, C::kABytes + C::kBBytes + sfb * (1 + chunks));
            tma_load_2d_u(a_dst, &tmA, fb, kt * 128, a_row);
            tma_load_2d_u(b_dst, &tmB, fb, kt * 128, b_row);
            bulk_load_u(sfa_base + stage * C::kSfaBytes, sfa_src, sfb, fb);
            bulk_load_u(sfb_base + stage * C::kSfbBytes, sfb_src, sfb, fb);
            if (C::kSfbChunks > 1 && chunks > 1)
              bulk_load_u(sfb_base + stage * C::kSfbBytes + 2048, sfb_src + sfb_chunk_stride, sfb, fb);
            sfa_src += 2048;
            sfb_src += 2048;
          } else {
            const int ls = kt - kt1;
            mbar_arrive_expect_tx_u(fb, C::kABytes + C::kBBytes);
            tma_load_2d_u(a_dst, &tmT, fb, ls * 64, a_row);
            tma_load_2d_u(b_dst, &tmLB, fb, ls * 64, b_row);
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
      // stage-0 descriptors; a stage adds its byte offset / 16 to the address field
      const uint64_t adesc0 = sdesc_k_sw128(sA), bdesc0 = sdesc_k_sw128(sB);
      const uint32_t sfr_base = smem_u32(sfready), empty_base = smem_u32(empty);
      const uint32_t accf = smem_u32(acc_full), acce = smem_u32(acc_empty);
      const int last_nk = p.nk64 - (p.num_kt - 1) * 4;
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
        WSTAT_T0();
        const bool got_acc = !*abort_flag && mbar_wait_u(acce, acc_phase ^ 1, p.timeout_ns);
        WSTAT_ADD(p, 2);
        if (!got_acc) {
          signal_abort(abort_flag, p.status);
          break;
        }
        tc_fence_after();
        uint32_t accumulate = 0;
        const uint32_t sfb_lane_col = (uint32_t)((ti.b_row0 & 127) >> 5);
        const int nsteps = (kt1 - kt0) + p.lora_steps;
        for (int i = 0; i < nsteps; ++i) {
          const int kt = kt0 + i;
          WSTAT_T0();
          // the stage's operands have landed and its scales are in tensor memory
          const bool got = !*abort_flag && mbar_wait_u(sfr_base + 8 * stage, phase, p.timeout_ns);
          WSTAT_ADD(p, 1);
          if (!got) {
            signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = adesc0 + (uint64_t)((stage * C::kABytes) >> 4);
          const uint64_t bdesc = bdesc0 + (uint64_t)((stage * C::kBBytes) >> 4);
          if (kt < kt1) {
            const int nk = kt == p.num_kt - 1 ? last_nk : 4;
            const uint32_t sfa_col = tmem + BN + stage * C::kSfColsPerStage;
            const uint32_t sfb_col = sfa_col + 16;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (j < nk) {
                tc_mma_nvfp4(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col + 4 * j,
                             sfb_col + j * C::kSfbColsPerK + sfb_lane_col, accumulate);
                accumulate = 1;
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tc_mma_bf16(tmem, adesc + 2 * j, bdesc + 2 * j, idesc_l, accumulate);
              accumulate = 1;
            }
          }
          tc_commit_u(empty_base + 8 * stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_u(accf);
        acc_phase ^= 1;
      }
      // all MMAs issued by this thread complete before TMEM is freed
      tc_commit(drain);
      mbar_wait(drain, 0, kDrainNs);
    }
  } else if (warp < 2 + kSfWarps) {
    // --------------------------------------------------- scales -> tensor memory --
    // Warp w writes TMEM lane quarter (w % 4).  Lane i of every quarter gets
    // line i of each 128x4 scale atom (rows i, i+32, i+64, i+96), so each
    // quarter holds the whole atom: per k-step, the A scales in 4 columns and
    // the B scales in 4 columns per 128-row chunk -- the layout the block-scaled
    // MMA reads (the same one tcgen05.cp .32x128b.warpx4 produces).
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + BN;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < num_tiles; u += gridDim.x) {
      const int kt0 = (u % ksplit) * kt_per;
      const int kt1 = min(p.num_kt, kt0 + kt_per);
      const int nsteps = (kt1 - kt0) + p.lora_steps;
      for (int i = 0; i < nsteps; ++i) {
        if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(&full[stage], phase, p.timeout_ns))) {
          if (lane == 0) signal_abort(abort_flag, p.status);
          ok = false;
          break;
        }
        if (kt0 + i < kt1) {
          const uint4 *fa = reinterpret_cast<const uint4 *>(sSFA + stage * C::kSfaBytes) + lane;
          const uint4 *fb = reinterpret_cast<const uint4 *>(sSFB + stage * C::kSfbBytes) + lane;
          uint32_t v[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w = fa[32 * j];              // atom j, line `lane`
            v[4 * j] = w.x; v[4 * j + 1] = w.y; v[4 * j + 2] = w.z; v[4 * j + 3] = w.w;
          }
          tmem_st_32x32b_x16(tq + stage * C::kSfColsPerStage, v);
#pragma unroll
          for (int h = 0; h < C::kSfbChunks; ++h) {
            // columns 16 + 16h .. : k-steps 2h', 2h'+1 for BN=256 (8 columns per k-step)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int col = 16 * h + 4 * t;        // column offset inside the B region
              const int j = col / C::kSfbColsPerK, c = (col % C::kSfbColsPerK) / 4;
              const uint4 w = fb[128 * c + 32 * j];  // chunk c (2048 B), atom j (512 B)
              v[4 * t] = w.x; v[4 * t + 1] = w.y; v[4 * t + 2] = w.z; v[4 * t + 3] = w.w;
            }
            tmem_st_32x32b_x16(tq + stage * C::kSfColsPerStage + 16 + 16 * h, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    // Warp w drains TMEM lane quarter (w % 4): each thread owns one accumulator
    // row, loads it in two halves and releases the accumulator after the second
    // half's loads, so the next tile's MMAs overlap the remaining stores.
    constexpr int kCh = BN / 64;            // 32-column chunks per half
    const int q = warp & 3;
    const int r = q * 32 + lane;            // accumulator row owned by this thread
    uint32_t acc_phase = 0;
    float sq = 0.0f;
    for (int u = blockIdx.x; u < num_tiles; u += gridDim.x) {
      const TileInfo ti = decode_tile<BN>(p, u / ksplit, nmt);
      const int ks = u % ksplit;
      WSTAT_T0();
      // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
      const bool got_full = __all_sync(0xffffffffu, !*abort_flag && mbar_wait(acc_full, acc_phase, p.timeout_ns));
      if (warp == 2 + kSfWarps && lane == 0) WSTAT_ADD(p, 3);
      if (!got_full) {
        if (lane == 0) signal_abort(abort_flag, p.status);
        break;
      }
      tc_fence_after();
      const float alpha = p.accumulate_d ? 1.0f : acc_scale(p.g_a, p.g_b, ti.e);
      const bool row_ok = r < ti.valid_rows;
      const int64_t orow = ti.out_row0 + r;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint32_t v[kCh][32];
        __syncwarp();
#pragma unroll
        for (int c = 0; c < kCh; ++c)
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (half * kCh + c) * 32, v[c]);
        tmem_ld_wait();
        if (half == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty);
        }
        if (!row_ok) continue;
#pragma unroll
        for (int c = 0; c < kCh; ++c) {
          const int64_t n = ti.n0 + (half * kCh + c) * 32;
          if (n >= p.N) break;
          float f[32];
#pragma unroll
          for (int i2 = 0; i2 < 32; ++i2) f[i2] = __fmul_rn(__uint_as_float(v[c][i2]), alpha);
          const bool full_chunk = n + 32 <= p.N;
          const int nvalid = full_chunk ? 32 : (int)(p.N - n);
          if (p.partial) {
            float *dst = p.partial + ((int64_t)ks * p.M + orow) * p.N + n;
            if (full_chunk && (reinterpret_cast<uintptr_t>(dst) & 31) == 0) {   // whole 32-byte sectors
#pragma unroll
              for (int i2 = 0; i2 < 32; i2 += 8)
                st_global_v8(dst + i2, __float_as_uint(f[i2]), __float_as_uint(f[i2 + 1]),
                             __float_as_uint(f[i2 + 2]), __float_as_uint(f[i2 + 3]), __float_as_uint(f[i2 + 4]),
                             __float_as_uint(f[i2 + 5]), __float_as_uint(f[i2 + 6]), __float_as_uint(f[i2 + 7]));
            } else {
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2)
                if (i2 < nvalid) dst[i2] = f[i2];
            }
          } else if (p.out_fp32) {
            float *dst = reinterpret_cast<float *>(p.d) + orow * p.ldd + n;
            if (p.accumulate_d) {
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2)
                if (i2 < nvalid) {
                  sq += f[i2] * f[i2];
                  dst[i2] = dst[i2] + f[i2];
                }
            } else if (full_chunk) {
              // whole 32-byte sectors per store where the row allows it
              if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
#pragma unroll
                for (int i2 = 0; i2 < 32; i2 += 8)
                  st_global_v8(dst + i2, __float_as_uint(f[i2]), __float_as_uint(f[i2 + 1]),
                               __float_as_uint(f[i2 + 2]), __float_as_uint(f[i2 + 3]), __float_as_uint(f[i2 + 4]),
                               __float_as_uint(f[i2 + 5]), __float_as_uint(f[i2 + 6]), __float_as_uint(f[i2 + 7]));
              } else {
#pragma unroll
                for (int i2 = 0; i2 < 32; i2 += 4)
                  *reinterpret_cast<float4 *>(dst + i2) = make_float4(f[i2], f[i2 + 1], f[i2 + 2], f[i2 + 3]);
              }
              if (p.sqnorm)
#pragma unroll
                for (int i2 = 0; i2 < 32; ++i2) sq += f[i2] * f[i2];
            } else {
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2)
                if (i2 < nvalid) {
                  dst[i2] = f[i2];
                  sq += f[i2] * f[i2];
                }
            }
          } else {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.d) + orow * p.ldd + n;
            if (p.accumulate_d) {
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2)
                if (i2 < nvalid) {
                  sq += f[i2] * f[i2];
                  dst[i2] = __float2bfloat16_rn(__fadd_rn(__bfloat162float(dst[i2]), f[i2]));
                }
            } else if (full_chunk) {
              uint32_t w[16];
#pragma unroll
              for (int i2 = 0; i2 < 16; ++i2) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * i2], f[2 * i2 + 1]);
                w[i2] = *reinterpret_cast<const uint32_t *>(&h2);
              }
              // whole 32-byte sectors per store where the row allows it
              if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
                st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
              } else {
#pragma unroll
                for (int i2 = 0; i2 < 16; i2 += 4)
                  *reinterpret_cast<uint4 *>(dst + 2 * i2) = make_uint4(w[i2], w[i2 + 1], w[i2 + 2], w[i2 + 3]);
              }
              if (p.sqnorm)
#pragma unroll
                for (int i2 = 0; i2 < 32; ++i2) sq += f[i2] * f[i2];
            } else {
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2)
                if (i2 < nvalid) {
                  dst[i2] = __float2bfloat16_rn(f[i2]);
                  sq += f[i2] * f[i2];
                }
            }
          }
        }
      }
      acc_phase ^= 1;
    }
    if (p.sqnorm) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
      if (lane == 0) atomicAdd(p.sqnorm, sq);
    }
  }
  __syncthreads();
#ifdef NVFP4_WAIT_STATS
  if (threadIdx.x == 0) {
    unsigned long long *c = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(p.status) + 64);
    atomicAdd(c + 4, (unsigned long long)(clock64() - kernel_t0));
    atomicAdd(c + 5, 1ull);
  }
#endif
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------ LoRA down --
// T'[row, j] = bf16( s_row * sum_k X[src(row), k] A[j, k] ), fp32 accumulation
// in TMEM (kind::f16, M=128, N=rank, K=16 per instruction).  s_row =
// (alpha/r) / (g_a g_b[e]) when the result feeds the FP4 accumulator, alpha/r
// for the standalone path.  Grouped mode gathers X rows with 16-byte cp.async
// copies issued by warps 2..5 (eight lanes per row: coalesced reads, written in
// the 128-byte swizzled arrangement the MMA descriptor expects), up to three
// stages in flight per thread; the A tiles still come by TMA.
constexpr int kLoraStages = 6;
constexpr int kLoraThreads = 192;
constexpr int kGatherThreads = 128;   // warps 2..5 gather X rows in grouped mode

// A stage holds two 64-wide K sub-tiles: [X0 | X1 | A0 | A1], X tiles 128 rows x 128 B.
constexpr int kLoraSub = 2;
__host__ __device__ constexpr int lora_stage_bytes(int rank) { return kLoraSub * (kBM * 128 + rank * 128); }
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
      // grouped: the producer's arrival + one per gathering thread
      mbar_init(&full[s], p.row_map ? 1 + kGatherThreads : 1);
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
  griddep_launch_dependents();
  griddep_wait();   // inputs of this kernel come from the previous one in the stream
  const int ksplit = p.ksplit > 1 ? p.ksplit : 1;
  const int num_tiles = (p.gtiles ? *p.gnum_mtiles : p.tiles_m) * ksplit;   // (tile, K range)
  // K range of a unit, in 64-wide steps, a multiple of the stage width
  const int k64_per = ((p.num_k64 + ksplit - 1) / ksplit + kLoraSub - 1) / kLoraSub * kLoraSub;

  const uint32_t x_sub = kBM * 128, a_sub = (uint32_t)p.rank * 128;
  if (warp == 0) {
    const uint32_t sbase = smem_u32(base);
    const uint32_t full_base = smem_u32(full), empty_base = smem_u32(empty);
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_par = 0;
    bool ok = true;
    // X is read again by the packing pass right after this one: ask L2 to keep it
    const uint64_t xpol = l2_policy_evict_last();
    for (int u = blockIdx.x; ok && u < num_tiles; u += gridDim.x) {
      const int t = u / ksplit;
      const int kb = (u % ksplit) * k64_per, ke = min(p.num_k64, kb + k64_per);
      const int nsteps = (ke - kb + kLoraSub - 1) / kLoraSub;
      const int64_t row0 = p.gtiles ? (int64_t)p.gtiles[t].a_row0 : (int64_t)t * kBM;
      const int a_row = p.gtiles ? p.gtiles[t].expert * p.rank : 0;   // this expert's A
      for (int st = 0; st < nsteps; ++st) {
        bool good = true;
        if (lane == 0)
          good = !*abort_flag && mbar_wait_u(empty_base + 8 * stage, phase ^ 1, p.timeout_ns);
        good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
        if (!good) {
          if (lane == 0) signal_abort(abort_flag, p.status);
          ok = false;
          break;
        }
        const uint32_t fb = full_base + 8 * stage;
        const uint32_t sx = sbase + stage * sbytes, sa = sx + kLoraSub * x_sub;
        const int k64 = kb + st * kLoraSub;
        const int nsub = min(kLoraSub, ke - k64);
        if (lane == 0) {
          mbar_arrive_expect_tx_u(fb, nsub * ((p.row_map ? 0 : x_sub) + a_sub));
          for (int j = 0; j < nsub; ++j) {
            tma_load_2d_u(sa + j * a_sub, &tmA, fb, (k64 + j) * 64, a_row);
            if (!p.row_map) tma_load_2d_hint_u(sx + j * x_sub, &tmX, fb, (k64 + j) * 64, (int)row0, xpol);
          }
        }
        __syncwarp();
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
      for (int s2 = 0; s2 < stages; ++s2)
        if (armed & (1u << s2)) mbar_wait(&full[s2], (armed_par >> s2) & 1, kDrainNs);
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kBM, p.rank);
      const uint64_t desc0 = sdesc_k_sw128(base);
      const uint32_t full_base = smem_u32(full), empty_base = smem_u32(empty);
      const uint32_t accf = smem_u32(acc_full), acce = smem_u32(acc_empty);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < num_tiles; u += gridDim.x) {
        const int kb = (u % ksplit) * k64_per, ke = min(p.num_k64, kb + k64_per);
        const int nsteps = (ke - kb + kLoraSub - 1) / kLoraSub;
        if (*abort_flag || !mbar_wait_u(acce, acc_phase ^ 1, p.timeout_ns)) {
          signal_abort(abort_flag, p.status);
          break;
        }
        tc_fence_after();
        for (int st = 0; st < nsteps; ++st) {
          if (*abort_flag || !mbar_wait_u(full_base + 8 * stage, phase, p.timeout_ns)) {
            signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const int nsub = min(kLoraSub, ke - (kb + st * kLoraSub));
          const uint64_t sdesc = desc0 + (uint64_t)((stage * sbytes) >> 4);
          for (int j = 0; j < nsub; ++j) {
            const uint64_t adesc = sdesc + ((j * x_sub) >> 4);
            const uint64_t bdesc = sdesc + ((kLoraSub * x_sub + j * a_sub) >> 4);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              tc_mma_bf16(tmem, adesc + 2 * q, bdesc + 2 * q, idesc, (st | j | q) != 0);
          }
          tc_commit_u(empty_base + 8 * stage);
          if (++stage == stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_u(accf);
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
    for (int u = blockIdx.x; ok && u < num_tiles; u += gridDim.x) {
      const int t = u / ksplit, ks = u % ksplit;
      const int kb = ks * k64_per, ke = min(p.num_k64, kb + k64_per);
      const int nsteps = (ke - kb + kLoraSub - 1) / kLoraSub;
      int64_t row0;
      int e = 0;
      if (p.row_map) {
        // gather this unit's X rows: thread r copies 16-byte chunk (r & 7) of
        // tile rows (r >> 3) + 16 i, i = 0..7 (token row_map[row0 + row];
        // padding rows read as zeros), so the eight lanes of a row read its
        // 128 contiguous bytes (coalesced) and land in the swizzled slots
        const int64_t g_row0 = p.gtiles ? (int64_t)p.gtiles[t].a_row0 : (int64_t)t * kBM;
        const int gc = r & 7, grow = r >> 3;
        const uint32_t swz = (uint32_t)((gc ^ (grow & 7)) << 4);
        int32_t srow[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          srow[i] = p.row_map[g_row0 + grow + 16 * i];
          if (!NVFP4_GUARD(srow[i] < p.x_rows, p.status)) srow[i] = -1;
        }
        int pend[3];
        int npend = 0;
        for (int st = 0; st < nsteps; ++st) {
          if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(&empty[stage], phase ^ 1, p.timeout_ns))) {
            if (lane == 0) signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          const int k64 = kb + st * kLoraSub;
          const int nsub = min(kLoraSub, ke - k64);
          const uint32_t dst0 = smem_u32(base + stage * sbytes) + (uint32_t)(grow * 128) + swz;
          for (int j = 0; j < nsub; ++j) {
            const int64_t kel = (int64_t)(k64 + j) * 64 + gc * 8;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const bool in = srow[i] >= 0 && kel < p.K;
              cp_async_16(dst0 + j * x_sub + (uint32_t)(i * 16 * 128),
                          in ? p.x + (int64_t)srow[i] * p.K + kel : p.x, in ? 16u : 0u);
            }
          }
          cp_async_commit();
          pend[npend++] = stage;
          if (npend == 3) {
            // the oldest group has landed: publish it to the MMA (async proxy)
            cp_async_wait<2>();
            fence_proxy_async_shared();
            mbar_arrive(&full[pend[0]]);
            pend[0] = pend[1];
            pend[1] = pend[2];
            npend = 2;
          }
          if (++stage == stages) {
            stage = 0;
            phase ^= 1;
          }
        }
        cp_async_wait<0>();
        fence_proxy_async_shared();
        for (int i = 0; i < npend; ++i) mbar_arrive(&full[pend[i]]);
        if (!ok) break;
      }
      if (scan) {
        // max |x| over this warp's 32 rows of every X tile, read from shared memory
        for (int st = 0; st < nsteps; ++st) {
          if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(&full[stage], phase, p.timeout_ns))) {
            if (lane == 0) signal_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          const int nsub = min(kLoraSub, ke - (kb + st * kLoraSub));
          for (int j = 0; j < nsub; ++j) {
            const uint4 *row = reinterpret_cast<const uint4 *>(base + stage * sbytes + j * x_sub + r * 128);
            // The tile is 128-byte swizzled (16-byte chunk c of row r sits at
            // c ^ (r & 7)); visiting chunks in the order i ^ (r & 7) makes the
            // eight lanes of each quarter-warp hit eight different chunks
            // (conflict-free); the max over the row is order-independent.
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = row[i ^ (r & 7)];
              m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
              m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
              m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
              m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
            }
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
          float4 *dst = reinterpret_cast<float4 *>(p.t_f32 + ((int64_t)ks * p.M + row) * p.rank + c * 32);
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
// Four consecutive outputs per thread and pass (N % 4 == 0): the partials of
// every K range are loaded before they are added, so the loads of a pass are
// in flight together; sums in K-range order as below.
__global__ void k_splitk_reduce4(const GemmParams p) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  constexpr int kMaxSplit = 16;
  const int64_t total = p.M * p.N, quads = total / 4;
  const float4 *part = reinterpret_cast<const float4 *>(p.partial);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < quads;
       i += (int64_t)gridDim.x * blockDim.x) {
    float4 v[kMaxSplit];
#pragma unroll
    for (int k = 0; k < kMaxSplit; ++k)
      if (k < p.ksplit) v[k] = part[k * quads + i];
    float4 s = v[0];
#pragma unroll
    for (int k = 1; k < kMaxSplit; ++k)
      if (k < p.ksplit) {
        s.x = __fadd_rn(s.x, v[k].x);
        s.y = __fadd_rn(s.y, v[k].y);
        s.z = __fadd_rn(s.z, v[k].z);
        s.w = __fadd_rn(s.w, v[k].w);
      }
    const int64_t e = 4 * i, m = e / p.N, n = e - m * p.N;
    if (p.out_fp32) {
      *reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.d) + m * p.ldd + n) = s;
    } else {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y), hi = __floats2bfloat162_rn(s.z, s.w);
      *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(p.d) + m * p.ldd + n) =
          make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
    }
  }
}

__global__ void k_splitk_reduce(const GemmParams p) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
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
  // the vector form: rows of whole quads, 16-byte partials, aligned output quads
  const bool quad = p.N % 4 == 0 && p.ldd % 4 == 0 && p.ksplit <= 16 &&
                    (reinterpret_cast<uintptr_t>(p.partial) & 15) == 0 &&
                    (reinterpret_cast<uintptr_t>(p.d) & (p.out_fp32 ? 15 : 7)) == 0;
  if (quad) {
    const int64_t quads = total / 4;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((quads + 255) / 256, (int64_t)num_sms * 8));
    return launch_pdl(k_splitk_reduce4, dim3(grid), dim3(256), 0, st, p);
  }
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)num_sms * 4));
  return launch_pdl(k_splitk_reduce, dim3(grid), dim3(256), 0, st, p);
}

// ----------------------------------------------------------------- launch --

template <int BN>
static cudaError_t launch_bn(const GemmParams &p, const GemmMaps &m, int num_sms, cudaStream_t st) {
  using C = GemmCfg<BN>;
  if (cudaError_t e = ensure_dynamic_smem((const void *)k_gemm_fp4<BN>, C::kSmemBytes); e != cudaSuccess) return e;
  int64_t tiles = (int64_t)p.tiles_n * (p.gtiles ? 0 : p.tiles_m) * std::max(1, p.ksplit);
  int grid = num_sms;
#ifdef NVFP4_WAIT_STATS
  if (const char *cap = getenv("NVFP4_GRID_CAP")) grid = std::max(1, std::min(grid, atoi(cap)));
#endif
  if (!p.gtiles) grid = (int)std::min<int64_t>(tiles, grid);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(k_gemm_fp4<BN>, dim3(grid), dim3(kGemmThreads), C::kSmemBytes, st, m.a, m.b, m.t, m.lb, p);
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
  if (cudaError_t e = ensure_dynamic_smem((const void *)k_lora_down, smem); e != cudaSuccess) return e;
  int grid = num_sms;
  if (!p.gtiles) grid = std::min(p.tiles_m * std::max(1, p.ksplit), num_sms);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(k_lora_down, dim3(grid), dim3(kLoraThreads), smem, st, m.x, m.a, p, stages);
}

}  // namespace nvfp4
