// gemm_skinny.cu -- the W4A4 product for a few activation rows (decode,
// M <= 32) on tcgen05, with the operands swapped.
//
// Same product as k_gemm_fp4 (gemm.cu): Y[m, n] = g_x g_w * sum_k
// e2m1(x_mk) sx(m, k/16) e2m1(w_nk) sw(n, k/16), both operands K-major with one
// E4M3 scale per 16 elements ("vroomfondel/glm-5.2-reap-504B-v2-W4A4" card,
// "Kernel choice" and "What this variant changes": at decode the projection is
// a stream of the weights).  Here the weights are the MMA's 128-row A operand
// and the <= 32 activation rows its B operand (N = 32): the accumulator holds
// Y^T for 128 output features, and a stage carries 16 KB of weights and only
// 4 KB of activations (24 KB with both scale atoms), so nine stages -- 144 KB
// of weights -- are in flight per SM instead of the six (96 KB) of the
// 128 x 128 tile whose A side would be the padded activation rows.
//
// A persistent kernel, one CTA per SM, 192 threads:
//   warp 0      producer (one thread): the stage's weight tile (128 rows x
//               256 codes) and activation tile (32 rows x 256 codes) by
//               TMA, their scale atoms by bulk copy.
//   warp 1      MMA issue (one thread): kind::mxf4nvf4 scale_vec::4X, M=128,
//               N=32, K=64, four per stage.
//   warps 2..5  scales -> tensor memory for every stage; after a unit's last
//               stage they drain the 128 x 32 accumulator and store Y (or the
//               unit's fp32 split-K partial) transposed: lane = feature n,
//               one store per activation row, coalesced across the warp.
// Work units are (128-feature tile, K range); K ranges are summed in order by
// the split-K pass.  Every wait is bounded.
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

constexpr int kSkThreads = 192;
constexpr int kSkStages = 9;
constexpr int kSkN = 32;                         // activation rows per MMA (B operand)
constexpr int kSkABytes = 128 * 128;             // 128 weight rows x 256 codes
constexpr int kSkBBytes = kSkN * 128;            // 32 activation rows x 256 codes
constexpr int kSkSfBytes = 4 * 512;              // one 128-row chunk, four 128x4 atoms
constexpr int kSkStageBytes = kSkABytes + kSkBBytes + 2 * kSkSfBytes;
constexpr int kSkSmemBytes = kSkStages * kSkStageBytes + 256 + 1024;
// TMEM: 32 accumulator columns, then per stage 16 columns of weight scales and
// 16 of activation scales (4 per K step each: lane i of every quarter holds
// line i of the atom, rows i, i+32, i+64, i+96 -- the MMA reads row r of an
// operand from lane r % 32, column r / 32 of its K step)
constexpr int kSkSfCols = 32;
constexpr int kSkTmemCols = 512;
constexpr uint64_t kSkDrainNs = 200000000ull;
static_assert(kSkN + kSkStages * kSkSfCols <= kSkTmemCols, "TMEM budget");
static_assert(kSkSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void sk_abort(volatile int *abort_flag, int *status) {
  *abort_flag = 1;
  record_timeout(status);
}

}  // namespace

// p.M activation rows (<= 32), p.N features, a_* = activations, b_* = weights
// (as for k_gemm_fp4); tmX: activation codes, box 128 B x 32 rows; tmW: weight
// codes, box 128 B x 128 rows.
__global__ void __launch_bounds__(kSkThreads, 1)
    k_gemm_fp4_skinny(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                      const GemmParams p) {
  constexpr int S = kSkStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sW = base;
  uint8_t *sX = sW + S * kSkABytes;
  uint8_t *sSFW = sX + S * kSkBBytes;
  uint8_t *sSFX = sSFW + S * kSkSfBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sSFX + S * kSkSfBytes);
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
      mbar_init(&sfready[s], 4);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 4);
    mbar_init(drain, 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kSkTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();
  // Inputs of this kernel come from the previous one in the stream (the
  // activation packing), which lets this grid start only after every kernel
  // before it has completed: the producer issues the weight tiles of its
  // first stages before its wait, every other thread waits here.
  if (warp != 0) griddep_wait();

  const int ksplit = p.ksplit > 1 ? p.ksplit : 1;
  const int num_units = p.tiles_n * ksplit;          // (128-feature tile, K range)
  const int kt_per = (p.num_kt + ksplit - 1) / ksplit;
  const int last_nk = p.nk64 - (p.num_kt - 1) * 4;   // K steps of the last 256-wide K tile

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const uint32_t w_base = smem_u32(sW), x_base = smem_u32(sX);
      const uint32_t sfw_base = smem_u32(sSFW), sfx_base = smem_u32(sSFX);
      const uint32_t full_base = smem_u32(full), empty_base = smem_u32(empty);
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      // the first unit's first stages (all free at entry): weights before the wait
      int pre = 0;
      if ((int)blockIdx.x < num_units) {
        const int nt = blockIdx.x / ksplit;
        const int kt0 = (blockIdx.x % ksplit) * kt_per, kt1 = min(p.num_kt, kt0 + kt_per);
        pre = min(S, kt1 - kt0);
        const uint8_t *sfw_src = p.b_sf + 512 * ((int64_t)nt * p.b_sf_katoms + (int64_t)kt0 * 4);
        for (int i = 0; i < pre; ++i) {
          const int kt = kt0 + i;
          const uint32_t fb = full_base + 8 * i;
          const uint32_t sfb = (uint32_t)((kt == p.num_kt - 1 ? last_nk : 4) * 512);
          mbar_arrive_expect_tx_u(fb, kSkABytes + kSkBBytes + 2 * sfb);
          tma_load_2d_u(w_base + i * kSkABytes, &tmW, fb, kt * 128, nt * 128);
          bulk_load_u(sfw_base + i * kSkSfBytes, sfw_src, sfb, fb);
          sfw_src += 2048;
        }
      }
      griddep_wait();
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const int nt = u / ksplit;
        const int kt0 = (u % ksplit) * kt_per, kt1 = min(p.num_kt, kt0 + kt_per);
        const uint8_t *sfw_src = p.b_sf + 512 * ((int64_t)nt * p.b_sf_katoms + (int64_t)kt0 * 4);
        const uint8_t *sfx_src = p.a_sf + 512 * ((int64_t)kt0 * 4);   // the rows' one 128-row chunk
        for (int kt = kt0; kt < kt1; ++kt) {
          const bool early = u == (int)blockIdx.x && kt - kt0 < pre;   // weights already in flight
          const bool got = early || (!*abort_flag && mbar_wait_u(empty_base + 8 * stage, phase ^ 1, p.timeout_ns));
          if (!got) {
            sk_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          const uint32_t fb = full_base + 8 * stage;
          const uint32_t sfb = (uint32_t)((kt == p.num_kt - 1 ? last_nk : 4) * 512);
          if (!early) {
            mbar_arrive_expect_tx_u(fb, kSkABytes + kSkBBytes + 2 * sfb);
            tma_load_2d_u(w_base + stage * kSkABytes, &tmW, fb, kt * 128, nt * 128);
            bulk_load_u(sfw_base + stage * kSkSfBytes, sfw_src, sfb, fb);
          }
          tma_load_2d_u(x_base + stage * kSkBBytes, &tmX, fb, kt * 128, 0);
          bulk_load_u(sfx_base + stage * kSkSfBytes, sfx_src, sfb, fb);
          sfw_src += 2048;
          sfx_src += 2048;
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == S) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every fill this thread started lands before the CTA may exit
      for (int s = 0; s < S; ++s)
        if (armed & (1u << s)) mbar_wait(&full[s], (armed_par >> s) & 1, kSkDrainNs);
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issue --
    if (lane == 0) {
      const uint32_t idesc = idesc_nvfp4(128, kSkN);
      const uint64_t wdesc0 = sdesc_k_sw128(sW), xdesc0 = sdesc_k_sw128(sX);
      const uint32_t sfr_base = smem_u32(sfready), empty_base = smem_u32(empty);
      const uint32_t accf = smem_u32(acc_full), acce = smem_u32(acc_empty);
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      if (p.stall_probe && !mbar_wait(never, 0, p.timeout_ns)) {
        sk_abort(abort_flag, p.status);   // expected: the expiry path under test
        ok = false;
      }
      for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
        const int kt0 = (u % ksplit) * kt_per, kt1 = min(p.num_kt, kt0 + kt_per);
        if (*abort_flag || !mbar_wait_u(acce, acc_phase ^ 1, p.timeout_ns)) {
          sk_abort(abort_flag, p.status);
          break;
        }
        tc_fence_after();
        uint32_t accumulate = 0;
        for (int kt = kt0; kt < kt1; ++kt) {
          // the stage's operands have landed and its scales are in tensor memory
          if (*abort_flag || !mbar_wait_u(sfr_base + 8 * stage, phase, p.timeout_ns)) {
            sk_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = kt == p.num_kt - 1 ? last_nk : 4;
          const uint64_t wdesc = wdesc0 + (uint64_t)((stage * kSkABytes) >> 4);
          const uint64_t xdesc = xdesc0 + (uint64_t)((stage * kSkBBytes) >> 4);
          const uint32_t sfw_col = tmem + kSkN + stage * kSkSfCols, sfx_col = sfw_col + 16;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j < nk) {
              tc_mma_nvfp4(tmem, wdesc + 2 * j, xdesc + 2 * j, idesc, sfw_col + 4 * j, sfx_col + 4 * j, accumulate);
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
      mbar_wait(drain, 0, kSkDrainNs);
    }
  } else {
    // ------------------------------- scales -> tensor memory, then epilogue --
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    const float alpha = acc_scale_of(p.g_a ? *p.g_a : 1.0f, p.g_b ? *p.g_b : 1.0f);
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
      const int nt = u / ksplit, ks = u % ksplit;
      const int kt0 = ks * kt_per, kt1 = min(p.num_kt, kt0 + kt_per);
      for (int kt = kt0; kt < kt1; ++kt) {
        if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(&full[stage], phase, p.timeout_ns))) {
          if (lane == 0) sk_abort(abort_flag, p.status);
          ok = false;
          break;
        }
        const uint4 *fw = reinterpret_cast<const uint4 *>(sSFW + stage * kSkSfBytes) + lane;
        const uint4 *fx = reinterpret_cast<const uint4 *>(sSFX + stage * kSkSfBytes) + lane;
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = fw[32 * j];                // atom j, line `lane`
          v[4 * j] = w.x; v[4 * j + 1] = w.y; v[4 * j + 2] = w.z; v[4 * j + 3] = w.w;
        }
        tmem_st_32x32b_x16(tq + kSkN + stage * kSkSfCols, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = fx[32 * j];
          v[4 * j] = w.x; v[4 * j + 1] = w.y; v[4 * j + 2] = w.z; v[4 * j + 3] = w.w;
        }
        tmem_st_32x32b_x16(tq + kSkN + stage * kSkSfCols + 16, v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfready[stage]);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok) break;
      // epilogue: thread = feature n0 + 32q + lane, its 32 columns = the activation rows
      if (!__all_sync(0xffffffffu, !*abort_flag && mbar_wait(acc_full, acc_phase, p.timeout_ns))) {
        if (lane == 0) sk_abort(abort_flag, p.status);
        break;
      }
      tc_fence_after();
      uint32_t acc[32];
      __syncwarp();
      tmem_ld_32x32b_x32(tq, acc);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      acc_phase ^= 1;
      const int row = q * 32 + lane;
      const int64_t n = (int64_t)nt * 128 + row;
      float f[kSkN];
#pragma unroll
      for (int m = 0; m < kSkN; ++m) f[m] = __fmul_rn(__uint_as_float(acc[m]), alpha);
      if (n < p.N) {
#pragma unroll
        for (int m = 0; m < kSkN; ++m) {
          if (m < p.M) {
            if (p.partial)
              p.partial[((int64_t)ks * p.M + m) * p.N + n] = f[m];
            else if (p.out_fp32)
              reinterpret_cast<float *>(p.d)[m * p.ldd + n] = f[m];
            else
              reinterpret_cast<__nv_bfloat16 *>(p.d)[m * p.ldd + n] = __float2bfloat16_rn(f[m]);
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kSkTmemCols);
  }
}

cudaError_t launch_gemm_fp4_skinny(const GemmParams &p, const CUtensorMap &x, const CUtensorMap &w, int num_sms,
                                   cudaStream_t st) {
  if (cudaError_t e = ensure_dynamic_smem((const void *)k_gemm_fp4_skinny, kSkSmemBytes); e != cudaSuccess) return e;
  const int64_t units = (int64_t)p.tiles_n * std::max(1, p.ksplit);
  const int64_t grid = std::min<int64_t>(units, num_sms);
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(k_gemm_fp4_skinny, dim3((unsigned)grid), dim3(kSkThreads), kSkSmemBytes, st, x, w, p);
}

}  // namespace nvfp4
