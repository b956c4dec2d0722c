// gemm_pair.cu -- the dense W4A4 GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same product as k_gemm_fp4 (gemm.cu): the W4A4 product of two NVFP4 operands
// with fp32 accumulation ("vroomfondel/glm-5.2-reap-504B-v2-W4A4" card, "Kernel
// choice"), both operands K-major with one E4M3 scale per 16 elements along K
// ("Getting GLM-5.2 NVFP4 Post-Training off the ground", "TN, NT, and what
// actually binds"), plus the bf16 LoRA up-projection as extra kind::f16 K
// steps (same page, TL;DR).
//
// Why pairs: one M=128 x N=256 x K=64 block-scaled MMA takes 128 cycles of the
// tensor pipe (measured), and its operands are 12 KB (+1.5 KB of scales): ~105
// B/cycle per SM from L2, while tile loads from L2 with every SM loading were
// measured at ~48-61 B/cycle per SM.  The pair MMA computes a 256 x 256 tile
// on two SMs: each SM supplies its own 128 A rows and half of the B tile and
// the instruction reads the other half from the peer's shared memory, so each
// SM loads 4 KB of A, 4 KB of B and 1.5 KB of scales per 128 cycles (~74
// B/cycle), and a stage is 38.9 KB instead of 54 KB (five stages in flight
// instead of four).  In steady state the stage copies arrive at ~56 B/cycle
// per SM, close to what bulk copies from L2 reach with every SM loading: that
// bandwidth, not the tensor pipe, bounds the kernel (~700 cycles a stage).
//
// A persistent kernel on clusters of two CTAs, one per SM, 384 threads each:
//   warps 0, 10, 11  producers (both CTAs), one thread each: its 128 A rows,
//               its 128-row half of B, and the scales of its A rows and of all
//               256 B rows (one issuing warp per stream: a single warp issuing
//               16 KB tile loads was measured at ~24 B/cycle per SM).
//   warp 1      leader CTA only: one thread waits on one barrier per stage --
//               both CTAs' tiles landed (the peer's loads complete on the
//               leader's barrier) and both CTAs' scale warps arrived -- then
//               issues the pair MMAs (kind::mxf4nvf4 scale_vec::4X, M=256,
//               N=256, K=64), two stages per loop iteration, and the LoRA
//               kind::f16 steps; each commit arrives on the barriers of both
//               CTAs (multicast).
//   warps 2..5  scales -> own tensor memory (tcgen05.st), then arrive on the
//               leader's stage barrier (remote arrive for the peer).
//   warps 6..9  epilogue: drain own 128 x 256 accumulator, arrive on the
//               leader's "accumulator free" barrier, scale, convert, store
//               (bf16 through shared-memory boxes and tensor stores).
// Every wait is bounded; on expiry a CTA records a timeout, drains its own
// copies (and, in the leader, its MMAs) and leaves its loops; the peer's waits
// then expire too.  Both CTAs meet at a cluster barrier before freeing TMEM.
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

namespace {

constexpr int kPairThreads = 384;
constexpr int kPairStages = 5;
constexpr int kPABytes = 128 * 128;            // this CTA's 128 A rows x 256 FP4 (or 64 bf16)
constexpr int kPBBytes = 128 * 128;            // this CTA's half of the B tile
constexpr int kPSfaBytes = 4 * 512;            // 128 A rows x 16 scales (four 128x4 atoms)
constexpr int kPSfbBytes = 2 * 4 * 512;        // 256 B rows x 16 scales (two 128-row chunks)
constexpr int kPStageBytes = kPABytes + kPBBytes + kPSfaBytes + kPSfbBytes;
constexpr int kPBarBytes = 256;
// epilogue staging for the bf16 output's tensor stores: per epilogue warp four
// 32 x 32 bf16 boxes (2 KB each), 1024-aligned
constexpr int kPStgBytes = 4 * 4 * 2048;
constexpr int kPSmemBytes = kPairStages * kPStageBytes + kPBarBytes + 1024 + kPStgBytes + 1024;
// TMEM columns of one stage's scales: 4 per K step for A, then 8 per K step
// for B.  The MMA of K step j reads the A scale of row r from lane r, column
// base + 4j + r/32, so lane quarter q needs only column base + 4j + q (one
// single-column store per K step); the B scales are replicated in every lane
// quarter.  Wider stores (.x4, .x16) need columns aligned to their width: the
// stage stride and both regions stay multiples of 16.
constexpr int kPSfaCols = 16;
constexpr int kPSfCols = kPSfaCols + 32;
static_assert(kPSfCols % 16 == 0 && kPSfaCols % 16 == 0, "TMEM store alignment");
constexpr int kPTmemCols = 512;
constexpr uint64_t kPDrainNs = 200000000ull;
static_assert(256 + kPairStages * kPSfCols <= kPTmemCols, "TMEM budget");
static_assert(kPSmemBytes <= 232448, "shared memory budget");

struct PairTile {
  int64_t m0, n0;      // first row of the unit's A (256 rows) and B (256 or 128 rows)
  bool half;           // a 256 x 128 unit: one half of a tail tile
};

// The work units of a launch.  256 x 256 tiles, n-tile major (the pairs
// running together share B tiles; A stays in L2), dealt round-robin to the
// pairs.  When the tiles leave a last wave that fills at most half of the
// pairs (and the host allows it), each tile of that wave is dealt as two
// 256 x 128 units instead, so that the last wave takes about half a tile's
// time on twice as many pairs.  Every role derives the same schedule from
// the grid size.
struct PairSchedule {
  int tiles_m2;        // 256-row tiles along M
  int split_from;      // units before this are whole tiles
  int num_units;
};

__device__ __forceinline__ PairSchedule pair_schedule(const GemmParams &p, int npairs) {
  PairSchedule s;
  s.tiles_m2 = (int)((p.M + 255) / 256);
  const int tiles = s.tiles_m2 * p.tiles_n;
  const int tail = tiles % npairs;
  const bool split = p.pair_half_tail && tail > 0 && 2 * tail <= npairs;
  s.split_from = split ? tiles - tail : tiles;
  s.num_units = split ? tiles + tail : tiles;
  return s;
}

__device__ __forceinline__ PairTile pair_tile(const PairSchedule &s, int u) {
  PairTile t;
  int v = u, sub = 0;
  t.half = u >= s.split_from;
  if (t.half) {
    v = s.split_from + ((u - s.split_from) >> 1);
    sub = (u - s.split_from) & 1;
  }
  t.n0 = (int64_t)(v / s.tiles_m2) * 256 + 128 * sub;
  t.m0 = (int64_t)(v % s.tiles_m2) * 256;
  return t;
}

// Optional wait statistics (compile with -DNVFP4_WAIT_STATS): cycles each role
// of each CTA of the pair spends in waits, summed over pairs into 64-bit
// counters at byte 64 of the workspace (the status word's reserved block):
// [8 * rank + role], roles 0 producer (stage free), 1 MMA (stage ready),
// 2 MMA (accumulator free), 3 scale warp (stage full), 4 epilogue (accumulator
// full), 5 kernel cycles, 6 CTAs.  Off in normal builds.
#ifdef NVFP4_WAIT_STATS
#define PSTAT_T0() const long long _ps_t0 = clock64()
#define PSTAT_ADD(p, rank, i)                                                                             \
  atomicAdd(reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>((p).status) + 64) + 8 * (rank) + (i), \
            (unsigned long long)(clock64() - _ps_t0))
#else
#define PSTAT_T0() (void)0
#define PSTAT_ADD(p, rank, i) (void)0
#endif

__device__ __forceinline__ void pair_abort(volatile int *abort_flag, int *status) {
  *abort_flag = 1;
  record_timeout(status);
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    k_gemm_fp4_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmT, const __grid_constant__ CUtensorMap tmLB,
                    const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmLBh,
                    const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  constexpr int S = kPairStages;
#ifdef NVFP4_WAIT_STATS
  const long long kernel_t0 = clock64();
#endif
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = base;
  uint8_t *sB = sA + S * kPABytes;
  uint8_t *sSFA = sB + S * kPBBytes;
  uint8_t *sSFB = sSFA + S * kPSfaBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sSFB + S * kPSfbBytes);
  uint8_t *stg = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(bars) + kPBarBytes + 1023) &
                                             ~uintptr_t(1023));
  // full (the leader's copy): both CTAs' A and B tiles landed -- the peer's
  // tile loads complete on the leader's barrier -- and both CTAs' scale warps
  // have written the stage's scales into tensor memory; sf_full: this CTA's scales
  // landed (small copies, so the scale warps fill tensor memory while the
  // tiles are still in flight)
  uint64_t *full = bars, *empty = bars + S, *sf_full = bars + 3 * S;
  uint64_t *acc_full = bars + 4 * S, *acc_empty = acc_full + 1, *drain = acc_full + 2;
  uint64_t *never = acc_full + 3;          // test hook: a barrier nothing arrives at
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 4);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // the leader's A and B producers (with the bytes of both CTAs) and the
      // scale warps of both CTAs: the MMA thread waits on one barrier a stage
      mbar_init(&full[s], 2 + 2 * 4);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_full[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 2 * 4);         // the epilogue warps of both CTAs (leader's copy used)
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
    if (p.pair_half_tail) {
      tma_prefetch_desc(&tmBh);
      if (p.lora_steps) tma_prefetch_desc(&tmLBh);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();      // both CTAs' barriers exist before any remote arrive or multicast commit
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();
  griddep_wait();      // inputs of this kernel come from the previous one in the stream

  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const PairSchedule sched = pair_schedule(p, npairs);
  const int num_units = sched.num_units;
  const int a_sf_chunks = (int)((p.M + 127) / 128);
  // the leader's barriers as cluster addresses (for the peer: its remote copy)
  const uint32_t full_l = mapa_shared(smem_u32(full), 0);
  const uint32_t acc_empty_l = mapa_shared(smem_u32(acc_empty), 0);

  if ((warp == 0 || warp >= 10) && lane == 0) {
    // ----------------------------------------------------------- producers --
    // Three threads in three warps, one per operand stream: warp 0 the A tile
    // (or T'), warp 10 the B half (or LB), warp 11 the scales.  Each waits for
    // the stage to be freed by the leader's multicast commit.
    const int role = warp == 0 ? 0 : warp - 9;            // 0: A, 1: B, 2: scales
    const uint32_t a_base = smem_u32(sA), b_base = smem_u32(sB);
    const uint32_t sfa_base = smem_u32(sSFA), sfb_base = smem_u32(sSFB);
    const uint32_t full_base = smem_u32(full), empty_base = smem_u32(empty);
    const uint32_t sff_base = smem_u32(sf_full);
    const int last_nk = p.num_kt ? p.nk64 - (p.num_kt - 1) * 4 : 0;
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_par = 0;
    bool ok = true;
    for (int u = pair; ok && u < num_units; u += npairs) {
      const PairTile t = pair_tile(sched, u);
      // a half unit's B is 128 rows: 64 in each CTA
      const int a_row = (int)(t.m0 + 128 * rank), b_row = (int)(t.n0 + (t.half ? 64 : 128) * rank);
      const uint32_t b_bytes = t.half ? kPBBytes / 2 : kPBBytes;
      const bool sfa_ok = (a_row >> 7) < a_sf_chunks;           // rows past the padded scales: codes are 0
      const int64_t chunk0 = t.n0 >> 7;
      const int chunks = !t.half && chunk0 + 1 < p.b_sf_row_chunks ? 2 : 1;  // B scale chunks read
      const uint8_t *sfa_src = p.a_sf + 512 * ((int64_t)(a_row >> 7) * p.a_sf_katoms);
      const uint8_t *sfb_src = p.b_sf + 512 * (chunk0 * p.b_sf_katoms);
      const int64_t sfb_chunk_stride = 512 * p.b_sf_katoms;
      const int nsteps = p.num_kt + p.lora_steps;
      for (int i = 0; i < nsteps; ++i) {
        PSTAT_T0();
        const bool got = !*abort_flag && mbar_wait_u(empty_base + 8 * stage, phase ^ 1, p.timeout_ns);
        if (role == 0) PSTAT_ADD(p, rank, 0);
        if (!got) {
          pair_abort(abort_flag, p.status);
          ok = false;
          break;
        }
        const uint32_t fb = full_base + 8 * stage, sfbar = sff_base + 8 * stage;
        if (role < 2) {
          // the leader expects both CTAs' tiles; the peer's land on the leader's barrier
          const CUtensorMap *tm = role == 0 ? (i < p.num_kt ? &tmA : &tmT)
                                            : t.half ? (i < p.num_kt ? &tmBh : &tmLBh)
                                                     : (i < p.num_kt ? &tmB : &tmLB);
          const uint32_t dst = role == 0 ? a_base + stage * kPABytes : b_base + stage * kPBBytes;
          const int c0 = i < p.num_kt ? i * 128 : (i - p.num_kt) * 64;
          const int c1 = role == 0 ? a_row : b_row;
          if (rank == 0) {
            mbar_arrive_expect_tx_u(fb, 2 * (role == 0 ? (uint32_t)kPABytes : b_bytes));
            tma_load_2d_u(dst, tm, fb, c0, c1);
          } else {
            tma_load_2d_pair_u(dst, tm, full_l + 8 * stage, c0, c1);
          }
        } else if (i < p.num_kt) {
          const int nk = i == p.num_kt - 1 ? last_nk : 4;
          const uint32_t sfb = nk * 512;
          mbar_arrive_expect_tx_u(sfbar, sfb * ((sfa_ok ? 1 : 0) + chunks));
          if (sfa_ok) bulk_load_u(sfa_base + stage * kPSfaBytes, sfa_src, sfb, sfbar);
          bulk_load_u(sfb_base + stage * kPSfbBytes, sfb_src, sfb, sfbar);
          if (chunks > 1) bulk_load_u(sfb_base + stage * kPSfbBytes + 2048, sfb_src + sfb_chunk_stride, sfb, sfbar);
          sfa_src += 2048;
          sfb_src += 2048;
        } else {
          mbar_arrive_u(sfbar);                 // no scales in a bf16 step: the phase completes at once
        }
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // every fill this thread started lands before the CTA may exit (the
    // peer's tiles are counted on the leader's barrier, which the leader's
    // producers drain; both CTAs' producers fill the same stages, each after
    // the same multicast commit)
    for (int s = 0; s < S; ++s)
      if ((armed & (1u << s)) && (role == 2 || rank == 0))
        mbar_wait(role == 2 ? &sf_full[s] : &full[s], (armed_par >> s) & 1, kPDrainNs);
  } else if (warp == 1) {
    // ----------------------------------------------- MMA issue (leader only) --
    if (lane == 0 && rank == 0) {
      uint32_t idesc = idesc_nvfp4(256, 256);
      uint32_t idesc_l = idesc_bf16(256, 256);
      const uint64_t adesc0 = sdesc_k_sw128(sA), bdesc0 = sdesc_k_sw128(sB);
      const uint32_t empty_base = smem_u32(empty);
      const uint32_t full_base = smem_u32(full);
      const uint32_t accf = smem_u32(acc_full), acce = smem_u32(acc_empty);
      const int last_nk = p.num_kt ? p.nk64 - (p.num_kt - 1) * 4 : 0;
      const int nsteps = p.num_kt + p.lora_steps;
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      if (p.stall_probe && !mbar_wait(never, 0, p.timeout_ns)) {
        pair_abort(abort_flag, p.status);   // expected: the expiry path under test
        ok = false;
      }
      // The issuing thread, not the tensor pipe, sets the pace: each MMA
      // instruction and each iteration's waits, commit and loop control cost
      // it tens to hundreds of cycles.  So one iteration takes two stages:
      // both stages' barriers are waited first (one barrier per stage: the
      // tiles and the scales), then the eight MMAs go out back to back with
      // a commit after each stage's four, and no flag is read per stage.
      auto issue_stage = [&](int st, int i, uint32_t &accumulate) {
        const uint64_t adesc = adesc0 + (uint64_t)((st * kPABytes) >> 4);
        const uint64_t bdesc = bdesc0 + (uint64_t)((st * kPBBytes) >> 4);
        if (i < p.num_kt) {
          const int nk = i == p.num_kt - 1 ? last_nk : 4;
          const uint32_t sfa_col = tmem + 256 + st * kPSfCols;
          const uint32_t sfb_col = sfa_col + kPSfaCols;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j < nk) {
              tc_mma_nvfp4_pair(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col + 4 * j, sfb_col + 8 * j,
                                accumulate);
              accumulate = 1;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_mma_bf16_pair(tmem, adesc + 2 * j, bdesc + 2 * j, idesc_l, accumulate);
            accumulate = 1;
          }
        }
        tc_commit_pair_mc(empty_base + 8 * st, 3);   // frees the stage in both CTAs
      };
      // one stage with all four K steps of FP4 (the first MMA accumulates
      // when `acc_first` is set)
      auto issue_full = [&](int st, uint32_t acc_first) {
        const uint64_t adesc = adesc0 + (uint64_t)((st * kPABytes) >> 4);
        const uint64_t bdesc = bdesc0 + (uint64_t)((st * kPBBytes) >> 4);
        const uint32_t sfa_col = tmem + 256 + st * kPSfCols;
        const uint32_t sfb_col = sfa_col + kPSfaCols;
        tc_mma_nvfp4_pair(tmem, adesc, bdesc, idesc, sfa_col, sfb_col, acc_first);
#pragma unroll
        for (int j = 1; j < 4; ++j)
          tc_mma_nvfp4_pair(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_col + 4 * j, sfb_col + 8 * j, 1u);
        tc_commit_pair_mc(empty_base + 8 * st, 3);   // frees the stage in both CTAs
      };
      const int nfull = p.num_kt - (last_nk < 4 ? 1 : 0);
      for (int u = pair; ok && u < num_units; u += npairs) {
        // a half unit: N = 128 (64 B rows in each CTA, one chunk of B scales)
        const bool half_unit = u >= sched.split_from;
        idesc = idesc_nvfp4(256, half_unit ? 128 : 256);
        idesc_l = idesc_bf16(256, half_unit ? 128 : 256);
        PSTAT_T0();
        const bool got_acc = !*abort_flag && mbar_wait_u(acce, acc_phase ^ 1, p.timeout_ns);
        PSTAT_ADD(p, rank, 2);
        if (!got_acc) {
          pair_abort(abort_flag, p.status);
          break;
        }
        tc_fence_after();
        uint32_t accumulate = 0;
        // pairs of full FP4 stages (all four K steps present), then the rest
        // (a partial last FP4 stage, the LoRA stages, bf16-only products) in
        // pairs of any kind
        int i = 0;
        for (; i + 2 <= nfull; i += 2) {
          const int stage1 = stage + 1 == S ? 0 : stage + 1;
          const uint32_t phase1 = stage + 1 == S ? phase ^ 1 : phase;
          PSTAT_T0();
          bool got = mbar_wait_u(full_base + 8 * stage, phase, p.timeout_ns);
          PSTAT_ADD(p, rank, 1);
          if (!got) {
            pair_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          issue_full(stage, accumulate);
          accumulate = 1;
          // the second stage's wait comes after the first stage's MMAs: the
          // stage it needs was freed by MMAs issued four stages back
          got = mbar_wait_u(full_base + 8 * stage1, phase1, p.timeout_ns);
          if (!got) {
            phase = phase1;
            stage = stage1;
            pair_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          issue_full(stage1, 1);
          phase = stage1 + 1 == S ? phase1 ^ 1 : phase1;
          stage = stage1 + 1 == S ? 0 : stage1 + 1;
        }
        for (; ok && i < nsteps; i += 2) {
          const int stage1 = stage + 1 == S ? 0 : stage + 1;
          const uint32_t phase1 = stage + 1 == S ? phase ^ 1 : phase;
          const bool two = i + 1 < nsteps;
          PSTAT_T0();
          const bool got = mbar_wait_u(full_base + 8 * stage, phase, p.timeout_ns) &&
                           (!two || mbar_wait_u(full_base + 8 * stage1, phase1, p.timeout_ns));
          PSTAT_ADD(p, rank, 1);
          if (!got) {
            pair_abort(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          issue_stage(stage, i, accumulate);
          stage = stage1;
          phase = phase1;
          if (two) {
            issue_stage(stage, i + 1, accumulate);
            phase = stage + 1 == S ? phase ^ 1 : phase;
            stage = stage + 1 == S ? 0 : stage + 1;
          }
        }
        if (!ok) break;
        tc_commit_pair_mc(accf, 3);                        // both CTAs' accumulators are ready
        acc_phase ^= 1;
      }
      // every MMA issued by this thread completes before TMEM is freed
      tc_commit_pair_mc(smem_u32(drain), 1);
      mbar_wait(drain, 0, kPDrainNs);
    }
  } else if (warp >= 2 && warp < 6) {
    // ------------------------------------------- scales -> own tensor memory --
    // Warp w writes lane quarter q = w % 4 of this CTA's tensor memory.  A
    // scales: row 32q + i (lane i) of K step j goes to column base + 4j + q
    // (the MMA of K step j reads lane r at column base + 4j + r/32).  B
    // scales: lane i of every quarter gets line i of each
    // 128x4 atom (rows i, i+32, i+64, i+96 of the chunk), 4 columns per atom --
    // every quarter holds all 256 B rows.  Then one arrive on the leader's
    // stage barrier.
    const int q = warp & 3;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + 256;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int u = pair; ok && u < num_units; u += npairs) {
      const int nsteps = p.num_kt + p.lora_steps;
      for (int i = 0; i < nsteps; ++i) {
        PSTAT_T0();
        bool got = __all_sync(0xffffffffu, !*abort_flag && mbar_wait(&sf_full[stage], phase, p.timeout_ns));
        if (got && i < p.num_kt) {
          const uint4 *fa = reinterpret_cast<const uint4 *>(sSFA + stage * kPSfaBytes) + lane;
          const uint4 *fb = reinterpret_cast<const uint4 *>(sSFB + stage * kPSfbBytes) + lane;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 w = fa[32 * j];                  // atom j, line `lane`: word q is row 32q + lane
            tmem_st_32x32b_x1(tq + stage * kPSfCols + 4 * j + q, q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
          }
          uint32_t v[16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // columns 16h .. 16h+15 of the B region: K steps 2h, 2h+1, both chunks
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int col = 16 * h + 4 * t;
              const int j = col / 8, c = (col % 8) / 4;
              const uint4 w = fb[128 * c + 32 * j];      // chunk c (2048 B), atom j (512 B)
              v[4 * t] = w.x; v[4 * t + 1] = w.y; v[4 * t + 2] = w.z; v[4 * t + 3] = w.w;
            }
            tmem_st_32x32b_x16(tq + stage * kPSfCols + kPSfaCols + 16 * h, v);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        if (warp == 2 && lane == 0) PSTAT_ADD(p, rank, 3);
        if (!got) {
          if (lane == 0) pair_abort(abort_flag, p.status);
          ok = false;
          break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(full_l + 8 * stage);
        if (++stage == S) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------------------ epilogue --
    // Warp w drains lane quarter w % 4 of this CTA's accumulator: each thread
    // owns one row, loads it in two halves of 128 columns (a half unit: one)
    // and releases the accumulator after the last half's loads, so that the
    // next unit's MMAs overlap the remaining stores.
    const int q = warp & 3;
    const int r = q * 32 + lane;
    uint32_t acc_phase = 0;
    const float alpha = acc_scale_of(p.g_a ? *p.g_a : 1.0f, p.g_b ? *p.g_b : 1.0f);
    for (int u = pair; u < num_units; u += npairs) {
      const PairTile t = pair_tile(sched, u);
      const int halves = t.half ? 1 : 2;
      // warp-uniform outcome: tcgen05.ld below is a warp-collective instruction
      PSTAT_T0();
      const bool got_full =
          __all_sync(0xffffffffu, !*abort_flag && mbar_wait_u(smem_u32(acc_full), acc_phase, p.timeout_ns));
      if (warp == 6 && lane == 0) PSTAT_ADD(p, rank, 4);
      if (!got_full) {
        if (lane == 0) pair_abort(abort_flag, p.status);
        break;
      }
      tc_fence_after();
      const int64_t orow = t.m0 + 128 * rank + r;
      const bool row_ok = orow < p.M;
#pragma unroll 1
      for (int half = 0; half < halves; ++half) {
        uint32_t v[4][32];
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(q * 32) << 16) + (half * 4 + c) * 32, v[c]);
        tmem_ld_wait();
        if (half == halves - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(acc_empty_l);
        }
        if (p.store_tma) {
          // bf16 through shared memory: this warp's four 32 x 32 boxes take
          // the half's four column chunks (row `lane` of each, its 16-byte
          // pieces at their 64-byte-swizzle positions: conflict-free), then
          // one fence and one lane issues the four tensor stores, which leave
          // out rows and columns outside D.  Half 0 goes out before half 1 is
          // loaded, so the accumulator is released after one pass of stores.
          if (lane == 0) bulk_wait_group_read<0>();   // the boxes' previous stores have read them
          __syncwarp();
          const uint32_t box0 = smem_u32(stg) + (uint32_t)(q * 4 * 2048);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            if (t.n0 + (half * 4 + c) * 32 < p.N) {
              uint32_t w[16];
#pragma unroll
              for (int i2 = 0; i2 < 16; ++i2) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[c][2 * i2]), alpha),
                                                                __fmul_rn(__uint_as_float(v[c][2 * i2 + 1]), alpha));
                w[i2] = *reinterpret_cast<const uint32_t *>(&h2);
              }
              const uint32_t row = box0 + (uint32_t)(c * 2048 + lane * 64);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                sts128(row + ((k ^ ((lane >> 1) & 3)) << 4), w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            }
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int64_t n = t.n0 + (half * 4 + c) * 32;
              if (n < p.N) tma_store_2d(&tmD, box0 + (uint32_t)(c * 2048), (int32_t)n, (int32_t)(t.m0 + 128 * rank + 32 * q));
            }
            bulk_commit_group();
          }
          continue;
        }
        if (!row_ok) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int64_t n = t.n0 + (half * 4 + c) * 32;
          if (n >= p.N) break;
          float f[32];
#pragma unroll
          for (int i2 = 0; i2 < 32; ++i2) f[i2] = __fmul_rn(__uint_as_float(v[c][i2]), alpha);
          const bool full_chunk = n + 32 <= p.N;
          const int nvalid = full_chunk ? 32 : (int)(p.N - n);
          if (p.out_fp32) {
            float *dst = reinterpret_cast<float *>(p.d) + orow * p.ldd + n;
            if (full_chunk && (reinterpret_cast<uintptr_t>(dst) & 31) == 0) {
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
          } else {
            __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.d) + orow * p.ldd + n;
            if (full_chunk && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
              uint32_t w[16];
#pragma unroll
              for (int i2 = 0; i2 < 16; ++i2) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(f[2 * i2], f[2 * i2 + 1]);
                w[i2] = *reinterpret_cast<const uint32_t *>(&h2);
              }
              if ((reinterpret_cast<uintptr_t>(dst) & 31) == 0) {   // whole 32-byte sectors
                st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
                st_global_v8(dst + 16, w[8], w[9], w[10], w[11], w[12], w[13], w[14], w[15]);
              } else {
#pragma unroll
                for (int i2 = 0; i2 < 16; i2 += 4)
                  *reinterpret_cast<uint4 *>(dst + 2 * i2) = make_uint4(w[i2], w[i2 + 1], w[i2 + 2], w[i2 + 3]);
              }
            } else {
#pragma unroll
              for (int i2 = 0; i2 < 32; ++i2)
                if (i2 < nvalid) dst[i2] = __float2bfloat16_rn(f[i2]);
            }
          }
        }
      }
      acc_phase ^= 1;
    }
    // every tensor store of this warp has written D before the CTA exits
    if (p.store_tma && lane == 0) bulk_wait_group_all();
    __syncwarp();
  }
  __syncthreads();
#ifdef NVFP4_WAIT_STATS
  if (threadIdx.x == 0) {
    unsigned long long *c = reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(p.status) + 64);
    atomicAdd(c + 8 * rank + 5, (unsigned long long)(clock64() - kernel_t0));
    atomicAdd(c + 8 * rank + 6, 1ull);
  }
#endif
  cluster_sync();      // the leader's MMAs are complete and no remote arrive is pending
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kPTmemCols);
  }
}

// How many CTA pairs of this kernel the device holds at once (clusters of two
// need two SMs of one GPC), queried once per device.
static int resident_pairs(int num_sms) {
  static std::mutex mu;
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  std::lock_guard<std::mutex> lk(mu);
  if (!cached[dev]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = kPSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (void *)k_gemm_fp4_pair, &cfg) != cudaSuccess || n <= 0) {
      cudaGetLastError();   // clear: fall back to every SM pair
      n = num_sms / 2;
    }
    cached[dev] = std::min(n, num_sms / 2);
  }
  return cached[dev];
}

cudaError_t launch_gemm_fp4_pair(const GemmParams &p, const GemmMaps &m, int num_sms, cudaStream_t st) {
  if (cudaError_t e = ensure_dynamic_smem((const void *)k_gemm_fp4_pair, kPSmemBytes); e != cudaSuccess) return e;
  const int64_t tiles = ((p.M + 255) / 256) * (int64_t)p.tiles_n;
  const int64_t resident = resident_pairs(num_sms);
  GemmParams q = p;
  q.store_tma = p.store_tma && m.has_d;
  // half units need the 64-row B maps, and every half of the last n-tile
  // must hold a column of D (so that its B scale chunk exists)
  q.pair_half_tail = m.has_half && p.N - (int64_t)(p.tiles_n - 1) * 256 > 128;
  // fewer tiles than pairs: as many pairs as tiles, or twice as many (every
  // tile dealt as two half units) when they fit
  int64_t pairs = std::min<int64_t>(tiles, resident);
  if (q.pair_half_tail && tiles < resident && 2 * tiles <= resident) pairs = 2 * tiles;
  if (pairs <= 0) return cudaSuccess;
  return launch_pdl(k_gemm_fp4_pair, dim3((unsigned)(2 * pairs)), dim3(kPairThreads), kPSmemBytes, st, m.a, m.b, m.t,
                    m.lb, m.has_half ? m.bh : m.b, m.has_half ? m.lbh : m.lb, m.has_d ? m.d : m.a, q);
}

}  // namespace nvfp4
