// gemv.cu -- batch-1 decode: y = (g_x g_w) sum_b sx_b sw_b sum_{k in b} e2m1(x_k) e2m1(w_nk)
//
// At batch size 1 the W4A4 projection is a GEMV whose time is the weight
// bandwidth ("vroomfondel/glm-5.2-reap-504B-v2-W4A4" card, "What this variant
// changes": o_proj 6144x16384 and q_b_proj 16384x2048 at bs 1), with the
// activation quantized per call under the static per-tensor input_scale
// ("How it was produced").  The CUDA-core path streams W once:
//   * every CTA quantizes the (tiny) X into shared memory with the static
//     scale, keeping each E2M1 value doubled as a signed 8-bit integer (the
//     grid {0,.5,1,1.5,2,3,4,6} x 2 is {0,1,2,3,4,6,8,12}), both signs of it,
//     and the E4M3 block scales as fp32;
//   * a warp reads 32 x 32 contiguous bytes of W codes (64 elements per lane)
//     and the matching 4-byte group of swizzled scales;
//   * four codes at a time become the doubled magnitudes of the positive
//     codes and, from the codes with their sign bits flipped, of the negative
//     codes, each by one byte permute whose sign-replicate mode zeroes the
//     other sign; two dp4a sum them against +x and -x: a 16-element block dot
//     product is an exact integer (4x the E2M1 dot), sx_b*sw_b is exact in
//     fp32 (two 4-bit significands) and so is their product with the block
//     dot; only the fp32 sum over blocks rounds.
// Rows longer than 2048 elements are split into 2048-element chunks; the chunk
// sums of a row are added in chunk order, inside the CTA for rows of up to
// 16384 elements and by a second kernel beyond (no atomics, deterministic).
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

constexpr int kGemvThreads = 256;
constexpr int kGemvChunk = 2048;   // K elements per (row, chunk) unit = 32 lanes x 64

// Doubled E2M1 magnitudes {0,1,2,3,4,6,8,12} as bytes of two words: byte c of
// (lo, hi) is 2*E2M1(c) for c = 0..7 (a byte-permute lookup table).
constexpr uint32_t kE2m1x2Lo = 0x03020100u, kE2m1x2Hi = 0x0C080604u;
constexpr int kMagic = 0x4B400000;   // fp32 bits of 1.5 * 2^23

// Byte permute with the selector's high bit per byte honoured: a selector
// nibble of 8..15 yields the sign of the selected byte replicated (0 for the
// non-negative table entries here), 0..7 the byte itself.
__device__ __forceinline__ uint32_t prmt_sx(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Same block quantizer as the row packing (kept local: tiny X, static scale).
// Writes the block's 16 values as signed bytes 2*E2M1 (xp, 4 words) and their
// negations (xn), and the E4M3 scale as fp32.
__device__ __forceinline__ void quant_x_block(const uint4 (&raw)[2], float g, float t6g,
                                              uint32_t (&xp)[4], uint32_t (&xn)[4], float &sx) {
  const uint32_t w[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w};
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m2 = __vmaxu2(m2, w[i] & 0x7FFF7FFFu);
  const float bamax = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
  uint32_t sb = 0;
  if (g > 0.0f) sb = cvt_e4m3(__fdiv_rn(bamax, t6g));
  sx = e4m3_to_f32(sb);
#pragma unroll
  for (int i = 0; i < 4; ++i) xp[i] = xn[i] = 0;
  if (sb == 0) return;
  const float senc = fminf(__frcp_rn(__fmul_rn(sx, g)), 3.402823466e38f);
  uint32_t cc[8];   // byte i: the codes of elements 2i (low nibble) and 2i + 1
#pragma unroll
  for (int i = 0; i < 8; ++i)
    cc[i] = cvt_e2m1x2(__fmul_rn(bf16lo(w[i]), senc), __fmul_rn(bf16hi(w[i]), senc));
#pragma unroll
  for (int hw = 0; hw < 2; ++hw) {
    // the eight codes of elements 8hw .. 8hw + 7, element k in nibble k
    const uint32_t c8 = __byte_perm(__byte_perm(cc[4 * hw], cc[4 * hw + 1], 0x0040),
                                    __byte_perm(cc[4 * hw + 2], cc[4 * hw + 3], 0x0040), 0x5410);
    const uint32_t c8n = c8 ^ 0x88888888u;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      // doubled magnitudes of the positive codes (mp) and of the negative ones
      // (mn); per byte one of them is zero, so the byte-wise differences mp - mn
      // and mn - mp need no borrow between bytes: with the minuend biased by
      // 0x80 the subtraction stays inside the byte, and the bias is toggled off
      const uint32_t mp = prmt_sx(kE2m1x2Lo, kE2m1x2Hi, c8 >> (16 * hh));
      const uint32_t mn = prmt_sx(kE2m1x2Lo, kE2m1x2Hi, c8n >> (16 * hh));
      xp[2 * hw + hh] = ((mp | 0x80808080u) - mn) ^ 0x80808080u;
      xn[2 * hw + hh] = ((mn | 0x80808080u) - mp) ^ 0x80808080u;
    }
  }
}

// A warp's task is R consecutive rows of one 2048-element K chunk (R = 2 when
// a row is one chunk, so twice the tasks are in flight; R = 4 otherwise).  Tasks
// are ordered row-major (all chunks of a row batch are adjacent), so a CTA
// streams whole rows.  With at most kWarps chunks per row, one CTA holds every
// chunk of its row batches at once: the warps' chunk sums meet in shared
// memory and are added in chunk order there.  Longer rows write fp32 chunk
// sums [chunk][m][n] that a second kernel adds in the same order.  The loads
// of the next task are issued before the arithmetic of the current one (two
// register buffers), and the first task's loads before the CTA quantizes X,
// so the weight stream starts at kernel entry.
constexpr int kWarps = kGemvThreads / 32;

template <int R>
struct GemvBatch {
  uint32_t c[R][8];   // 64 codes of each row for this lane
  uint32_t sf[R];     // the 4 block scales of this lane's 64 codes
  int32_t n0, g4;     // first row of the task; this lane's 64-element group (-1: none)
};

template <int R>
__device__ __forceinline__ void gemv_load(const GemvParams &p, int32_t n0, int32_t kc, int32_t g4_total,
                                          int lane, GemvBatch<R> &B) {
  B.n0 = n0;
  const int32_t g4 = kc * (kGemvChunk / 64) + lane;
  B.g4 = g4 < g4_total ? g4 : -1;
  const int64_t row_bytes = p.K / 2;
#pragma unroll
  for (int j = 0; j < R; ++j) {
    const int32_t n = n0 + j;
    if (B.g4 >= 0 && n < p.N) {
      asm volatile(
          "ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
          : "=r"(B.c[j][0]), "=r"(B.c[j][1]), "=r"(B.c[j][2]), "=r"(B.c[j][3]), "=r"(B.c[j][4]),
            "=r"(B.c[j][5]), "=r"(B.c[j][6]), "=r"(B.c[j][7])
          : "l"(p.w_codes + (int64_t)n * row_bytes + (int64_t)B.g4 * 32));
      B.sf[j] = __ldg(reinterpret_cast<const uint32_t *>(
          p.w_sf + 512 * ((int64_t)(n >> 7) * p.w_sf_katoms + B.g4) + 16 * (n & 31) + 4 * ((n & 127) >> 5)));
    }
  }
}

// The chunk sums of the task's rows: on return lane m (< MX) holds row j's
// sum for activation row m in out[j].  Blocks outer, rows inner: the lane's X
// words of a block are read from shared memory once for all rows.
template <int MX, int R>
__device__ __forceinline__ void gemv_compute(const GemvParams &p, const GemvBatch<R> &B, const uint32_t *xs,
                                             const float *sxs, int64_t G4, int64_t nblk, int lane,
                                             float (&out)[R]) {
  float acc[R][MX];
#pragma unroll
  for (int j = 0; j < R; ++j)
#pragma unroll
    for (int m = 0; m < MX; ++m) acc[j][m] = 0.0f;
  if (B.g4 >= 0) {
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
      uint32_t pw[MX][4], nw[MX][4];
      float sx[MX];
#pragma unroll
      for (int m = 0; m < MX; ++m) {
        const uint4 *xq = reinterpret_cast<const uint4 *>(xs + m * (p.K / 2));
        const uint4 xp = xq[(0 * 4 + bb) * G4 + B.g4], xn = xq[(1 * 4 + bb) * G4 + B.g4];
        pw[m][0] = xp.x; pw[m][1] = xp.y; pw[m][2] = xp.z; pw[m][3] = xp.w;
        nw[m][0] = xn.x; nw[m][1] = xn.y; nw[m][2] = xn.z; nw[m][3] = xn.w;
        sx[m] = sxs[m * nblk + bb * G4 + B.g4];
      }
#pragma unroll
      for (int j = 0; j < R; ++j) {
        if (B.n0 + j >= p.N) continue;
        // the E4M3 scale byte shifted into fp32 bits 20..27 reads as its value
        // times 2^-120 (a subnormal for exponent 0, still exact); the X scales
        // carry the 2^120 back, so no conversion instruction is needed
        const float sw = __uint_as_float(((B.sf[j] >> (8 * bb)) & 0xFFu) << 20);
        // per group of four codes: the doubled magnitudes of the positive
        // codes (negative ones read 0) and of the negative codes (positive
        // ones read 0), each by one table lookup in sign-replicate mode
        uint32_t mpos[4], mneg[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t w = B.c[j][2 * bb + h], wn = w ^ 0x88888888u;
          mpos[2 * h] = prmt_sx(kE2m1x2Lo, kE2m1x2Hi, w);
          mpos[2 * h + 1] = prmt_sx(kE2m1x2Lo, kE2m1x2Hi, w >> 16);
          mneg[2 * h] = prmt_sx(kE2m1x2Lo, kE2m1x2Hi, wn);
          mneg[2 * h + 1] = prmt_sx(kE2m1x2Lo, kE2m1x2Hi, wn >> 16);
        }
#pragma unroll
        for (int m = 0; m < MX; ++m) {
          // two independent chains; the first starts at the bits of 1.5 * 2^23,
          // so their sum read as fp32 is 1.5 * 2^23 + isum (|isum| <= 2304)
          int ipos = kMagic, ineg = 0;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            ipos = __dp4a((int)mpos[q], (int)pw[m][q], ipos);
            ineg = __dp4a((int)mneg[q], (int)nw[m][q], ineg);
          }
          const float fsum = __fsub_rn(__int_as_float(ipos + ineg), 12582912.0f);   // isum, exact
          // isum/4 (the E2M1 dot) times sx*sw, both exact: one rounding in the fma
          acc[j][m] = __fmaf_rn(fsum, __fmul_rn(sw, sx[m]), acc[j][m]);
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < R; ++j) {
#pragma unroll
    for (int m = 0; m < MX; ++m)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[j][m] += __shfl_xor_sync(0xffffffffu, acc[j][m], o);
    float v = acc[j][0];
#pragma unroll
    for (int m = 1; m < MX; ++m)
      if (lane == m) v = acc[j][m];
    out[j] = v;
  }
}

__device__ __forceinline__ void gemv_store(const GemvParams &p, int64_t m, int64_t n, float y) {
  if (p.out_fp32) reinterpret_cast<float *>(p.d)[m * p.ldd + n] = y;
  else reinterpret_cast<__nv_bfloat16 *>(p.d)[m * p.ldd + n] = __float2bfloat16_rn(y);
}

// Work units.  In-CTA mode (nchunks <= kWarps): a unit is rbu = kWarps / nchunks
// row batches x nchunks chunks, warp w taking row batch w / nchunks, chunk
// w % nchunks (warps past rbu * nchunks idle).  Global mode: a unit is one task.
struct GemvPlan {
  int32_t nchunks, rbu, units, g4_total;
  bool in_cta;
};

template <int R>
__device__ __forceinline__ GemvPlan gemv_plan(const GemvParams &p, int nchunks) {
  GemvPlan q;
  q.nchunks = nchunks;
  q.in_cta = nchunks <= kWarps;
  const int32_t nb = (int32_t)((p.N + R - 1) / R);
  q.rbu = q.in_cta ? kWarps / nchunks : 1;
  q.units = q.in_cta ? (nb + q.rbu - 1) / q.rbu : nb * nchunks;
  q.g4_total = (int32_t)(p.K / 64);
  return q;
}

// L2 prefetch of a unit's weights: in-CTA mode (thread 0) the unit's rows are
// contiguous, all K; the unit that starts a 128-row group also takes the
// group's swizzled scale atoms.  Global mode (one task per warp) fetches the
// task's R row pieces of one chunk from lanes 0..R-1.
template <int R>
__device__ __forceinline__ void gemv_prefetch(const GemvParams &p, const GemvPlan &q, int32_t unit, int lane) {
  if (unit >= q.units) return;
  const int64_t row_bytes = p.K / 2;
  if (q.in_cta) {
    if (threadIdx.x != 0) return;
    const int64_t n0 = (int64_t)unit * q.rbu * R;
    const int64_t span = (int64_t)q.rbu * R, rows = p.N - n0 < span ? p.N - n0 : span;
    if (rows <= 0) return;
    prefetch_l2_bulk(p.w_codes + n0 * row_bytes, (uint32_t)(rows * row_bytes));
    if ((n0 & 127) == 0) prefetch_l2_bulk(p.w_sf + (n0 >> 7) * p.w_sf_katoms * 512, (uint32_t)(p.w_sf_katoms * 512));
  } else {
    const int64_t n = (int64_t)(unit / q.nchunks) * R + lane;
    const int64_t k0 = (int64_t)(unit % q.nchunks) * (kGemvChunk / 2);
    const int64_t piece = row_bytes - k0 < kGemvChunk / 2 ? row_bytes - k0 : kGemvChunk / 2;
    if (lane < R && n < p.N) prefetch_l2_bulk(p.w_codes + n * row_bytes + k0, (uint32_t)piece);
  }
}

// resident CTAs per SM the register budget is held to: three for the
// one-row-of-X two-row tasks, two up to two X rows (at most 128 registers)
constexpr int gemv_min_ctas(int mx, int r) { return mx == 1 && r == 2 ? 3 : mx <= 2 ? 2 : 1; }

template <int MX, int R>
__global__ void __launch_bounds__(kGemvThreads, gemv_min_ctas(MX, R)) k_gemv(const GemvParams p, int nchunks, float *partial) {
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const GemvPlan q = gemv_plan<R>(p, nchunks);
  const int32_t ustep = q.in_cta ? (int32_t)gridDim.x : (int32_t)gridDim.x * kWarps;
  int32_t u = q.in_cta ? (int32_t)blockIdx.x : (int32_t)blockIdx.x * kWarps + w;
  // The weight stream starts before the wait on the previous grid: an L2
  // prefetch of the first unit (a cache hint, safe against that grid's
  // writes) overlaps that grid's tail.
  gemv_prefetch<R>(p, q, u, lane);
  griddep_wait();   // inputs may come from the previous kernel in the stream
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float red[2][kWarps][R][4];   // in-CTA chunk sums, double-buffered
  const int64_t K = p.K, nblk = K / 16;
  // Shared layout chosen so that the 32 lanes of a warp, which take 32
  // consecutive 64-element groups g4, read consecutive 16-byte words:
  //   xs  [m][h][bb][g4] = the 16 values of block 4*g4 + bb as signed bytes
  //                        2*E2M1 (h = 0) and their negations (h = 1)
  //   sxs [m][bb][g4]    = E4M3 block scale * 2^118 as fp32 (1/4: the values are
  //                        doubled; 2^120: the weight scales' bit placement)
  const int64_t G4 = K / 64;
  uint32_t *xs = reinterpret_cast<uint32_t *>(smem);             // MX * K/2 words
  float *sxs = reinterpret_cast<float *>(xs + MX * (K / 2));    // MX * K/16 floats

  // this warp's task in unit u (in-CTA) / task index (global)
  const bool active = !q.in_cta || w < q.rbu * q.nchunks;
  const int32_t my_kc = q.in_cta ? w % q.nchunks : 0, my_rb = q.in_cta ? w / q.nchunks : 0;
  auto task_of = [&](int32_t unit, int32_t &n0, int32_t &kc) {
    if (q.in_cta) {
      n0 = (unit * q.rbu + my_rb) * R;
      kc = my_kc;
    } else {
      n0 = (unit / q.nchunks) * R;
      kc = unit % q.nchunks;
    }
  };

  GemvBatch<R> A, B;
  if (active && u < q.units) {   // weights in flight first
    int32_t n0, kc;
    task_of(u, n0, kc);
    gemv_load(p, n0, kc, q.g4_total, lane, A);
  }

  const float g = *p.g_x;
  const float t6g = __fmul_rn(6.0f, g);
  const int32_t nb32 = (int32_t)nblk;
  // a thread's X blocks: all loads first, then the arithmetic (one L2
  // round trip instead of one per block)
  constexpr int kXDepth = 4;
  for (int32_t i0 = threadIdx.x; i0 < MX * nb32; i0 += kXDepth * blockDim.x) {
    uint4 raw[kXDepth][2];
#pragma unroll
    for (int r = 0; r < kXDepth; ++r) {
      const int32_t i = i0 + r * (int32_t)blockDim.x;
      if (i < MX * nb32) {
        const int32_t m = i / nb32, bk = i - m * nb32;
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + m * p.ldx + (int64_t)bk * 16);
        raw[r][0] = __ldg(src);
        raw[r][1] = __ldg(src + 1);
      }
    }
#pragma unroll
    for (int r = 0; r < kXDepth; ++r) {
      const int32_t i = i0 + r * (int32_t)blockDim.x;
      if (i < MX * nb32) {
        const int32_t m = i / nb32, bk = i - m * nb32;
        uint32_t xpv[4], xnv[4];
        float sx;
        quant_x_block(raw[r], g, t6g, xpv, xnv, sx);
        const int64_t g4 = bk >> 2, bb = bk & 3;
        uint4 *dst = reinterpret_cast<uint4 *>(xs + m * (K / 2));
        dst[(0 * 4 + bb) * G4 + g4] = make_uint4(xpv[0], xpv[1], xpv[2], xpv[3]);
        dst[(1 * 4 + bb) * G4 + g4] = make_uint4(xnv[0], xnv[1], xnv[2], xnv[3]);
        // with the 1/4 of the doubled values and the 2^120 of the weight scales (exact)
        sxs[m * nblk + bb * G4 + g4] = __fmul_rn(sx, 0x1p118f);
      }
    }
  }
  __syncthreads();

  const float alpha = __fmul_rn(g, *p.g_w);
  int buf = 0;
  // one unit: this warp's task (batch `cur`, prefetching the next unit into
  // `nxt`), then the output of the unit
  auto run_unit = [&](int32_t unit, const GemvBatch<R> &cur, GemvBatch<R> &nxt) {
    const int32_t un = unit + ustep;
    if (active && un < q.units) {
      int32_t n0, kc;
      task_of(un, n0, kc);
      gemv_load(p, n0, kc, q.g4_total, lane, nxt);
    }
    float v[R];
    if (active) gemv_compute<MX, R>(p, cur, xs, sxs, G4, nblk, lane, v);
    if (!q.in_cta) {
      const int32_t kc = unit % q.nchunks;
#pragma unroll
      for (int j = 0; j < R; ++j)
        if (cur.n0 + j < p.N && lane < MX) partial[((int64_t)kc * MX + lane) * p.N + cur.n0 + j] = v[j];
    } else if (q.nchunks == 1) {
      if (active)
#pragma unroll
        for (int j = 0; j < R; ++j)
          if (cur.n0 + j < p.N && lane < MX) gemv_store(p, lane, cur.n0 + j, __fmul_rn(v[j], alpha));
    } else {
      if (active && lane < MX)
#pragma unroll
        for (int j = 0; j < R; ++j) red[buf][w][j][lane] = v[j];
      __syncthreads();
      // chunk sums of each output added in chunk order
      const int t = threadIdx.x;
      if (t < q.rbu * R * MX) {
        const int rbl = t / (R * MX), j = (t / MX) % R, m = t % MX;
        const int64_t n = (int64_t)(unit * q.rbu + rbl) * R + j;
        if (n < p.N) {
          float sum = 0.0f;
          for (int kc = 0; kc < q.nchunks; ++kc) sum = __fadd_rn(sum, red[buf][rbl * q.nchunks + kc][j][m]);
          gemv_store(p, m, n, __fmul_rn(sum, alpha));
        }
      }
      buf ^= 1;
    }
  };
  // units are CTA-uniform in in-CTA mode (every thread takes the same path
  // to the barrier); in global mode they are per warp and no barrier is used
  while (u < q.units) {
    run_unit(u, A, B);
    u += ustep;
    if (u >= q.units) break;
    run_unit(u, B, A);
    u += ustep;
  }
}

__global__ void k_gemv_reduce(const GemvParams p, int nchunks, int mx, const float *partial) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  const float alpha = __fmul_rn(*p.g_x, *p.g_w);
  const int64_t total = (int64_t)mx * p.N;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / p.N, n = i % p.N;
    float s = 0.0f;
    for (int kc = 0; kc < nchunks; ++kc) s = __fadd_rn(s, partial[(kc * mx + m) * p.N + n]);
    gemv_store(p, m, n, __fmul_rn(s, alpha));
  }
}

size_t gemv_smem_bytes(int64_t M, int64_t K) { return (size_t)M * (K / 2) * 4 + (size_t)M * (K / 16) * 4; }
// a warp covers 2048 elements of a row (32 lanes x 64): longer rows are split
int gemv_chunks(int64_t K) { return (int)((K + kGemvChunk - 1) / kGemvChunk); }
size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int c = gemv_chunks(K);
  return c > kWarps ? (size_t)c * M * N * sizeof(float) : 0;
}

template <int MX, int R>
static cudaError_t launch_mxr(const GemvParams &p, int nchunks, int num_sms, cudaStream_t st, float *partial) {
  const size_t smem = gemv_smem_bytes(MX, p.K);
  if (cudaError_t e = ensure_dynamic_smem((const void *)k_gemv<MX, R>, smem); e != cudaSuccess) return e;
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv<MX, R>, kGemvThreads, smem);
  per_sm = std::max(1, std::min(per_sm, 8));
  // one wave of resident CTAs (or fewer when there is less work)
  const int64_t nb = (p.N + R - 1) / R;
  const int64_t ctas_needed = nchunks <= kWarps ? (nb + kWarps / nchunks - 1) / (kWarps / nchunks)
                                                : (nb * nchunks + kWarps - 1) / kWarps;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)num_sms * per_sm, ctas_needed));
  return launch_pdl(k_gemv<MX, R>, dim3(grid), dim3(kGemvThreads), smem, st, p, nchunks, partial);
}

template <int MX>
static cudaError_t launch_mx(const GemvParams &p, int num_sms, cudaStream_t st, float *partial) {
  const int nchunks = gemv_chunks(p.K);
  // rows of one chunk: two-row tasks (twice the tasks in flight); longer rows: four
  cudaError_t e = nchunks == 1 ? launch_mxr<MX, 2>(p, nchunks, num_sms, st, partial)
                               : launch_mxr<MX, 4>(p, nchunks, num_sms, st, partial);
  if (e != cudaSuccess || nchunks <= kWarps) return e;
  return launch_pdl(k_gemv_reduce, dim3(num_sms), dim3(256), 0, st, p, nchunks, (int)MX, (const float *)partial);
}

cudaError_t launch_gemv_ws(const GemvParams &p, int num_sms, cudaStream_t st, float *partial) {
  switch (p.M) {
    case 1: return launch_mx<1>(p, num_sms, st, partial);
    case 2: return launch_mx<2>(p, num_sms, st, partial);
    case 3: return launch_mx<3>(p, num_sms, st, partial);
    case 4: return launch_mx<4>(p, num_sms, st, partial);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4
