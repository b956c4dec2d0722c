// gemv.cu -- batch-1 decode: y = (g_x g_w) sum_b sx_b sw_b sum_{k in b} e2m1(x_k) e2m1(w_nk)
//
// At batch size 1 the W4A4 projection is a GEMV whose time is the weight
// bandwidth ("vroomfondel/glm-5.2-reap-504B-v2-W4A4" card, "What this variant
// changes": o_proj 6144x16384 and q_b_proj 16384x2048 at bs 1), with the
// activation quantized per call under the static per-tensor input_scale
// ("How it was produced").  The CUDA-core path streams W once:
//   * every CTA quantizes the (tiny) X into shared memory with the static
//     scale, keeping the E2M1 values as exact fp16 pairs and the E4M3 block
//     scales as fp32;
//   * a warp reads 32 x 32 contiguous bytes of W codes (64 elements per lane)
//     and the matching 4-byte group of swizzled scales;
//   * a 16-element block dot product of E2M1 values is exact in fp16x2 (every
//     partial sum is a multiple of 1/4 below 512), sx_b*sw_b is exact in fp32
//     (two 4-bit significands) and so is their product with the block dot;
//     only the fp32 sum over blocks rounds.
// Long rows (K > 4096) are split into 2048-element chunks written as fp32
// partials and summed in order by a second kernel (no atomics, deterministic).
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

constexpr int kGemvThreads = 256;
constexpr int kGemvChunk = 2048;   // K elements per (row, chunk) unit = 32 lanes x 64
constexpr int kRows = 4;           // units (rows) a warp has in flight

// Same block quantizer as the row packing (kept local: tiny X, static scale).
__device__ __forceinline__ void quant_x_block(const __nv_bfloat16 *src, float g, float t6g,
                                              uint32_t (&h2)[8], float &sx) {
  uint32_t w[8];
  const uint4 a = __ldg(reinterpret_cast<const uint4 *>(src));
  const uint4 b = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  uint32_t m2 = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) m2 = __vmaxu2(m2, w[i] & 0x7FFF7FFFu);
  const float bamax = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
  uint32_t sb = 0;
  if (g > 0.0f) sb = cvt_e4m3(__fdiv_rn(bamax, t6g));
  sx = e4m3_to_f32(sb);
  if (sb == 0) {
#pragma unroll
    for (int i = 0; i < 8; ++i) h2[i] = 0;
    return;
  }
  const float senc = fminf(__frcp_rn(__fmul_rn(sx, g)), 3.402823466e38f);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    h2[i] = e2m1x2_to_h2(cvt_e2m1x2(__fmul_rn(bf16lo(w[i]), senc), __fmul_rn(bf16hi(w[i]), senc)));
}

template <int MX>
__global__ void __launch_bounds__(kGemvThreads) k_gemv(const GemvParams p, int nchunks, float *partial) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int64_t K = p.K, nblk = K / 16;
  // Shared layout chosen so that the 32 lanes of a warp, which take 32
  // consecutive 64-element groups g4, read consecutive 16-byte words:
  //   xs  [m][half h][bb][g4] = 4 half2 (elements 8h..8h+7 of block 4*g4 + bb)
  //   sxs [m][bb][g4]         = E4M3 block scale as fp32
  const int64_t G4 = K / 64;
  uint32_t *xs = reinterpret_cast<uint32_t *>(smem);             // MX * K/2 words
  float *sxs = reinterpret_cast<float *>(xs + MX * (K / 2));    // MX * K/16 floats

  const float g = *p.g_x;
  const float t6g = __fmul_rn(6.0f, g);
  for (int64_t i = threadIdx.x; i < MX * nblk; i += blockDim.x) {
    const int m = (int)(i / nblk);
    const int64_t b = i % nblk;
    uint32_t h2[8];
    float sx;
    quant_x_block(p.x + m * p.ldx + b * 16, g, t6g, h2, sx);
    const int64_t g4 = b >> 2, bb = b & 3;
    uint4 *dst = reinterpret_cast<uint4 *>(xs + m * (K / 2));
    dst[(0 * 4 + bb) * G4 + g4] = make_uint4(h2[0], h2[1], h2[2], h2[3]);
    dst[(1 * 4 + bb) * G4 + g4] = make_uint4(h2[4], h2[5], h2[6], h2[7]);
    sxs[m * nblk + bb * G4 + g4] = sx;
  }
  __syncthreads();

  const float alpha = __fmul_rn(g, *p.g_w);
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (kGemvThreads / 32) + (threadIdx.x >> 5);
  const int64_t nwarps = (int64_t)gridDim.x * (kGemvThreads / 32);
  const int64_t units = p.N * nchunks;
  const int64_t row_bytes = K / 2;
  const int64_t g4_total = K / 64;
  // A warp takes kRows consecutive units (consecutive rows of one K chunk) and
  // issues all of their loads before any arithmetic, so every lane keeps
  // kRows x 32 bytes of weights in flight.
  for (int64_t u0 = warp * kRows; u0 < units; u0 += nwarps * kRows) {
    uint32_t c[kRows][8];
    uint32_t sf4[kRows];
    int64_t n[kRows], g4v[kRows];
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      const int64_t u = u0 + j;
      const int64_t kc = u / p.N;
      n[j] = u % p.N;
      g4v[j] = kc * (kGemvChunk / 64) + lane;
      const bool live = u < units && g4v[j] < g4_total && g4v[j] < (kc + 1) * (kGemvChunk / 64);
      if (!live) g4v[j] = -1;
      if (live) {
        asm volatile(
            "ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=r"(c[j][0]), "=r"(c[j][1]), "=r"(c[j][2]), "=r"(c[j][3]), "=r"(c[j][4]),
              "=r"(c[j][5]), "=r"(c[j][6]), "=r"(c[j][7])
            : "l"(p.w_codes + n[j] * row_bytes + g4v[j] * 32));
        sf4[j] = __ldg(reinterpret_cast<const uint32_t *>(
            p.w_sf + 512 * ((n[j] >> 7) * p.w_sf_katoms + g4v[j]) + 16 * (n[j] & 31) +
            4 * ((n[j] & 127) >> 5)));
      }
    }
#pragma unroll
    for (int j = 0; j < kRows; ++j) {
      float acc[MX];
#pragma unroll
      for (int m = 0; m < MX; ++m) acc[m] = 0.0f;
      if (g4v[j] >= 0) {
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const float sw = e4m3_to_f32((sf4[j] >> (8 * bb)) & 0xFF);
          uint32_t wh[8];   // wh[i] = elements 2i, 2i+1 of the block (same order as X)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            wh[i] = e2m1x2_to_h2(c[j][2 * bb] >> (8 * i));
            wh[4 + i] = e2m1x2_to_h2(c[j][2 * bb + 1] >> (8 * i));
          }
#pragma unroll
          for (int m = 0; m < MX; ++m) {
            const uint4 *xp = reinterpret_cast<const uint4 *>(xs + m * (K / 2));
            const uint4 x0 = xp[(0 * 4 + bb) * G4 + g4v[j]], x1 = xp[(1 * 4 + bb) * G4 + g4v[j]];
            const uint32_t xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            __half2 s2 = __float2half2_rn(0.0f);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              s2 = __hfma2(*reinterpret_cast<const __half2 *>(&wh[i]),
                           *reinterpret_cast<const __half2 *>(&xv[i]), s2);
            const float dot = __fadd_rn(__low2float(s2), __high2float(s2));
            acc[m] = __fmaf_rn(dot, __fmul_rn(sw, sxs[m * nblk + bb * G4 + g4v[j]]), acc[m]);
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MX; ++m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
      const int64_t u = u0 + j;
      if (u < units && lane < MX) {
        float v = acc[0];
#pragma unroll
        for (int m = 1; m < MX; ++m)
          if (lane == m) v = acc[m];
        const int64_t kc = u / p.N;
        if (nchunks == 1) {
          const float y = __fmul_rn(v, alpha);
          if (p.out_fp32) reinterpret_cast<float *>(p.d)[lane * p.ldd + n[j]] = y;
          else reinterpret_cast<__nv_bfloat16 *>(p.d)[lane * p.ldd + n[j]] = __float2bfloat16_rn(y);
        } else {
          partial[(kc * MX + lane) * p.N + n[j]] = v;
        }
      }
    }
  }
}

__global__ void k_gemv_reduce(const GemvParams p, int nchunks, int mx, const float *partial) {
  const float alpha = __fmul_rn(*p.g_x, *p.g_w);
  const int64_t total = (int64_t)mx * p.N;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / p.N, n = i % p.N;
    float s = 0.0f;
    for (int kc = 0; kc < nchunks; ++kc) s = __fadd_rn(s, partial[(kc * mx + m) * p.N + n]);
    const float y = __fmul_rn(s, alpha);
    if (p.out_fp32) reinterpret_cast<float *>(p.d)[m * p.ldd + n] = y;
    else reinterpret_cast<__nv_bfloat16 *>(p.d)[m * p.ldd + n] = __float2bfloat16_rn(y);
  }
}

size_t gemv_smem_bytes(int64_t M, int64_t K) { return (size_t)M * (K / 2) * 4 + (size_t)M * (K / 16) * 4; }
int gemv_chunks(int64_t K) { return K > 4096 ? (int)((K + kGemvChunk - 1) / kGemvChunk) : 1; }
size_t gemv_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int c = gemv_chunks(K);
  return c > 1 ? (size_t)c * M * N * sizeof(float) : 0;
}

template <int MX>
static cudaError_t launch_mx(const GemvParams &p, int num_sms, cudaStream_t st, float *partial) {
  const size_t smem = gemv_smem_bytes(MX, p.K);
  static size_t configured = 48 * 1024;
  if (smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(k_gemv<MX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  const int nchunks = gemv_chunks(p.K);
  int per_sm = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_gemv<MX>, kGemvThreads, smem);
  per_sm = std::max(1, std::min(per_sm, 8));
  const int64_t warps_needed = (p.N * nchunks + 8 * kRows - 1) / (8 * kRows);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)num_sms * per_sm, warps_needed));
  k_gemv<MX><<<grid, kGemvThreads, smem, st>>>(p, nchunks, partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || nchunks == 1) return e;
  k_gemv_reduce<<<num_sms, 256, 0, st>>>(p, nchunks, MX, partial);
  return cudaGetLastError();
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
