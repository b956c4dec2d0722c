// dequant.cu -- NVFP4 -> bf16 (optionally transposed), the weight rebuild of
// the frozen-base backward ("Getting GLM-5.2 NVFP4 Post-Training off the
// ground", "Why can't we just transpose the one copy?" and "For a frozen
// QLoRA base": keep the rowwise packing only and dequantize it to bf16,
// transposed, for the Dgrad contraction).
//
// Per element, IEEE fp32, one rounding per operation:
//   s_dec = E4M3(sb) * g;   v = E2M1(code) * s_dec;   out = bf16_rn(v)
// HBM-bound: 0.5625 B read + 2 B written per element.
#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {

__device__ __forceinline__ uint32_t scale_word(const uint8_t *sf, int sf_swz, int64_t r, int64_t blk0,
                                               int64_t nblk) {
  // the 4 scales of blocks blk0 .. blk0+3 (blk0 % 4 == 0) of row r, as one word
  if (sf_swz) {
    const int64_t sfc_pad = (nblk + 3) & ~int64_t(3);
    const int64_t off = 512 * ((r >> 7) * (sfc_pad >> 2) + (blk0 >> 2)) + 16 * (r & 31) + 4 * ((r & 127) >> 5);
    return __ldg(reinterpret_cast<const uint32_t *>(sf + off));
  }
  return __ldg(reinterpret_cast<const uint32_t *>(sf + r * nblk + blk0));
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// Transposed: thread = (row pair 2p, 2p+1; 64-column chunk).  Consecutive
// threads take consecutive row pairs, so each store instruction writes 32
// consecutive bf16 pairs of one output row (coalesced).
__global__ void __launch_bounds__(256) k_dequant_t(const uint8_t *__restrict__ codes,
                                                   const uint8_t *__restrict__ sf, int sf_swz,
                                                   const float *__restrict__ gp, int64_t rows, int64_t cols,
                                                   __nv_bfloat16 *__restrict__ out, int64_t ldo) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  const float g = *gp;
  const int64_t pairs = rows / 2, chunks = cols / 64, nblk = cols / 16;
  const int64_t total = pairs * chunks;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pr = t % pairs, ch = t / pairs;
    const int64_t r0 = 2 * pr;
    uint4 c[2][2];
    uint32_t sw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 *src = reinterpret_cast<const uint4 *>(codes + (r0 + h) * (cols / 2) + ch * 32);
      c[h][0] = __ldg(src);
      c[h][1] = __ldg(src + 1);
      sw[h] = scale_word(sf, sf_swz, r0 + h, ch * 4, nblk);
    }
    uint32_t *dst = reinterpret_cast<uint32_t *>(out + (ch * 64) * ldo + r0);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float sd[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) sd[h] = __fmul_rn(e4m3_to_f32((sw[h] >> (8 * b)) & 0xFF), g);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        // code byte i of block b: elements 16b + 2i, 16b + 2i + 1
        float lo[2], hi[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 q = c[h][b >> 1];
          const uint32_t w = (b & 1) ? ((i < 4) ? q.z : q.w) : ((i < 4) ? q.x : q.y);
          const uint32_t h2 = e2m1x2_to_h2(w >> (8 * (i & 3)));
          lo[h] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF))), sd[h]);
          hi[h] = __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 >> 16))), sd[h]);
        }
        const int64_t j = 16 * b + 2 * i;
        dst[(j * ldo) >> 1] = bf16x2_bits(lo[0], lo[1]);
        dst[((j + 1) * ldo) >> 1] = bf16x2_bits(hi[0], hi[1]);
      }
    }
  }
}

// Row-major: thread = (row, 64-column chunk), 128 bytes of bf16 out as four
// 32-byte stores where the row allows it.
__global__ void __launch_bounds__(256) k_dequant_n(const uint8_t *__restrict__ codes,
                                                   const uint8_t *__restrict__ sf, int sf_swz,
                                                   const float *__restrict__ gp, int64_t rows, int64_t cols,
                                                   __nv_bfloat16 *__restrict__ out, int64_t ldo) {
  griddep_launch_dependents();
  griddep_wait();   // inputs may come from the previous kernel in the stream
  const float g = *gp;
  const int64_t chunks = cols / 64, nblk = cols / 16;
  const int64_t total = rows * chunks;
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = t / chunks, ch = t % chunks;
    const uint4 *src = reinterpret_cast<const uint4 *>(codes + r * (cols / 2) + ch * 32);
    const uint4 c2[2] = {__ldg(src), __ldg(src + 1)};
    const uint32_t sw = scale_word(sf, sf_swz, r, ch * 4, nblk);
    uint4 *dst = reinterpret_cast<uint4 *>(out + r * ldo + ch * 64);
    const bool whole = (reinterpret_cast<uintptr_t>(dst) & 31) == 0;   // 32-byte stores fill sectors
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float sd = __fmul_rn(e4m3_to_f32((sw >> (8 * b)) & 0xFF), g);
      const uint4 q = c2[b >> 1];
      const uint32_t wv[2] = {(b & 1) ? q.z : q.x, (b & 1) ? q.w : q.y};
      uint32_t o[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t h2 = e2m1x2_to_h2(wv[i >> 2] >> (8 * (i & 3)));
        o[i] = bf16x2_bits(__fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF))), sd),
                           __fmul_rn(__half2float(__ushort_as_half((unsigned short)(h2 >> 16))), sd));
      }
      if (whole) {
        st_global_v8(dst + 2 * b, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
      } else {
        dst[2 * b] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * b + 1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  }
}

cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *sf, int sf_swz, const float *g, int64_t rows,
                           int64_t cols, int transpose, __nv_bfloat16 *out, int64_t ldo, int num_sms,
                           cudaStream_t st) {
  const int64_t work = transpose ? (rows / 2) * (cols / 64) : rows * (cols / 64);
  const int64_t ctas = std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, (int64_t)num_sms * 8));
  if (transpose)
    return launch_pdl(k_dequant_t, dim3((unsigned)ctas), dim3(256), 0, st, codes, sf, sf_swz, g, rows, cols, out, ldo);
  else
    return launch_pdl(k_dequant_n, dim3((unsigned)ctas), dim3(256), 0, st, codes, sf, sf_swz, g, rows, cols, out, ldo);
}

}  // namespace nvfp4
