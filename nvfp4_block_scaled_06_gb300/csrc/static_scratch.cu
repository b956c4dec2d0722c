// static_scratch.cu -- nvfp4_quantize_noalloc: the quantize entry point for
// callers that cannot allocate device memory.
//
// The dynamic global scale needs scratch for the per-part amax maxima.  The
// ordinary entry point takes it from the caller's workspace; this one uses a
// file-scope device array instead, so the caller passes only inputs and
// outputs.  The array is part of the library image: every GPU that loads the
// library holds it (64 KiB) until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "internal.h"

namespace {

// Capacity in 32-bit words: one word per (matrix, part); a matrix of R rows
// uses min(R, 512) parts, so e.g. 32 matrices of >= 512 rows fit exactly.
constexpr size_t kScratchWords = 16384;

static __device__ __align__(256) uint32_t g_amax_scratch[kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_scratch_ptr[kMaxDevices] = {};

// The device address of g_amax_scratch on the current device, looked up once
// per device with that device current (the host-side symbol is only a stand-in
// and must never be handed to a kernel).
nvfp4_status scratch_for_current_device(uint32_t **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_amax_scratch) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint32_t *>(p);
  }
  *out = g_scratch_ptr[dev];
  return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status nvfp4_quantize_noalloc(const nvfp4_quant_args *args, nvfp4_stream stream) {
  if (!args || args->batch < 1 || args->rows < 1) return NVFP4_ERR_INVALID_ARG;
  if (!args->global_scale_in) {
    // reject before any device work: batch x parts must fit the static array
    const size_t need = (size_t)args->batch * (size_t)nvfp4::amax_parts_for(args->rows);
    if (need > kScratchWords) return NVFP4_ERR_WORKSPACE;
  }
  uint32_t *scratch = nullptr;
  nvfp4_status s = scratch_for_current_device(&scratch);
  if (s != NVFP4_OK) return s;
  return nvfp4::quantize_with_amax_scratch(args, scratch, kScratchWords,
                                            reinterpret_cast<cudaStream_t>(stream));
}
