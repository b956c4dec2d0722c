// static_scratch.cu -- nvfp4_quantize_noalloc: the quantize entry point for
// callers that cannot allocate device memory.
//
// The dynamic global scale needs scratch for the per-part amax maxima.  The
// ordinary entry point takes it from the caller's workspace; this one uses a
// file-scope device array instead, so the caller passes only inputs and
// outputs.  The array is part of the library image: every GPU that loads the
// library holds it (64 KiB of amax words plus a 256-byte status block) until
// the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/nvfp4.h"
#include "internal.h"

namespace {

// Capacity in 32-bit words: one word per (matrix, part); a matrix of R rows
// uses min(R, 512) parts, so e.g. 32 matrices of >= 512 rows fit exactly.
constexpr size_t kScratchWords = 16384;
// Words reserved ahead of the amax words: word 0 is this entry point's device
// status word (what the packing kernels' bounded waits write on expiry); the
// block keeps the amax words 256-byte aligned.
constexpr size_t kStatusWords = 64;

// Status block, then the amax words.  Zero when the library is loaded.
static __device__ __align__(256) uint32_t g_noalloc_scratch[kStatusWords + kScratchWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_scratch_ptr[kMaxDevices] = {};

// The device address of g_noalloc_scratch on the current device, looked up
// once per device with that device current (the host-side symbol is only a
// stand-in and must never be handed to a kernel).
nvfp4_status scratch_for_current_device(uint32_t **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint32_t *>(p);
  }
  *out = g_scratch_ptr[dev];
  return NVFP4_OK;
}

}  // namespace

namespace nvfp4 {
nvfp4_status noalloc_status_word(int **out) {
  uint32_t *base = nullptr;
  if (nvfp4_status s = scratch_for_current_device(&base); s != NVFP4_OK) return s;
  *out = reinterpret_cast<int *>(base);
  return NVFP4_OK;
}
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize_noalloc(const nvfp4_quant_args *args, nvfp4_stream stream) {
  if (!args || args->batch < 1 || args->rows < 1) return NVFP4_ERR_INVALID_ARG;
  if (!args->global_scale_in) {
    // reject before any device work: batch x parts must fit the static array
    const size_t need = (size_t)args->batch * (size_t)nvfp4::amax_parts_for(args->rows);
    if (need > kScratchWords) return NVFP4_ERR_WORKSPACE;
  }
  uint32_t *base = nullptr;
  nvfp4_status s = scratch_for_current_device(&base);
  if (s != NVFP4_OK) return s;
  // `workspace` is not used: the status word and the amax words are the array's
  return nvfp4::quantize_with_amax_scratch(args, base + kStatusWords, kScratchWords,
                                            reinterpret_cast<int *>(base),
                                            reinterpret_cast<cudaStream_t>(stream));
}
