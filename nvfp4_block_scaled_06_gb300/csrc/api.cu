// api.cu -- the extern "C" entry points of libnvfp4 (declared in include/nvfp4.h).
//
// Host side only: argument validation, workspace carving, tensor-map encoding
// and kernel sequencing on the caller's stream.  Nothing here allocates device
// memory; scratch lives in the caller's workspace, whose first 256 bytes hold
// the device status word written by bounded in-kernel waits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/nvfp4.h"
#include "internal.h"

using namespace nvfp4;

namespace {

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

struct DevInfo {
  int sms = 0;
  int major = 0, minor = 0;
  bool ok = false;
};

constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

nvfp4_status device_info(DevInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo &d = g_dev[dev];
  if (!d.ok) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    d.ok = true;
  }
  *out = d;
  if (d.major != 10 || d.minor != 3) return NVFP4_ERR_UNSUPPORTED_DEVICE;
  return NVFP4_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline int64_t pad_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Bump allocator over the caller's workspace; offsets are 256-byte aligned.
struct Carve {
  uint8_t *base;
  size_t off = 256;   // [0, 256): status word
  explicit Carve(void *b) : base(static_cast<uint8_t *>(b)) {}
  template <class T>
  T *take(size_t bytes) {
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += (bytes + 255) / 256 * 256;
    return p;
  }
};

size_t sf_swizzled_bytes(int64_t rows, int64_t cols) {
  return (size_t)pad_up(rows, 128) * (size_t)pad_up(cols / 16, 4);
}

// The last CUDA runtime error this thread saw inside the library (for
// nvfp4_last_cuda_error).
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

nvfp4_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4_OK;
  g_last_cuda_error = e;
  return NVFP4_ERR_CUDA;
}

// K ranges of the fused LoRA-down + amax pass (fp32 partials, summed in order
// by the packing kernel): two ranges put 2x as many SMs on the pass over X.
// Every range must hold at least one 128-wide stage, so short K uses one.
int lora_split_for(int64_t K) { return ceil_div(K, 64) >= 8 ? 2 : 1; }

// Records an optional caller-owned cudaEvent_t on the stream (profiling hook).
cudaError_t mark(void *ev, cudaStream_t st) {
  return ev ? cudaEventRecord(reinterpret_cast<cudaEvent_t>(ev), st) : cudaSuccess;
}

// ---------------------------------------------------------------- quantize --
struct QuantPlan {
  size_t ws = 0;
  uint32_t *amax = nullptr;
  int nparts = 0;
};

nvfp4_status plan_quantize(const nvfp4_quant_args *a, QuantPlan *pl) {
  Carve c(a->workspace);
  if (!a->global_scale_in) {
    pl->nparts = amax_parts_for(a->rows);
    pl->amax = c.take<uint32_t>((size_t)a->batch * pl->nparts * 4);
  }
  pl->ws = c.off;
  return NVFP4_OK;
}

nvfp4_status validate_quantize(const nvfp4_quant_args *a) {
  if (!a || !a->src) return NVFP4_ERR_INVALID_ARG;
  if (a->batch < 1 || a->rows < 1 || a->cols < 1) return NVFP4_ERR_INVALID_ARG;
  if (a->pack < NVFP4_PACK_ROW || a->pack > NVFP4_PACK_BOTH) return NVFP4_ERR_INVALID_ARG;
  if (a->sf_layout != NVFP4_SF_LINEAR && a->sf_layout != NVFP4_SF_SWIZZLED) return NVFP4_ERR_INVALID_ARG;
  const bool row = a->pack & NVFP4_PACK_ROW, col = a->pack & NVFP4_PACK_COL;
  if (row && (!a->codes_row || !a->sf_row)) return NVFP4_ERR_INVALID_ARG;
  if (col && (!a->codes_col || !a->sf_col)) return NVFP4_ERR_INVALID_ARG;
  if (!a->global_scale_in && !a->global_scale_out) return NVFP4_ERR_INVALID_ARG;
  if (a->ld < a->cols || (a->batch > 1 && a->batch_stride < a->rows * a->ld)) return NVFP4_ERR_INVALID_ARG;
  if (a->cols % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (col && a->rows % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->rows > (1ll << 31) || a->cols > (1ll << 31)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  // the tiled kernel (column packing) indexes rows and columns in 32 bits
  if (col && (a->rows >= (1ll << 30) || a->cols >= (1ll << 30))) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a->src, 16) || a->ld % 8 != 0 || (a->batch > 1 && a->batch_stride % 8 != 0))
    return NVFP4_ERR_ALIGNMENT;
  for (const void *p : {(const void *)a->codes_row, (const void *)a->sf_row, (const void *)a->codes_col,
                        (const void *)a->sf_col})
    if (p && !aligned(p, 16)) return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

// `status`: the device status word that the packing kernels' bounded waits
// write (the workspace's first word, or the workspace-free entry point's own).
nvfp4_status run_quantize(const nvfp4_quant_args *a, const QuantPlan &pl, int *status, int sms, cudaStream_t st) {
  QuantParams p{};
  p.src = static_cast<const __nv_bfloat16 *>(a->src);
  p.rows = a->rows;
  p.cols = a->cols;
  p.ld = a->ld;
  p.bstride = a->batch > 1 ? a->batch_stride : 0;
  p.batch = a->batch;
  p.g_in = a->global_scale_in;
  p.g_out = a->global_scale_out;
  p.amax_part = pl.amax;
  p.nparts = pl.nparts;
  p.sf_swizzled = a->sf_layout == NVFP4_SF_SWIZZLED;
  const bool row = a->pack & NVFP4_PACK_ROW, col = a->pack & NVFP4_PACK_COL;
  if (row) {
    p.codes_row = a->codes_row;
    p.sf_row = a->sf_row;
    p.codes_row_bstride = (int64_t)nvfp4_codes_bytes(a->rows, a->cols);
    p.sf_row_bstride = (int64_t)nvfp4_sf_bytes(a->rows, a->cols, a->sf_layout);
  }
  if (col) {
    p.codes_col = a->codes_col;
    p.sf_col = a->sf_col;
    p.codes_col_bstride = (int64_t)nvfp4_codes_bytes(a->cols, a->rows);
    p.sf_col_bstride = (int64_t)nvfp4_sf_bytes(a->cols, a->rows, a->sf_layout);
  }
  p.dst_rows = a->rows;
  p.status = status;
  p.timeout_ns = g_timeout_ns.load();
  p.stall_probe = p.timeout_ns == 0;
  if (!a->global_scale_in) {
    cudaError_t e = launch_amax(p, st);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (cudaError_t e_ = mark(a->prof_begin, st); e_ != cudaSuccess) return cuda_status(e_);
  cudaError_t e = col ? launch_quant_tiles(p, sms, st) : launch_quant_rows(p, sms, st);
  if (e == cudaSuccess) e = mark(a->prof_end, st);
  return cuda_status(e);
}

// -------------------------------------------------------------------- GEMM --
bool map2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
           uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_rows) {
  return make_map_2d(m, dt, base, inner, rows, pitch_bytes, box_inner, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

// The pair kernel's bf16 output leaves through tensor stores of 32 x 32 boxes
// (64-byte swizzle) when D's base and pitch allow a tensor map and its rows
// end on a 16-byte boundary (a store clips the last box of a row only at 16
// bytes: with N % 8 != 0 it would write up to 7 columns past N); otherwise
// the epilogue threads store their rows directly.
void map_pair_d(GemmMaps *maps, GemmParams *p) {
  maps->has_d = false;
  p->store_tma = 0;
  if (p->out_fp32 || p->ksplit > 1 || p->M < 32 || p->N < 32 || p->N % 8 != 0) return;
  if ((reinterpret_cast<uintptr_t>(p->d) & 15) != 0 || (p->ldd * 2) % 16 != 0) return;
  if (!make_map_2d(&maps->d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p->d, p->N, p->M, p->ldd * 2, 32, 32,
                   CU_TENSOR_MAP_SWIZZLE_64B))
    return;
  maps->has_d = true;
  p->store_tma = 1;
}

int pick_bn(int64_t M, int64_t N, int sms) {
  if (N <= 128) return 128;
  const int64_t t256 = ceil_div(M, 128) * ceil_div(N, 256);
  if (t256 < sms && N % 128 == 0) return 128;
  return 256;
}

struct GemmPlan {
  size_t ws = 0;
  bool gemv = false;
  float *gemv_partial = nullptr;
  // in-call quantization of A
  uint8_t *aq_codes = nullptr, *aq_sf = nullptr;
  float *aq_g = nullptr;
  uint32_t *aq_amax = nullptr;
  int aq_nparts = 0;
  __nv_bfloat16 *t = nullptr;   // T' [M][rank]
  float *t32 = nullptr;         // T [lsplit][M][rank] fp32 (dynamic X with LoRA: amax in the same pass)
  int lsplit = 1;
  int bn = 256, ksplit = 1;
  bool pair = false;            // dense product on CTA pairs (256 x 256 tiles)
  bool skinny = false;          // a few rows, weights as the MMA's A operand
  float *partial = nullptr;     // split-K partials [ksplit][M][N]
};

// A few activation rows quantized in the call (decode) take the operand-swapped
// kernel: the weights fill the 128-row side of the MMA, the rows (<= 32) its
// N = 32 side, and a stage carries 24 KB instead of 36 KB.
bool use_skinny(const nvfp4_gemm_args *a) { return a->M <= 32 && a->a_bf16 && !a->lora_a; }

// K ranges for the operand-swapped kernel: enough units (128-feature tiles x
// K ranges) to occupy the SMs, at least four 256-wide K tiles per range.
int pick_skinny_ksplit(int64_t N, int64_t K, int sms) {
  const int64_t tiles = ceil_div(N, 128), nkt = ceil_div(K, 256);
  int64_t ks = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(sms / tiles, nkt / 4), 16));
  const int64_t per = ceil_div(nkt, ks);   // every K range non-empty
  return (int)ceil_div(nkt, per);
}

// The pair kernel serves every dense product with at least one full 256-row
// pair tile and no K split (the small-M decode products keep the 1-SM kernel,
// whose 128-row tiles waste less).
bool use_pair(int64_t M, int ksplit) { return M >= 256 && ksplit == 1; }

// K is split when the output has too few tiles to occupy the SMs (small-M
// decode); the caller's SM count is taken from the device at plan time.
int pick_ksplit(int64_t M, int64_t N, int64_t K, int bn, int sms, bool lora) {
  if (lora) return 1;
  const int64_t tiles = ceil_div(M, 128) * ceil_div(N, bn);
  const int64_t nkt = ceil_div(K, 256);
  if (tiles * 2 > sms || nkt < 8) return 1;
  int64_t ks = std::max<int64_t>(1, (sms + tiles / 2) / tiles);
  ks = std::max<int64_t>(1, std::min<int64_t>(std::min<int64_t>(ks, nkt / 4), 16));
  const int64_t per = ceil_div(nkt, ks);   // every K range non-empty
  return (int)ceil_div(nkt, per);
}

int plan_sms() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 148;
}

bool use_gemv(const nvfp4_gemm_args *a) {
  return a->a_bf16 && a->a_global_scale && a->M <= 4 && a->K % 64 == 0 && !a->lora_a &&
         aligned(a->b_codes, 32) && gemv_smem_bytes(a->M, a->K) <= 200 * 1024;
}

nvfp4_status plan_gemm(const nvfp4_gemm_args *a, GemmPlan *pl) {
  Carve c(a->workspace);
  if (use_gemv(a)) {
    pl->gemv = true;
    const size_t pb = gemv_workspace_bytes(a->M, a->N, a->K);
    if (pb) pl->gemv_partial = c.take<float>(pb);
    pl->ws = c.off;
    return NVFP4_OK;
  }
  if (a->a_bf16) {
    // rows up to the next multiple of 128: the GEMM's A tiles then never
    // reach past the buffer (tensor loads of mostly out-of-range boxes were
    // measured slow: o_proj M = 8 took 23.6 against 20.4 us per call)
    pl->aq_codes = c.take<uint8_t>((size_t)pad_up(a->M, 128) * a->K / 2);
    pl->aq_sf = c.take<uint8_t>(sf_swizzled_bytes(a->M, a->K));
    pl->aq_g = c.take<float>(4);
    if (!a->a_global_scale) {
      pl->aq_nparts = amax_parts_for(a->M);
      // sized for either producer of the partials: the amax kernel or the LoRA pass's grid
      pl->aq_amax = c.take<uint32_t>((size_t)std::max(pl->aq_nparts, 1024) * 4);
    }
  }
  if (a->lora_a) pl->t = c.take<__nv_bfloat16>((size_t)a->M * a->rank * 2);
  // with X quantized in the call, the LoRA-down pass goes first (it reads X
  // from HBM, and takes the amax when the scale is dynamic) and the packing
  // pass reads X from L2 after it
  if (a->lora_a && a->a_bf16 && !a->lora_x) {
    pl->lsplit = lora_split_for(a->K);
    pl->t32 = c.take<float>((size_t)pl->lsplit * a->M * a->rank * 4);
  }
  const int sms = plan_sms();
  pl->bn = pick_bn(a->M, a->N, sms);
  pl->skinny = use_skinny(a);
  pl->ksplit = pl->skinny ? pick_skinny_ksplit(a->N, a->K, sms)
                          : pick_ksplit(a->M, a->N, a->K, pl->bn, sms, a->lora_a != nullptr);
  pl->pair = !pl->skinny && use_pair(a->M, pl->ksplit);
  if (pl->ksplit > 1) pl->partial = c.take<float>((size_t)pl->ksplit * a->M * a->N * 4);
  pl->ws = c.off;
  return NVFP4_OK;
}

nvfp4_status validate_gemm(const nvfp4_gemm_args *a) {
  if (!a || !a->b_codes || !a->b_sf || !a->b_global_scale || !a->d) return NVFP4_ERR_INVALID_ARG;
  if (a->M < 1 || a->N < 1 || a->K < 1) return NVFP4_ERR_INVALID_ARG;
  if (a->out_dtype != NVFP4_OUT_BF16 && a->out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
  if (a->ldd < a->N) return NVFP4_ERR_INVALID_ARG;
  if (!a->a_bf16 && (!a->a_codes || !a->a_sf || !a->a_global_scale)) return NVFP4_ERR_INVALID_ARG;
  if ((a->a_bf16 || a->lora_x) && a->lda < a->K) return NVFP4_ERR_INVALID_ARG;
  if (a->K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->M > (1ll << 31) - 256 || a->N > (1ll << 31) - 256 || a->K > (1ll << 24))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->lora_a || a->lora_b) {
    if (!a->lora_a || !a->lora_b || (!a->lora_x && !a->a_bf16)) return NVFP4_ERR_INVALID_ARG;
    if (a->rank < 32 || a->rank > 256 || a->rank % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(a->lora_a, 16) || !aligned(a->lora_b, 16)) return NVFP4_ERR_ALIGNMENT;
    if (a->lora_x && !aligned(a->lora_x, 16)) return NVFP4_ERR_ALIGNMENT;
  }
  const int64_t dalign = a->out_dtype == NVFP4_OUT_BF16 ? 8 : 4;
  if (!aligned(a->d, 16) || a->ldd % dalign != 0) return NVFP4_ERR_ALIGNMENT;
  if (!aligned(a->b_codes, 16) || !aligned(a->b_sf, 16)) return NVFP4_ERR_ALIGNMENT;
  if (a->a_codes && (!aligned(a->a_codes, 16) || !aligned(a->a_sf, 16))) return NVFP4_ERR_ALIGNMENT;
  if ((a->a_bf16 || a->lora_x) && a->lda % 8 != 0) return NVFP4_ERR_ALIGNMENT;
  if (a->a_bf16 && !aligned(a->a_bf16, 16)) return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

nvfp4_status check_workspace(void *ws, size_t have, size_t need) {
  if (!ws || have < need || !aligned(ws, 256)) return NVFP4_ERR_WORKSPACE;
  return NVFP4_OK;
}

nvfp4_status run_gemm(const nvfp4_gemm_args *a, const GemmPlan &pl, int sms, cudaStream_t st) {
  int *status = static_cast<int *>(a->workspace);
  const uint64_t tmo = g_timeout_ns.load();
  if (pl.gemv) {
    GemvParams g{};
    g.M = a->M;
    g.N = a->N;
    g.K = a->K;
    g.x = static_cast<const __nv_bfloat16 *>(a->a_bf16);
    g.ldx = a->lda;
    g.g_x = a->a_global_scale;
    g.w_codes = a->b_codes;
    g.w_sf = a->b_sf;
    g.w_sf_katoms = pad_up(a->K / 16, 4) / 4;
    g.g_w = a->b_global_scale;
    g.d = a->d;
    g.ldd = a->ldd;
    g.out_fp32 = a->out_dtype == NVFP4_OUT_FP32;
    if (cudaError_t e_ = mark(a->prof_begin, st); e_ != cudaSuccess) return cuda_status(e_);
    cudaError_t e = launch_gemv_ws(g, sms, st, pl.gemv_partial);
    if (e == cudaSuccess) e = mark(a->prof_end, st);
    return cuda_status(e);
  }
  const uint8_t *a_codes = a->a_codes, *a_sf = a->a_sf;
  const float *g_a = a->a_global_scale;
  const void *xb = a->lora_x ? a->lora_x : a->a_bf16;
  const int bn = pl.bn;
  const int b_box = pl.pair ? 128 : bn;   // a CTA of a pair loads half of the 256-row B tile
  GemmMaps maps;
  int lora_steps = 0;
  LoraDownMaps lm;
  LoraDownParams lp{};
  if (a->lora_a) {
    if (!map2d(&lm.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xb, a->K, a->M, a->lda * 2, 64, 128) ||
        !map2d(&lm.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->lora_a, a->K, a->rank, a->K * 2, 64, a->rank) ||
        !map2d(&maps.t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pl.t, a->rank, a->M, a->rank * 2, 64, 128) ||
        !map2d(&maps.lb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->lora_b, a->rank, a->N, a->rank * 2, 64, b_box))
      return NVFP4_ERR_CUDA;
    lp.M = a->M;
    lp.K = a->K;
    lp.rank = a->rank;
    lp.num_k64 = (int)ceil_div(a->K, 64);
    lp.lora_scale = a->alpha / (float)a->rank;
    lp.g_b = a->b_global_scale;
    lp.t_out = pl.t;
    lp.tiles_m = (int)ceil_div(a->M, 128);
    lp.status = status;
    lp.timeout_ns = tmo;
    lora_steps = a->rank / 64 + (a->rank % 64 ? 1 : 0);
  }
  if (a->a_bf16) {
    QuantParams q{};
    q.src = static_cast<const __nv_bfloat16 *>(a->a_bf16);
    q.rows = a->M;
    q.cols = a->K;
    q.ld = a->lda;
    q.batch = 1;
    q.g_in = a->a_global_scale;
    q.g_out = pl.aq_g;
    q.amax_part = pl.aq_amax;
    q.nparts = pl.aq_nparts;
    q.codes_row = pl.aq_codes;
    q.sf_row = pl.aq_sf;
    q.sf_swizzled = 1;
    q.dst_rows = a->M;
    q.status = status;
    q.timeout_ns = tmo;
    if (pl.t32) {
      // one pass over X forms T = X A^T (fp32) and, for a dynamic scale, the
      // amax partials; the packing pass then derives g (or takes the static
      // one), quantizes X and rounds T' = bf16(T s)
      lp.amax_part = a->a_global_scale ? nullptr : pl.aq_amax;
      lp.t_f32 = pl.t32;
      lp.ksplit = pl.lsplit;
      if (cudaError_t e_ = launch_lora_down(lp, lm, sms, st); e_ != cudaSuccess) return cuda_status(e_);
      q.nparts = std::min(lp.tiles_m * pl.lsplit, sms);
      q.t_f32 = pl.t32;
      q.t_splits = pl.lsplit;
      q.t_out = pl.t;
      q.rank = a->rank;
      q.lora_scale = lp.lora_scale;
      q.g_b = a->b_global_scale;
    } else if (!a->a_global_scale) {
      if (cudaError_t e_ = launch_amax(q, st); e_ != cudaSuccess) return cuda_status(e_);
    }
    if (cudaError_t e_ = launch_quant_rows(q, sms, st); e_ != cudaSuccess) return cuda_status(e_);
    a_codes = pl.aq_codes;
    a_sf = pl.aq_sf;
    g_a = pl.aq_g;
  }
  if (a->lora_a && !pl.t32) {
    lp.g_a = g_a;
    if (cudaError_t e_ = launch_lora_down(lp, lm, sms, st); e_ != cudaSuccess) return cuda_status(e_);
  }
  // X quantized in the call: A spans the padded rows of its workspace buffer.
  // Their codes are whatever the buffer held, but their block scales are 0
  // (the packing writes every scale of the last 128-row atom), so they add
  // exactly 0 to accumulator rows that are never stored.
  const int64_t a_rows = a->a_bf16 ? pad_up(a->M, 128) : a->M;
  if (!map2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, a->K / 2, a_rows, a->K / 2, 128, 128) ||
      !map2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->b_codes, a->K / 2, a->N, a->K / 2, 128, b_box))
    return NVFP4_ERR_CUDA;
  if (!a->lora_a) {
    maps.t = maps.a;
    maps.lb = maps.b;
  }
  GemmParams p{};
  p.M = a->M;
  p.N = a->N;
  p.K = a->K;
  p.num_kt = (int)ceil_div(a->K, 256);
  p.nk64 = (int)ceil_div(a->K, 64);
  p.a_sf = a_sf;
  p.b_sf = a->b_sf;
  p.a_sf_katoms = pad_up(a->K / 16, 4) / 4;
  p.b_sf_katoms = p.a_sf_katoms;
  p.b_sf_row_chunks = ceil_div(a->N, 128);
  p.g_a = g_a;
  p.g_b = a->b_global_scale;
  p.d = a->d;
  p.ldd = a->ldd;
  p.out_fp32 = a->out_dtype == NVFP4_OUT_FP32;
  p.lora_steps = lora_steps;
  p.tiles_m = (int)ceil_div(a->M, 128);
  p.tiles_n = (int)ceil_div(a->N, bn);
  p.ksplit = pl.ksplit;
  p.partial = pl.partial;
  p.status = status;
  p.timeout_ns = tmo;
  p.stall_probe = tmo == 0;
  if (pl.skinny) {
    // the activation rows as the MMA's B operand: boxes of 32 rows of the
    // 128-row padded buffer; the weights keep their 128-row boxes
    CUtensorMap mx;
    if (!map2d(&mx, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_codes, a->K / 2, a_rows, a->K / 2, 128, 32) ||
        !map2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->b_codes, a->K / 2, a->N, a->K / 2, 128, 128))
      return NVFP4_ERR_CUDA;
    p.tiles_n = (int)ceil_div(a->N, 128);
    if (cudaError_t e_ = mark(a->prof_begin, st); e_ != cudaSuccess) return cuda_status(e_);
    cudaError_t e = launch_gemm_fp4_skinny(p, mx, maps.b, sms, st);
    if (e == cudaSuccess && pl.ksplit > 1) e = launch_splitk_reduce(p, sms, st);
    if (e == cudaSuccess) e = mark(a->prof_end, st);
    return cuda_status(e);
  }
  if (pl.pair) {
    p.tiles_n = (int)ceil_div(a->N, 256);
    map_pair_d(&maps, &p);
    // 64-row B boxes for the half units of a short last wave
    maps.has_half = map2d(&maps.bh, CU_TENSOR_MAP_DATA_TYPE_UINT8, a->b_codes, a->K / 2, a->N, a->K / 2, 128, 64) &&
                    (!a->lora_a || map2d(&maps.lbh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->lora_b, a->rank, a->N,
                                         a->rank * 2, 64, 64));
    if (!a->lora_a) maps.lbh = maps.bh;
  }
  if (cudaError_t e_ = mark(a->prof_begin, st); e_ != cudaSuccess) return cuda_status(e_);
  cudaError_t e = pl.pair ? launch_gemm_fp4_pair(p, maps, sms, st) : launch_gemm_fp4(p, maps, bn, sms, st);
  if (e == cudaSuccess && pl.ksplit > 1) e = launch_splitk_reduce(p, sms, st);
  if (e == cudaSuccess) e = mark(a->prof_end, st);
  return cuda_status(e);
}

// ------------------------------------------------------------------ grouped --
struct GroupedPlan {
  size_t ws = 0;
  int nchunks = 0;
  int64_t prow_max = 0;
  int32_t *hist = nullptr, *counts = nullptr, *offsets = nullptr, *poffsets = nullptr, *goffsets = nullptr;
  int32_t *row_map = nullptr, *nmt = nullptr;
  GroupTile *gtiles = nullptr;
  uint32_t *amax = nullptr;
  int nparts = 0;
  float *g_x = nullptr;
  uint8_t *xq = nullptr, *xsf = nullptr;      // grouped, padded A operand
  uint8_t *xq_tok = nullptr, *xsf_tok = nullptr;  // X quantized once per token (linear scales)
  __nv_bfloat16 *t = nullptr;
};

nvfp4_status plan_grouped(const nvfp4_grouped_args *a, GroupedPlan *pl) {
  Carve c(a->workspace);
  const int64_t P = a->num_tokens * a->top_k;
  pl->nchunks = (int)ceil_div(P, 1024);
  pl->prow_max = pad_up(P + a->num_experts * 127, 128);
  if (a->expert_ids) {
    pl->hist = c.take<int32_t>((size_t)pl->nchunks * a->num_experts * 4);
    pl->counts = c.take<int32_t>((size_t)a->num_experts * 4);
    pl->offsets = c.take<int32_t>((size_t)(a->num_experts + 1) * 4);
  } else {
    pl->goffsets = c.take<int32_t>((size_t)(a->num_experts + 1) * 4);
  }
  pl->poffsets = c.take<int32_t>((size_t)(a->num_experts + 1) * 4);
  pl->row_map = c.take<int32_t>((size_t)pl->prow_max * 4);
  pl->gtiles = c.take<GroupTile>((size_t)(pl->prow_max / 128) * sizeof(GroupTile));
  pl->nmt = c.take<int32_t>(4);
  if (!a->x_codes) {
    if (!a->x_global_scale) {
      pl->nparts = amax_parts_for(a->num_tokens);
      pl->amax = c.take<uint32_t>((size_t)pl->nparts * 4);
    }
    pl->g_x = c.take<float>(4);
    pl->xq_tok = c.take<uint8_t>((size_t)a->num_tokens * a->K / 2);
    pl->xsf_tok = c.take<uint8_t>((size_t)a->num_tokens * (a->K / 16));
  }
  pl->xq = c.take<uint8_t>((size_t)pl->prow_max * a->K / 2);
  pl->xsf = c.take<uint8_t>(sf_swizzled_bytes(pl->prow_max, a->K));
  if (a->lora_a) pl->t = c.take<__nv_bfloat16>((size_t)pl->prow_max * a->rank * 2);
  pl->ws = c.off;
  return NVFP4_OK;
}

nvfp4_status validate_grouped(const nvfp4_grouped_args *a) {
  if (!a || !a->w_codes || !a->w_sf || !a->w_global_scale || !a->d) return NVFP4_ERR_INVALID_ARG;
  // routing: expert ids (grouped here, perm_out required) or offsets + perm given
  const bool ids = a->expert_ids != nullptr, given = a->offsets_in && a->perm_in;
  if (ids == given || (!given && (a->offsets_in || a->perm_in))) return NVFP4_ERR_INVALID_ARG;
  if (ids && !a->perm_out) return NVFP4_ERR_INVALID_ARG;
  // activations: bf16 rows, or packed rows with their global scale
  if (a->x_codes || a->x_sf) {
    if (!a->x_codes || !a->x_sf || !a->x_global_scale) return NVFP4_ERR_INVALID_ARG;
  } else if (!a->x_bf16) {
    return NVFP4_ERR_INVALID_ARG;
  }
  if ((a->lora_a || a->lora_b) && !a->x_bf16) return NVFP4_ERR_INVALID_ARG;
  if (a->out_dtype != NVFP4_OUT_BF16 && a->out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
  if (a->num_tokens < 1 || a->top_k < 1 || a->num_experts < 1 || a->N < 1 || a->K < 1)
    return NVFP4_ERR_INVALID_ARG;
  if (a->num_experts > 1024 || a->top_k > a->num_experts) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->N % 256 != 0 || a->K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->num_tokens * a->top_k > (1ll << 30) || a->num_experts * a->N > (1ll << 31) - 256)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->lora_a || a->lora_b) {
    if (!a->lora_a || !a->lora_b) return NVFP4_ERR_INVALID_ARG;
    if (a->rank < 32 || a->rank > 256 || a->rank % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(a->lora_a, 16) || !aligned(a->lora_b, 16)) return NVFP4_ERR_ALIGNMENT;
  }
  const void *ptrs[] = {a->x_bf16, a->w_codes, a->w_sf, a->d, a->x_codes, a->x_sf, a->offsets_in, a->perm_in};
  for (const void *q : ptrs)
    if (q && !aligned(q, 16)) return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

// The expert products of a grouped operand already in the padded layout: the
// optional per-expert LoRA down pass (X rows gathered through row_map) and the
// grouped W4A4 GEMM with the fused LoRA up-projection, D in grouped row order.
struct GroupedProducts {
  int64_t E, N, K, prow_max;
  int64_t out_rows;               // rows of d (the pairs)
  const uint8_t *aq, *asf;        // padded A codes / swizzled scales
  const float *g_a;
  const int32_t *row_map;         // padded row -> row of x_src (-1: padding)
  const GroupTile *gtiles;
  const int32_t *nmt;
  const void *x_src;              // bf16 source rows of the LoRA input [x_rows][K]
  int64_t x_rows;
  const void *w_codes, *w_sf;
  const float *w_g;
  const void *lora_a, *lora_b;
  int32_t rank;
  float alpha;
  __nv_bfloat16 *t;               // [prow_max][rank] T' scratch
  void *d;                        // [P][N], bf16 or fp32
  int out_fp32;
  void *prof_begin, *prof_end;
};

nvfp4_status run_grouped_products(const GroupedProducts &g, int *status, uint64_t tmo, int sms,
                                  cudaStream_t st) {
  const int bn = 256;
  GemmMaps maps;
  if (!map2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.aq, g.K / 2, g.prow_max, g.K / 2, 128, 128) ||
      !map2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, g.w_codes, g.K / 2, g.E * g.N, g.K / 2, 128, bn))
    return NVFP4_ERR_CUDA;
  maps.t = maps.a;
  maps.lb = maps.b;
  int lora_steps = 0;
  if (g.lora_a) {
    LoraDownMaps lm;
    if (!make_map_2d(&lm.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.x_src, g.K, g.x_rows, g.K * 2, 64, 1,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !map2d(&lm.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.lora_a, g.K, g.E * g.rank, g.K * 2, 64, g.rank) ||
        !map2d(&maps.t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.t, g.rank, g.prow_max, g.rank * 2, 64, 128) ||
        !map2d(&maps.lb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g.lora_b, g.rank, g.E * g.N, g.rank * 2, 64, bn))
      return NVFP4_ERR_CUDA;
    LoraDownParams lp{};
    lp.M = g.prow_max;
    lp.K = g.K;
    lp.rank = g.rank;
    lp.num_k64 = (int)ceil_div(g.K, 64);
    lp.lora_scale = g.alpha / (float)g.rank;
    lp.g_a = g.g_a;
    lp.g_b = g.w_g;
    lp.t_out = g.t;
    lp.gtiles = g.gtiles;
    lp.gnum_mtiles = g.nmt;
    lp.row_map = g.row_map;
    lp.x = static_cast<const __nv_bfloat16 *>(g.x_src);
    lp.x_rows = g.x_rows;
    lp.status = status;
    lp.timeout_ns = tmo;
    if (cudaError_t e_ = launch_lora_down(lp, lm, sms, st); e_ != cudaSuccess) return cuda_status(e_);
    lora_steps = g.rank / 64 + (g.rank % 64 ? 1 : 0);
  }
  GemmParams p{};
  p.M = g.prow_max;
  p.N = g.N;
  p.K = g.K;
  p.num_kt = (int)ceil_div(g.K, 256);
  p.nk64 = (int)ceil_div(g.K, 64);
  p.a_sf = g.asf;
  p.b_sf = static_cast<const uint8_t *>(g.w_sf);
  p.a_sf_katoms = pad_up(g.K / 16, 4) / 4;
  p.b_sf_katoms = p.a_sf_katoms;
  p.b_sf_row_chunks = g.E * g.N / 128;
  p.g_a = g.g_a;
  p.g_b = g.w_g;
  p.d = g.d;
  p.ldd = g.N;
  p.out_fp32 = g.out_fp32;
  p.lora_steps = lora_steps;
  p.tiles_n = (int)(g.N / bn);
  p.gtiles = g.gtiles;
  p.gnum_mtiles = g.nmt;
  p.out_rows = g.out_rows;
  p.status = status;
  p.timeout_ns = tmo;
  p.stall_probe = tmo == 0;
  if (cudaError_t e_ = mark(g.prof_begin, st); e_ != cudaSuccess) return cuda_status(e_);
  cudaError_t e = launch_gemm_fp4(p, maps, bn, sms, st);
  if (e == cudaSuccess) e = mark(g.prof_end, st);
  return cuda_status(e);
}

nvfp4_status run_grouped(const nvfp4_grouped_args *a, const GroupedPlan &pl, int sms, cudaStream_t st) {
  int *status = static_cast<int *>(a->workspace);
  const uint64_t tmo = g_timeout_ns.load();
  const int64_t P = a->num_tokens * a->top_k;
  if (a->expert_ids) {
    RouteParams r{};
    r.expert_ids = a->expert_ids;
    r.pairs = P;
    r.top_k = (int)a->top_k;
    r.num_experts = (int)a->num_experts;
    r.chunk = 1024;
    r.nchunks = pl.nchunks;
    r.hist = pl.hist;
    r.counts = pl.counts;
    r.offsets = pl.offsets;
    r.poffsets = pl.poffsets;
    r.perm = a->perm_out;
    r.row_map = pl.row_map;
    r.padded_rows_max = pl.prow_max;
    r.gtiles = pl.gtiles;
    r.gnum_mtiles = pl.nmt;
    r.offsets_out = a->expert_offsets_out;
    r.status = status;
    if (cudaError_t e_ = launch_route(r, st); e_ != cudaSuccess) return cuda_status(e_);
  } else {
    // the caller's grouping: padded layout from its offsets, row_map -> token through its perm
    if (cudaError_t e_ = launch_layout_from_offsets(a->offsets_in, (int)a->num_experts, P, pl.prow_max, pl.goffsets,
                                                    pl.poffsets, pl.gtiles, pl.nmt, pl.row_map, a->perm_in,
                                                    (int)a->top_k, sms, st, status);
        e_ != cudaSuccess)
      return cuda_status(e_);
    if (a->perm_out && a->perm_out != a->perm_in &&
        cudaMemcpyAsync(a->perm_out, a->perm_in, (size_t)P * 4, cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    if (a->expert_offsets_out && cudaMemcpyAsync(a->expert_offsets_out, pl.goffsets, (size_t)(a->num_experts + 1) * 4,
                                                 cudaMemcpyDeviceToDevice, st) != cudaSuccess)
      return NVFP4_ERR_CUDA;
  }
  if (a->x_codes) {
    // activations already quantized per token row (linear scales) with x_global_scale
    if (cudaError_t e_ = launch_gather_packed(a->x_codes, a->x_sf, pl.row_map, pl.prow_max, pl.nmt, a->K, pl.xq,
                                              pl.xsf, sms, st, a->num_tokens, status);
        e_ != cudaSuccess)
      return cuda_status(e_);
    GroupedProducts gp;
    gp.E = a->num_experts;
    gp.N = a->N;
    gp.K = a->K;
    gp.prow_max = pl.prow_max;
  gp.out_rows = P;
    gp.out_rows = P;
    gp.aq = pl.xq;
    gp.asf = pl.xsf;
    gp.g_a = a->x_global_scale;
    gp.row_map = pl.row_map;
    gp.gtiles = pl.gtiles;
    gp.nmt = pl.nmt;
    gp.x_src = a->x_bf16;
    gp.x_rows = a->num_tokens;
    gp.w_codes = a->w_codes;
    gp.w_sf = a->w_sf;
    gp.w_g = a->w_global_scale;
    gp.lora_a = a->lora_a;
    gp.lora_b = a->lora_b;
    gp.rank = a->rank;
    gp.alpha = a->alpha;
    gp.t = pl.t;
    gp.d = a->d;
    gp.out_fp32 = a->out_dtype == NVFP4_OUT_FP32;
    gp.prof_begin = a->prof_begin;
    gp.prof_end = a->prof_end;
    return run_grouped_products(gp, status, tmo, sms, st);
  }

  QuantParams q{};
  q.src = static_cast<const __nv_bfloat16 *>(a->x_bf16);
  q.rows = a->num_tokens;
  q.cols = a->K;
  q.ld = a->K;
  q.batch = 1;
  q.g_in = a->x_global_scale;
  q.g_out = pl.g_x;
  q.amax_part = pl.amax;
  q.nparts = pl.nparts;
  // every token row is quantized once (one tensor-wide g), then its codes and
  // scales are copied to each of its top_k rows of the grouped operand
  q.codes_row = pl.xq_tok;
  q.sf_row = pl.xsf_tok;
  q.sf_swizzled = 0;
  q.dst_rows = a->num_tokens;
  q.status = status;
  q.timeout_ns = tmo;
  if (!a->x_global_scale) {
    if (cudaError_t e_ = launch_amax(q, st); e_ != cudaSuccess) return cuda_status(e_);
  }
  if (cudaError_t e_ = launch_quant_rows(q, sms, st); e_ != cudaSuccess) return cuda_status(e_);
  if (cudaError_t e_ = launch_gather_packed(pl.xq_tok, pl.xsf_tok, pl.row_map, pl.prow_max, pl.nmt, a->K, pl.xq,
                                            pl.xsf, sms, st, a->num_tokens, status);
      e_ != cudaSuccess)
    return cuda_status(e_);
  GroupedProducts gp;
  gp.E = a->num_experts;
  gp.N = a->N;
  gp.K = a->K;
  gp.prow_max = pl.prow_max;
  gp.out_rows = P;
  gp.aq = pl.xq;
  gp.asf = pl.xsf;
  gp.g_a = a->x_global_scale ? a->x_global_scale : pl.g_x;
  gp.row_map = pl.row_map;
  gp.gtiles = pl.gtiles;
  gp.nmt = pl.nmt;
  gp.x_src = a->x_bf16;
  gp.x_rows = a->num_tokens;
  gp.w_codes = a->w_codes;
  gp.w_sf = a->w_sf;
  gp.w_g = a->w_global_scale;
  gp.lora_a = a->lora_a;
  gp.lora_b = a->lora_b;
  gp.rank = a->rank;
  gp.alpha = a->alpha;
  gp.t = pl.t;
  gp.d = a->d;
  gp.out_fp32 = a->out_dtype == NVFP4_OUT_FP32;
  gp.prof_begin = a->prof_begin;
  gp.prof_end = a->prof_end;
  return run_grouped_products(gp, status, tmo, sms, st);
}

// ------------------------------------------------------- MoE down + combine --
struct MoeDownPlan {
  size_t ws = 0;
  int64_t prow_max = 0;
  int32_t *goffsets = nullptr, *poffsets = nullptr, *row_map = nullptr, *nmt = nullptr, *inv = nullptr;
  GroupTile *gtiles = nullptr;
  uint32_t *amax = nullptr;
  int nparts = 0;
  float *g_h = nullptr;
  uint8_t *hq = nullptr, *hsf = nullptr;
  __nv_bfloat16 *t = nullptr, *d = nullptr;
};

void plan_moe_down(const nvfp4_moe_down_args *a, MoeDownPlan *pl) {
  Carve c(a->workspace);
  const int64_t P = a->num_tokens * a->top_k;
  pl->prow_max = pad_up(P + a->num_experts * 127, 128);
  pl->goffsets = c.take<int32_t>((size_t)(a->num_experts + 1) * 4);
  pl->poffsets = c.take<int32_t>((size_t)(a->num_experts + 1) * 4);
  pl->row_map = c.take<int32_t>((size_t)pl->prow_max * 4);
  pl->gtiles = c.take<GroupTile>((size_t)(pl->prow_max / 128) * sizeof(GroupTile));
  pl->nmt = c.take<int32_t>(4);
  pl->inv = c.take<int32_t>((size_t)P * 4);
  if (!a->h_global_scale) {
    pl->nparts = amax_parts_for(P);
    pl->amax = c.take<uint32_t>((size_t)pl->nparts * 4);
  }
  pl->g_h = c.take<float>(4);
  pl->hq = c.take<uint8_t>((size_t)pl->prow_max * a->K / 2);
  pl->hsf = c.take<uint8_t>(sf_swizzled_bytes(pl->prow_max, a->K));
  if (a->lora_a) pl->t = c.take<__nv_bfloat16>((size_t)pl->prow_max * a->rank * 2);
  pl->d = c.take<__nv_bfloat16>((size_t)P * a->N * 2);
  pl->ws = c.off;
}

nvfp4_status validate_moe_down(const nvfp4_moe_down_args *a) {
  if (!a || !a->h || !a->perm || !a->expert_offsets || !a->route_weights || !a->w_codes || !a->w_sf ||
      !a->w_global_scale || !a->y)
    return NVFP4_ERR_INVALID_ARG;
  if (a->num_tokens < 1 || a->top_k < 1 || a->num_experts < 1 || a->N < 1 || a->K < 1)
    return NVFP4_ERR_INVALID_ARG;
  if (a->num_experts > 1024 || a->top_k > a->num_experts) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->N % 256 != 0 || a->K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->num_tokens * a->top_k > (1ll << 30) || a->num_experts * a->N > (1ll << 31) - 256)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->lora_a || a->lora_b) {
    if (!a->lora_a || !a->lora_b) return NVFP4_ERR_INVALID_ARG;
    if (a->rank < 32 || a->rank > 256 || a->rank % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(a->lora_a, 16) || !aligned(a->lora_b, 16)) return NVFP4_ERR_ALIGNMENT;
  }
  if (!aligned(a->h, 16) || !aligned(a->w_codes, 16) || !aligned(a->w_sf, 16) || !aligned(a->y, 16))
    return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

nvfp4_status run_moe_down(const nvfp4_moe_down_args *a, const MoeDownPlan &pl, int sms, cudaStream_t st) {
  int *status = static_cast<int *>(a->workspace);
  const uint64_t tmo = g_timeout_ns.load();
  const int64_t P = a->num_tokens * a->top_k;
  if (cudaError_t e_ = launch_layout_from_offsets(a->expert_offsets, (int)a->num_experts, P, pl.prow_max,
                                                  pl.goffsets, pl.poffsets, pl.gtiles, pl.nmt, pl.row_map,
                                                  nullptr, 0, sms, st, status);
      e_ != cudaSuccess)
    return cuda_status(e_);
  // h is quantized once (one tensor-wide g) straight into the padded layout:
  // padded row r takes grouped row row_map[r]
  QuantParams q{};
  q.src = static_cast<const __nv_bfloat16 *>(a->h);
  q.rows = P;
  q.cols = a->K;
  q.ld = a->K;
  q.batch = 1;
  q.g_in = a->h_global_scale;
  q.g_out = pl.g_h;
  q.amax_part = pl.amax;
  q.nparts = pl.nparts;
  q.codes_row = pl.hq;
  q.sf_row = pl.hsf;
  q.sf_swizzled = 1;
  q.row_map = pl.row_map;
  q.dst_rows = pl.prow_max;
  q.num_mtiles = pl.nmt;   // rows past the routed layout are never read
  q.status = status;
  q.timeout_ns = tmo;
  if (!a->h_global_scale) {
    if (cudaError_t e_ = launch_amax(q, st); e_ != cudaSuccess) return cuda_status(e_);
  }
  if (cudaError_t e_ = launch_quant_rows(q, sms, st); e_ != cudaSuccess) return cuda_status(e_);
  GroupedProducts gp;
  gp.E = a->num_experts;
  gp.N = a->N;
  gp.K = a->K;
  gp.prow_max = pl.prow_max;
  gp.out_rows = P;
  gp.aq = pl.hq;
  gp.asf = pl.hsf;
  gp.g_a = a->h_global_scale ? a->h_global_scale : pl.g_h;
  gp.row_map = pl.row_map;
  gp.gtiles = pl.gtiles;
  gp.nmt = pl.nmt;
  gp.x_src = a->h;
  gp.x_rows = P;
  gp.w_codes = a->w_codes;
  gp.w_sf = a->w_sf;
  gp.w_g = a->w_global_scale;
  gp.lora_a = a->lora_a;
  gp.lora_b = a->lora_b;
  gp.rank = a->rank;
  gp.alpha = a->alpha;
  gp.t = pl.t;
  gp.d = pl.d;
  gp.out_fp32 = 0;
  gp.prof_begin = a->prof_begin;
  gp.prof_end = a->prof_end;
  nvfp4_status s = run_grouped_products(gp, status, tmo, sms, st);
  if (s != NVFP4_OK) return s;
  return cuda_status(launch_moe_combine(pl.d, a->perm, pl.inv, a->route_weights, a->num_tokens,
                                        (int)a->top_k, a->N, static_cast<__nv_bfloat16 *>(a->y), sms, st,
                                        status));
}

// --------------------------------------------------------------------- LoRA --
struct LoraPlan {
  size_t ws = 0;
  __nv_bfloat16 *t = nullptr;
};

nvfp4_status plan_lora(const nvfp4_lora_args *a, LoraPlan *pl) {
  Carve c(a->workspace);
  pl->t = c.take<__nv_bfloat16>((size_t)a->M * a->rank * 2);
  pl->ws = c.off;
  return NVFP4_OK;
}

nvfp4_status validate_lora(const nvfp4_lora_args *a) {
  if (!a || !a->x || !a->lora_a || !a->lora_b || !a->y) return NVFP4_ERR_INVALID_ARG;
  if (a->M < 1 || a->N < 1 || a->K < 1 || a->ldx < a->K || a->ldy < a->N) return NVFP4_ERR_INVALID_ARG;
  if (a->y_dtype != NVFP4_OUT_BF16 && a->y_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
  if (a->rank < 32 || a->rank > 256 || a->rank % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->K % 8 != 0 || a->M > (1ll << 31) - 256 || a->N > (1ll << 31) - 256) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a->x, 16) || !aligned(a->lora_a, 16) || !aligned(a->lora_b, 16) || !aligned(a->y, 16) ||
      a->ldx % 8 != 0)
    return NVFP4_ERR_ALIGNMENT;
  if (a->y_dtype == NVFP4_OUT_FP32 ? a->ldy % 4 != 0 : a->ldy % 8 != 0) return NVFP4_ERR_ALIGNMENT;
  if (a->delta_sq_norm_out && !aligned(a->delta_sq_norm_out, 4)) return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

nvfp4_status run_lora(const nvfp4_lora_args *a, const LoraPlan &pl, int sms, cudaStream_t st) {
  int *status = static_cast<int *>(a->workspace);
  const uint64_t tmo = g_timeout_ns.load();
  const int bn = a->N <= 128 ? 128 : 256;
  LoraDownMaps lm;
  GemmMaps maps;
  if (!map2d(&lm.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->x, a->K, a->M, a->ldx * 2, 64, 128) ||
      !map2d(&lm.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->lora_a, a->K, a->rank, a->K * 2, 64, a->rank) ||
      !map2d(&maps.t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pl.t, a->rank, a->M, a->rank * 2, 64, 128) ||
      !map2d(&maps.lb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->lora_b, a->rank, a->N, a->rank * 2, 64, bn))
    return NVFP4_ERR_CUDA;
  maps.a = maps.t;
  maps.b = maps.lb;
  LoraDownParams lp{};
  lp.M = a->M;
  lp.K = a->K;
  lp.rank = a->rank;
  lp.num_k64 = (int)ceil_div(a->K, 64);
  lp.lora_scale = a->alpha / (float)a->rank;
  lp.t_out = pl.t;
  lp.tiles_m = (int)ceil_div(a->M, 128);
  lp.status = status;
  lp.timeout_ns = tmo;
  if (cudaError_t e_ = launch_lora_down(lp, lm, sms, st); e_ != cudaSuccess) return cuda_status(e_);
  if (a->delta_sq_norm_out && cudaMemsetAsync(a->delta_sq_norm_out, 0, 4, st) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  GemmParams p{};
  p.M = a->M;
  p.N = a->N;
  p.K = 0;
  p.num_kt = 0;
  p.nk64 = 0;
  p.d = a->y;
  p.ldd = a->ldy;
  p.out_fp32 = a->y_dtype == NVFP4_OUT_FP32;
  p.accumulate_d = 1;
  p.sqnorm = a->delta_sq_norm_out;
  p.lora_steps = a->rank / 64 + (a->rank % 64 ? 1 : 0);
  p.tiles_m = (int)ceil_div(a->M, 128);
  p.tiles_n = (int)ceil_div(a->N, bn);
  p.status = status;
  p.timeout_ns = tmo;
  p.stall_probe = tmo == 0;
  return cuda_status(launch_gemm_fp4(p, maps, bn, sms, st));
}

// ---------------------------------------------------------------- dequant --
nvfp4_status validate_dequant(const nvfp4_dequant_args *a) {
  if (!a || !a->codes || !a->sf || !a->global_scale || !a->out) return NVFP4_ERR_INVALID_ARG;
  if (a->rows < 1 || a->cols < 1) return NVFP4_ERR_INVALID_ARG;
  if (a->sf_layout != NVFP4_SF_LINEAR && a->sf_layout != NVFP4_SF_SWIZZLED) return NVFP4_ERR_INVALID_ARG;
  if (a->cols % 64 != 0 || (a->transpose && a->rows % 2 != 0)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->ldo < (a->transpose ? a->rows : a->cols)) return NVFP4_ERR_INVALID_ARG;
  // transposed rows are written as bf16 pairs (4-byte words), untransposed as 16-byte vectors
  if (!aligned(a->codes, 16) || !aligned(a->sf, 16) || !aligned(a->out, 16) ||
      a->ldo % (a->transpose ? 2 : 8) != 0)
    return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

// ------------------------------------------------------------------ dgrad --
// A bf16 tensor-core GEMM D[M][Nout] = A[M][Kc] B[Nout][Kc]^T on the FP4 GEMM
// kernel with no FP4 steps: every pipeline stage is a 64-wide kind::f16 step
// (the path the LoRA up-projection uses), fp32 accumulation, scale 1.
nvfp4_status run_bf16_gemm(int64_t M, int64_t Nout, int64_t Kc, const void *A, int64_t lda, const void *B,
                           int64_t ldb, void *D, int64_t ldd, int out_fp32, int *status, void *prof_begin,
                           void *prof_end, int sms, cudaStream_t st) {
  const uint64_t tmo = g_timeout_ns.load();
  const int bn = pick_bn(M, Nout, sms);
  const bool pair = use_pair(M, 1);
  GemmMaps maps;
  if (!map2d(&maps.t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, Kc, M, lda * 2, 64, 128) ||
      !map2d(&maps.lb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, Kc, Nout, ldb * 2, 64, pair ? 128 : bn))
    return NVFP4_ERR_CUDA;
  maps.a = maps.t;
  maps.b = maps.lb;
  GemmParams p{};
  p.M = M;
  p.N = Nout;
  p.K = 0;
  p.num_kt = 0;
  p.nk64 = 0;
  p.d = D;
  p.ldd = ldd;
  p.out_fp32 = out_fp32;
  p.lora_steps = (int)ceil_div(Kc, 64);
  p.tiles_m = (int)ceil_div(M, 128);
  p.tiles_n = (int)ceil_div(Nout, pair ? 256 : bn);
  p.ksplit = 1;
  p.status = status;
  p.timeout_ns = tmo;
  p.stall_probe = tmo == 0;
  if (pair) {
    map_pair_d(&maps, &p);
    // 64-row B boxes for the half units of a short last wave
    maps.has_half = map2d(&maps.lbh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, B, Kc, Nout, ldb * 2, 64, 64);
    maps.bh = maps.lbh;
  }
  if (cudaError_t e_ = mark(prof_begin, st); e_ != cudaSuccess) return cuda_status(e_);
  cudaError_t e = pair ? launch_gemm_fp4_pair(p, maps, sms, st) : launch_gemm_fp4(p, maps, bn, sms, st);
  if (e == cudaSuccess) e = mark(prof_end, st);
  return cuda_status(e);
}

nvfp4_gemm_args dgrad_as_gemm(const nvfp4_dgrad_args *a) {
  nvfp4_gemm_args g{};
  g.M = a->M;
  g.N = a->K;   // output columns
  g.K = a->N;   // contraction
  g.a_bf16 = a->dy;
  g.lda = a->lddy;
  g.a_global_scale = a->dy_global_scale;
  g.b_codes = static_cast<const uint8_t *>(a->wcol_codes);
  g.b_sf = static_cast<const uint8_t *>(a->wcol_sf);
  g.b_global_scale = a->w_global_scale;
  g.out_dtype = a->out_dtype;
  g.d = a->dx;
  g.ldd = a->lddx;
  g.workspace = a->workspace;
  g.workspace_bytes = a->workspace_bytes;
  g.prof_begin = a->prof_begin;
  g.prof_end = a->prof_end;
  return g;
}

nvfp4_status validate_dgrad(const nvfp4_dgrad_args *a) {
  if (!a || !a->dy || !a->dx || !a->w_global_scale) return NVFP4_ERR_INVALID_ARG;
  if (a->M < 1 || a->N < 1 || a->K < 1 || a->lddy < a->N || a->lddx < a->K) return NVFP4_ERR_INVALID_ARG;
  if (a->out_dtype != NVFP4_OUT_BF16 && a->out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
  if (a->N % 64 != 0 || a->K % 64 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->M > (1ll << 31) - 256 || a->N > (1ll << 24) || a->K > (1ll << 31) - 256)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->mode == NVFP4_DGRAD_DEQUANT_BF16) {
    if (!a->w_codes || !a->w_sf) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(a->w_codes, 16) || !aligned(a->w_sf, 16)) return NVFP4_ERR_ALIGNMENT;
  } else if (a->mode == NVFP4_DGRAD_FP4_COLPACK) {
    if (!a->wcol_codes || !a->wcol_sf) return NVFP4_ERR_INVALID_ARG;
    const nvfp4_gemm_args g = dgrad_as_gemm(a);
    return validate_gemm(&g);
  } else {
    return NVFP4_ERR_INVALID_ARG;
  }
  if (!aligned(a->dy, 16) || a->lddy % 8 != 0) return NVFP4_ERR_ALIGNMENT;
  const int64_t dalign = a->out_dtype == NVFP4_OUT_BF16 ? 8 : 4;
  if (!aligned(a->dx, 16) || a->lddx % dalign != 0) return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

size_t dgrad_workspace(const nvfp4_dgrad_args *a) {
  if (a->mode == NVFP4_DGRAD_FP4_COLPACK) {
    nvfp4_gemm_args g = dgrad_as_gemm(a);
    g.workspace = nullptr;
    GemmPlan pl;
    plan_gemm(&g, &pl);
    return pl.ws;
  }
  Carve c(nullptr);
  c.take<__nv_bfloat16>((size_t)a->K * a->N * 2);   // W^T in bf16
  return c.off;
}

nvfp4_status run_dgrad(const nvfp4_dgrad_args *a, int sms, cudaStream_t st) {
  if (a->mode == NVFP4_DGRAD_FP4_COLPACK) {
    const nvfp4_gemm_args g = dgrad_as_gemm(a);
    GemmPlan pl;
    plan_gemm(&g, &pl);
    return run_gemm(&g, pl, sms, st);
  }
  Carve c(a->workspace);
  __nv_bfloat16 *wt = c.take<__nv_bfloat16>((size_t)a->K * a->N * 2);
  if (cudaError_t e_ = launch_dequant(static_cast<const uint8_t *>(a->w_codes),
                                      static_cast<const uint8_t *>(a->w_sf), 1, a->w_global_scale, a->N,
                                      a->K, 1, wt, a->N, sms, st);
      e_ != cudaSuccess)
    return cuda_status(e_);
  return run_bf16_gemm(a->M, a->K, a->N, a->dy, a->lddy, wt, a->N, a->dx, a->lddx,
                       a->out_dtype == NVFP4_OUT_FP32, static_cast<int *>(a->workspace), a->prof_begin,
                       a->prof_end, sms, st);
}

// ------------------------------------------------------------------ wgrad --
struct WgradPlan {
  size_t ws = 0;
  uint8_t *dy_codes = nullptr, *dy_sf = nullptr, *x_codes = nullptr, *x_sf = nullptr;
  float *g_dy = nullptr, *g_x = nullptr;
  uint8_t *q_dy_ws = nullptr, *q_x_ws = nullptr, *gemm_ws = nullptr;
  size_t q_dy_bytes = 0, q_x_bytes = 0, gemm_bytes = 0;
};

nvfp4_quant_args wgrad_quant(const void *src, int64_t M, int64_t cols, int64_t ld, const float *g_in,
                             float *g_out, uint8_t *codes, uint8_t *sf, void *ws, size_t ws_bytes) {
  nvfp4_quant_args q{};
  q.src = src;
  q.batch = 1;
  q.rows = M;
  q.cols = cols;
  q.ld = ld;
  q.pack = NVFP4_PACK_COL;
  q.sf_layout = NVFP4_SF_SWIZZLED;
  q.global_scale_in = g_in;
  q.global_scale_out = g_out;
  q.codes_col = codes;
  q.sf_col = sf;
  q.workspace = ws;
  q.workspace_bytes = ws_bytes;
  return q;
}

nvfp4_gemm_args wgrad_gemm(const nvfp4_wgrad_args *a, const WgradPlan &pl) {
  nvfp4_gemm_args g{};
  g.M = a->N;   // rows of dW
  g.N = a->K;   // columns of dW
  g.K = a->M;   // contraction over the tokens
  g.a_codes = pl.dy_codes;
  g.a_sf = pl.dy_sf;
  g.a_global_scale = pl.g_dy;
  g.b_codes = pl.x_codes;
  g.b_sf = pl.x_sf;
  g.b_global_scale = pl.g_x;
  g.out_dtype = a->out_dtype;
  g.d = a->dw;
  g.ldd = a->lddw;
  g.workspace = pl.gemm_ws;
  g.workspace_bytes = pl.gemm_bytes;
  g.prof_begin = a->prof_begin;
  g.prof_end = a->prof_end;
  return g;
}

void plan_wgrad(const nvfp4_wgrad_args *a, WgradPlan *pl) {
  Carve c(a->workspace);
  pl->dy_codes = c.take<uint8_t>((size_t)a->N * a->M / 2);
  pl->dy_sf = c.take<uint8_t>(sf_swizzled_bytes(a->N, a->M));
  pl->g_dy = c.take<float>(4);
  pl->x_codes = c.take<uint8_t>((size_t)a->K * a->M / 2);
  pl->x_sf = c.take<uint8_t>(sf_swizzled_bytes(a->K, a->M));
  pl->g_x = c.take<float>(4);
  {
    nvfp4_quant_args q = wgrad_quant(a->dy, a->M, a->N, a->lddy, a->dy_global_scale, pl->g_dy, pl->dy_codes,
                                     pl->dy_sf, nullptr, 0);
    QuantPlan qp;
    plan_quantize(&q, &qp);
    pl->q_dy_bytes = qp.ws;
    pl->q_dy_ws = c.take<uint8_t>(qp.ws);
  }
  {
    nvfp4_quant_args q = wgrad_quant(a->x, a->M, a->K, a->ldx, a->x_global_scale, pl->g_x, pl->x_codes,
                                     pl->x_sf, nullptr, 0);
    QuantPlan qp;
    plan_quantize(&q, &qp);
    pl->q_x_bytes = qp.ws;
    pl->q_x_ws = c.take<uint8_t>(qp.ws);
  }
  {
    nvfp4_gemm_args g = wgrad_gemm(a, *pl);
    g.workspace = nullptr;
    GemmPlan gp;
    plan_gemm(&g, &gp);
    pl->gemm_bytes = gp.ws;
    pl->gemm_ws = c.take<uint8_t>(gp.ws);
  }
  pl->ws = c.off;
}

nvfp4_status validate_wgrad(const nvfp4_wgrad_args *a) {
  if (!a || !a->dy || !a->x || !a->dw) return NVFP4_ERR_INVALID_ARG;
  if (a->M < 1 || a->N < 1 || a->K < 1 || a->lddy < a->N || a->ldx < a->K || a->lddw < a->K)
    return NVFP4_ERR_INVALID_ARG;
  if (a->out_dtype != NVFP4_OUT_BF16 && a->out_dtype != NVFP4_OUT_FP32) return NVFP4_ERR_INVALID_ARG;
  if (a->M % 32 != 0 || a->N % 16 != 0 || a->K % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (a->M > (1ll << 24) || a->N > (1ll << 31) - 256 || a->K > (1ll << 31) - 256)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned(a->dy, 16) || !aligned(a->x, 16) || a->lddy % 8 != 0 || a->ldx % 8 != 0)
    return NVFP4_ERR_ALIGNMENT;
  const int64_t dalign = a->out_dtype == NVFP4_OUT_BF16 ? 8 : 4;
  if (!aligned(a->dw, 16) || a->lddw % dalign != 0) return NVFP4_ERR_ALIGNMENT;
  return NVFP4_OK;
}

nvfp4_status run_wgrad(const nvfp4_wgrad_args *a, const WgradPlan &pl, int sms, cudaStream_t st) {
  const nvfp4_quant_args qd = wgrad_quant(a->dy, a->M, a->N, a->lddy, a->dy_global_scale, pl.g_dy, pl.dy_codes,
                                          pl.dy_sf, pl.q_dy_ws, pl.q_dy_bytes);
  const nvfp4_quant_args qx = wgrad_quant(a->x, a->M, a->K, a->ldx, a->x_global_scale, pl.g_x, pl.x_codes,
                                          pl.x_sf, pl.q_x_ws, pl.q_x_bytes);
  nvfp4_status s;
  QuantPlan qp;
  plan_quantize(&qd, &qp);
  if ((s = run_quantize(&qd, qp, static_cast<int *>(qd.workspace), sms, st)) != NVFP4_OK) return s;
  plan_quantize(&qx, &qp);
  if ((s = run_quantize(&qx, qp, static_cast<int *>(qx.workspace), sms, st)) != NVFP4_OK) return s;
  const nvfp4_gemm_args g = wgrad_gemm(a, pl);
  GemmPlan gp;
  plan_gemm(&g, &gp);
  return run_gemm(&g, gp, sms, st);
}

}  // namespace

namespace nvfp4 {
cudaError_t ensure_dynamic_smem(const void *func, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // one record per (device, function) for the whole process; the lock is held
  // across the attribute call so that two threads never race a smaller value
  // past a larger one
  static std::mutex mu;
  static std::vector<std::pair<const void *, size_t>> done[kMaxDevices];
  std::lock_guard<std::mutex> lk(mu);
  for (auto &f : done[dev])
    if (f.first == func) {
      if (f.second >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
      if (e == cudaSuccess) f.second = bytes;
      return e;
    }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done[dev].emplace_back(func, bytes);
  return e;
}

bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                 uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_pitch_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, const uint64_t (&dims)[3],
                 const uint64_t (&strides_bytes)[2], const uint32_t (&box)[3]) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  const cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
  const cuuint32_t bx[3] = {box[0], box[1], box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, dt, 3, const_cast<void *>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace nvfp4

namespace nvfp4 {
// nvfp4_quantize with the amax scratch supplied by the caller of this function
// (the workspace-free entry point); `words` is the scratch capacity.
nvfp4_status quantize_with_amax_scratch(const nvfp4_quant_args *a, uint32_t *scratch, size_t words,
                                        int *status, cudaStream_t st) {
  nvfp4_status s = validate_quantize(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  QuantPlan pl;
  if (!a->global_scale_in) {
    pl.nparts = amax_parts_for(a->rows);
    if ((size_t)a->batch * (size_t)pl.nparts > words) return NVFP4_ERR_WORKSPACE;
    pl.amax = scratch;
  }
  return run_quantize(a, pl, status, d.sms, st);
}
}  // namespace nvfp4

// =============================================================== C ABI ==
extern "C" {

size_t nvfp4_codes_bytes(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return 0;
  return (size_t)rows * (size_t)cols / 2;
}

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols, int32_t sf_layout) {
  if (rows < 0 || cols < 0) return 0;
  if (sf_layout == NVFP4_SF_SWIZZLED) return sf_swizzled_bytes(rows, cols);
  return (size_t)rows * (size_t)(cols / 16);
}

const char *nvfp4_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

const char *nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case NVFP4_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case NVFP4_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case NVFP4_ERR_CUDA: return "CUDA runtime error";
    case NVFP4_ERR_TIMEOUT: return "an in-kernel wait timed out";
    case NVFP4_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103";
    case NVFP4_ERR_DEVICE_BOUNDS: return "a device-side index check failed";
  }
  return "unknown status";
}

int32_t nvfp4_version(void) { return 0x000100; }

uint64_t nvfp4_set_wait_timeout_ns(uint64_t ns) { return g_timeout_ns.exchange(ns); }

nvfp4_status nvfp4_read_device_status(void *workspace, nvfp4_stream stream) {
  if (!workspace) {
    // the status word of nvfp4_quantize_noalloc on the current device
    int *w = nullptr;
    if (nvfp4_status s = noalloc_status_word(&w); s != NVFP4_OK) return s;
    workspace = w;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaError_t e_ = cudaStreamSynchronize(st); e_ != cudaSuccess) return cuda_status(e_);
  if (cudaError_t e_ = cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost); e_ != cudaSuccess) return cuda_status(e_);
  if (v != 0) {
    if (cudaError_t e_ = cudaMemset(workspace, 0, sizeof(int)); e_ != cudaSuccess) return cuda_status(e_);
  }
  return static_cast<nvfp4_status>(v);
}

size_t nvfp4_quantize_workspace_bytes(const nvfp4_quant_args *a) {
  if (!a) return 0;
  nvfp4_quant_args c = *a;
  c.workspace = nullptr;
  QuantPlan pl;
  plan_quantize(&c, &pl);
  return pl.ws;
}

nvfp4_status nvfp4_quantize(const nvfp4_quant_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_quantize(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  QuantPlan pl;
  plan_quantize(a, &pl);
  if ((s = check_workspace(a->workspace, a->workspace_bytes, pl.ws)) != NVFP4_OK) return s;
  return run_quantize(a, pl, static_cast<int *>(a->workspace), d.sms, reinterpret_cast<cudaStream_t>(stream));
}

size_t nvfp4_gemm_workspace_bytes(const nvfp4_gemm_args *a) {
  if (!a) return 0;
  nvfp4_gemm_args c = *a;
  c.workspace = nullptr;
  GemmPlan pl;
  plan_gemm(&c, &pl);
  return pl.ws;
}

nvfp4_status nvfp4_gemm(const nvfp4_gemm_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_gemm(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  GemmPlan pl;
  plan_gemm(a, &pl);
  if ((s = check_workspace(a->workspace, a->workspace_bytes, pl.ws)) != NVFP4_OK) return s;
  return run_gemm(a, pl, d.sms, reinterpret_cast<cudaStream_t>(stream));
}

size_t nvfp4_grouped_workspace_bytes(const nvfp4_grouped_args *a) {
  if (!a) return 0;
  nvfp4_grouped_args c = *a;
  c.workspace = nullptr;
  GroupedPlan pl;
  plan_grouped(&c, &pl);
  return pl.ws;
}

nvfp4_status nvfp4_grouped_gemm(const nvfp4_grouped_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_grouped(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  GroupedPlan pl;
  plan_grouped(a, &pl);
  if ((s = check_workspace(a->workspace, a->workspace_bytes, pl.ws)) != NVFP4_OK) return s;
  return run_grouped(a, pl, d.sms, reinterpret_cast<cudaStream_t>(stream));
}

size_t nvfp4_lora_workspace_bytes(const nvfp4_lora_args *a) {
  if (!a) return 0;
  nvfp4_lora_args c = *a;
  c.workspace = nullptr;
  LoraPlan pl;
  plan_lora(&c, &pl);
  return pl.ws;
}

nvfp4_status nvfp4_lora_epilogue(const nvfp4_lora_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_lora(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  LoraPlan pl;
  plan_lora(a, &pl);
  if ((s = check_workspace(a->workspace, a->workspace_bytes, pl.ws)) != NVFP4_OK) return s;
  return run_lora(a, pl, d.sms, reinterpret_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_dequantize(const nvfp4_dequant_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_dequant(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  return cuda_status(launch_dequant(static_cast<const uint8_t *>(a->codes), static_cast<const uint8_t *>(a->sf),
                                    a->sf_layout == NVFP4_SF_SWIZZLED, a->global_scale, a->rows, a->cols,
                                    a->transpose, static_cast<__nv_bfloat16 *>(a->out), a->ldo, d.sms,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

size_t nvfp4_dgrad_workspace_bytes(const nvfp4_dgrad_args *a) {
  if (!a) return 0;
  return dgrad_workspace(a);
}

nvfp4_status nvfp4_dgrad(const nvfp4_dgrad_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_dgrad(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  if ((s = check_workspace(a->workspace, a->workspace_bytes, dgrad_workspace(a))) != NVFP4_OK) return s;
  return run_dgrad(a, d.sms, reinterpret_cast<cudaStream_t>(stream));
}

size_t nvfp4_wgrad_workspace_bytes(const nvfp4_wgrad_args *a) {
  if (!a) return 0;
  nvfp4_wgrad_args c = *a;
  c.workspace = nullptr;
  WgradPlan pl;
  plan_wgrad(&c, &pl);
  return pl.ws;
}

nvfp4_status nvfp4_wgrad(const nvfp4_wgrad_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_wgrad(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  WgradPlan pl;
  plan_wgrad(a, &pl);
  if ((s = check_workspace(a->workspace, a->workspace_bytes, pl.ws)) != NVFP4_OK) return s;
  return run_wgrad(a, pl, d.sms, reinterpret_cast<cudaStream_t>(stream));
}

size_t nvfp4_moe_down_workspace_bytes(const nvfp4_moe_down_args *a) {
  if (!a) return 0;
  nvfp4_moe_down_args c = *a;
  c.workspace = nullptr;
  MoeDownPlan pl;
  plan_moe_down(&c, &pl);
  return pl.ws;
}

nvfp4_status nvfp4_moe_down_combine(const nvfp4_moe_down_args *a, nvfp4_stream stream) {
  nvfp4_status s = validate_moe_down(a);
  if (s != NVFP4_OK) return s;
  DevInfo d;
  if ((s = device_info(&d)) != NVFP4_OK) return s;
  MoeDownPlan pl;
  plan_moe_down(a, &pl);
  if ((s = check_workspace(a->workspace, a->workspace_bytes, pl.ws)) != NVFP4_OK) return s;
  return run_moe_down(a, pl, d.sms, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
