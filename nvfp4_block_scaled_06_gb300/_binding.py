"""ctypes binding of libnvfp4 (include/nvfp4.h).  Argument marshalling only.

The structures below mirror the C structs field for field.  Every compute step
runs inside the CUDA library; this module only fills argument structs with
device pointers, allocates outputs and workspaces through torch, and raises
on a non-OK status.  If the shared library is missing, ``load()`` raises: there
is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# NVFP4_CHECKED=1 selects the build with device-side index checks
# (python -m nvfp4_block_scaled_06_gb300.build --checked).
CHECKED = os.environ.get("NVFP4_CHECKED", "") not in ("", "0")
LIB_PATH = os.path.join(HERE, "libnvfp4_checked.so" if CHECKED else "libnvfp4.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_ALIGNMENT, ERR_WORKSPACE, ERR_CUDA, \
    ERR_TIMEOUT, ERR_UNSUPPORTED_DEVICE, ERR_DEVICE_BOUNDS = range(9)
SF_LINEAR, SF_SWIZZLED = 0, 1
PACK_ROW, PACK_COL, PACK_BOTH = 1, 2, 3
OUT_BF16, OUT_FP32 = 0, 1

EXPORTS = [
    "nvfp4_quantize", "nvfp4_quantize_workspace_bytes", "nvfp4_gemm",
    "nvfp4_gemm_workspace_bytes", "nvfp4_grouped_gemm", "nvfp4_grouped_workspace_bytes",
    "nvfp4_lora_epilogue", "nvfp4_lora_workspace_bytes", "nvfp4_codes_bytes",
    "nvfp4_sf_bytes", "nvfp4_status_string", "nvfp4_read_device_status",
    "nvfp4_set_wait_timeout_ns", "nvfp4_version", "nvfp4_quantize_noalloc",
    "nvfp4_last_cuda_error", "nvfp4_dequantize", "nvfp4_dgrad", "nvfp4_dgrad_workspace_bytes",
    "nvfp4_wgrad", "nvfp4_wgrad_workspace_bytes", "nvfp4_moe_down_combine",
    "nvfp4_moe_down_workspace_bytes",
]

DGRAD_DEQUANT_BF16, DGRAD_FP4_COLPACK = 0, 1


class QuantArgs(C.Structure):
    _fields_ = [
        ("src", C.c_void_p),
        ("batch", C.c_int64), ("rows", C.c_int64), ("cols", C.c_int64),
        ("ld", C.c_int64), ("batch_stride", C.c_int64),
        ("pack", C.c_int32), ("sf_layout", C.c_int32),
        ("global_scale_in", C.c_void_p), ("global_scale_out", C.c_void_p),
        ("codes_row", C.c_void_p), ("sf_row", C.c_void_p),
        ("codes_col", C.c_void_p), ("sf_col", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
        ("prof_begin", C.c_void_p), ("prof_end", C.c_void_p),
    ]


class GemmArgs(C.Structure):
    _fields_ = [
        ("M", C.c_int64), ("N", C.c_int64), ("K", C.c_int64),
        ("a_codes", C.c_void_p), ("a_sf", C.c_void_p), ("a_global_scale", C.c_void_p),
        ("a_bf16", C.c_void_p), ("lda", C.c_int64),
        ("b_codes", C.c_void_p), ("b_sf", C.c_void_p), ("b_global_scale", C.c_void_p),
        ("out_dtype", C.c_int32),
        ("d", C.c_void_p), ("ldd", C.c_int64),
        ("lora_x", C.c_void_p), ("lora_a", C.c_void_p), ("lora_b", C.c_void_p),
        ("rank", C.c_int32), ("alpha", C.c_float),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
        ("prof_begin", C.c_void_p), ("prof_end", C.c_void_p),
    ]


class GroupedArgs(C.Structure):
    _fields_ = [
        ("num_tokens", C.c_int64), ("top_k", C.c_int64), ("num_experts", C.c_int64),
        ("N", C.c_int64), ("K", C.c_int64),
        ("expert_ids", C.c_void_p), ("x_bf16", C.c_void_p), ("x_global_scale", C.c_void_p),
        ("w_codes", C.c_void_p), ("w_sf", C.c_void_p), ("w_global_scale", C.c_void_p),
        ("lora_a", C.c_void_p), ("lora_b", C.c_void_p),
        ("rank", C.c_int32), ("alpha", C.c_float),
        ("d", C.c_void_p), ("perm_out", C.c_void_p), ("expert_offsets_out", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
        ("prof_begin", C.c_void_p), ("prof_end", C.c_void_p),
        ("x_codes", C.c_void_p), ("x_sf", C.c_void_p),
        ("offsets_in", C.c_void_p), ("perm_in", C.c_void_p),
        ("out_dtype", C.c_int32),
    ]


class LoraArgs(C.Structure):
    _fields_ = [
        ("M", C.c_int64), ("N", C.c_int64), ("K", C.c_int64),
        ("x", C.c_void_p), ("ldx", C.c_int64),
        ("lora_a", C.c_void_p), ("lora_b", C.c_void_p),
        ("rank", C.c_int32), ("alpha", C.c_float),
        ("y_dtype", C.c_int32),
        ("y", C.c_void_p), ("ldy", C.c_int64),
        ("delta_sq_norm_out", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
    ]


class DequantArgs(C.Structure):
    _fields_ = [
        ("codes", C.c_void_p), ("sf", C.c_void_p),
        ("sf_layout", C.c_int32),
        ("global_scale", C.c_void_p),
        ("rows", C.c_int64), ("cols", C.c_int64),
        ("transpose", C.c_int32),
        ("out", C.c_void_p), ("ldo", C.c_int64),
    ]


class DgradArgs(C.Structure):
    _fields_ = [
        ("M", C.c_int64), ("N", C.c_int64), ("K", C.c_int64),
        ("mode", C.c_int32),
        ("dy", C.c_void_p), ("lddy", C.c_int64),
        ("w_codes", C.c_void_p), ("w_sf", C.c_void_p),
        ("wcol_codes", C.c_void_p), ("wcol_sf", C.c_void_p),
        ("w_global_scale", C.c_void_p), ("dy_global_scale", C.c_void_p),
        ("out_dtype", C.c_int32),
        ("dx", C.c_void_p), ("lddx", C.c_int64),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
        ("prof_begin", C.c_void_p), ("prof_end", C.c_void_p),
    ]


class WgradArgs(C.Structure):
    _fields_ = [
        ("M", C.c_int64), ("N", C.c_int64), ("K", C.c_int64),
        ("dy", C.c_void_p), ("lddy", C.c_int64),
        ("x", C.c_void_p), ("ldx", C.c_int64),
        ("dy_global_scale", C.c_void_p), ("x_global_scale", C.c_void_p),
        ("out_dtype", C.c_int32),
        ("dw", C.c_void_p), ("lddw", C.c_int64),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
        ("prof_begin", C.c_void_p), ("prof_end", C.c_void_p),
    ]


class MoeDownArgs(C.Structure):
    _fields_ = [
        ("num_tokens", C.c_int64), ("top_k", C.c_int64), ("num_experts", C.c_int64),
        ("N", C.c_int64), ("K", C.c_int64),
        ("h", C.c_void_p), ("perm", C.c_void_p), ("expert_offsets", C.c_void_p),
        ("route_weights", C.c_void_p), ("h_global_scale", C.c_void_p),
        ("w_codes", C.c_void_p), ("w_sf", C.c_void_p), ("w_global_scale", C.c_void_p),
        ("lora_a", C.c_void_p), ("lora_b", C.c_void_p),
        ("rank", C.c_int32), ("alpha", C.c_float),
        ("y", C.c_void_p),
        ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
        ("prof_begin", C.c_void_p), ("prof_end", C.c_void_p),
    ]


_lib = None


def load(path: str | None = None):
    """Load libnvfp4.so (raises if it is missing or lacks an export)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"{os.path.basename(p)} not found at {p}: build it first (python -m nvfp4_block_scaled_06_gb300.build"
            f"{' --checked' if CHECKED else ''})")
    lib = C.CDLL(p)
    for name in EXPORTS:
        if not hasattr(lib, name):
            raise RuntimeError(f"libnvfp4.so lacks export {name}")
    vp = C.c_void_p
    for fn, wsq, st in [("nvfp4_quantize", "nvfp4_quantize_workspace_bytes", QuantArgs),
                        ("nvfp4_gemm", "nvfp4_gemm_workspace_bytes", GemmArgs),
                        ("nvfp4_grouped_gemm", "nvfp4_grouped_workspace_bytes", GroupedArgs),
                        ("nvfp4_lora_epilogue", "nvfp4_lora_workspace_bytes", LoraArgs),
                        ("nvfp4_dgrad", "nvfp4_dgrad_workspace_bytes", DgradArgs),
                        ("nvfp4_wgrad", "nvfp4_wgrad_workspace_bytes", WgradArgs),
                        ("nvfp4_moe_down_combine", "nvfp4_moe_down_workspace_bytes", MoeDownArgs)]:
        f = getattr(lib, fn)
        f.argtypes = [C.POINTER(st), vp]
        f.restype = C.c_int
        w = getattr(lib, wsq)
        w.argtypes = [C.POINTER(st)]
        w.restype = C.c_size_t
    lib.nvfp4_dequantize.argtypes = [C.POINTER(DequantArgs), vp]
    lib.nvfp4_dequantize.restype = C.c_int
    lib.nvfp4_quantize_noalloc.argtypes = [C.POINTER(QuantArgs), vp]
    lib.nvfp4_quantize_noalloc.restype = C.c_int
    lib.nvfp4_codes_bytes.argtypes = [C.c_int64, C.c_int64]
    lib.nvfp4_codes_bytes.restype = C.c_size_t
    lib.nvfp4_sf_bytes.argtypes = [C.c_int64, C.c_int64, C.c_int32]
    lib.nvfp4_sf_bytes.restype = C.c_size_t
    lib.nvfp4_status_string.argtypes = [C.c_int]
    lib.nvfp4_status_string.restype = C.c_char_p
    lib.nvfp4_last_cuda_error.argtypes = []
    lib.nvfp4_last_cuda_error.restype = C.c_char_p
    lib.nvfp4_read_device_status.argtypes = [vp, vp]
    lib.nvfp4_read_device_status.restype = C.c_int
    lib.nvfp4_set_wait_timeout_ns.argtypes = [C.c_uint64]
    lib.nvfp4_set_wait_timeout_ns.restype = C.c_uint64
    lib.nvfp4_version.argtypes = []
    lib.nvfp4_version.restype = C.c_int32
    if path is None:
        _lib = lib
    return lib


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        lib = load()
        msg = f"{where}: {lib.nvfp4_status_string(status).decode()} (status {status})"
        if status == ERR_CUDA:
            msg += f": {lib.nvfp4_last_cuda_error().decode()}"
        super().__init__(msg)
        self.status = status


def check(status: int, where: str):
    if status != OK:
        raise NVFP4Error(status, where)
