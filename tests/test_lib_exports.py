"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/nvfp4.h declares, and rejects bad arguments on the host before any
device work (status codes only; no compute call is made here)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clib():
    from nvfp4_block_scaled_06_gb300 import build as b
    b.build()
    from nvfp4_block_scaled_06_gb300 import _binding
    return _binding.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(clib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(clib, n), n
    from nvfp4_block_scaled_06_gb300._binding import EXPORTS
    assert sorted(EXPORTS) == names


def test_size_queries(clib):
    assert clib.nvfp4_codes_bytes(2048, 6144) == 2048 * 3072
    assert clib.nvfp4_sf_bytes(2048, 6144, 0) == 2048 * 384
    # swizzled: rows padded to 128, scale columns padded to 4
    assert clib.nvfp4_sf_bytes(37, 80, 1) == 128 * 8
    assert clib.nvfp4_status_string(4).decode().startswith("workspace")
    assert clib.nvfp4_version() == 0x000100
    assert clib.nvfp4_last_cuda_error().decode() == "no error"


def test_host_validation_without_device(clib):
    from nvfp4_block_scaled_06_gb300._binding import (ERR_ALIGNMENT, ERR_INVALID_ARG,
                                                       ERR_UNSUPPORTED_SHAPE, GemmArgs,
                                                       GroupedArgs, LoraArgs, QuantArgs)
    nullq = C.cast(None, C.POINTER(QuantArgs))
    assert clib.nvfp4_quantize(nullq, None) == ERR_INVALID_ARG
    q = QuantArgs(src=4096, batch=1, rows=16, cols=24, ld=24, pack=1, sf_layout=1,
                  global_scale_out=4096, codes_row=4096, sf_row=4096)
    assert clib.nvfp4_quantize(C.byref(q), None) == ERR_UNSUPPORTED_SHAPE      # cols % 16
    q.cols, q.ld = 32, 32
    q.src = 4104                                                              # not 16-aligned
    assert clib.nvfp4_quantize(C.byref(q), None) == ERR_ALIGNMENT
    g = GemmArgs(M=8, N=8, K=48, a_codes=4096, a_sf=4096, a_global_scale=4096, b_codes=4096,
                 b_sf=4096, b_global_scale=4096, d=4096, ldd=8)
    assert clib.nvfp4_gemm(C.byref(g), None) == ERR_UNSUPPORTED_SHAPE          # K % 32
    g.K = 64
    g.lora_a, g.lora_b, g.lora_x, g.lda, g.rank = 4096, 4096, 4096, 64, 48
    assert clib.nvfp4_gemm(C.byref(g), None) == ERR_UNSUPPORTED_SHAPE          # rank % 32
    gr = GroupedArgs(num_tokens=4, top_k=2, num_experts=8, N=200, K=64, expert_ids=4096,
                     x_bf16=4096, w_codes=4096, w_sf=4096, w_global_scale=4096, d=4096,
                     perm_out=4096)
    assert clib.nvfp4_grouped_gemm(C.byref(gr), None) == ERR_UNSUPPORTED_SHAPE  # N % 256
    lo = LoraArgs(M=4, N=8, K=64, x=4096, ldx=64, lora_a=4096, lora_b=4096, rank=64,
                  y=4096, ldy=8, y_dtype=3)
    assert clib.nvfp4_lora_epilogue(C.byref(lo), None) == ERR_INVALID_ARG      # bad dtype


def test_workspace_queries_need_no_device(clib):
    from nvfp4_block_scaled_06_gb300._binding import GemmArgs, GroupedArgs
    g = GemmArgs(M=8192, N=2048, K=6144, a_bf16=4096, lda=6144, b_codes=4096, b_sf=4096,
                 b_global_scale=4096, d=4096, ldd=2048, lora_a=4096, lora_b=4096, rank=64,
                 alpha=128.0)
    ws = clib.nvfp4_gemm_workspace_bytes(C.byref(g))
    # X codes + swizzled scales + T' (bf16 [M, r]) + small scalars
    assert ws >= 8192 * 3072 + 8192 * 384 + 8192 * 64 * 2
    gr = GroupedArgs(num_tokens=4096, top_k=8, num_experts=256, N=2048, K=6144)
    assert clib.nvfp4_grouped_workspace_bytes(C.byref(gr)) > 32768 * 3072


def test_product_package_does_not_import_oracle():
    pkg = os.path.join(ROOT, "nvfp4_block_scaled_06_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.replace("the oracle", ""), f


def test_grouped_input_forms_validation(clib):
    """The grouped call's routing and activation forms are checked on the host:
    exactly one routing form (expert ids + perm_out, or offsets + perm), packed
    activations with their scales and global scale, bf16 rows with a LoRA, a
    known output dtype.  Valid forms pass validation (and then fail for the
    missing device, or the missing workspace, never with INVALID_ARG)."""
    from nvfp4_block_scaled_06_gb300._binding import ERR_INVALID_ARG, GroupedArgs, OUT_FP32

    def grouped(**kw):
        base = dict(num_tokens=4, top_k=2, num_experts=8, N=256, K=64, w_codes=4096, w_sf=4096,
                    w_global_scale=4096, d=4096)
        base.update(kw)
        return clib.nvfp4_grouped_gemm(C.byref(GroupedArgs(**base)), None)

    ids = dict(expert_ids=4096, perm_out=4096)
    given = dict(offsets_in=4096, perm_in=4096)
    bf16 = dict(x_bf16=4096)
    packed = dict(x_codes=4096, x_sf=4096, x_global_scale=4096)
    assert grouped(**bf16) == ERR_INVALID_ARG                                   # no routing
    assert grouped(**ids, **given, **bf16) == ERR_INVALID_ARG                   # both routings
    assert grouped(expert_ids=4096, **bf16) == ERR_INVALID_ARG                  # ids without perm_out
    assert grouped(**ids, offsets_in=4096, **bf16) == ERR_INVALID_ARG           # ids + half of given
    assert grouped(offsets_in=4096, **bf16) == ERR_INVALID_ARG                  # offsets without perm
    assert grouped(**ids) == ERR_INVALID_ARG                                    # no activations
    assert grouped(**ids, x_codes=4096, x_global_scale=4096) == ERR_INVALID_ARG  # codes without scales
    assert grouped(**ids, x_codes=4096, x_sf=4096) == ERR_INVALID_ARG           # packed without g_x
    assert grouped(**ids, **packed, lora_a=4096, lora_b=4096, rank=64) == ERR_INVALID_ARG  # LoRA needs bf16 X
    assert grouped(**ids, **bf16, out_dtype=7) == ERR_INVALID_ARG                # unknown output dtype
    for form in (dict(**ids, **bf16), dict(**given, **packed), dict(**ids, **packed, x_bf16=4096,
                 lora_a=4096, lora_b=4096, rank=64), dict(**given, **bf16, out_dtype=OUT_FP32)):
        assert grouped(**form) != ERR_INVALID_ARG, form


def test_empty_operands_rejected_before_any_launch(clib):
    """An empty operand (a zero size) is NVFP4_ERR_INVALID_ARG on every entry
    point, decided on the host before anything is launched or written; the
    same arguments with the size restored pass that check (they then fail for
    the missing workspace or device, never with INVALID_ARG)."""
    from nvfp4_block_scaled_06_gb300._binding import (ERR_INVALID_ARG, DequantArgs, DgradArgs, GemmArgs,
                                                       GroupedArgs, LoraArgs, MoeDownArgs, QuantArgs, WgradArgs)
    P = 4096                                       # a 16-byte aligned stand-in pointer (never dereferenced)
    cases = [
        (clib.nvfp4_quantize, QuantArgs, dict(src=P, batch=1, rows=32, cols=64, ld=64, pack=1, sf_layout=1,
                                              global_scale_out=P, codes_row=P, sf_row=P),
         ("batch", "rows", "cols")),
        (clib.nvfp4_gemm, GemmArgs, dict(M=8, N=8, K=64, a_codes=P, a_sf=P, a_global_scale=P, b_codes=P,
                                         b_sf=P, b_global_scale=P, d=P, ldd=8),
         ("M", "N", "K")),
        (clib.nvfp4_grouped_gemm, GroupedArgs, dict(num_tokens=4, top_k=2, num_experts=8, N=256, K=64,
                                                    expert_ids=P, x_bf16=P, w_codes=P, w_sf=P,
                                                    w_global_scale=P, d=P, perm_out=P),
         ("num_tokens", "top_k", "num_experts", "N", "K")),
        (clib.nvfp4_lora_epilogue, LoraArgs, dict(M=4, N=8, K=64, x=P, ldx=64, lora_a=P, lora_b=P, rank=64,
                                                  alpha=128.0, y_dtype=0, y=P, ldy=8),
         ("M", "N", "K")),
        (clib.nvfp4_dequantize, DequantArgs, dict(codes=P, sf=P, sf_layout=1, global_scale=P, rows=32, cols=64,
                                                  out=P, ldo=64),
         ("rows", "cols")),
        (clib.nvfp4_dgrad, DgradArgs, dict(M=8, N=64, K=64, mode=0, dy=P, lddy=64, w_codes=P, w_sf=P,
                                           w_global_scale=P, dx=P, lddx=64),
         ("M", "N", "K")),
        (clib.nvfp4_wgrad, WgradArgs, dict(M=32, N=16, K=16, dy=P, lddy=16, x=P, ldx=16, dw=P, lddw=16),
         ("M", "N", "K")),
        (clib.nvfp4_moe_down_combine, MoeDownArgs, dict(num_tokens=4, top_k=2, num_experts=8, N=256, K=64,
                                                        h=P, perm=P, expert_offsets=P, route_weights=P,
                                                        w_codes=P, w_sf=P, w_global_scale=P, y=P),
         ("num_tokens", "top_k", "num_experts", "N", "K")),
    ]
    for fn, cls, base, sizes in cases:
        assert fn(C.byref(cls(**base)), None) != ERR_INVALID_ARG, (fn.__name__, "baseline")
        for name in sizes:
            args = cls(**dict(base, **{name: 0}))
            assert fn(C.byref(args), None) == ERR_INVALID_ARG, (fn.__name__, name)


def test_size_limits_on_the_host(clib):
    """The largest sizes each entry point takes (indices stay within the
    kernels' 32-bit fields) pass the host checks; one step past them is
    NVFP4_ERR_UNSUPPORTED_SHAPE, decided before any launch."""
    from nvfp4_block_scaled_06_gb300._binding import (ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, GemmArgs,
                                                       GroupedArgs, QuantArgs)
    P = 4096
    bad = (ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE)

    def gemm(**kw):
        base = dict(M=8, N=8, K=64, a_codes=P, a_sf=P, a_global_scale=P, b_codes=P, b_sf=P,
                    b_global_scale=P, d=P, ldd=8)
        base.update(kw)
        base["ldd"] = max(base["ldd"], base["N"] + (-base["N"]) % 8)
        return clib.nvfp4_gemm(C.byref(GemmArgs(**base)), None)

    top = (1 << 31) - 256
    assert gemm(M=top) not in bad and gemm(M=top + 1) == ERR_UNSUPPORTED_SHAPE
    assert gemm(N=top) not in bad and gemm(N=top + 8) == ERR_UNSUPPORTED_SHAPE
    assert gemm(K=1 << 24) not in bad and gemm(K=(1 << 24) + 32) == ERR_UNSUPPORTED_SHAPE

    def quant(**kw):
        base = dict(src=P, batch=1, rows=32, cols=64, ld=64, pack=1, sf_layout=1, global_scale_out=P,
                    codes_row=P, sf_row=P, codes_col=P, sf_col=P)
        base.update(kw)
        base["ld"] = max(base["ld"], base["cols"])
        return clib.nvfp4_quantize(C.byref(QuantArgs(**base)), None)

    assert quant(rows=1 << 31) not in bad and quant(rows=(1 << 31) + 16) == ERR_UNSUPPORTED_SHAPE
    # the column packing indexes rows and columns in 32 bits
    assert quant(pack=3, rows=(1 << 30) - 16) not in bad and quant(pack=3, rows=1 << 30) == ERR_UNSUPPORTED_SHAPE

    def grouped(**kw):
        base = dict(num_tokens=4, top_k=2, num_experts=8, N=256, K=64, expert_ids=P, x_bf16=P, w_codes=P,
                    w_sf=P, w_global_scale=P, d=P, perm_out=P)
        base.update(kw)
        return clib.nvfp4_grouped_gemm(C.byref(GroupedArgs(**base)), None)

    assert grouped(num_experts=1024) not in bad and grouped(num_experts=1025) == ERR_UNSUPPORTED_SHAPE
    assert grouped(top_k=8, num_experts=8) not in bad and grouped(top_k=9, num_experts=8) == ERR_UNSUPPORTED_SHAPE
    assert grouped(num_tokens=1 << 27, top_k=8) not in bad
    assert grouped(num_tokens=(1 << 27) + 1, top_k=8) == ERR_UNSUPPORTED_SHAPE
