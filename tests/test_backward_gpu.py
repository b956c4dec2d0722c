"""nvfp4_dequantize, nvfp4_dgrad and nvfp4_wgrad on the GPU against the oracle.

Dequantization is bit-exact (the oracle's fp32 decode order, then bf16).  The
Dgrad products are checked like the forward GEMM: fp32 out |dX - dX_or| <=
2e-5 S, bf16 out within one bf16 ulp of max(|dX_or|, 2e-5 S), S = sum_n
|dY_nm W_nk| of the operands the product actually uses (the dequantized bf16
weight, or both FP4 operands)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from helpers import assert_bits_equal, assert_gemm_close, dev_bf16, host_bits
from oracle import nvfp4_oracle as o
from synth import f32_to_bf16_bits, make_case

pytestmark = pytest.mark.gpu


def upload_packed(codes, sf_lin, g, layout="swizzled"):
    rows = codes.shape[0]
    sf = o.sf_swizzle(sf_lin) if layout == "swizzled" else sf_lin.reshape(-1)
    return (torch.from_numpy(np.ascontiguousarray(codes)).cuda(),
            torch.from_numpy(np.ascontiguousarray(sf)).cuda(),
            torch.tensor([float(g)], dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("layout", ["swizzled", "linear"])
@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("shape", [(256, 512), (300, 192), (2, 64), (130, 1088)])
def test_dequantize_bit_exact(shape, transpose, layout):
    R, C = shape
    rng = np.random.default_rng(R * 7 + C)
    w = f32_to_bf16_bits((rng.standard_normal((R, C)) * 0.05).astype(np.float32))
    w[0, :16] = 0                                    # a zero block: scale 0
    codes, sf, g = o.quantize(w)
    c, s, gg = upload_packed(codes, sf, g, layout)
    out = nv.nvfp4_dequantize(c, s, gg, R, C, transpose=transpose, sf_layout=layout)
    torch.cuda.synchronize()
    want = o.dequantize_bf16(codes, sf, g)
    assert_bits_equal(host_bits(out), want.T if transpose else want, f"dequant {shape} t={transpose}")


def test_dequantize_matches_device_quantizer_output():
    """Codes and scales from nvfp4_quantize, rebuilt on the device: the same bits as the oracle's."""
    c = make_case("dgrad", M=16, N=384, K=1024)
    q = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
    out = nv.nvfp4_dequantize(q["codes_row"][0], q["sf_row"][0], q["global_scale"], 384, 1024, transpose=True)
    torch.cuda.synchronize()
    codes, sf, g = o.quantize(c["w"])
    assert_bits_equal(host_bits(out), o.dequantize_bf16(codes, sf, g).T, "device-packed dequant")


def dgrad_oracle_bf16(dy_bits, codes, sf, g):
    what = o.bf16_to_f32(o.dequantize_bf16(codes, sf, g)).astype(np.float64)    # [N, K]
    dy = o.bf16_to_f32(dy_bits).astype(np.float64)
    return dy @ what, np.abs(dy) @ np.abs(what)


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (300, 256, 640), (1, 128, 128), (129, 1024, 256),
                                   (2560, 256, 2048)])
def test_dgrad_dequant_bf16(M, N, K, out_dtype):
    c = make_case("dgrad", M=M, N=N, K=K)
    codes, sf, g = o.quantize(c["w"])
    w = upload_packed(codes, sf, g)
    dx = nv.nvfp4_dgrad(dev_bf16(c["dy"]), N, K, w=w, out_dtype=out_dtype)
    y_or, S = dgrad_oracle_bf16(c["dy"], codes, sf, g)
    assert_gemm_close(dx, y_or, S, what=f"dgrad bf16 {M}x{N}x{K}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (300, 256, 640), (129, 1024, 256)])
def test_dgrad_fp4_colpack(M, N, K, out_dtype):
    c = make_case("dgrad", M=M, N=N, K=K)
    col = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="col", sf_layout="swizzled")
    wcol = (col["codes_col"][0], col["sf_col"][0], col["global_scale"])
    dx = nv.nvfp4_dgrad(dev_bf16(c["dy"]), N, K, wcol=wcol, out_dtype=out_dtype)
    dyq = o.quantize(c["dy"])                        # blocks of 16 along N
    wq = o.quantize_colwise(c["w"])                  # W^T, blocks along N, same g
    y_or = o.linear_fp64(dyq, wq)
    S = o.error_scale(dyq, wq)
    assert_gemm_close(dx, y_or, S, what=f"dgrad fp4 {M}x{N}x{K}")


def test_dgrad_full_size_sampled_rows():
    """dY [8192,2048], W [2048,6144] (the prefill linear's backward), both modes, 64 rows."""
    from synth import torch_case
    t = torch_case("dgrad")
    M, N, K = t["M"], t["N"], t["K"]
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], np.random.default_rng(4).choice(M, 60, replace=False)]))
    ridx = torch.from_numpy(rows).cuda()
    wb = host_bits(t["w"])
    dyb = host_bits(t["dy"])[rows]
    q = nv.nvfp4_quantize(t["w"], pack="both", sf_layout="swizzled")
    dx1 = nv.nvfp4_dgrad(t["dy"], N, K, w=(q["codes_row"][0], q["sf_row"][0], q["global_scale"]))
    dx2 = nv.nvfp4_dgrad(t["dy"], N, K, wcol=(q["codes_col"][0], q["sf_col"][0], q["global_scale"]))
    torch.cuda.synchronize()
    codes, sf, g = o.quantize(wb)
    y1, S1 = dgrad_oracle_bf16(dyb, codes, sf, g)
    assert_gemm_close(dx1[ridx], y1, S1, what="dgrad bf16 full")
    gdy = o.global_scale(host_bits(t["dy"]))
    dyq = o.quantize(dyb, gdy)
    wq = o.quantize_colwise(wb, g)
    assert_gemm_close(dx2[ridx], o.linear_fp64(dyq, wq), o.error_scale(dyq, wq), what="dgrad fp4 full")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (96, 208, 640), (544, 128, 48)])
def test_wgrad_fp4(M, N, K, out_dtype):
    """dW = dY^T X with both operands quantized along M (their column packings)."""
    rng = np.random.default_rng(M + N + K)
    dy = f32_to_bf16_bits((rng.standard_normal((M, N)) * 0.01).astype(np.float32))
    x = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    dw = nv.nvfp4_wgrad(dev_bf16(dy), dev_bf16(x), out_dtype=out_dtype)
    a = o.quantize_colwise(dy)       # dY^T [N, M], blocks along M
    b = o.quantize_colwise(x)        # X^T  [K, M]
    assert_gemm_close(dw, o.linear_fp64(a, b), o.error_scale(a, b), what=f"wgrad {M}x{N}x{K}")


def test_wgrad_static_scales():
    rng = np.random.default_rng(31)
    M, N, K = 128, 256, 256
    dy = f32_to_bf16_bits((rng.standard_normal((M, N)) * 0.01).astype(np.float32))
    x = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    gdy, gx = np.float32(0.05 / 2688), np.float32(4.0 / 2688)
    dw = nv.nvfp4_wgrad(dev_bf16(dy), dev_bf16(x), out_dtype=torch.float32,
                        dy_global_scale=torch.tensor([float(gdy)], device="cuda"),
                        x_global_scale=torch.tensor([float(gx)], device="cuda"))
    a = o.quantize_colwise(dy, gdy)
    b = o.quantize_colwise(x, gx)
    assert_gemm_close(dw, o.linear_fp64(a, b), o.error_scale(a, b), what="wgrad static")


def _padded(rows, cols, pad, dtype, fill=7.0):
    full = torch.full((rows, cols + pad), fill, dtype=dtype, device="cuda")
    return full, full[:, :cols]


def _strided_bf16(bits, pad):
    """A device bf16 view of `bits` whose rows are `pad` elements wider (the
    extra columns hold large values the call must not read)."""
    R, C = bits.shape
    big = np.full((R, C + pad), 0x4480, np.uint16)              # bf16 1024.0
    big[:, :C] = bits
    return dev_bf16(big)[:, :C]


@pytest.mark.parametrize("transpose", [False, True])
def test_dequantize_into_padded_rows(transpose):
    R, C = 300, 192
    rng = np.random.default_rng(77)
    w = f32_to_bf16_bits((rng.standard_normal((R, C)) * 0.05).astype(np.float32))
    codes, sf, g = o.quantize(w)
    c, s, gg = upload_packed(codes, sf, g)
    orows, ocols = (C, R) if transpose else (R, C)
    full, out = _padded(orows, ocols, 8, torch.bfloat16)
    nv.nvfp4_dequantize(c, s, gg, R, C, transpose=transpose, out=out)
    torch.cuda.synchronize()
    want = o.dequantize_bf16(codes, sf, g)
    assert_bits_equal(host_bits(out.contiguous()), want.T if transpose else want, "padded dequant")
    assert torch.all(full[:, ocols:] == 7.0), "padding columns written"


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["bf16", "fp4"])
def test_dgrad_strided_dy_padded_dx(mode, out_dtype):
    """dY with rows wider than N (the extra columns must not be read) and dX
    written into rows wider than K (the padding must not be written)."""
    M, N, K = 300, 256, 640
    c = make_case("dgrad", M=M, N=N, K=K)
    dy = _strided_bf16(c["dy"], 16)
    full, out = _padded(M, K, 8, out_dtype)
    if mode == "bf16":
        codes, sf, g = o.quantize(c["w"])
        nv.nvfp4_dgrad(dy, N, K, w=upload_packed(codes, sf, g), out_dtype=out_dtype, out=out)
        y_or, S = dgrad_oracle_bf16(c["dy"], codes, sf, g)
    else:
        col = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="col", sf_layout="swizzled")
        nv.nvfp4_dgrad(dy, N, K, wcol=(col["codes_col"][0], col["sf_col"][0], col["global_scale"]),
                       out_dtype=out_dtype, out=out)
        dyq = o.quantize(c["dy"])
        wq = o.quantize_colwise(c["w"])
        y_or, S = o.linear_fp64(dyq, wq), o.error_scale(dyq, wq)
    torch.cuda.synchronize()
    assert_gemm_close(out, y_or, S, what=f"dgrad {mode} strided")
    assert torch.all(full[:, K:] == 7.0), "padding columns written"


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_wgrad_strided_inputs_padded_dw(out_dtype):
    M, N, K = 256, 208, 640
    rng = np.random.default_rng(91)
    dyb = f32_to_bf16_bits((rng.standard_normal((M, N)) * 0.01).astype(np.float32))
    xb = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    full, out = _padded(N, K, 8, out_dtype)
    nv.nvfp4_wgrad(_strided_bf16(dyb, 24), _strided_bf16(xb, 16), out_dtype=out_dtype, out=out)
    torch.cuda.synchronize()
    a = o.quantize_colwise(dyb)
    b = o.quantize_colwise(xb)
    assert_gemm_close(out, o.linear_fp64(a, b), o.error_scale(a, b), what="wgrad strided")
    assert torch.all(full[:, K:] == 7.0), "padding columns written"
