"""nvfp4_gemm / nvfp4_lora_epilogue on the GPU against the oracle.

Tolerances (fp64 oracle Y_or, S = sum_k |x_hat w_hat| per output):
  fp32 out: |Y - Y_or| <= 2e-5 S;  bf16 out: |Y - bf16(Y_or)| <= ulp(max(|Y_or|, 2e-5 S));
  with the LoRA branch both add 2^-8 (alpha/r) sum_j |T_j||B_nj| (bf16 rounding of
  the scaled T before the tensor-core step)."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from helpers import (assert_bits_equal, assert_gemm_close, dev_bf16, host_bits,
                     lora_bf16_term, u8)
from oracle import nvfp4_oracle as o
from synth import f32_to_bf16_bits, make_case

pytestmark = pytest.mark.gpu


def quant_dev(bits, static=None):
    gs = None if static is None else torch.tensor([static], dtype=torch.float32, device="cuda")
    out = nv.nvfp4_quantize(dev_bf16(bits), pack="row", sf_layout="swizzled", global_scale=gs)
    return out["codes_row"], out["sf_row"], out["global_scale"]


def oracle_linear(x_bits, w_bits, lora=None, xg=None):
    xq = o.quantize(x_bits, xg)
    wq = o.quantize(w_bits)
    y = o.linear_fp64(xq, wq, x_bits, lora)
    s = o.error_scale(xq, wq)
    term = None if lora is None else lora_bf16_term(x_bits, *lora)
    return y, s, term


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_tiny_config_packed_operands(out_dtype):
    c = make_case("tiny")                          # X[32,512] with outliers, W[256,512]
    xc, xs, xg = quant_dev(c["x"])
    wc, ws, wg = quant_dev(c["w"])
    y = nv.nvfp4_gemm(wc, ws, wg, 256, 512, a_codes=xc, a_sf=xs, a_global_scale=xg,
                      out_dtype=out_dtype)
    y_or, S, _ = oracle_linear(c["x"], c["w"])
    assert_gemm_close(y, y_or, S, what="tiny")


@pytest.mark.parametrize("M,N,K", [(300, 320, 544), (128, 256, 256), (1, 128, 32),
                                   (513, 1024, 2048), (200, 640, 1056)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_ragged_gemm(M, N, K, out_dtype):
    rng = np.random.default_rng(M + N + K)
    xb = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    wb = f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    xc, xs, xg = quant_dev(xb)
    wc, ws, wg = quant_dev(wb)
    y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_codes=xc, a_sf=xs, a_global_scale=xg,
                      out_dtype=out_dtype)
    y_or, S, _ = oracle_linear(xb, wb)
    assert_gemm_close(y, y_or, S, what=f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(260, 333, 512), (512, 96, 256), (384, 1030, 768)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_pair_gemm_ragged_columns_and_padded_output(M, N, K, out_dtype):
    """The CTA-pair GEMM (M >= 256) with N not a multiple of the 32-column
    store boxes, written into an output whose rows are wider than N: every
    element of the product within tolerance, the padding columns untouched."""
    rng = np.random.default_rng(M * 7 + N)
    xb = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    wb = f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    xc, xs, xg = quant_dev(xb)
    wc, ws, wg = quant_dev(wb)
    pad = (8 - N % 8) % 8 + 8                      # row pitch a multiple of 8 elements
    full = torch.full((M, N + pad), 7.0, dtype=out_dtype, device="cuda")
    out = full[:, :N]
    y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_codes=xc, a_sf=xs, a_global_scale=xg, out_dtype=out_dtype, out=out)
    torch.cuda.synchronize()
    y_or, S, _ = oracle_linear(xb, wb)
    assert_gemm_close(y, y_or, S, what=f"pair gemm {M}x{N}x{K}")
    assert torch.all(full[:, N:] == 7.0), "padding columns written"


@pytest.mark.parametrize("M,N,K,rank", [(2560, 2048, 512, 0), (4864, 1536, 256, 64), (5120, 968, 512, 32),
                                         (1024, 1792, 512, 64), (2304, 864, 256, 0)])
def test_pair_gemm_half_width_last_wave(M, N, K, rank):
    """The CTA-pair schedule whose last wave of 256 x 256 tiles fills at most
    half of the pairs deals those tiles as 256 x 128 halves (with 76 resident
    pairs: 80 tiles leave 4, 114 leave 38; 32 tiles all run as 64 halves; a
    last n-tile of 200 columns splits into 128 + 72, one of 96 columns keeps
    whole tiles): every element of Y within tolerance, with and without the
    LoRA steps, whatever the number of resident pairs."""
    rng = np.random.default_rng(M + 3 * N + K)
    xb = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    wb = f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    wc, ws, wg = quant_dev(wb)
    if rank:
        la = f32_to_bf16_bits((rng.standard_normal((rank, K)) * 0.02).astype(np.float32))
        lb = f32_to_bf16_bits((rng.standard_normal((N, rank)) * 0.02).astype(np.float32))
        lora = dict(a=dev_bf16(la), b=dev_bf16(lb), alpha=128.0)
        y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(xb), lora=lora)
        y_or, S, term = oracle_linear(xb, wb, (la, lb, 128.0))
    else:
        xc, xs, xg = quant_dev(xb)
        y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_codes=xc, a_sf=xs, a_global_scale=xg)
        y_or, S, term = oracle_linear(xb, wb)
    torch.cuda.synchronize()
    assert_gemm_close(y, y_or, S, term, what=f"half-width last wave {M}x{N}x{K} r{rank}")


@pytest.mark.parametrize("M,N,K,static", [(1, 333, 2048, True), (3, 1030, 20480, True), (8, 333, 512, False),
                                          (64, 1030, 4096, False), (32, 333, 16384, True)])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_padded_output_rows_every_path(M, N, K, static, out_dtype):
    """Outputs with rows wider than N on the other GEMM paths (CUDA-core GEMV
    with one or several chunk passes, the 1-SM tcgen05 GEMM with and without
    split K): the product within tolerance, the padding columns untouched."""
    c = make_case("decode_q_b_proj", M=M, N=N, K=K)
    wc, ws, wg = quant_dev(c["w"])
    pad = (8 - N % 8) % 8 + 8
    full = torch.full((M, N + pad), 7.0, dtype=out_dtype, device="cuda")
    if static:
        sx = 16.0 / 2688.0
        gx = torch.tensor([sx], dtype=torch.float32, device="cuda")
        nv.nvfp4_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(c["x"]), a_global_scale=gx, out_dtype=out_dtype,
                      out=full[:, :N])
        y_or, S, _ = oracle_linear(c["x"], c["w"], xg=np.float32(sx))
    else:
        xc, xs, xg = quant_dev(c["x"])
        nv.nvfp4_gemm(wc, ws, wg, N, K, a_codes=xc, a_sf=xs, a_global_scale=xg, out_dtype=out_dtype,
                      out=full[:, :N])
        y_or, S, _ = oracle_linear(c["x"], c["w"])
    torch.cuda.synchronize()
    assert_gemm_close(full[:, :N], y_or, S, what=f"padded {M}x{N}x{K}")
    assert torch.all(full[:, N:] == 7.0), "padding columns written"


def test_bf16_input_dynamic_matches_packed_path():
    c = make_case("prefill", M=384, N=512, K=1024)
    wc, ws, wg = quant_dev(c["w"])
    x = dev_bf16(c["x"])
    y1 = nv.nvfp4_gemm(wc, ws, wg, 512, 1024, a_bf16=x)
    xc, xs, xg = quant_dev(c["x"])
    y2 = nv.nvfp4_gemm(wc, ws, wg, 512, 1024, a_codes=xc, a_sf=xs, a_global_scale=xg)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("rank", [64, 32, 128])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_prefill_lora_small(rank, out_dtype):
    M, N, K = 320, 512, 1024
    c = make_case("prefill", M=M, N=N, K=K, rank=rank)
    wc, ws, wg = quant_dev(c["w"])
    lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=128.0)
    y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(c["x"]), lora=lora, out_dtype=out_dtype)
    y_or, S, term = oracle_linear(c["x"], c["w"], (c["lora_a"], c["lora_b"], 128.0))
    assert_gemm_close(y, y_or, S, term, what=f"lora r{rank}")


@pytest.mark.parametrize("M", [320, 96])
def test_prefill_lora_static_input_scale(M):
    """The prefill linear with a static input scale (no maximum pass: X is
    packed first and the LoRA-down pass reads it on its own) on the CTA-pair
    path (M = 320) and the 1-SM path (M = 96)."""
    N, K, r = 512, 1024, 64
    c = make_case("prefill", M=M, N=N, K=K, rank=r)
    wc, ws, wg = quant_dev(c["w"])
    sx = np.float32(16.0 / 2688.0)
    gx = torch.tensor([float(sx)], dtype=torch.float32, device="cuda")
    lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=128.0)
    y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(c["x"]), a_global_scale=gx, lora=lora)
    y_or, S, term = oracle_linear(c["x"], c["w"], (c["lora_a"], c["lora_b"], 128.0), xg=sx)
    assert_gemm_close(y, y_or, S, term, what=f"static-scale lora M{M}")


def test_prefill_full_size_sampled_rows():
    """X[8192,6144], W[2048,6144], LoRA r64 alpha 128, bf16 out: 96 sampled rows."""
    c = make_case("prefill")
    wc, ws, wg = quant_dev(c["w"])
    lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=128.0)
    y = nv.nvfp4_gemm(wc, ws, wg, 2048, 6144, a_bf16=dev_bf16(c["x"]), lora=lora)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, 127, 128, 8191],
                                     np.random.default_rng(1).choice(8192, 92, replace=False)]))
    gx = o.global_scale(c["x"])
    xq = o.quantize(c["x"][rows], gx)
    wq = o.quantize(c["w"])
    lo = (c["lora_a"], c["lora_b"], 128.0)
    y_or = o.linear_fp64(xq, wq, c["x"][rows], lo)
    S = o.error_scale(xq, wq)
    term = lora_bf16_term(c["x"][rows], *lo)
    assert_gemm_close(y[torch.from_numpy(rows).cuda()], y_or, S, term, what="prefill full")


@pytest.mark.parametrize("M,K", [(1, 2048), (2, 2048), (4, 2048), (8, 2048), (32, 2048),
                                 (1, 3072), (3, 4096), (1, 1088)])
def test_decode_static_scale(M, K):
    """Decode: X quantized per call with a static input_scale (GEMV for M <= 4;
    rows longer than 2048 are split into chunks summed in order)."""
    N = 1024
    c = make_case("decode_q_b_proj", M=M, N=N, K=K)
    static = 16.0 / 2688.0
    wc, ws, wg = quant_dev(c["w"])
    gx = torch.tensor([static], dtype=torch.float32, device="cuda")
    for od in (torch.bfloat16, torch.float32):
        y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(c["x"]), a_global_scale=gx,
                          out_dtype=od)
        y_or, S, _ = oracle_linear(c["x"], c["w"], xg=np.float32(static))
        assert_gemm_close(y, y_or, S, what=f"decode M{M}")


@pytest.mark.parametrize("M,N,K", [(1, 520, 6144), (2, 520, 10240), (4, 520, 16384), (3, 776, 2112),
                                   (1, 264, 20480), (2, 264, 18432)])
def test_decode_chunked_rows(M, N, K):
    """Decode GEMV with rows of several 2048-element chunks: 3, 5, 8 and 2
    chunks are summed inside one CTA (6, 5, 8 and 8 busy warps, ragged last
    unit), 10 and 9 chunks through fp32 chunk sums and the ordered second pass."""
    c = make_case("decode_q_b_proj", M=M, N=N, K=K)
    static = 16.0 / 2688.0
    wc, ws, wg = quant_dev(c["w"])
    gx = torch.tensor([static], dtype=torch.float32, device="cuda")
    y_or, S, _ = oracle_linear(c["x"], c["w"], xg=np.float32(static))
    for od in (torch.bfloat16, torch.float32):
        y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(c["x"]), a_global_scale=gx,
                          out_dtype=od)
        assert_gemm_close(y, y_or, S, what=f"decode M{M} N{N} K{K}")


@pytest.mark.parametrize("M,N,K,static", [(8, 1024, 2048, True), (8, 768, 16384, True), (40, 512, 1024, False),
                                          (300, 512, 512, False), (8, 200, 3072, True), (24, 968, 2560, False),
                                          (2, 520, 4096, False)])
def test_in_call_x_padding_rows_ignored(M, N, K, static):
    """X quantized in the call is packed into the workspace with its rows
    padded to 128, and the GEMM's tiles span the padding: whatever those
    rows' codes hold (the workspace is filled with 0xFF, code -6 in every
    nibble, before each call), their zero block scales keep them out of every
    stored row of Y.  M <= 32 on the operand-swapped kernel (K ranges summed
    in clusters of 2 and 3, ragged N, or by the split-K pass for 16 ranges),
    M = 40 on the 1-SM kernel and a ragged last row tile on the CTA-pair
    kernel."""
    c = make_case("decode_q_b_proj", M=M, N=N, K=K)
    wc, ws, wg = quant_dev(c["w"])
    sx = np.float32(16.0 / 2688.0)
    gx = torch.tensor([float(sx)], dtype=torch.float32, device="cuda") if static else None
    call, y = nv.prepare_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(c["x"]), a_global_scale=gx)
    for _ in range(2):
        call.workspace[256:].fill_(0xFF)
        call()
        torch.cuda.synchronize()
        y_or, S, _ = oracle_linear(c["x"], c["w"], xg=sx if static else None)
        assert_gemm_close(y, y_or, S, what=f"padded-row X M{M} N{N} K{K}")


@pytest.mark.parametrize("name", ["decode_q_b_proj", "decode_o_proj"])
def test_decode_full_weights_sampled(name):
    """The decode projections at their real shapes and M = 1, 8, 32: the GEMV
    for M = 1, the tcgen05 GEMM with X quantized in the call for M = 8 and 32
    (for o_proj, K = 16384, with the K ranges summed by the split-K pass)."""
    c = make_case(name, M=32)
    N, K = c["N"], c["K"]
    static = np.float32(16.0 / 2688.0)
    wc, ws, wg = quant_dev(c["w"])
    gx = torch.tensor([float(static)], dtype=torch.float32, device="cuda")
    cols = np.unique(np.concatenate([[0, 127, 128, 255, 256, N - 1],
                                     np.random.default_rng(2).choice(N, 250, replace=False)]))
    # the sampled rows of W, quantized with the whole tensor's global scale
    wq = o.quantize(c["w"][cols], o.global_scale(c["w"]))
    for M in (1, 8, 32):
        x = np.ascontiguousarray(c["x"][:M])
        for od in (torch.float32, torch.bfloat16):
            y = nv.nvfp4_gemm(wc, ws, wg, N, K, a_bf16=dev_bf16(x), a_global_scale=gx,
                              out_dtype=od)
            torch.cuda.synchronize()
            xq = o.quantize(x, static)
            y_or = o.linear_fp64(xq, wq)
            S = o.error_scale(xq, wq)
            assert_gemm_close(y[:, torch.from_numpy(cols).cuda()], y_or, S, what=f"{name} M{M} {od}")


@pytest.mark.parametrize("ydtype", [torch.bfloat16, torch.float32])
def test_lora_epilogue_in_place_and_norm(ydtype):
    M, N, K, r = 300, 384, 512, 64
    c = make_case("prefill", M=M, N=N, K=K, rank=r)
    rng = np.random.default_rng(9)
    y0 = rng.standard_normal((M, N)).astype(np.float32)
    y = torch.from_numpy(y0).to("cuda", ydtype)
    ybase = y.double().cpu().numpy()
    norm = nv.nvfp4_lora_epilogue(y, dev_bf16(c["x"]), dev_bf16(c["lora_a"]),
                                  dev_bf16(c["lora_b"]), 128.0, want_norm=True)
    torch.cuda.synchronize()
    d, _ = o.lora_delta_fp64(c["x"], c["lora_a"], c["lora_b"], 128.0)
    term = lora_bf16_term(c["x"], c["lora_a"], c["lora_b"], 128.0)
    got = y.double().cpu().numpy()
    tol = term + 2e-5 * np.abs(d) + 1e-30
    if ydtype == torch.bfloat16:
        tol = tol + o.bf16_ulp(np.abs(ybase + d) + 1e-30)
    assert np.all(np.abs(got - (ybase + d)) <= tol)
    want = float(np.sum(d * d))
    assert abs(float(norm) - want) <= 2e-2 * want


@pytest.mark.parametrize("ydtype", [torch.bfloat16, torch.float32])
def test_lora_epilogue_strided_x_padded_y(ydtype):
    """The standalone LoRA epilogue with X rows wider than K (extra elements
    large: a read of them would change T) and Y rows wider than N (the padding
    must stay as it was)."""
    M, N, K, r = 260, 333, 512, 32
    c = make_case("prefill", M=M, N=N, K=K, rank=r)
    big = np.full((M, K + 16), 0x4480, np.uint16)
    big[:, :K] = c["x"]
    x = dev_bf16(big)[:, :K]
    rng = np.random.default_rng(19)
    pad = (8 - N % 8) % 8 + 8
    full = torch.full((M, N + pad), 7.0, dtype=ydtype, device="cuda")
    full[:, :N] = torch.from_numpy(rng.standard_normal((M, N)).astype(np.float32)).to("cuda", ydtype)
    y = full[:, :N]
    ybase = y.double().cpu().numpy()
    nv.nvfp4_lora_epilogue(y, x, dev_bf16(c["lora_a"]), dev_bf16(c["lora_b"]), 64.0)
    torch.cuda.synchronize()
    d, _ = o.lora_delta_fp64(c["x"], c["lora_a"], c["lora_b"], 64.0)
    term = lora_bf16_term(c["x"], c["lora_a"], c["lora_b"], 64.0)
    got = y.double().cpu().numpy()
    tol = term + 2e-5 * np.abs(d) + 1e-30
    if ydtype == torch.bfloat16:
        tol = tol + o.bf16_ulp(np.abs(ybase + d) + 1e-30)
    assert np.all(np.abs(got - (ybase + d)) <= tol)
    assert torch.all(full[:, N:] == 7.0), "padding columns written"


def test_timeout_path_reports_and_recovers():
    """A zero wait budget makes in-kernel waits expire: the call must report
    NVFP4_ERR_TIMEOUT through the status word and leave the context usable."""
    M, N, K = 1024, 2048, 8192
    rng = np.random.default_rng(11)
    xb = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    wb = f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    xc, xs, xg = quant_dev(xb)
    wc, ws, wg = quant_dev(wb)
    call, y = nv.prepare_gemm(wc, ws, wg, N, K, a_codes=xc, a_sf=xs, a_global_scale=xg)
    old = nv.set_wait_timeout_ns(0)
    try:
        call()
        st = nv.read_device_status(call.workspace)
    finally:
        nv.set_wait_timeout_ns(old)
    assert st == 6, st
    call()
    assert nv.read_device_status(call.workspace) == 0
    # first 64 rows, quantized with the whole tensor's global scale
    y_or, S, _ = oracle_linear(xb[:64], wb, xg=o.global_scale(xb))
    assert_gemm_close(y[:64], y_or, S, what="after timeout")
