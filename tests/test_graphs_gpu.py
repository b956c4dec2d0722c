"""The calls captured into CUDA graphs (a serving loop replays one graph per
step): after capture the input buffers are refilled with new data and the
graph replayed; every output must be bit-identical to an eager call on the
same data.  Covers the programmatic-dependency launches, the workspace-carved
scratch and the in-call memsets under stream capture."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from helpers import dev_bf16
from synth import f32_to_bf16_bits, make_case

pytestmark = pytest.mark.gpu


def _bits(rng, shape, scale):
    return f32_to_bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def _capture(call):
    """Warm the call up (attributes set outside capture), then capture it."""
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


def _same(a, b, what):
    assert torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8)), what


def test_graph_prefill_dynamic_with_lora():
    M, N, K, r = 384, 512, 1024, 64
    c = make_case("prefill", M=M, N=N, K=K, rank=r)
    wq = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
    x = dev_bf16(c["x"])
    lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=128.0)
    call, y = nv.prepare_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x, lora=lora)
    g = _capture(call)
    rng = np.random.default_rng(1)
    for step in range(2):
        x.copy_(dev_bf16(_bits(rng, (M, K), 1.0 + step)))
        g.replay()
        torch.cuda.synchronize()
        want = nv.nvfp4_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x.clone(),
                             lora=lora)
        torch.cuda.synchronize()
        _same(y, want, f"prefill replay {step}")


def test_graph_decode_gemv_static_scale():
    M, N, K = 1, 1024, 16384          # CUDA-core GEMV, chunk sums in the CTA
    c = make_case("decode_q_b_proj", M=M, N=N, K=K)
    wq = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
    gx = torch.tensor([16.0 / 2688.0], dtype=torch.float32, device="cuda")
    x = dev_bf16(c["x"])
    call, y = nv.prepare_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x,
                              a_global_scale=gx)
    g = _capture(call)
    rng = np.random.default_rng(2)
    x.copy_(dev_bf16(_bits(rng, (M, K), 0.5)))
    g.replay()
    torch.cuda.synchronize()
    want = nv.nvfp4_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x.clone(),
                         a_global_scale=gx)
    torch.cuda.synchronize()
    _same(y, want, "decode replay")


def test_graph_decode_operand_swapped_split_k():
    """M = 8 rows with a static scale on a long K: the operand-swapped tcgen05
    GEMM (weights issued before its wait on the activation packing) and the
    split-K pass, captured and replayed on new rows."""
    M, N, K = 8, 768, 16384
    c = make_case("decode_o_proj", M=M, N=N, K=K)
    wq = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
    gx = torch.tensor([16.0 / 2688.0], dtype=torch.float32, device="cuda")
    x = dev_bf16(c["x"])
    call, y = nv.prepare_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x,
                              a_global_scale=gx)
    g = _capture(call)
    rng = np.random.default_rng(5)
    for step in range(2):
        x.copy_(dev_bf16(_bits(rng, (M, K), 0.5 + step)))
        g.replay()
        torch.cuda.synchronize()
        want = nv.nvfp4_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x.clone(),
                             a_global_scale=gx)
        torch.cuda.synchronize()
        _same(y, want, f"operand-swapped replay {step}")


def test_graph_quantize_batched_both():
    E, R, C = 3, 256, 768
    rng = np.random.default_rng(3)
    w = dev_bf16(_bits(rng, (E, R, C), 0.02))
    call, out = nv.prepare_quantize(w, pack="both", sf_layout="swizzled")
    g = _capture(call)
    w.copy_(dev_bf16(_bits(rng, (E, R, C), 0.07)))
    g.replay()
    torch.cuda.synchronize()
    want = nv.nvfp4_quantize(w.clone(), pack="both", sf_layout="swizzled")
    torch.cuda.synchronize()
    for k in ("codes_row", "sf_row", "codes_col", "sf_col", "global_scale"):
        _same(out[k], want[k], f"quantize replay {k}")


def test_graph_grouped_routing_and_lora():
    c = make_case("grouped", T=96, E=16, N=256, K=512, rank=64)
    E, N, K = c["E"], c["N"], c["K"]
    q = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
    ids = torch.from_numpy(c["expert_ids"]).cuda()
    x = dev_bf16(c["x"])
    lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=c["alpha"])
    call, (d, perm, offs) = nv.prepare_grouped(ids, x, q["codes_row"], q["sf_row"], q["global_scale"], N, K, E,
                                               lora=lora)
    g = _capture(call)
    rng = np.random.default_rng(4)
    ids.copy_(torch.from_numpy(rng.integers(0, E, size=ids.shape).astype(np.int32)))
    x.copy_(dev_bf16(_bits(rng, tuple(x.shape), 1.0)))
    g.replay()
    torch.cuda.synchronize()
    d2, perm2, offs2 = nv.nvfp4_grouped_gemm(ids.clone(), x.clone(), q["codes_row"], q["sf_row"],
                                             q["global_scale"], N, K, E, lora=lora)
    torch.cuda.synchronize()
    _same(perm, perm2, "grouped perm")
    _same(offs, offs2, "grouped offsets")
    _same(d, d2, "grouped D")


def test_concurrent_streams_match_serial():
    """Two calls on two streams at once (the persistent kernels share the
    SMs; none of them waits on another grid): each result bit-identical to
    the same call run alone."""
    M, N, K, r = 512, 1024, 2048, 64
    c = make_case("prefill", M=M, N=N, K=K, rank=r)
    wq = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
    x = dev_bf16(c["x"])
    lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=128.0)
    rng = np.random.default_rng(6)
    w2 = dev_bf16(_bits(rng, (4, 512, 1536), 0.05))
    call1, y = nv.prepare_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x, lora=lora)
    call2, q = nv.prepare_quantize(w2, pack="both", sf_layout="swizzled")
    call1()
    call2()
    torch.cuda.synchronize()
    y_alone = y.clone()
    q_alone = {k: v.clone() for k, v in q.items() if k != "workspace"}
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        s1.wait_stream(torch.cuda.current_stream())
        s2.wait_stream(torch.cuda.current_stream())
        for _ in range(4):
            call1(s1)
            call2(s2)
        torch.cuda.synchronize()
        _same(y, y_alone, "gemm on a concurrent stream")
        for k, v in q_alone.items():
            _same(q[k], v, f"quantize on a concurrent stream: {k}")
