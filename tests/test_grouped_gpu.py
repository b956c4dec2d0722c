"""nvfp4_grouped_gemm on the GPU against the oracle: the stable grouping
(perm, offsets) exactly, the grouped outputs within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from helpers import assert_gemm_close, dev_bf16, host_bits, lora_bf16_term
from oracle import nvfp4_oracle as o
from synth import make_case

pytestmark = pytest.mark.gpu


def quant_experts(w_bits):
    out = nv.nvfp4_quantize(dev_bf16(w_bits), pack="row", sf_layout="swizzled")
    return out["codes_row"], out["sf_row"], out["global_scale"]


def run_case(c, with_lora, rows=None):
    E, N, K, r = c["E"], c["N"], c["K"], c["rank"]
    wc, ws, wg = quant_experts(c["w"])
    ids = torch.from_numpy(c["expert_ids"]).cuda()
    lora = None
    if with_lora:
        lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=c["alpha"])
    d, perm, offs = nv.nvfp4_grouped_gemm(ids, dev_bf16(c["x"]), wc, ws, wg, N, K, E, lora=lora)
    torch.cuda.synchronize()
    counts, offsets, perm_or = o.group_rows(c["expert_ids"], E)
    assert np.array_equal(perm.cpu().numpy(), perm_or)
    assert np.array_equal(offs.cpu().numpy(), offsets)
    # oracle rows
    xq = o.quantize(c["x"])
    wq = [o.quantize(c["w"][e]) for e in range(E)] if rows is None else None
    if rows is None:
        rows = np.arange(perm_or.size)
    experts_needed = sorted({int(c["expert_ids"].reshape(-1)[perm_or[i]]) for i in rows})
    wcodes, wsf, wgs = {}, {}, {}
    for e in experts_needed:
        q = o.quantize(c["w"][e])
        wcodes[e], wsf[e], wgs[e] = q
    lo = None if not with_lora else (c["lora_a"], c["lora_b"], c["alpha"])
    y_or, S = o.grouped_linear_rows(rows, c["x"], xq, wcodes, wsf, wgs, perm_or,
                                    c["expert_ids"], c["topk"], lo)
    term = None
    if with_lora:
        flat = c["expert_ids"].reshape(-1)
        term = np.stack([lora_bf16_term(c["x"][perm_or[i] // c["topk"]][None],
                                        c["lora_a"][flat[perm_or[i]]], c["lora_b"][flat[perm_or[i]]],
                                        c["alpha"])[0] for i in rows])
    assert_gemm_close(d[torch.from_numpy(np.asarray(rows)).cuda()], y_or, S, term, what="grouped")


@pytest.mark.parametrize("with_lora", [False, True])
def test_grouped_small_all_rows(with_lora):
    c = make_case("grouped", T=96, E=16, N=256, K=512, rank=64)
    run_case(c, with_lora)


def test_grouped_skewed_many_experts():
    c = make_case("grouped", T=256, E=64, N=512, K=256, rank=32)
    run_case(c, True)


def test_grouped_full_size_sampled():
    """4096 tokens, 256 experts of [2048,6144], top-8, Zipf-skewed routing, LoRA r64
    (inputs drawn on the device; the sampled rows' inputs are copied back)."""
    from synth import torch_case
    t = torch_case("grouped")
    E, N, K, topk = t["E"], t["N"], t["K"], t["topk"]
    out = nv.nvfp4_quantize(t["w"], pack="row", sf_layout="swizzled")
    lora = dict(a=t["lora_a"], b=t["lora_b"], alpha=t["alpha"])
    d, perm, offs = nv.nvfp4_grouped_gemm(t["expert_ids"], t["x"], out["codes_row"],
                                          out["sf_row"], out["global_scale"], N, K, E, lora=lora)
    torch.cuda.synchronize()
    ids = t["expert_ids"].cpu().numpy()
    counts, offsets, perm_or = o.group_rows(ids, E)
    assert np.array_equal(perm.cpu().numpy(), perm_or)
    assert np.array_equal(offs.cpu().numpy(), offsets)
    heavy = np.argsort(-counts)[:2]
    rng = np.random.default_rng(5)
    rows = set(rng.choice(perm_or.size, 40, replace=False).tolist())
    for e in heavy:                          # edges of the two heaviest experts' row ranges
        rows |= {int(offsets[e]), int(offsets[e + 1] - 1), int(offsets[e]) + 127}
    rows = np.array(sorted(rows))
    xb = host_bits(t["x"])
    xq = o.quantize(xb)
    flat = ids.reshape(-1)
    need = sorted({int(flat[perm_or[i]]) for i in rows})
    wc, wsf, wgs, la, lb = {}, {}, {}, {}, {}
    for e in need:
        wc[e], wsf[e], wgs[e] = o.quantize(host_bits(t["w"][e]))
        la[e], lb[e] = host_bits(t["lora_a"][e]), host_bits(t["lora_b"][e])
    y_or, S = o.grouped_linear_rows(rows, xb, xq, wc, wsf, wgs, perm_or, ids, topk,
                                    (la, lb, t["alpha"]))
    term = np.stack([lora_bf16_term(xb[perm_or[i] // topk][None], la[flat[perm_or[i]]],
                                    lb[flat[perm_or[i]]], t["alpha"])[0] for i in rows])
    assert_gemm_close(d[torch.from_numpy(rows).cuda()], y_or, S, term, what="grouped full")


def test_grouped_input_forms_identical():
    """The three input forms of the grouped call give the same bits: bf16 rows
    with a static global scale; the same rows packed beforehand (codes + linear
    scales, the quantizer's output) with that scale; and the grouping passed in
    as offsets + perm instead of expert ids."""
    c = make_case("grouped", T=200, E=24, N=512, K=512, rank=32)
    E, N, K, topk = c["E"], c["N"], c["K"], c["topk"]
    wc, ws, wg = quant_experts(c["w"])
    ids = torch.from_numpy(c["expert_ids"]).cuda()
    x = dev_bf16(c["x"])
    q = nv.nvfp4_quantize(x, pack="row", sf_layout="linear")
    g = q["global_scale"]
    d1, perm1, offs1 = nv.nvfp4_grouped_gemm(ids, x, wc, ws, wg, N, K, E, x_global_scale=g)
    d2, perm2, offs2 = nv.nvfp4_grouped_gemm(ids, None, wc, ws, wg, N, K, E, x_global_scale=g,
                                             x_packed=(q["codes_row"], q["sf_row"]))
    d3, perm3, offs3 = nv.nvfp4_grouped_gemm(None, None, wc, ws, wg, N, K, E, x_global_scale=g,
                                             x_packed=(q["codes_row"], q["sf_row"]),
                                             routing=(offs1, perm1), top_k=topk)
    torch.cuda.synchronize()
    assert torch.equal(perm1, perm2) and torch.equal(offs1, offs2)
    assert torch.equal(perm3, perm1) and torch.equal(offs3, offs1)
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))
    assert torch.equal(d1.view(torch.int16), d3.view(torch.int16))
    # and the packed form against the oracle (the static scale is the tensor's own)
    counts, offsets, perm_or = o.group_rows(c["expert_ids"], E)
    assert np.array_equal(perm1.cpu().numpy(), perm_or)
    xq = o.quantize(c["x"])
    wq = {e: o.quantize(c["w"][e]) for e in range(E)}
    rows = np.arange(perm_or.size)
    y_or, S = o.grouped_linear_rows(rows, c["x"], xq, {e: wq[e][0] for e in wq},
                                    {e: wq[e][1] for e in wq}, {e: wq[e][2] for e in wq}, perm_or,
                                    c["expert_ids"], topk, None)
    assert_gemm_close(d2, y_or, S, None, what="grouped packed input")


@pytest.mark.parametrize("with_lora", [False, True])
def test_grouped_fp32_output(with_lora):
    """out_dtype fp32 within the fp32 tolerance of the oracle; the bf16 output
    is that fp32 result rounded to nearest even."""
    c = make_case("grouped", T=96, E=16, N=256, K=512, rank=64)
    E, N, K = c["E"], c["N"], c["K"]
    wc, ws, wg = quant_experts(c["w"])
    ids = torch.from_numpy(c["expert_ids"]).cuda()
    x = dev_bf16(c["x"])
    lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=c["alpha"]) if with_lora else None
    d32, perm, _ = nv.nvfp4_grouped_gemm(ids, x, wc, ws, wg, N, K, E, lora=lora,
                                         out_dtype=torch.float32)
    d16, _, _ = nv.nvfp4_grouped_gemm(ids, x, wc, ws, wg, N, K, E, lora=lora)
    torch.cuda.synchronize()
    assert d32.dtype == torch.float32
    assert torch.equal(d32.to(torch.bfloat16).view(torch.int16), d16.view(torch.int16))
    counts, offsets, perm_or = o.group_rows(c["expert_ids"], E)
    xq = o.quantize(c["x"])
    wq = {e: o.quantize(c["w"][e]) for e in range(E)}
    rows = np.arange(perm_or.size)
    lo = (c["lora_a"], c["lora_b"], c["alpha"]) if with_lora else None
    y_or, S = o.grouped_linear_rows(rows, c["x"], xq, {e: wq[e][0] for e in wq},
                                    {e: wq[e][1] for e in wq}, {e: wq[e][2] for e in wq}, perm_or,
                                    c["expert_ids"], c["topk"], lo)
    term = None
    if with_lora:
        flat = c["expert_ids"].reshape(-1)
        term = np.stack([lora_bf16_term(c["x"][perm_or[i] // c["topk"]][None],
                                        c["lora_a"][flat[perm_or[i]]], c["lora_b"][flat[perm_or[i]]],
                                        c["alpha"])[0] for i in rows])
    assert_gemm_close(d32, y_or, S, term, what="grouped fp32")


def test_grouped_given_routing_inconsistent():
    """Given routing is device data the host cannot check: offsets that step
    backwards or past the pair count, and perm entries outside [0, P), are
    clamped (counts cumulatively to P, such pairs as padding).  The call
    succeeds, the sanitized offsets come back, and the rows the clamped layout
    does hold are computed as usual."""
    c = make_case("grouped", T=64, E=8, N=256, K=256, rank=32)
    E, N, K, topk = c["E"], c["N"], c["K"], c["topk"]
    P = c["T"] * topk
    wc, ws, wg = quant_experts(c["w"])
    ids = torch.from_numpy(c["expert_ids"]).cuda()
    x = dev_bf16(c["x"])
    d_ref, perm_ref, offs_ref = nv.nvfp4_grouped_gemm(ids, x, wc, ws, wg, N, K, E)
    bad_offs = offs_ref.clone()
    bad_offs[3] = bad_offs[2] - 7            # expert 2 count negative -> 0
    bad_offs[E] = P + 1000                   # last expert past the end
    bad_perm = perm_ref.clone()
    bad_perm[0] = -3
    bad_perm[1] = P + 5
    d, perm, offs = nv.nvfp4_grouped_gemm(None, x, wc, ws, wg, N, K, E,
                                          routing=(bad_offs, bad_perm), top_k=topk)
    torch.cuda.synchronize()
    # the sanitized layout: counts of the given offsets clamped to [0, P] cumulatively
    given = bad_offs.cpu().numpy().astype(np.int64)
    cnt = np.clip(np.diff(given), 0, P)
    want = np.zeros(E + 1, np.int64)
    for e in range(E):
        want[e + 1] = min(want[e] + cnt[e], P)
    assert np.array_equal(offs.cpu().numpy(), want)
    # rows whose expert range and pair are both intact match the consistent call
    ref_o = offs_ref.cpu().numpy()
    pr = bad_perm.cpu().numpy()
    for e in range(E):
        for i in range(int(want[e]), int(want[e + 1])):
            j = i - int(want[e]) + int(ref_o[e])          # the same row of the consistent call
            if 0 <= pr[i] < P and j < ref_o[e + 1] and int(pr[i]) == int(perm_ref[j]):
                assert torch.equal(d[i].view(torch.int16), d_ref[j].view(torch.int16)), (e, i)


def test_grouped_single_expert_top1():
    """Degenerate routing: top-1 with every token on one expert (three m-tiles,
    the last one ragged) and the other 15 experts empty."""
    c = make_case("grouped", T=300, E=16, topk=1, N=256, K=512, rank=32)
    c["expert_ids"] = np.full((300, 1), 5, np.int32)
    run_case(c, True)


def test_grouped_repeated_expert_in_a_token():
    """top-2 with both slots of every third token on the same expert: two pairs
    of one token in one expert's rows, kept in pair order."""
    c = make_case("grouped", T=128, E=8, topk=2, N=256, K=256, rank=32)
    ids = c["expert_ids"].copy()
    ids[::3, 1] = ids[::3, 0]
    c["expert_ids"] = ids
    run_case(c, False)
