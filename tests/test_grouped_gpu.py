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
