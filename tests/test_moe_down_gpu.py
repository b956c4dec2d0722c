"""nvfp4_moe_down_combine on the GPU against the oracle.

y[t] = sum_j w[t,j] D[row of (t, j)], D = the W4A4 down-projection of the
grouped rows (+ LoRA).  The library stores D in bf16 before the combine (as the
up-projection stores its grouped output), so the tolerance of y is
sum_j |w_tj| (2^-8 |D_tj| + 2e-5 S_tj + LoRA term) + one bf16 ulp of y."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from helpers import dev_bf16, lora_bf16_term
from oracle import nvfp4_oracle as o
from synth import make_case

pytestmark = pytest.mark.gpu


def run_case(c, with_lora, static=None):
    T, E, k, N, K = c["T"], c["E"], c["topk"], c["N"], c["K"]
    counts, offsets, perm = o.group_rows(c["expert_ids"], E)
    wq = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
    lora = None
    if with_lora:
        lora = dict(a=dev_bf16(c["lora_a"]), b=dev_bf16(c["lora_b"]), alpha=c["alpha"])
    hs = None if static is None else torch.tensor([static], dtype=torch.float32, device="cuda")
    y = nv.nvfp4_moe_down_combine(
        dev_bf16(c["h"]), torch.from_numpy(perm.astype(np.int32)).cuda(),
        torch.from_numpy(offsets.astype(np.int32)).cuda(), torch.from_numpy(c["route_weights"]).cuda(),
        wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, E, h_global_scale=hs, lora=lora)
    torch.cuda.synchronize()
    flat = c["expert_ids"].reshape(-1)
    row_e = flat[perm]
    hq = o.quantize(c["h"], None if static is None else np.float32(static))
    wl = [o.quantize(c["w"][e]) for e in range(E)]
    lo = None if not with_lora else (c["lora_a"], c["lora_b"], c["alpha"])
    d_or, S = o.grouped_input_rows(c["h"], hq, row_e, [q[0] for q in wl], [q[1] for q in wl],
                                   [q[2] for q in wl], lo)
    y_or = o.moe_combine(d_or, perm, c["route_weights"], k)
    term = 2.0 ** -8 * np.abs(d_or) + 2e-5 * S
    if with_lora:
        term = term + np.stack([lora_bf16_term(c["h"][i:i + 1], c["lora_a"][row_e[i]], c["lora_b"][row_e[i]],
                                               c["alpha"])[0] for i in range(len(perm))])
    tol = o.moe_combine(term, perm, np.abs(c["route_weights"]), k) + o.bf16_ulp(np.abs(y_or) + 1e-30)
    got = y.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - y_or)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{bad.shape[0]} outside tolerance; first {bad[:3].tolist()} "
                           f"err {err[tuple(bad[0])]:.4g} tol {tol[tuple(bad[0])]:.4g}")


@pytest.mark.parametrize("with_lora", [False, True])
def test_moe_down_small(with_lora):
    run_case(make_case("moe_down", T=96, E=16, N=256, K=512, rank=64), with_lora)


def test_moe_down_skewed_static_scale():
    run_case(make_case("moe_down", T=200, E=40, topk=4, N=512, K=256, rank=32), True,
             static=np.float32(4.0 / 2688.0))
