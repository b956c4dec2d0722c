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


def test_moe_down_full_size_sampled():
    """The benchmarked shape: h[32768,2048] in grouped order, 256 experts
    W2_e[6144,2048], top-8 of 256 with the Zipf-skewed routing, LoRA r64, the
    launch configuration the benchmark times.  The oracle evaluates sampled
    tokens x sampled output columns: tokens routed to the two heaviest experts,
    tokens routed to experts that hold a single row, and seeded random ones;
    columns at both ends, at the 256-wide tile edges and seeded random ones.
    Each touched expert's global scale is its whole matrix's amax / 2688, taken
    on the host from a host copy of that matrix."""
    from synth import torch_case
    c = torch_case("moe_down", seed=0, device="cuda")
    T, E, k, N, K, r, alpha = c["T"], c["E"], c["topk"], c["N"], c["K"], c["rank"], c["alpha"]
    ids = c["expert_ids"].cpu().numpy()
    counts, offsets, perm = o.group_rows(ids, E)
    wq = nv.nvfp4_quantize(c["w"], pack="row", sf_layout="swizzled")
    lora = dict(a=c["lora_a"], b=c["lora_b"], alpha=alpha)
    y = nv.nvfp4_moe_down_combine(
        c["h"], torch.from_numpy(perm.astype(np.int32)).cuda(),
        torch.from_numpy(offsets.astype(np.int32)).cuda(), c["route_weights"],
        wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, E, lora=lora)
    torch.cuda.synchronize()
    del wq

    rng = np.random.default_rng(5)
    heavy = np.argsort(-counts, kind="stable")[:2]
    single = np.flatnonzero(counts == 1)
    pick = set()
    for e in heavy:
        pick.update(rng.choice(np.flatnonzero((ids == e).any(axis=1)), 3, replace=False).tolist())
    for e in single[:4]:
        pick.update(np.flatnonzero((ids == e).any(axis=1)).tolist())
    pick.update(rng.choice(T, 6, replace=False).tolist())
    tokens = np.array(sorted(pick))
    cols = np.unique(np.concatenate([[0, 255, 256, 511, N - 256, N - 1],
                                     rng.choice(N, 90, replace=False)]))

    def bits(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    h_bits = bits(c["h"])
    g_h = o.global_scale(h_bits)
    inv = np.empty(T * k, np.int64)
    inv[perm] = np.arange(T * k)
    pairs = (tokens[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    rows = inv[pairs]
    row_e = ids.reshape(-1)[pairs]
    w_rows = {}
    for e in np.unique(row_e):
        we = bits(c["w"][int(e)])
        w_rows[int(e)] = o.quantize(np.ascontiguousarray(we[cols]), o.global_scale(we))
    la, lb = bits(c["lora_a"]), bits(c["lora_b"])
    d_or, S, lt = [], [], []
    for i, e in zip(rows, row_e):
        e = int(e)
        hb = h_bits[i:i + 1]
        hr = o.quantize(hb, g_h)
        lo = (la[e], np.ascontiguousarray(lb[e][cols]), alpha)
        d_or.append(o.linear_fp64(hr, w_rows[e], hb, lo)[0])
        S.append(o.error_scale(hr, w_rows[e], hb, lo)[0])
        lt.append(lora_bf16_term(hb, la[e], lo[1], alpha)[0])
    d_or, S, lt = np.array(d_or), np.array(S), np.array(lt)
    wts = c["route_weights"].cpu().numpy()[tokens]
    ident = np.arange(len(pairs))
    y_or = o.moe_combine(d_or, ident, wts, k)
    term = 2.0 ** -8 * np.abs(d_or) + 2e-5 * S + lt
    tol = o.moe_combine(term, ident, np.abs(wts), k) + o.bf16_ulp(np.abs(y_or) + 1e-30)
    got = y[torch.from_numpy(tokens).cuda()][:, torch.from_numpy(cols).cuda()].float().cpu().numpy()
    err = np.abs(got.astype(np.float64) - y_or)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{bad.shape[0]} of {err.size} outside tolerance; first {bad[:3].tolist()} "
                           f"err {err[tuple(bad[0])]:.4g} tol {tol[tuple(bad[0])]:.4g}")
    assert len(tokens) >= 10 and counts[heavy[0]] > 1000 and len(single) >= 1


def test_moe_down_single_expert_top1():
    """Degenerate routing: top-1, every token on one expert, 15 experts empty."""
    c = make_case("moe_down", T=300, E=16, topk=1, N=256, K=512, rank=32)
    c["expert_ids"] = np.full((300, 1), 3, np.int32)
    run_case(c, True)
