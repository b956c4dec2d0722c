"""Seeded synthetic inputs shaped like the layers the NVFP4 pages describe.

This module is shared by the tests, the benchmark and the oracle's callers.
It holds no NVFP4 arithmetic: it only draws random numbers, rounds them to
bf16 storage and builds the MoE routing table that the library takes as an
input.  Every tensor is drawn from its own child of ``SeedSequence(seed)``,
spawned in a fixed order, so a given (config, seed) always yields the same
bytes.

Two backends draw the same recipe:

* ``numpy``  - PCG64 streams; used for every case the oracle checks in full.
* ``torch``  - a seeded ``torch.Generator`` on the target device; used for the
  full-size benchmark workloads (gigabytes of weights), where drawing on the
  host would dominate the run.  Parity at those sizes is checked on sampled
  outputs whose inputs are copied back to the host.

Recipes (shapes and distributions follow the pages' layers: hidden 6144,
256 routed experts with top-8 routing, o_proj 6144x16384, q_b_proj
16384x2048; LoRA rank 64 with alpha 128):

* tiny:      W[256,512] ~N(0,0.02); X[32,512] ~N(0,1) with exactly
             round(0.01*numel) entries, drawn without replacement, x20.
* decode:    W[N,K] ~N(0,0.02) for (N,K) in {(16384,2048), (6144,16384)};
             X[M,K] ~N(0,1), M in {1,8,32}.
* quantize:  32 x W[2048,6144] ~N(0,0.02); in every row exactly 6 entries
             (round(0.001*6144)), drawn without replacement, x50.
* prefill:   X[8192,6144] ~N(0,1); W[2048,6144] ~N(0,0.02); LoRA down
             weight A_w[64,6144] ~N(0,0.01) and up weight B_w[2048,64]
             ~N(0,0.01), both stored in the Linear-weight layout
             (out_features x in_features); alpha = 128.
* grouped:   X[4096,6144] ~N(0,1); 256 experts W_e[2048,6144] ~N(0,0.02);
             per-expert LoRA A_e[64,6144], B_e[2048,64] ~N(0,0.01);
             routing logits N(0,1)[4096,256] plus bias_e = -1.1*ln(rank_e)
             (rank_e a seeded permutation of 1..256: the log of a Zipf(1.1)
             pmf), top-8 per token by logit, ties to the lower expert id.
* dgrad:     the backward of the prefill linear: W[2048,6144] ~N(0,0.02),
             dY[8192,2048] ~N(0,0.01) (gradient-sized values).
* moe_down:  h[32768,2048] ~N(0,1) (the activated up-projection output, in
             grouped order); 256 experts W2_e[6144,2048] ~N(0,0.02); LoRA
             A_e[64,2048], B_e[6144,64] ~N(0,0.01); routing as grouped; gate
             weights = softmax over each token's selected scores.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "CONFIGS", "f32_to_bf16_bits", "bf16_bits_to_f32", "Draw", "make_case",
    "route_top_k",
]

#: Shapes of the five workloads (see module docstring for distributions).
CONFIGS = {
    "tiny": dict(M=32, N=256, K=512),
    "decode_q_b_proj": dict(N=16384, K=2048, Ms=(1, 8, 32)),
    "decode_o_proj": dict(N=6144, K=16384, Ms=(1, 8, 32)),
    "quantize": dict(E=32, N=2048, K=6144),
    "prefill": dict(M=8192, N=2048, K=6144, rank=64, alpha=128.0),
    "grouped": dict(T=4096, E=256, topk=8, N=2048, K=6144, rank=64, alpha=128.0),
    # the backward of the prefill linear: dX [M, K] = dY [M, N] W [N, K]
    "dgrad": dict(M=8192, N=2048, K=6144),
    # the routed experts' down-projection W2_e [6144, 2048] after the grouped
    # up-projection, and the gate-weighted combine
    "moe_down": dict(T=4096, E=256, topk=8, N=6144, K=2048, rank=64, alpha=128.0),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); uint16 bits.

    Storage rounding of the synthetic draws only.  NaN is not expected here.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    rounded = (u + 0x7FFF + lsb) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


class Draw:
    """Fixed-order child streams of ``SeedSequence(seed)`` (numpy backend)."""

    def __init__(self, seed: int = 0, n_children: int = 64):
        self._children = np.random.SeedSequence(seed).spawn(n_children)
        self._next = 0

    def rng(self) -> np.random.Generator:
        ss = self._children[self._next]
        self._next += 1
        return np.random.Generator(np.random.PCG64(ss))

    def normal_bf16(self, shape, sigma: float) -> np.ndarray:
        g = self.rng()
        v = g.standard_normal(size=shape, dtype=np.float32) * np.float32(sigma)
        return f32_to_bf16_bits(v)


def _outliers_global(bits: np.ndarray, frac: float, mult: float, g: np.random.Generator):
    """Multiply exactly round(frac*numel) entries, drawn without replacement, by mult."""
    flat = bf16_bits_to_f32(bits).ravel()
    n = int(round(frac * flat.size))
    idx = g.choice(flat.size, size=n, replace=False)
    flat[idx] *= np.float32(mult)
    return f32_to_bf16_bits(flat.reshape(bits.shape)), np.sort(idx)


def _outliers_per_row(bits: np.ndarray, per_row: int, mult: float, g: np.random.Generator):
    """In every row multiply exactly ``per_row`` entries (no replacement) by mult."""
    v = bf16_bits_to_f32(bits).copy()
    rows, cols = v.shape[-2], v.shape[-1]
    v2 = v.reshape(-1, cols)
    keys = g.random(size=v2.shape, dtype=np.float32)
    idx = np.argpartition(keys, per_row, axis=1)[:, :per_row]
    r = np.arange(v2.shape[0])[:, None]
    v2[r, idx] *= np.float32(mult)
    return f32_to_bf16_bits(v2.reshape(v.shape))


def route_top_k(logits: np.ndarray, bias: np.ndarray, k: int) -> np.ndarray:
    """Top-k experts per token by (logit + bias); ties go to the lower expert id.

    Softmax is monotone, so the top-k of the softmax equals the top-k of the
    biased logits.  Returns int32 [tokens, k] in decreasing-score order.
    """
    s = logits.astype(np.float64) + bias.astype(np.float64)[None, :]
    # lexsort: last key is primary.  Sort by (-score, expert id).
    E = s.shape[1]
    ids = np.broadcast_to(np.arange(E), s.shape)
    order = np.lexsort((ids, -s), axis=1)
    return order[:, :k].astype(np.int32)


def zipf_bias(E: int, g: np.random.Generator, s: float = 1.1) -> np.ndarray:
    """bias_e = -s*ln(rank_e) with rank a seeded permutation of 1..E."""
    rank = g.permutation(E) + 1
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


def gate_weights(scores: np.ndarray, experts: np.ndarray) -> np.ndarray:
    """Gate weights of the chosen experts: softmax over each token's selected
    scores (fp32 inputs to the combine)."""
    sel = np.take_along_axis(np.asarray(scores, np.float64), experts, axis=1)
    e = np.exp(sel - sel.max(axis=1, keepdims=True))
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def make_case(name: str, seed: int = 0, **over) -> dict:
    """Draw one workload with the numpy backend; returns uint16 bf16 bits.

    ``over`` may shrink shapes (e.g. M=..., N=..., E=...) for small parity
    cases; the distributions stay those of the named workload.
    """
    d = Draw(seed)
    if name == "tiny":
        c = dict(CONFIGS["tiny"], **over)
        w = d.normal_bf16((c["N"], c["K"]), 0.02)
        x = d.normal_bf16((c["M"], c["K"]), 1.0)
        x, out_idx = _outliers_global(x, 0.01, 20.0, d.rng())
        return dict(x=x, w=w, outlier_index=out_idx, **c)
    if name in ("decode_q_b_proj", "decode_o_proj"):
        c = dict(CONFIGS[name], **over)
        M = over.get("M", 1)
        w = d.normal_bf16((c["N"], c["K"]), 0.02)
        x = d.normal_bf16((M, c["K"]), 1.0)
        return dict(x=x, w=w, M=M, N=c["N"], K=c["K"])
    if name == "quantize":
        c = dict(CONFIGS["quantize"], **over)
        w = d.normal_bf16((c["E"], c["N"], c["K"]), 0.02)
        per_row = over.get("per_row", int(round(0.001 * c["K"])))
        w = _outliers_per_row(w, per_row, 50.0, d.rng())
        return dict(w=w, per_row=per_row, **c)
    if name == "prefill":
        c = dict(CONFIGS["prefill"], **over)
        x = d.normal_bf16((c["M"], c["K"]), 1.0)
        w = d.normal_bf16((c["N"], c["K"]), 0.02)
        a = d.normal_bf16((c["rank"], c["K"]), 0.01)
        b = d.normal_bf16((c["N"], c["rank"]), 0.01)
        return dict(x=x, w=w, lora_a=a, lora_b=b, **c)
    if name == "dgrad":
        c = dict(CONFIGS["dgrad"], **over)
        w = d.normal_bf16((c["N"], c["K"]), 0.02)
        dy = d.normal_bf16((c["M"], c["N"]), 0.01)
        return dict(w=w, dy=dy, **c)
    if name == "moe_down":
        c = dict(CONFIGS["moe_down"], **over)
        P = c["T"] * c["topk"]
        h = d.normal_bf16((P, c["K"]), 1.0)
        w = d.normal_bf16((c["E"], c["N"], c["K"]), 0.02)
        a = d.normal_bf16((c["E"], c["rank"], c["K"]), 0.01)
        b = d.normal_bf16((c["E"], c["N"], c["rank"]), 0.01)
        g = d.rng()
        logits = g.standard_normal(size=(c["T"], c["E"]), dtype=np.float32)
        bias = zipf_bias(c["E"], d.rng())
        experts = route_top_k(logits, bias, c["topk"])
        weights = gate_weights(logits + bias, experts)
        return dict(h=h, w=w, lora_a=a, lora_b=b, expert_ids=experts, route_weights=weights, **c)
    if name == "grouped":
        c = dict(CONFIGS["grouped"], **over)
        x = d.normal_bf16((c["T"], c["K"]), 1.0)
        w = d.normal_bf16((c["E"], c["N"], c["K"]), 0.02)
        a = d.normal_bf16((c["E"], c["rank"], c["K"]), 0.01)
        b = d.normal_bf16((c["E"], c["N"], c["rank"]), 0.01)
        g = d.rng()
        logits = g.standard_normal(size=(c["T"], c["E"]), dtype=np.float32)
        bias = zipf_bias(c["E"], d.rng())
        experts = route_top_k(logits, bias, c["topk"])
        return dict(x=x, w=w, lora_a=a, lora_b=b, expert_ids=experts, **c)
    raise KeyError(name)


# ----------------------------------------------------------------------------
# torch backend (device-side draws for full-size benchmark workloads)
# ----------------------------------------------------------------------------

def torch_normal_bf16(shape, sigma: float, gen, device):
    """Draw N(0, sigma) on ``device`` with generator ``gen``; bf16 tensor (RNE)."""
    import torch
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return (v * sigma).to(torch.bfloat16)


def torch_outliers_per_row(t, per_row: int, mult: float, gen):
    """In every row of a bf16 tensor multiply ``per_row`` entries by ``mult``."""
    import torch
    cols = t.shape[-1]
    flat = t.view(-1, cols)
    keys = torch.rand(flat.shape, generator=gen, device=t.device, dtype=torch.float32)
    idx = keys.topk(per_row, dim=1, largest=False).indices
    vals = flat.gather(1, idx).float() * mult
    flat.scatter_(1, idx, vals.to(torch.bfloat16))
    return t


def torch_outliers_global(t, frac: float, mult: float, gen):
    import torch
    flat = t.view(-1)
    n = int(round(frac * flat.numel()))
    keys = torch.rand(flat.numel(), generator=gen, device=t.device, dtype=torch.float32)
    idx = keys.topk(n, largest=False).indices
    flat[idx] = (flat[idx].float() * mult).to(torch.bfloat16)
    return t


def torch_route_top_k(T: int, E: int, k: int, gen, device):
    """Routing with the recipe of ``route_top_k`` drawn on device."""
    import torch
    logits = torch.randn((T, E), generator=gen, device=device, dtype=torch.float32)
    perm = torch.randperm(E, generator=gen, device=device) + 1
    bias = -1.1 * torch.log(perm.double())
    s = logits.double() + bias[None, :]
    # stable descending sort keeps the lower expert id first among ties
    order = torch.sort(s, dim=1, descending=True, stable=True).indices
    return order[:, :k].to(torch.int32).contiguous()


def torch_route_top_k_weights(T: int, E: int, k: int, gen, device):
    """``torch_route_top_k`` plus the gate weights (softmax over the selected scores)."""
    import torch
    logits = torch.randn((T, E), generator=gen, device=device, dtype=torch.float32)
    perm = torch.randperm(E, generator=gen, device=device) + 1
    bias = -1.1 * torch.log(perm.double())
    s = logits.double() + bias[None, :]
    order = torch.sort(s, dim=1, descending=True, stable=True).indices[:, :k]
    w = torch.softmax(torch.gather(s, 1, order), dim=1).float()
    return order.to(torch.int32).contiguous(), w.contiguous()


def pad_up(v: int, m: int) -> int:
    return (v + m - 1) // m * m


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def log2_int(v: int) -> int:
    return int(math.log2(v))


def torch_case(name: str, seed: int = 0, device="cuda", **over) -> dict:
    """The named workload drawn on ``device`` (same recipe, torch Philox streams).

    Returns torch tensors (bf16 / int32).  Used for full-size benchmark inputs."""
    import torch
    gen = torch.Generator(device=device).manual_seed(seed)
    if name == "prefill":
        c = dict(CONFIGS["prefill"], **over)
        return dict(x=torch_normal_bf16((c["M"], c["K"]), 1.0, gen, device),
                    w=torch_normal_bf16((c["N"], c["K"]), 0.02, gen, device),
                    lora_a=torch_normal_bf16((c["rank"], c["K"]), 0.01, gen, device),
                    lora_b=torch_normal_bf16((c["N"], c["rank"]), 0.01, gen, device), **c)
    if name == "grouped":
        c = dict(CONFIGS["grouped"], **over)
        return dict(x=torch_normal_bf16((c["T"], c["K"]), 1.0, gen, device),
                    w=torch_normal_bf16((c["E"], c["N"], c["K"]), 0.02, gen, device),
                    lora_a=torch_normal_bf16((c["E"], c["rank"], c["K"]), 0.01, gen, device),
                    lora_b=torch_normal_bf16((c["E"], c["N"], c["rank"]), 0.01, gen, device),
                    expert_ids=torch_route_top_k(c["T"], c["E"], c["topk"], gen, device), **c)
    if name == "moe_down":
        c = dict(CONFIGS["moe_down"], **over)
        P = c["T"] * c["topk"]
        ids, wts = torch_route_top_k_weights(c["T"], c["E"], c["topk"], gen, device)
        return dict(h=torch_normal_bf16((P, c["K"]), 1.0, gen, device),
                    w=torch_normal_bf16((c["E"], c["N"], c["K"]), 0.02, gen, device),
                    lora_a=torch_normal_bf16((c["E"], c["rank"], c["K"]), 0.01, gen, device),
                    lora_b=torch_normal_bf16((c["E"], c["N"], c["rank"]), 0.01, gen, device),
                    expert_ids=ids, route_weights=wts, **c)
    if name == "dgrad":
        c = dict(CONFIGS["dgrad"], **over)
        return dict(w=torch_normal_bf16((c["N"], c["K"]), 0.02, gen, device),
                    dy=torch_normal_bf16((c["M"], c["N"]), 0.01, gen, device), **c)
    if name == "quantize":
        c = dict(CONFIGS["quantize"], **over)
        w = torch_normal_bf16((c["E"], c["N"], c["K"]), 0.02, gen, device)
        torch_outliers_per_row(w, int(round(0.001 * c["K"])), 50.0, gen)
        return dict(w=w, **c)
    if name in ("decode_q_b_proj", "decode_o_proj"):
        c = dict(CONFIGS[name], **over)
        M = over.get("M", 1)
        return dict(w=torch_normal_bf16((c["N"], c["K"]), 0.02, gen, device),
                    x=torch_normal_bf16((M, c["K"]), 1.0, gen, device), M=M, N=c["N"], K=c["K"])
    if name == "tiny":
        c = dict(CONFIGS["tiny"], **over)
        w = torch_normal_bf16((c["N"], c["K"]), 0.02, gen, device)
        x = torch_normal_bf16((c["M"], c["K"]), 1.0, gen, device)
        torch_outliers_global(x, 0.01, 20.0, gen)
        return dict(x=x, w=w, **c)
    raise KeyError(name)
