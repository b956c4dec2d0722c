"""The seeded input generators follow the stated recipe: the same seed gives the
same tensors, the draws have the stated scales, the outliers are exactly as
many as stated, routing picks k distinct experts by biased score with a
skewed (Zipf) load, and the gate weights of a token sum to 1.  Reduced shapes,
the distributions of the named workloads; CPU only."""
import numpy as np

from synth import bf16_bits_to_f32, gate_weights, make_case, route_top_k, zipf_bias


def test_same_seed_same_tensors_other_seed_differs():
    a = make_case("prefill", seed=0, M=64, N=128, K=256)
    b = make_case("prefill", seed=0, M=64, N=128, K=256)
    c = make_case("prefill", seed=1, M=64, N=128, K=256)
    for k in ("x", "w", "lora_a", "lora_b"):
        assert np.array_equal(a[k], b[k]), k
        assert not np.array_equal(a[k], c[k]), k


def test_prefill_scales():
    c = make_case("prefill", seed=0, M=256, N=256, K=1024)
    for k, sigma in (("x", 1.0), ("w", 0.02), ("lora_a", 0.01), ("lora_b", 0.01)):
        v = bf16_bits_to_f32(c[k]).astype(np.float64)
        assert abs(v.mean()) < 0.02 * sigma * 5, k
        assert abs(v.std() / sigma - 1.0) < 0.03, (k, v.std())


def test_tiny_outliers_exact_count():
    c = make_case("tiny", seed=0)
    x = bf16_bits_to_f32(c["x"])
    idx = c["outlier_index"]
    assert len(idx) == int(round(0.01 * x.size)) and len(np.unique(idx)) == len(idx)
    # the x20 entries dominate: their magnitudes are those of N(0, 20^2) draws
    big = np.abs(x.ravel()[idx])
    rest = np.abs(np.delete(x.ravel(), idx))
    assert np.median(big) > 10 * np.median(rest)


def test_quantize_rows_carry_their_outliers():
    c = make_case("quantize", seed=0, E=2, N=64)
    assert c["per_row"] == int(round(0.001 * c["K"])) == 6
    w = bf16_bits_to_f32(c["w"]).reshape(-1, c["K"])
    # every row holds x50 entries: its largest magnitude is far above 0.02-sigma draws
    assert np.all(np.abs(w).max(axis=1) > 0.2)
    # and the bulk keeps the 0.02 scale
    assert abs(np.median(np.abs(w)) / (0.02 * 0.6745) - 1.0) < 0.05


def test_routing_distinct_sorted_and_skewed():
    g = np.random.default_rng(7)
    T, E, k = 2048, 64, 8
    logits = g.standard_normal((T, E)).astype(np.float32)
    bias = zipf_bias(E, np.random.default_rng(8))
    ex = route_top_k(logits, bias, k)
    assert ex.shape == (T, k)
    assert all(len(set(r)) == k for r in ex)
    s = logits.astype(np.float64) + bias.astype(np.float64)
    sel = np.take_along_axis(s, ex.astype(np.int64), axis=1)
    assert np.all(np.diff(sel, axis=1) <= 0)                  # decreasing score
    kth = sel[:, -1:]
    others = np.where(np.isin(np.arange(E)[None, :], ex, invert=True), s, -np.inf)
    assert np.all(others <= kth)                               # nothing better left out
    load = np.bincount(ex.ravel(), minlength=E)
    assert load.max() > 3 * load.mean()                        # Zipf(1.1) skew
    w = gate_weights(s, ex)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6) and np.all(w > 0)


def test_grouped_case_routing_shape():
    c = make_case("grouped", seed=0, T=256, E=16, N=128, K=256, rank=32)
    ex = c["expert_ids"]
    assert ex.shape == (256, c["topk"]) and ex.dtype == np.int32
    assert ex.min() >= 0 and ex.max() < 16


# ---- the device-side generators of the benchmark inputs (run here on the CPU)

def test_torch_case_same_recipe_on_cpu():
    import torch
    from synth import torch_case
    a = torch_case("prefill", seed=3, device="cpu", M=256, N=256, K=1024)
    b = torch_case("prefill", seed=3, device="cpu", M=256, N=256, K=1024)
    for k, sigma in (("x", 1.0), ("w", 0.02), ("lora_a", 0.01), ("lora_b", 0.01)):
        assert torch.equal(a[k], b[k]), k
        assert a[k].dtype == torch.bfloat16
        v = a[k].double()
        assert abs(v.std().item() / sigma - 1.0) < 0.03, (k, v.std().item())
    q = torch_case("quantize", seed=0, device="cpu", E=2, N=64)
    w = q["w"].float().reshape(-1, q["K"])
    assert bool((w.abs().amax(dim=1) > 0.2).all())
    g = torch_case("grouped", seed=0, device="cpu", T=2048, E=64, N=128, K=256, rank=32)
    ex = g["expert_ids"]
    assert ex.dtype == torch.int32 and ex.shape == (2048, 8)
    assert all(len(set(r.tolist())) == 8 for r in ex)
    load = torch.bincount(ex.reshape(-1).long(), minlength=64)
    assert load.max().item() > 3 * load.float().mean().item()
    m = torch_case("moe_down", seed=0, device="cpu", T=256, E=16, N=128, K=256, rank=32)
    assert torch.allclose(m["route_weights"].sum(dim=1), torch.ones(256), atol=1e-6)
