"""nvfp4_quantize on the GPU against the oracle: codes, scales and the global
scale bit-exact, for the row, column and both packings, linear and swizzled
scale layouts, dynamic and static global scales, ragged and degenerate shapes."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from helpers import assert_bits_equal, dev_bf16, host_bits, u8
from oracle import nvfp4_oracle as o
from synth import f32_to_bf16_bits, make_case

pytestmark = pytest.mark.gpu


def oracle_pack(bits, g, layout):
    codes, sf, g = o.quantize(bits, g)
    return codes, (o.sf_swizzle(sf) if layout == "swizzled" else sf.reshape(-1)), g


def check_quantize(bits, pack, layout, static=None):
    """bits: uint16 [R, C] or [B, R, C]."""
    x = dev_bf16(bits)
    gs = None if static is None else torch.tensor(static, dtype=torch.float32, device="cuda")
    out = nv.nvfp4_quantize(x, pack=pack, sf_layout=layout, global_scale=gs)
    torch.cuda.synchronize()
    b3 = bits if bits.ndim == 3 else bits[None]
    g_gpu = out["global_scale"].cpu().numpy().reshape(-1)
    for b in range(b3.shape[0]):
        sel = (lambda t: t[b]) if bits.ndim == 3 else (lambda t: t)
        g_or = None if static is None else np.float32(static[b])
        if pack in ("row", "both"):
            c, s, g = oracle_pack(b3[b], g_or, layout)
            assert g_gpu[b] == g, (b, g_gpu[b], g)
            assert_bits_equal(u8(sel(out["codes_row"])), c, f"codes_row[{b}]")
            assert_bits_equal(u8(sel(out["sf_row"])), s, f"sf_row[{b}]")
        if pack in ("col", "both"):
            gg = o.global_scale(b3[b]) if g_or is None else g_or
            c, s, g = oracle_pack(np.ascontiguousarray(b3[b].T), gg, layout)
            assert_bits_equal(u8(sel(out["codes_col"])), c, f"codes_col[{b}]")
            assert_bits_equal(u8(sel(out["sf_col"])), s, f"sf_col[{b}]")


@pytest.mark.parametrize("layout", ["swizzled", "linear"])
@pytest.mark.parametrize("pack", ["row", "col", "both"])
def test_tiny_activation_with_outliers(pack, layout):
    check_quantize(make_case("tiny")["x"], pack, layout)          # [32, 512], 1% x20


@pytest.mark.parametrize("layout", ["swizzled", "linear"])
def test_expert_weights_batched_both(layout):
    w = make_case("quantize", E=3, N=256, K=384)["w"]              # 6 x50 outliers per row
    check_quantize(w, "both", layout)


@pytest.mark.parametrize("pack", ["col", "both"])
def test_batched_dynamic_every_matrix(pack):
    """A batch with dynamic scales and the column packing: every matrix's g,
    codes and scales against the oracle.  Ragged tiles in both dimensions, a
    different scale per matrix and the outlier of matrix b in a different tile
    region each time, so that a maximum taken over the wrong matrix or a
    missed region changes g."""
    E, R, C = 9, 208, 1040
    rng = np.random.default_rng(11)
    x = rng.standard_normal((E, R, C)).astype(np.float32)
    for b in range(E):
        x[b] *= 0.05 * (b + 1)
        x[b, (37 * b) % R, (211 * b + 5) % C] = 40.0 * (b + 2) * (-1) ** b
    bits = f32_to_bf16_bits(x)
    check_quantize(bits, pack, "swizzled")
    check_quantize(bits, pack, "linear")


@pytest.mark.parametrize("pack", ["row", "col", "both"])
def test_strided_batched_input(pack):
    """Input rows wider than the matrix and matrices further apart than their
    rows (a view into a larger buffer whose extra elements are large: a read
    of them would change g and the codes), dynamic scales, every matrix
    against the oracle."""
    E, R, C = 3, 208, 1040
    rng = np.random.default_rng(23)
    bits = f32_to_bf16_bits((rng.standard_normal((E, R, C)) * 0.1).astype(np.float32))
    big = np.full((E, R + 2, C + 16), 0x4480, np.uint16)          # bf16 1024.0 outside the view
    big[:, :R, :C] = bits
    x = dev_bf16(big)[:, :R, :C]
    out = nv.nvfp4_quantize(x, pack=pack, sf_layout="swizzled")
    torch.cuda.synchronize()
    g_gpu = out["global_scale"].cpu().numpy().reshape(-1)
    for b in range(E):
        if pack in ("row", "both"):
            c, s_, g = oracle_pack(bits[b], None, "swizzled")
            assert g_gpu[b] == g, (b, g_gpu[b], g)
            assert_bits_equal(u8(out["codes_row"][b]), c, f"codes_row[{b}]")
            assert_bits_equal(u8(out["sf_row"][b]), s_, f"sf_row[{b}]")
        if pack in ("col", "both"):
            gg = o.global_scale(bits[b])
            assert g_gpu[b] == gg, (b, g_gpu[b], gg)
            c, s_, _ = oracle_pack(np.ascontiguousarray(bits[b].T), gg, "swizzled")
            assert_bits_equal(u8(out["codes_col"][b]), c, f"codes_col[{b}]")
            assert_bits_equal(u8(out["sf_col"][b]), s_, f"sf_col[{b}]")


@pytest.mark.parametrize("pack", ["row", "both"])
def test_block_maxima_at_e4m3_rounding_ties(pack):
    """Block maxima on every E4M3 value, on every midpoint between two
    neighbours (exact ties of the scale's round-to-nearest-even), and one bf16
    step either side of each midpoint.  The tensor maximum 448 gives
    g = fl(448/2688) = fl(1/6) and fl(6 g) = 1 exactly, so each block's
    quotient bamax / (6 g) is bamax itself and the ties are exact: the scale
    codes near rounding boundaries, where a fast approximate quotient cannot
    decide, are checked bit for bit against the oracle."""
    v = o.E4M3_VALUES.astype(np.float64)
    mids = (v[1:] + v[:-1]) / 2                      # exact in bf16 (four significant bits)
    mb = f32_to_bf16_bits(mids.astype(np.float32)).astype(np.int64)
    tb = np.concatenate([f32_to_bf16_bits(v[1:].astype(np.float32)).astype(np.int64), mb, mb - 1, mb + 1])
    tvals = o.bf16_to_f32(tb.astype(np.uint16)).astype(np.float64)
    nblk = len(tvals) + 1
    cols = 512
    rows = (nblk * 16 + cols - 1) // cols
    rows = (rows + 15) // 16 * 16
    rng = np.random.default_rng(5)
    x = np.zeros(rows * cols, np.float64)
    x[0] = 448.0                                     # block 0: the tensor maximum
    for i, tv in enumerate(tvals):
        blk = x[(i + 1) * 16:(i + 2) * 16]
        blk[:] = rng.uniform(-1.0, 1.0, 16) * tv * 0.9
        blk[rng.integers(16)] = tv * (1 if i % 2 else -1)
    bits = f32_to_bf16_bits(x.reshape(rows, cols).astype(np.float32))
    check_quantize(bits, pack, "linear")


@pytest.mark.parametrize("shape", [(16, 16), (1, 16), (300, 208), (144, 80), (48, 1040)])
@pytest.mark.parametrize("pack", ["row", "both"])
def test_ragged_shapes(shape, pack):
    R, Cc = shape
    if pack == "both" and R % 16:
        pytest.skip("column packing needs rows % 16 == 0")
    rng = np.random.default_rng(R * 1000 + Cc)
    bits = f32_to_bf16_bits(rng.standard_normal((R, Cc)).astype(np.float32) * 0.3)
    check_quantize(bits, pack, "swizzled")
    check_quantize(bits, pack, "linear")


def test_static_scale_saturation_and_zero_blocks():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[3, :16] = 0.0                      # an all-zero block
    x[4, :16] = -0.0                     # negative zeros
    x[5, 16:32] = 1e-30                  # tiny block: scale rounds to zero
    x[6, 32] = -1e-3                     # signed zero code in a live block
    x[6, 33] = 50.0
    bits = f32_to_bf16_bits(x)
    for static in ([1.0 / 2688.0], [1e-4], [5.0]):   # ordinary, saturating, coarse
        check_quantize(bits, "both", "swizzled", static=static)
    check_quantize(bits, "both", "swizzled")


def test_all_zero_tensor_gives_zero_scale():
    bits = f32_to_bf16_bits(np.zeros((32, 64), np.float32))
    check_quantize(bits, "both", "swizzled")
    check_quantize(bits, "row", "linear")


def test_grid_representable_round_trip_on_device():
    """The oracle's exact round-trip tensor re-quantizes to itself on the GPU too."""
    rng = np.random.default_rng(3)
    R, C = 128, 256
    g = np.float32(2.0 ** -10)
    sfc = rng.integers(1, 127, size=(R, C // 16)).astype(np.uint8)
    sfc[0, 0] = 126
    mag = rng.integers(0, 8, size=(R, C))
    mag.reshape(R, C // 16, 16)[:, :, 0] = 7
    sign = rng.integers(0, 2, size=(R, C))
    vals = (np.where(sign, -1.0, 1.0) * o.E2M1_MAGNITUDES[mag]).reshape(R, C // 16, 16)
    x = (vals * o.E4M3_VALUES[sfc][:, :, None] * float(g)).reshape(R, C)
    bits = f32_to_bf16_bits(x.astype(np.float32))
    out = nv.nvfp4_quantize(dev_bf16(bits), pack="row", sf_layout="linear")
    assert_bits_equal(u8(out["sf_row"]).reshape(R, C // 16), sfc, "round-trip scales")
    assert float(out["global_scale"][0]) == float(g)


def test_full_size_expert_sweep_sampled():
    """32 x [2048, 6144] expert weights (row + column packings, swizzled);
    every global scale checked, two whole matrices checked bit for bit."""
    E, N, K = 32, 2048, 6144
    gen = torch.Generator(device="cuda").manual_seed(0)
    from synth import torch_normal_bf16, torch_outliers_per_row
    w = torch_normal_bf16((E, N, K), 0.02, gen, "cuda")
    torch_outliers_per_row(w, 6, 50.0, gen)
    out = nv.nvfp4_quantize(w, pack="both", sf_layout="swizzled")
    torch.cuda.synchronize()
    g_gpu = out["global_scale"].cpu().numpy()
    amax = w.abs().amax(dim=(1, 2)).float().cpu().numpy()
    assert np.array_equal(g_gpu, (amax / np.float32(2688)).astype(np.float32))
    for e in (0, E - 1):
        bits = host_bits(w[e])
        c, s, g = oracle_pack(bits, None, "swizzled")
        assert g == g_gpu[e]
        assert_bits_equal(u8(out["codes_row"][e]), c, f"codes_row[{e}]")
        assert_bits_equal(u8(out["sf_row"][e]), s, f"sf_row[{e}]")
        c, s, _ = oracle_pack(np.ascontiguousarray(bits.T), g, "swizzled")
        assert_bits_equal(u8(out["codes_col"][e]), c, f"codes_col[{e}]")
        assert_bits_equal(u8(out["sf_col"][e]), s, f"sf_col[{e}]")
