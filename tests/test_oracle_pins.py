"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages state (grid maximum 6, scale maximum 448, amax/(6*448), the ~0.09
round-trip error, the [[1,2,3],[4,5,6]] transpose example), a library routine
for a special case (torch's float8_e4m3fn conversion), an independent bit-level
derivation, or brute force on tiny inputs.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import nvfp4_oracle as o
from synth import bf16_bits_to_f32, f32_to_bf16_bits, make_case

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bits(x):
    return f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


# --- format tables -----------------------------------------------------------

def test_e2m1_grid_from_bit_fields():
    # E2M1: 2 exponent bits with bias 1, 1 mantissa bit; exponent 0 subnormal.
    vals = []
    for code in range(8):
        e, m = code >> 1, code & 1
        vals.append(m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    assert vals == list(o.E2M1_MAGNITUDES)
    # the pages' grid {0, +-0.5, +-1, +-1.5, +-2, +-3, +-4, +-6}; max 6 = the 6 of 6*448
    assert sorted(set(vals)) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_table_matches_torch_float8():
    codes = torch.arange(127, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(ref, o.E4M3_VALUES)
    assert o.E4M3_VALUES.max() == 448.0          # the 448 of 6*448
    assert o.E4M3_VALUES[1] == 2.0 ** -9         # smallest subnormal
    assert float(o.GLOBAL_DIVISOR) == 6 * 448


def test_e4m3_rounding_matches_torch_below_saturation():
    rng = np.random.default_rng(1)
    q = np.concatenate([
        rng.uniform(0, 464, 20000).astype(np.float32),
        np.exp2(rng.uniform(-12, 8.8, 20000)).astype(np.float32),
        # exact midpoints between neighbouring E4M3 values (ties to even)
        ((o.E4M3_VALUES[1:] + o.E4M3_VALUES[:-1]) / 2).astype(np.float32),
        o.E4M3_VALUES.astype(np.float32),
    ])
    q = q[q < 464]       # torch does not saturate: 480 and above become NaN
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.e4m3_encode(q), ref)


def test_e4m3_saturates_to_448():
    q = np.array([448.0, 463.9, 464.0, 480.0, 1e6, np.inf], dtype=np.float32)
    assert np.all(o.E4M3_VALUES[o.e4m3_encode(q)] == 448.0)


def _e2m1_by_bits(v: float) -> int:
    """Independent RNE to E2M1 via the fp32 bit pattern (round the 23-bit
    mantissa to 1 bit, handle the subnormal range and saturation)."""
    v = abs(float(np.float32(v)))
    if v >= 6.0:
        return 7
    if v < 1.0:                              # subnormal range: multiples of 0.5
        fr = Fraction(v) * 2
        n = math.floor(fr)
        rem = fr - n
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
            n += 1
        return n                              # 0, 1 or 2 (=1.0)
    b = int(np.array(v, dtype=np.float32).view(np.uint32))
    exp = ((b >> 23) & 0xFF) - 127            # 0, 1 or 2
    mant = b & 0x7FFFFF
    keep = mant >> 22                         # 1 mantissa bit kept
    rest = mant & ((1 << 22) - 1)
    half = 1 << 21
    if rest > half or (rest == half and keep & 1):
        keep += 1
    code = ((exp + 1) << 1) + keep            # overflow of keep carries into exp
    return min(code, 7)


def test_e2m1_rounding_matches_bitlevel_derivation():
    rng = np.random.default_rng(2)
    v = np.concatenate([
        rng.uniform(0, 7, 20000), np.exp2(rng.uniform(-8, 3, 5000)),
        (o.E2M1_MAGNITUDES[1:] + o.E2M1_MAGNITUDES[:-1]) / 2,
        o.E2M1_MAGNITUDES,
    ]).astype(np.float32)
    got = o.e2m1_encode_magnitude(v)
    ref = np.array([_e2m1_by_bits(x) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e2m1_ties_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_ties.txt"))
            if l.strip() and not l.startswith("#")]
    for v, want in rows:
        code = o.e2m1_encode_magnitude(np.array([float(v)], np.float32))[0]
        assert o.E2M1_MAGNITUDES[code] == float(want), v


# --- quantization --------------------------------------------------------------

def test_global_scale_rule_and_amax_block():
    c = make_case("tiny")
    x = c["x"]
    xf = bf16_bits_to_f32(x)
    amax = np.abs(xf).max()
    codes, sf, g = o.quantize(x)
    # weight_scale_2 = amax/(6*448), the fp32 quotient
    assert g == np.float32(float(amax) / 2688.0) or abs(float(g) - float(amax) / 2688) <= 2 ** -24 * float(g)
    # the block holding amax gets the largest scale and its largest code (6)
    r, k = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert o.E4M3_VALUES[sf[r, k // 16]] == 448.0
    nib = o.unpack_codes(codes)[r, k]
    assert nib & 7 == 7 and ((nib >> 3) == (xf[r, k] < 0))
    # and the dequantized amax is within E4M3/E2M1 rounding of amax
    assert abs(6 * 448 * float(g) - amax) <= 1e-6 * amax


def test_exact_round_trip_of_grid_representable_tensor():
    """x = code * sb * g with a block at (6, 448) re-quantizes to itself."""
    rng = np.random.default_rng(3)
    R, C = 64, 256
    g = np.float32(2.0 ** -10)
    sfc = rng.integers(1, 127, size=(R, C // 16)).astype(np.uint8)
    sfc[0, 0] = 126                                   # 448: fixes amax = 2688 g
    mag = rng.integers(0, 8, size=(R, C))
    sign = rng.integers(0, 2, size=(R, C))
    mag.reshape(R, C // 16, 16)[:, :, 0] = 7          # every block holds a 6
    vals = (np.where(sign, -1.0, 1.0) * o.E2M1_MAGNITUDES[mag]).reshape(R, C // 16, 16)
    x = (vals * o.E4M3_VALUES[sfc][:, :, None] * float(g)).reshape(R, C)
    xb = bits(x)
    assert np.array_equal(bf16_bits_to_f32(xb).astype(np.float64), x)  # bf16-exact
    codes, sf, g2 = o.quantize(xb)
    assert g2 == g
    assert np.array_equal(sf, sfc)
    want = (sign << 3 | mag).astype(np.uint8)
    want[mag == 0] = (sign[mag == 0] << 3)
    assert np.array_equal(o.unpack_codes(codes), want)
    assert np.array_equal(o.dequantize(codes, sf, g2), x)


def test_round_trip_relative_error_is_about_0_09():
    # ordinary weights: N(0, 0.02) without outliers (the card's "ordinary NVFP4 fidelity")
    w = make_case("prefill", M=1, N=1024, rank=1)["w"]
    codes, sf, g = o.quantize(w)
    wf = bf16_bits_to_f32(w).astype(np.float64)
    err = o.dequantize(codes, sf, g) - wf
    fro = np.linalg.norm(err) / np.linalg.norm(wf)
    mean_abs = np.abs(err).mean() / np.abs(wf).mean()
    assert 0.08 <= fro <= 0.11 and 0.08 <= mean_abs <= 0.11, (fro, mean_abs)


def test_transpose_example_golden():
    w = np.zeros((16, 16), np.float32)
    w[0, :3] = [1, 2, 3]
    w[1, :3] = [4, 5, 6]
    wb = bits(w)
    _, sf_r, g = o.quantize(wb)
    _, sf_c, g_c = o.quantize_colwise(wb)
    assert g == g_c == np.float32(np.float32(6) / np.float32(2688))
    rows = [l.split() for l in open(os.path.join(GOLDEN, "transpose_example.txt"))
            if l.strip() and not l.startswith("#")]
    for kind, i, val in rows:
        sf = sf_r if kind == "row" else sf_c
        assert o.E4M3_VALUES[sf[int(i), 0]] == float(val), (kind, i)
    # the column scale set is not a relabelling of the row scales
    assert set(o.E4M3_VALUES[sf_c[:3, 0]]) != set(o.E4M3_VALUES[sf_r[:2, 0]])


def test_colwise_is_quantization_of_transpose_not_of_codes():
    c = make_case("quantize", E=1, N=64, K=96)
    w = c["w"][0]
    cc, sc, gc = o.quantize_colwise(w)
    cr, sr, gr = o.quantize(np.ascontiguousarray(w.T), o.global_scale(w))
    assert np.array_equal(cc, cr) and np.array_equal(sc, sr) and gc == gr
    # and its blocks really run along N: block maxima of W[:, k] columns
    wf = np.abs(bf16_bits_to_f32(w))
    colmax = wf.reshape(64 // 16, 16, 96).max(axis=1).T      # [K, N/16]
    q = (colmax / np.float32(6 * gc)).astype(np.float32)
    ref = torch.from_numpy(q).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(sc, ref)


def test_zero_blocks_signs_and_static_scale():
    x = np.zeros((2, 32), np.float32)
    x[0, :16] = -0.0
    x[1, 16] = 6.0
    x[1, 17] = -1e-3        # rounds to a signed zero code (reading: sign kept)
    codes, sf, g = o.quantize(bits(x))
    assert sf[0, 0] == 0 and sf[0, 1] == 0 and sf[1, 0] == 0   # all-zero blocks
    assert np.all(o.unpack_codes(codes)[0] == 0)               # +0 when sb == 0
    u = o.unpack_codes(codes)[1]
    assert u[16] == 7 and u[17] == 8
    # all-zero tensor: g = 0, every scale and code zero
    c0, s0, g0 = o.quantize(bits(np.zeros((3, 16))))
    assert g0 == 0 and not c0.any() and not s0.any()
    # static global scale: out-of-range blocks saturate at 448 and code 6
    cs, ss, gs = o.quantize(bits(np.full((1, 16), 100.0)), np.float32(1e-3))
    assert o.E4M3_VALUES[ss[0, 0]] == 448 and np.all(o.unpack_codes(cs) == 7)


def test_bytes_per_element_is_4_5_bits():
    assert o.bytes_per_element() * 8 == 4.5
    c, s, _ = o.quantize(make_case("tiny")["w"])
    assert (c.nbytes + s.nbytes) / (256 * 512) == 0.5625


# --- scale layouts ---------------------------------------------------------------

def test_swizzle_is_a_padded_bijection():
    rng = np.random.default_rng(4)
    for R, Cs in [(1, 1), (37, 5), (128, 4), (300, 24)]:
        sf = rng.integers(1, 256, size=(R, Cs)).astype(np.uint8)
        buf = o.sf_swizzle(sf)
        pR, pC = o.sf_swizzled_shape(R, Cs)
        assert buf.size == pR * pC
        assert np.array_equal(o.sf_unswizzle(buf, R, Cs), sf)
        assert np.count_nonzero(buf) == np.count_nonzero(sf)  # padding is zero
    # atom structure: rows r, r+32, r+64, r+96 share one 16-byte line
    sf = np.arange(128 * 4, dtype=np.int64).reshape(128, 4).astype(np.uint8)
    buf = o.sf_swizzle(sf)
    assert list(buf[:16]) == [0, 1, 2, 3, 128, 129, 130, 131, 0, 1, 2, 3, 128, 129, 130, 131]


# --- products ------------------------------------------------------------------

def _decode_by_bits(packed, sf, g):
    """Independent dequantization: nibbles via bit fields, scales via torch fp8."""
    R, H = packed.shape
    sfv = torch.from_numpy(sf.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    out = np.zeros((R, 2 * H))
    for r in range(R):
        for j in range(2 * H):
            nib = (int(packed[r, j // 2]) >> (4 * (j % 2))) & 0xF
            e, m = (nib >> 1) & 3, nib & 1
            mag = m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1)
            out[r, j] = (-mag if nib & 8 else mag) * sfv[r, j // 16] * float(g)
    return out


def test_gemm_and_lora_match_brute_force():
    c = make_case("prefill", M=3, N=5, K=32, rank=4)
    xq = o.quantize(c["x"])
    wq = o.quantize(c["w"])
    y = o.linear_fp64(xq, wq, c["x"], (c["lora_a"], c["lora_b"], 8.0))
    xd = _decode_by_bits(*xq)
    wd = _decode_by_bits(*wq)
    xf = bf16_bits_to_f32(c["x"]).astype(float)
    af = bf16_bits_to_f32(c["lora_a"]).astype(float)
    bf = bf16_bits_to_f32(c["lora_b"]).astype(float)
    for m in range(3):
        t = [math.fsum(xf[m, k] * af[j, k] for k in range(32)) for j in range(4)]
        for n in range(5):
            base = math.fsum(xd[m, k] * wd[n, k] for k in range(32))
            lo = (8.0 / 4) * math.fsum(t[j] * bf[n, j] for j in range(4))
            assert abs(y[m, n] - (base + lo)) <= 1e-12 * (abs(base) + abs(lo) + 1e-30)


def test_error_scale_bounds_the_sum():
    c = make_case("tiny", M=4, N=8)
    xq, wq = o.quantize(c["x"]), o.quantize(c["w"])
    s = o.error_scale(xq, wq)
    y = o.linear_fp64(xq, wq)
    assert np.all(s >= np.abs(y) - 1e-12)


def test_bf16_rounding_of_fp64():
    rng = np.random.default_rng(5)
    v32 = (rng.standard_normal(5000) * 10).astype(np.float32)
    ref = torch.from_numpy(v32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(o.round_fp64_to_bf16(v32.astype(np.float64)), ref)
    # a value just above an fp64 tie rounds up, an exact tie goes to even
    # bf16 spacing at 1.0 is 2^-7: 1 + 2^-8 is a tie (to even: 1.0)
    assert o.round_fp64_to_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert o.round_fp64_to_bf16(np.array([1 + 2 ** -8 + 2 ** -40]))[0] == 1 + 2 ** -7
    assert o.round_fp64_to_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    assert o.bf16_ulp(np.array([1.0]))[0] == 2 ** -7


def test_group_rows_matches_brute_force():
    c = make_case("grouped", T=64, E=16, K=16, N=16)
    ids = c["expert_ids"]
    counts, offsets, perm = o.group_rows(ids, 16)
    lists = {e: [] for e in range(16)}
    for t in range(ids.shape[0]):
        for s in range(ids.shape[1]):
            lists[int(ids[t, s])].append(t * ids.shape[1] + s)
    brute = [p for e in range(16) for p in sorted(lists[e])]
    assert list(perm) == brute
    assert list(counts) == [len(lists[e]) for e in range(16)]
    assert offsets[-1] == ids.size
    # every token's slots hold distinct experts
    assert all(len(set(r)) == r.size for r in ids)


# --- dequantization to bf16 (the backward's rebuilt weight) ---------------------

def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(21)
    v = (rng.standard_normal(20000) * np.exp(rng.uniform(-20, 20, 20000))).astype(np.float32)
    v[:8] = [0.0, -0.0, 1.0, 1.00390625, 1.005859375, 1.01171875, -3.0, 65504.0]   # ties included
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.f32_to_bf16_rne(v), want)


def test_dequantize_bf16_exact_when_scales_are_powers_of_two():
    # g a power of two: every fp32 product is exact, so the bf16 result is the
    # nearest bf16 of the exact value (an independent rounding routine)
    rng = np.random.default_rng(22)
    R, C = 64, 256
    w = f32_to_bf16_bits((rng.standard_normal((R, C)) * 0.05).astype(np.float32))
    codes, sf, _ = o.quantize(w, np.float32(2.0 ** -12))
    got = o.dequantize_bf16(codes, sf, np.float32(2.0 ** -12))
    exact = o.dequantize(codes, sf, 2.0 ** -12)
    want = o.f32_to_bf16_rne(exact.astype(np.float32))     # exact in fp32 (<= 7 significant bits)
    assert np.array_equal(got, want)
    assert np.array_equal(bf16_bits_to_f32(got).astype(np.float64), exact)


def test_dequantize_bf16_within_two_roundings_for_any_scale():
    rng = np.random.default_rng(23)
    R, C = 32, 512
    w = f32_to_bf16_bits((rng.standard_normal((R, C)) * 0.3).astype(np.float32))
    codes, sf, g = o.quantize(w)                              # g = amax / 2688, not a power of two
    got = bf16_bits_to_f32(o.dequantize_bf16(codes, sf, g)).astype(np.float64)
    exact = o.dequantize(codes, sf, g)
    # fp32 rounding of s_dec and of the product (2 x 2^-24), then bf16 (2^-8)
    bound = np.abs(exact) * (2.0 ** -8 + 3 * 2.0 ** -24) + 1e-45
    assert np.all(np.abs(got - exact) <= bound)
    assert np.mean(got == exact) < 1.0                       # the roundings do act


def test_dequantize_bf16_requantizes_to_the_same_codes():
    # grid-representable tensor (power-of-two g): dequantize then quantize is the identity
    rng = np.random.default_rng(24)
    R, C = 48, 128
    g = np.float32(2.0 ** -9)
    sfc = rng.integers(1, 127, size=(R, C // 16)).astype(np.uint8)
    mag = rng.integers(0, 8, size=(R, C))
    mag.reshape(R, C // 16, 16)[:, :, 0] = 7                  # each block reaches 6 * sb
    sign = rng.integers(0, 2, size=(R, C))
    vals = (np.where(sign, -1.0, 1.0) * o.E2M1_MAGNITUDES[mag]).reshape(R, C // 16, 16)
    x = (vals * o.E4M3_VALUES[sfc][:, :, None] * float(g)).reshape(R, C)
    codes, sf, _ = o.quantize(f32_to_bf16_bits(x.astype(np.float32)), g)
    back = o.dequantize_bf16(codes, sf, g)
    codes2, sf2, _ = o.quantize(back, g)
    assert np.array_equal(codes2, codes) and np.array_equal(sf2, sf)


def test_dequantize_bf16_signed_zero_and_zero_scale():
    codes = np.zeros((1, 8), np.uint8)
    codes[0, 0] = 0x08 | (0x01 << 4)      # element 0 = -0, element 1 = +0.5
    sf = np.array([[56]], np.uint8)       # E4M3 code 56 = 1.0
    out = o.dequantize_bf16(codes, sf, np.float32(1.0))
    assert out[0, 0] == 0x8000 and out[0, 1] == 0x3F00 and np.all(out[0, 2:] == 0)
    out0 = o.dequantize_bf16(codes, np.array([[0]], np.uint8), np.float32(1.0))
    assert out0[0, 1] == 0 and out0[0, 0] == 0x8000   # zero scale: +-0 by the code's sign


def test_moe_combine_matches_brute_force():
    rng = np.random.default_rng(41)
    T, k, E, N = 12, 3, 5, 4
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)])
    counts, offsets, perm = o.group_rows(ids, E)
    d_rows = rng.standard_normal((T * k, N))
    w = rng.random((T, k))
    y = o.moe_combine(d_rows, perm, w, k)
    for t in range(T):
        want = np.zeros(N)
        for j in range(k):
            g = int(np.flatnonzero(perm == t * k + j)[0])    # the grouped row holding pair (t, j)
            assert ids.reshape(-1)[perm[g]] == ids[t, j]
            want += w[t, j] * d_rows[g]
        assert np.allclose(y[t], want, rtol=0, atol=1e-12)


def test_grouped_input_rows_is_the_per_expert_linear():
    rng = np.random.default_rng(42)
    P, K, N, E = 6, 64, 32, 3
    h = f32_to_bf16_bits(rng.standard_normal((P, K)).astype(np.float32))
    ws = [f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.1).astype(np.float32)) for _ in range(E)]
    row_e = np.array([0, 0, 1, 2, 2, 2])
    hq = o.quantize(h)
    wq = [o.quantize(w) for w in ws]
    d, _ = o.grouped_input_rows(h, hq, row_e, [q[0] for q in wq], [q[1] for q in wq], [q[2] for q in wq])
    hd = o.dequantize(*hq)
    for i in range(P):   # brute force: one dot product per output
        wd = o.dequantize(*wq[row_e[i]])
        for n in range(N):
            assert abs(d[i, n] - sum(hd[i, kk] * wd[n, kk] for kk in range(K))) <= 1e-12 * (1 + abs(d[i, n]))
