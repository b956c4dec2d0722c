"""Pin of the quantizer's operation order (reading R1) at global scales that are
not powers of two.

The pages fix the format (E2M1 codes, one E4M3 scale per 16 elements along
the contraction axis, one fp32 global scale g = amax/(6*448): "vroomfondel/
glm-5.2-reap-504B-v2-W4A4" card, "How it was produced"; "GLM-5.2-NVFP4" card,
"Quantization recipe") but not the fp32 operation order.  Reading R1 fixes it:

    t = fl(6 g);  q = fl(bamax / t);  sb = E4M3(q);
    s_dec = fl(sb * g);  s_enc = fl(1 / s_dec);  v = fl(x * s_enc);  code = E2M1(v)

At a power-of-two g every plausible order gives the same codes, so this file
works at non-power-of-two g only.  The truth here is an independent derivation
in exact rationals (fractions.Fraction): every step is computed exactly and
then rounded to fp32 by an explicit round-half-even on the binary exponent,
and E4M3 / E2M1 are rounded from their bit fields (exponent and mantissa),
not by a search over a value table as the oracle does.

Coverage: every E4M3 scale code 1..126, and in each of its blocks the bf16
neighbours of every E2M1 grid point and of every midpoint between two
adjacent codes, at three static scales and one dynamic (amax) scale.

Sensitivity: a seeded search selects inputs on which plausible slips of the
order change the result (x / s_dec instead of x * s_enc; 1/s_dec or 6g or
sb*g left unrounded, i.e. a float64 promotion; bamax/6/g in place of
bamax/(6g)).  The exact derivation with each slip applied must differ from
R1 on those inputs -- so an oracle making that slip would fail here -- and the
oracle must agree with R1 on all of them.
"""
from fractions import Fraction as Fr

import numpy as np
import pytest

from oracle import nvfp4_oracle as o

FLT_MAX = Fr(2) ** 127 * (2 - Fr(1, 2 ** 23))


# ----------------------------------------------------- exact arithmetic --

def _floor_log2(a: Fr) -> int:
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fr(2) ** e > a:
        e -= 1
    elif Fr(2) ** (e + 1) <= a:
        e += 1
    return e


def f32(x: Fr) -> Fr:
    """Exact fp32 round-to-nearest-even of a rational (finite results only)."""
    if x == 0:
        return Fr(0)
    a = abs(x)
    e = max(_floor_log2(a), -126)          # subnormals share the exponent -126 quantum
    quantum = Fr(2) ** (e - 23)
    r = round(a / quantum) * quantum       # Fraction.__round__: ties to even
    assert r <= FLT_MAX
    return r if x > 0 else -r


def e4m3_code(q: Fr) -> int:
    """E4M3 (bias 7, 3 mantissa bits, subnormals, max 448) round-half-even and
    saturating, from the bit fields."""
    if q <= 0:
        return 0
    if q >= 448:
        return 126
    e = _floor_log2(q)
    if e < -6:                              # subnormal: m * 2^-9, m = 0..7
        m = round(q / Fr(2) ** -9)
        return 8 if m == 8 else m           # m == 8 is 2^-6, the first normal
    m = round(q / Fr(2) ** (e - 3))         # 8..16
    if m == 16:
        e, m = e + 1, 8
    code = ((e + 7) << 3) | (m - 8)
    return min(code, 126)


def e4m3_value(code: int) -> Fr:
    e, m = code >> 3, code & 7
    return Fr(m, 2 ** 9) if e == 0 else (1 + Fr(m, 8)) * Fr(2) ** (e - 7)


def e2m1_code(v: Fr) -> int:
    """E2M1 magnitude code (bias 1, 1 mantissa bit, max 6), round-half-even and
    saturating, from the bit fields."""
    if v >= 6:
        return 7
    if v < 1:
        return round(v / Fr(1, 2))          # 0, 1 (0.5) or 2 (1.0)
    e = _floor_log2(v)                      # 0, 1, 2
    m = round(v / Fr(2) ** (e - 1))         # 2..4
    if m == 4:
        e, m = e + 1, 2
    if e > 2:
        return 7
    return ((e + 1) << 1) | (m - 2)


def bf16_value(bits: int) -> Fr:
    f = np.array([bits], dtype=np.uint32) << 16
    return Fr(float(f.view(np.float32)[0]))


SLIPS = ("divide", "senc_f64", "t_f64", "sdec_f64", "q_div6_then_g")


def derive(block_bits, g: Fr, slip=None):
    """Scale code and 16 codes of one block by R1 (or with one slip applied)."""
    xs = [bf16_value(int(b)) for b in block_bits]
    bamax = max(abs(x) for x in xs)
    if g == 0:
        return 0, [0] * len(xs)
    t = 6 * g if slip == "t_f64" else f32(6 * g)
    if slip == "q_div6_then_g":
        q = f32(f32(bamax / 6) / g)
    else:
        q = f32(bamax / t)
    sb = e4m3_code(q)
    if sb == 0:
        return 0, [0] * len(xs)
    s_dec = e4m3_value(sb) * g if slip == "sdec_f64" else f32(e4m3_value(sb) * g)
    s_enc = 1 / s_dec if slip == "senc_f64" else min(f32(1 / s_dec), FLT_MAX)
    codes = []
    for b, x in zip(block_bits, xs):
        v = f32(abs(x) / s_dec) if slip == "divide" else f32(abs(x) * s_enc)
        codes.append(((int(b) >> 15) << 3) | e2m1_code(v))
    return sb, codes


# --------------------------------------------------------------- inputs --

def _bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bits (input construction only)."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) & 0xFFFF).astype(np.uint16)


def _neighbours(target: float) -> list:
    """The bf16 values just below and just above a positive target."""
    b = int(_bf16_bits(np.array([target], np.float32))[0])
    out = {b - 1, b, b + 1}
    return sorted(x for x in out if 0 < x < 0x7F80)


E2M1_POINTS = [0.5, 1, 1.5, 2, 3, 4, 6]
E2M1_MIDS = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5]


def coverage_blocks(g: Fr):
    """Blocks for every scale code 1..126: the first element sets the block
    maximum (so q rounds to that code), the rest sit next to every E2M1 grid
    point and midpoint at that scale, with alternating signs."""
    t = f32(6 * g)
    blocks = []
    for sb in range(1, 127):
        bam = _neighbours(float(e4m3_value(sb) * t))
        bam = [b for b in bam if e4m3_code(f32(bf16_value(b) / t)) == sb]
        if not bam:
            continue
        lead = bam[len(bam) // 2]
        lead_v = bf16_value(lead)
        s_dec = f32(e4m3_value(sb) * g)
        vals = []
        for p in E2M1_POINTS + E2M1_MIDS:
            for nb in _neighbours(float(p * s_dec)):
                if bf16_value(nb) <= lead_v:
                    vals.append(nb)
        for i in range(0, len(vals), 15):
            chunk = vals[i:i + 15]
            chunk = [c | (0x8000 if (j % 2) else 0) for j, c in enumerate(chunk)]
            chunk += [0] * (15 - len(chunk))
            blocks.append([lead] + chunk)
    return np.array(blocks, dtype=np.uint16)


def _f32_np(x):
    return np.asarray(x, dtype=np.float32)


def discriminating_cases(rng, n_g=4000):
    """Seeded search (plain numpy fp32/fp64, selection only) for (g, sb, x)
    where a slip of the order could change a code; each case is confirmed
    with the exact derivation by the test itself."""
    cases = {s: [] for s in SLIPS}
    # random non-power-of-two static scales spanning the useful range
    gs = _f32_np(np.exp(rng.uniform(np.log(1e-5), np.log(1e-1), n_g)))
    gs = gs[np.frexp(gs)[0] != 0.5]
    sbv = np.array([float(e4m3_value(c)) for c in range(1, 127)])
    # element-level slips: x next to an E2M1 midpoint at scale s_dec
    for gi in range(len(gs)):
        g = gs[gi]
        s_dec = _f32_np(_f32_np(sbv) * g)
        s_enc = _f32_np(np.float32(1.0) / s_dec)
        for B in E2M1_MIDS:
            tgt = _f32_np(B * s_dec.astype(np.float64))
            for d in (-1, 0, 1):
                xb = _bf16_bits(tgt).astype(np.int64) + d
                x = (xb.astype(np.uint32) << 16).view(np.float32)
                v1 = _f32_np(x * s_enc)
                v_div = _f32_np(x / s_dec)
                v_64 = x.astype(np.float64) * (1.0 / s_dec.astype(np.float64))
                for name, v2 in (("divide", v_div), ("senc_f64", v_64)):
                    hit = (np.minimum(v1, v2) <= B) & (np.maximum(v1, v2) >= B) & (v1 != v2)
                    for k in np.flatnonzero(hit):
                        if len(cases[name]) < 60:
                            cases[name].append((float(g), k + 1, int(xb[k])))
        if all(len(cases[s]) >= 60 for s in ("divide", "senc_f64")):
            break
    # scale-level slips: for a block maximum `bam` and an E4M3 midpoint M, scan
    # the fp32 scales next to the one that puts bam / (6g) exactly on M
    mids = (sbv[:-1] + sbv[1:]) / 2
    bams = np.unique(_bf16_bits(_f32_np(np.exp(rng.uniform(np.log(1e-3), np.log(10.0), 64)))))
    for bb in bams:
        bam = float((np.array([bb], np.uint32) << 16).view(np.float32)[0])
        g0 = _f32_np(bam / mids / 6.0)
        for k in range(-48, 49):
            g = (g0.view(np.int32) + k).view(np.float32)
            t = _f32_np(np.float32(6.0) * g)
            q1 = _f32_np(np.float32(bam) / t)
            alts = (("t_f64", _f32_np(bam / (6.0 * g.astype(np.float64)))),
                    ("q_div6_then_g", _f32_np(_f32_np(np.float32(bam) / np.float32(6.0)) / g)))
            for name, q2 in alts:
                hit = (np.minimum(q1, q2) <= mids) & (np.maximum(q1, q2) >= mids) & (q1 != q2)
                for j in np.flatnonzero(hit):
                    if len(cases[name]) < 60 and np.frexp(g[j])[0] != 0.5:
                        cases[name].append((float(g[j]), None, int(bb)))
        if len(cases["t_f64"]) >= 60 and len(cases["q_div6_then_g"]) >= 60:
            break
    for gi in range(len(gs)):
        g = gs[gi]
        # s_dec rounding: x next to a midpoint where sb*g is inexact (f64 vs f32)
        s_dec32 = _f32_np(_f32_np(sbv) * g)
        s_dec64 = sbv * float(g)
        for B in E2M1_MIDS:
            xb = _bf16_bits(_f32_np(B * s_dec64)).astype(np.int64)
            for d in (-1, 0, 1):
                x = ((xb + d).astype(np.uint32) << 16).view(np.float32)
                v1 = _f32_np(x * _f32_np(np.float32(1.0) / s_dec32))
                v2 = _f32_np(x * _f32_np(1.0 / s_dec64))
                hit = (np.minimum(v1, v2) <= B) & (np.maximum(v1, v2) >= B) & (v1 != v2)
                for k in np.flatnonzero(hit):
                    if len(cases["sdec_f64"]) < 60:
                        cases["sdec_f64"].append((float(g), k + 1, int(xb[k] + d)))
        if all(len(cases[s]) >= 60 for s in SLIPS):
            break
    return cases


def block_for_case(g: float, sb, xbits: int):
    """One 16-element block: a leading element that fixes the scale code (or,
    for the scale-level slips, the candidate block maximum itself), the case's
    element, and its negation."""
    gF = Fr(g)
    t = f32(6 * gF)
    if sb is None:                           # the block maximum is the case
        return np.array([xbits, xbits | 0x8000] + [0] * 14, np.uint16)
    lead = [b for b in _neighbours(float(e4m3_value(sb) * t))
            if e4m3_code(f32(bf16_value(b) / t)) == sb]
    if not lead or bf16_value(xbits) > bf16_value(lead[-1]):
        return None
    return np.array([lead[-1], xbits, xbits | 0x8000] + [0] * 13, np.uint16)


def oracle_block_codes(block_bits: np.ndarray, g: float):
    codes, sf, g_used = o.quantize(block_bits.reshape(1, 16), np.float32(g))
    assert float(g_used) == float(np.float32(g))
    un = np.empty(16, np.uint8)
    un[0::2] = codes[0] & 0xF
    un[1::2] = codes[0] >> 4
    return int(sf[0, 0]), [int(c) for c in un]


# ---------------------------------------------------------------- tests --

STATIC_G = [np.float32(0.0123456), np.float32(3.3e-3), np.float32(np.pi / 2688.0)]


@pytest.mark.parametrize("g", STATIC_G)
def test_every_scale_code_and_grid_boundary_static_scale(g):
    assert np.frexp(g)[0] != 0.5, "g must not be a power of two"
    blocks = coverage_blocks(Fr(float(g)))
    assert len(blocks) >= 200
    codes, sf, _ = o.quantize(blocks, g)
    seen_sb = set()
    for i, blk in enumerate(blocks):
        sb, want = derive(blk, Fr(float(g)))
        got_sf = int(sf[i, 0])
        got = [(int(codes[i, j // 2]) >> (4 * (j % 2))) & 0xF for j in range(16)]
        assert got_sf == sb, (i, got_sf, sb)
        assert got == want, (i, got, want)
        seen_sb.add(sb)
    assert seen_sb == set(range(1, 127))


def test_every_scale_code_dynamic_scale():
    """The dynamic rule with a non-power-of-two amax: g = fl(amax / 2688)."""
    g_target = Fr(float(np.float32(np.float32(3.140625) / np.float32(2688.0))))
    blocks = coverage_blocks(g_target)
    # a block holding amax itself (its q rounds to 448)
    amax_bits = int(_bf16_bits(np.array([3.140625], np.float32))[0])
    blocks = np.vstack([blocks, np.array([[amax_bits] + [0] * 15], np.uint16)])
    assert max(bf16_value(int(b)) for b in blocks[:, 0]) == Fr(3.140625)
    codes, sf, g = o.quantize(blocks)
    assert Fr(float(g)) == f32(Fr(3.140625) / 2688) == g_target
    for i, blk in enumerate(blocks):
        sb, want = derive(blk, g_target)
        got = [(int(codes[i, j // 2]) >> (4 * (j % 2))) & 0xF for j in range(16)]
        assert int(sf[i, 0]) == sb and got == want, i
    assert int(sf[-1, 0]) == 126 and (int(codes[-1, 0]) & 0xF) == 7


def test_order_slips_are_detected_and_the_oracle_follows_r1():
    rng = np.random.default_rng(20251203)
    cases = discriminating_cases(rng)
    for slip in SLIPS:
        differs = agrees = 0
        for g, sb, xbits in cases[slip]:
            blk = block_for_case(g, sb, xbits)
            if blk is None:
                continue
            r1 = derive(blk, Fr(g))
            assert oracle_block_codes(blk, g) == r1, (slip, g, sb, xbits)
            agrees += 1
            if derive(blk, Fr(g), slip=slip) != r1:
                differs += 1
        # the pin has teeth: each slip changes the result on some of these inputs
        assert differs >= 5, (slip, differs, agrees)


def test_exact_helpers_against_fixed_points():
    """The exact helpers themselves, on values fixed by the formats."""
    assert [e2m1_code(Fr(v)) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)] == list(range(8))
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5: 6}
    assert all(e2m1_code(Fr(k)) == v for k, v in ties.items())
    assert e2m1_code(Fr(100)) == 7
    assert e4m3_value(126) == 448 and e4m3_value(1) == Fr(1, 512) and e4m3_value(8) == Fr(1, 64)
    assert all(e4m3_code(e4m3_value(c)) == c for c in range(127))
    assert e4m3_code(Fr(1000)) == 126
    assert f32(Fr(1, 3)) == Fr(float(np.float32(1 / 3)))
    assert f32(Fr(1) + Fr(1, 2 ** 24)) == 1          # tie to even
    assert f32(Fr(1) + Fr(3, 2 ** 24)) == 1 + Fr(1, 2 ** 22)
