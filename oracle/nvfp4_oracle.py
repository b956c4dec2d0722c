"""NVFP4 oracle: a plain, slow, obviously correct CPU statement of the method.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may.  It shares no code, tables or constants with the CUDA
library: its conversion tables are enumerated here from the format
definitions and its roundings are nearest-value searches over those tables.

Sources (web pages, cited by title and section):

* [P1] "Getting GLM-5.2 NVFP4 Post-Training off the ground" -- sections
  "Going deeper: why a 4-bit weight needs two copies", "Why can't we just
  transpose the one copy?", "TN, NT, and what actually binds", "The bottom
  line", "For a frozen QLoRA base", "A model no kernel wanted to serve", TL;DR.
* [P2] "GLM-5.2-NVFP4" model card -- "Quantization recipe".
* [P3] "vroomfondel/glm-5.2-reap-504B-v2-W4A4" model card -- "How it was
  produced (data-free, no re-calibration)", "Kernel choice: cutlass W4A4".

What the pages fix: E2M1 values with one FP8 E4M3 scale per 16 consecutive
elements along the contraction axis and one FP32 per-tensor global scale
(P1 "Going deeper"; P2 "Quantization recipe"); the global scale rule
weight_scale_2 = amax / (6*448) and "linear block scales" (P3 "How it was
produced"); blocks are 1-D runs along the contraction axis, so the transposed
operand is a separate quantization of the high-precision values (P1 "Why
can't we just transpose"); values bit-packed two per byte (same section); a
static per-tensor input_scale for the W4A4 path (P3 "How it was produced");
a bf16 LoRA of rank 64 over the frozen 4-bit base (P1 TL;DR).

Readings where the pages are silent (each listed in the design notes):

R1  Scale arithmetic is IEEE fp32, one rounding per operation, in this order:
    g = amax / 2688;  q = bamax / (6*g);  sb = E4M3(q);  s_dec = sb*g;
    s_enc = 1/s_dec;  v = x * s_enc;  code = E2M1(v).
R2  E4M3 and E2M1 conversions round to nearest, ties to the even code, and
    saturate to the largest finite value (448 and 6).  E4M3 subnormals
    (down to 2^-9) are used.
R3  amax == 0 gives g = 0; g == 0 or q rounding to zero gives sb = 0, and a
    block with sb == 0 stores every code as +0.  s_enc larger than the
    largest fp32 value (s_dec == 0 or tiny) is clamped to that value.
R4  The code's sign bit is the sign bit of x (so -0.1 encodes as 0x8).
R5  Packing: element 2j in the low nibble, 2j+1 in the high nibble of byte j.
R6  "Linear" scales are [rows, cols/16] row-major.  The "swizzled" layout
    (rows padded to 128, scale columns padded to 4, 512-byte atoms of
    128x4) follows the public tensor-core block-scaling layout; the pages
    only say the values are "swizzled for the tensor-core tile".  Padding is 0.
R7  The product uses the unquantized bf16 X for the LoRA branch:
    Y = dq(Xq) dq(Wq)^T + (alpha/r) (X A^T) B^T, with A stored [r, K] and B
    stored [N, r] (the Linear-weight layout); fp64 throughout.
R8  Grouped rows are ordered by expert id, then by (token, slot) index.
R9  Dequantization to bf16 (the backward's rebuilt weight, [P1] "Why can't
    we just transpose the one copy?" / "For a frozen QLoRA base") is IEEE
    fp32 in the quantizer's decode order, s_dec = sb*g then v = E2M1*s_dec,
    rounded once more to bf16 (nearest, ties to even).  The Dgrad product
    dX = dY W contracts over N with fp32 accumulation.

R10 The routed down-projection takes its input already in the grouped order
    of the up-projection's output, quantized once with one tensor-wide g;
    the combine weights each expert output by its gate weight
    (y[t] = sum_j w[t,j] D[t,j]; [P3] "How it was produced": REAP saliency
    gate_weight x ||expert_output||), summed over the slots in order.

Parity of the swizzled layout and nibble order is pinned only through the
hardware (the tensor core consumes them); everything else is pinned by the
tests in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "E2M1_MAGNITUDES", "E4M3_VALUES", "GLOBAL_DIVISOR", "bf16_to_f32",
    "e2m1_encode_magnitude", "e4m3_encode", "global_scale", "quantize",
    "quantize_colwise", "dequantize", "sf_swizzle", "sf_unswizzle",
    "gemm_fp64", "lora_delta_fp64", "linear_fp64", "error_scale",
    "round_fp64_to_bf16", "bf16_ulp", "group_rows", "grouped_linear_rows",
    "dequantize_bf16", "f32_to_bf16_rne", "grouped_input_rows", "moe_combine",
]

# ---------------------------------------------------------------------------
# Format tables (enumerated from the format definitions).
# ---------------------------------------------------------------------------

#: E2M1 magnitudes for codes 0..7 (1 sign bit | 2 exponent bits | 1 mantissa
#: bit, bias 1, no inf/nan).  Largest value 6: the "6" in 6*448 [P3].
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def _e4m3_table() -> np.ndarray:
    """Values of E4M3 codes 0..126 (sign 0): 4 exponent bits (bias 7), 3 mantissa
    bits, subnormals for exponent field 0; code 127 (0x7F) is NaN and excluded.
    Largest finite value 448: the "448" in 6*448 [P3]."""
    vals = []
    for code in range(127):
        e, m = code >> 3, code & 7
        if e == 0:
            vals.append(m * 2.0 ** -9)
        else:
            vals.append((1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


E4M3_VALUES = _e4m3_table()

#: 6 * 448: the largest E2M1 magnitude times the largest E4M3 scale [P3].
GLOBAL_DIVISOR = np.float32(2688.0)

_F32 = np.float32
_FLT_MAX = np.float32(np.finfo(np.float32).max)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32, exact."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _nearest_code(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the table value nearest to ``mag`` (>= 0), ties to the even
    index, values above the table's last entry saturating to it (R2).

    ``table`` is ascending and its index is the code, so the even index is the
    even mantissa: this is round-to-nearest-even on the format's own grid.
    """
    mag = np.minimum(np.asarray(mag, dtype=np.float64), table[-1])
    hi = np.searchsorted(table, mag, side="left")
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - table[lo]
    d_hi = table[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    return np.where(pick_hi, hi, lo).astype(np.uint8)


def e2m1_encode_magnitude(v_abs: np.ndarray) -> np.ndarray:
    """|v| -> E2M1 magnitude code 0..7 (R2)."""
    return _nearest_code(v_abs, E2M1_MAGNITUDES)


def e4m3_encode(q: np.ndarray) -> np.ndarray:
    """q >= 0 -> E4M3 code 0..126 (R2)."""
    return _nearest_code(q, E4M3_VALUES)


# ---------------------------------------------------------------------------
# Quantization [P3 "How it was produced"; P2 "Quantization recipe";
# P1 "Going deeper" and "Why can't we just transpose"].
# ---------------------------------------------------------------------------

def global_scale(x_bits: np.ndarray) -> np.float32:
    """weight_scale_2 = amax / (6*448) in fp32 [P3]; amax == 0 gives 0 (R3)."""
    amax = np.max(np.abs(bf16_to_f32(x_bits))) if x_bits.size else _F32(0)
    return _F32(_F32(amax) / GLOBAL_DIVISOR)


def quantize(x_bits: np.ndarray, g: np.float32 | None = None):
    """Quantize a bf16 matrix [R, C] to NVFP4 with 1x16 blocks along C.

    Returns (codes uint8 [R, C/2] packed per R5, sf uint8 [R, C/16] linear E4M3
    codes, g float32).  ``g`` given = static global scale (the W4A4 input_scale
    of P3); ``g`` None = dynamic, from the tensor's amax.
    """
    x = bf16_to_f32(x_bits)
    R, C = x.shape
    assert C % 16 == 0, "blocks of 16 along the contraction axis"
    g = global_scale(x_bits) if g is None else _F32(g)
    blocks = x.reshape(R, C // 16, 16)
    bamax = np.max(np.abs(blocks), axis=2) if C else np.zeros((R, 0), np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        t = _F32(_F32(6.0) * g)                          # R1
        q = (bamax / t).astype(np.float32)               # R1
        sb_code = e4m3_encode(np.nan_to_num(q, nan=0.0, posinf=np.inf))
        if g == 0:
            sb_code[:] = 0                               # R3
        sb = E4M3_VALUES[sb_code].astype(np.float32)
        s_dec = (sb * g).astype(np.float32)              # R1
        s_enc = (_F32(1.0) / s_dec).astype(np.float32)   # R1
        s_enc = np.minimum(s_enc, _FLT_MAX)              # R3
        v = (blocks * s_enc[:, :, None]).astype(np.float32)
    mag = e2m1_encode_magnitude(np.abs(v))
    sign = np.signbit(blocks).astype(np.uint8) << 3     # R4
    codes = (sign | mag).astype(np.uint8)
    codes[sb_code == 0] = 0                               # R3
    codes = codes.reshape(R, C)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)   # R5
    return packed, sb_code.astype(np.uint8), g


def quantize_colwise(w_bits: np.ndarray, g: np.float32 | None = None):
    """The columnwise (transposed) packing of W [N, K]: 16x1 blocks along N.

    This is the quantization of W^T [K, N], a separate quantization from the
    bf16 values with its own block scales [P1 "Why can't we just transpose" /
    "The bottom line"]; it shares the tensor's global scale.
    Returns (codes [K, N/2], sf [K, N/16], g).
    """
    g = global_scale(w_bits) if g is None else _F32(g)
    return quantize(np.ascontiguousarray(w_bits.T), g)


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    """[R, C/2] packed bytes -> [R, C] 4-bit codes (R5)."""
    R, H = packed.shape
    out = np.empty((R, 2 * H), dtype=np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out


def dequantize(packed: np.ndarray, sf: np.ndarray, g) -> np.ndarray:
    """x_hat = E2M1(code) * E4M3(sb) * g, exact in fp64."""
    codes = unpack_codes(packed)
    R, C = codes.shape
    mag = E2M1_MAGNITUDES[codes & 7]
    sgn = np.where(codes & 8, -1.0, 1.0)
    scale = E4M3_VALUES[sf.astype(np.int64)] * float(g)       # [R, C/16]
    elem = (sgn * mag).reshape(R, C // 16, 16)
    return (elem * scale[:, :, None]).reshape(R, C)


def f32_to_bf16_rne(v: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest, ties to even (finite
    inputs): add 0x7FFF plus the lowest kept bit, keep the top 16 bits."""
    u = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> 16) & 1
    return (((u + 0x7FFF + keep_lsb) >> 16) & 0xFFFF).astype(np.uint16)


def dequantize_bf16(packed: np.ndarray, sf: np.ndarray, g) -> np.ndarray:
    """R9: bf16 bit patterns of fl32(E2M1(code) * fl32(E4M3(sb) * g)).

    ``packed`` [R, C/2] codes (R5), ``sf`` [R, C/16] linear E4M3 codes."""
    codes = unpack_codes(packed)
    R, C = codes.shape
    mag = E2M1_MAGNITUDES[codes & 7].astype(np.float32)
    elem = np.where(codes & 8, -mag, mag).astype(np.float32)          # sign of code (R4)
    s_dec = (E4M3_VALUES[sf.astype(np.int64)].astype(np.float32) * _F32(g)).astype(np.float32)
    v = (elem.reshape(R, C // 16, 16) * s_dec[:, :, None]).astype(np.float32)
    return f32_to_bf16_rne(v.reshape(R, C))


# ---------------------------------------------------------------------------
# Swizzled block-scale layout (R6).
# ---------------------------------------------------------------------------

def sf_swizzled_shape(rows: int, sf_cols: int):
    return (rows + 127) // 128 * 128, (sf_cols + 3) // 4 * 4


def sf_swizzle(sf: np.ndarray) -> np.ndarray:
    """Linear scales [R, Cs] -> flat swizzled buffer (R6).

    Scale (r, c) lives in atom (r // 128, c // 4) at byte
    512 * (atom_row * (padCs // 4) + atom_col) + 16*(r % 32) + 4*((r % 128)//32) + c % 4.
    """
    R, Cs = sf.shape
    pR, pC = sf_swizzled_shape(R, Cs)
    out = np.zeros(pR * pC, dtype=np.uint8)
    r = np.arange(R)[:, None]
    c = np.arange(Cs)[None, :]
    off = (512 * ((r // 128) * (pC // 4) + c // 4) + 16 * (r % 32)
           + 4 * ((r % 128) // 32) + c % 4)
    out[off.ravel()] = sf.ravel()
    return out


def sf_unswizzle(buf: np.ndarray, rows: int, sf_cols: int) -> np.ndarray:
    pR, pC = sf_swizzled_shape(rows, sf_cols)
    r = np.arange(rows)[:, None]
    c = np.arange(sf_cols)[None, :]
    off = (512 * ((r // 128) * (pC // 4) + c // 4) + 16 * (r % 32)
           + 4 * ((r % 128) // 32) + c % 4)
    return np.asarray(buf).reshape(-1)[off]


# ---------------------------------------------------------------------------
# Products [P3 "Kernel choice" (scaled_fp4_mm: W4A4 product of the two
# quantized operands); P1 TL;DR and "A model no kernel wanted to serve"
# (bf16 LoRA over the frozen NVFP4 base, delta added to the base output)].
# ---------------------------------------------------------------------------

def gemm_fp64(a_hat: np.ndarray, b_hat: np.ndarray) -> np.ndarray:
    """Y[m, n] = sum_k a_hat[m, k] * b_hat[n, k] (both K-major), fp64."""
    return np.asarray(a_hat, np.float64) @ np.asarray(b_hat, np.float64).T


def lora_delta_fp64(x_bits, a_bits, b_bits, alpha: float):
    """(alpha/r) * (X A^T) B^T with X [M,K], A [r,K], B [N,r] bf16 (R7).

    Returns (delta [M,N], T [M,r]) in fp64."""
    x = bf16_to_f32(x_bits).astype(np.float64)
    a = bf16_to_f32(a_bits).astype(np.float64)
    b = bf16_to_f32(b_bits).astype(np.float64)
    r = a.shape[0]
    t = x @ a.T
    return (alpha / r) * (t @ b.T), t


def linear_fp64(xq, w_q, x_bits=None, lora=None):
    """W4A4 linear: dq(Xq) dq(Wq)^T [+ LoRA].

    ``xq`` and ``w_q`` are (codes, linear sf, g) triples from ``quantize``;
    ``lora`` = (a_bits, b_bits, alpha) applied to the bf16 ``x_bits``.
    """
    y = gemm_fp64(dequantize(*xq), dequantize(*w_q))
    if lora is not None:
        d, _ = lora_delta_fp64(x_bits, *lora)
        y = y + d
    return y


def error_scale(xq, w_q, x_bits=None, lora=None):
    """S = sum_k |x_hat_k w_hat_k| + (alpha/r) sum_j |T_j| |B_jn| per output.

    The per-element scale of the fp32 tolerance 2e-5*S; the LoRA term is the
    reading used when the adapter branch is present."""
    s = np.abs(dequantize(*xq)) @ np.abs(dequantize(*w_q)).T
    if lora is not None:
        a_bits, b_bits, alpha = lora
        _, t = lora_delta_fp64(x_bits, a_bits, b_bits, alpha)
        b = bf16_to_f32(b_bits).astype(np.float64)
        s = s + (alpha / a_bits.shape[0]) * (np.abs(t) @ np.abs(b).T)
    return s


# ---------------------------------------------------------------------------
# bf16 rounding of fp64 results (for comparing bf16 outputs).
# ---------------------------------------------------------------------------

def round_fp64_to_bf16(v: np.ndarray) -> np.ndarray:
    """Nearest bf16 value (8 significant bits, ties to even) of fp64 ``v``,
    returned as fp64.  Normal range only (|v| in [2^-126, 2^127])."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                 # v = m * 2^e, |m| in [0.5, 1)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (normal range)."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(v == 0, 2.0 ** -126, v))
    return np.ldexp(1.0, e - 8)


# ---------------------------------------------------------------------------
# Grouped MoE rows [P2 "GLM-5.2-NVFP4": 256 routed experts, 8 per token;
# P1 "A model no kernel wanted to serve": per-expert LoRA over the FP4 experts].
# ---------------------------------------------------------------------------

def group_rows(expert_ids: np.ndarray, num_experts: int):
    """Stable grouping of (token, slot) pairs by expert (R8).

    Returns (counts [E], offsets [E+1], perm [T*k]) where grouped row i is the
    flat pair index perm[i] = token*k + slot."""
    flat = np.asarray(expert_ids).reshape(-1).astype(np.int64)
    perm = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=num_experts)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    return counts, offsets, perm


def grouped_linear_rows(rows, x_bits, xq, w_codes, w_sf, w_g, perm, expert_ids,
                        topk, lora=None):
    """Oracle output for selected grouped rows.

    ``rows``: grouped row indices to evaluate.  ``xq`` = (codes, sf, g) of the
    whole X (one tensor-wide scale).  ``w_codes/w_sf/w_g`` index by expert.
    ``lora`` = (A [E,r,K], B [E,N,r], alpha).  Returns fp64 [len(rows), N] and
    the matching error scale S."""
    flat = np.asarray(expert_ids).reshape(-1)
    out, scale = [], []
    for i in rows:
        p = int(perm[i])
        t, e = p // topk, int(flat[p])
        xr = (xq[0][t:t + 1], xq[1][t:t + 1], xq[2])
        wr = (w_codes[e], w_sf[e], w_g[e])
        lo = None
        if lora is not None:
            lo = (lora[0][e], lora[1][e], lora[2])
        out.append(linear_fp64(xr, wr, x_bits[t:t + 1], lo)[0])
        scale.append(error_scale(xr, wr, x_bits[t:t + 1], lo)[0])
    return np.array(out), np.array(scale)


def grouped_input_rows(h_bits, hq, row_expert, w_codes, w_sf, w_g, lora=None):
    """Oracle output of every row of an input that is already in grouped order
    (the down-projection: row i of ``h`` meets expert ``row_expert[i]``).

    ``hq`` = (codes, sf, g) of the whole h (one tensor-wide scale).  Returns
    fp64 D [P, N] and its error scale S."""
    out, scale = [], []
    for i, e in enumerate(np.asarray(row_expert)):
        e = int(e)
        hr = (hq[0][i:i + 1], hq[1][i:i + 1], hq[2])
        wr = (w_codes[e], w_sf[e], w_g[e])
        lo = None if lora is None else (lora[0][e], lora[1][e], lora[2])
        out.append(linear_fp64(hr, wr, h_bits[i:i + 1], lo)[0])
        scale.append(error_scale(hr, wr, h_bits[i:i + 1], lo)[0])
    return np.array(out), np.array(scale)


def moe_combine(d_rows, perm, weights, topk):
    """y[t] = sum over slots j of w[t, j] * D[grouped row of pair t*topk + j]
    (the routed experts' outputs weighted by their gate weights), fp64.

    ``perm[i]`` is the pair index of grouped row i (R8)."""
    P = len(perm)
    inv = np.empty(P, dtype=np.int64)
    inv[np.asarray(perm, dtype=np.int64)] = np.arange(P)
    T = P // topk
    w = np.asarray(weights, dtype=np.float64).reshape(T, topk)
    y = np.zeros((T, d_rows.shape[1]))
    for j in range(topk):
        y += w[:, j:j + 1] * d_rows[inv[np.arange(T) * topk + j]]
    return y


def bytes_per_element() -> float:
    """4-bit code + one 8-bit scale per 16 elements = 4.5 bits (P1 "The 4-bit
    base that was actually using 8-bit memory": the per-16 scales on top of
    the 4-bit values)."""
    return 0.5 + 1.0 / 16.0


