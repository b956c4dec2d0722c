"""NVFP4 W4A4 linear layer for sm_103a (GB300): Python binding of libnvfp4.

The functions here carry the names of the C entry points in include/nvfp4.h
and only marshal arguments: outputs and workspaces are allocated with torch on
the input's device, pointers go into the C argument structs, and the library
launches every kernel on the current (or given) torch stream.  A missing
library raises; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes as C

import torch

from ._binding import (DGRAD_DEQUANT_BF16, DGRAD_FP4_COLPACK, EXPORTS, DequantArgs, DgradArgs,
                       GemmArgs, GroupedArgs, LoraArgs, MoeDownArgs, NVFP4Error, OUT_BF16, OUT_FP32,
                       PACK_BOTH, PACK_COL, PACK_ROW, QuantArgs, SF_LINEAR, SF_SWIZZLED, WgradArgs,
                       check, load)

__all__ = [
    "load", "NVFP4Error", "nvfp4_quantize", "nvfp4_gemm", "nvfp4_grouped_gemm",
    "nvfp4_lora_epilogue", "nvfp4_codes_bytes", "nvfp4_sf_bytes", "read_device_status",
    "set_wait_timeout_ns", "Prepared", "prepare_gemm", "prepare_quantize", "prepare_grouped",
    "SF_LINEAR", "SF_SWIZZLED", "PACK_ROW", "PACK_COL", "PACK_BOTH", "EXPORTS",
    "nvfp4_dequantize", "nvfp4_dgrad", "prepare_dgrad", "nvfp4_wgrad", "prepare_wgrad",
    "nvfp4_moe_down_combine", "prepare_moe_down",
]

_PACK = {"row": PACK_ROW, "col": PACK_COL, "both": PACK_BOTH}
_SF = {"linear": SF_LINEAR, "swizzled": SF_SWIZZLED}


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ws(nbytes: int, device) -> torch.Tensor:
    # zero-filled: the first 4 bytes are the device status word
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def nvfp4_codes_bytes(rows: int, cols: int) -> int:
    return int(load().nvfp4_codes_bytes(rows, cols))


def nvfp4_sf_bytes(rows: int, cols: int, sf_layout: str = "swizzled") -> int:
    return int(load().nvfp4_sf_bytes(rows, cols, _SF[sf_layout]))


def set_wait_timeout_ns(ns: int) -> int:
    return int(load().nvfp4_set_wait_timeout_ns(int(ns)))


def read_device_status(workspace, stream=None) -> int:
    """Status word of a workspace (synchronizes the stream, clears the word);
    workspace=None reads the workspace-free quantize call's own status word."""
    return int(load().nvfp4_read_device_status(_p(workspace), _stream(stream)))


class Prepared:
    """A filled argument struct and its C function: call() re-launches it.

    Holds references to every tensor the struct points to."""

    def __init__(self, fn, args, keep, where):
        self.fn, self.args, self.keep, self.where = fn, args, keep, where
        self._ref = C.byref(args)

    def __call__(self, stream=None):
        check(self.fn(self._ref, _stream(stream)), self.where)


# ----------------------------------------------------------------- quantize --

def prepare_quantize(src: torch.Tensor, pack: str = "row", sf_layout: str = "swizzled",
                     global_scale: torch.Tensor | None = None) -> tuple[Prepared, dict]:
    lib = load()
    if src.dtype != torch.bfloat16 or not src.is_cuda:
        raise TypeError("src must be a CUDA bf16 tensor")
    batched = src.dim() == 3
    s3 = src if batched else src.unsqueeze(0)
    B, R, Cc = s3.shape
    if s3.stride(2) != 1:
        raise ValueError("src must have unit stride along columns")
    dev = src.device
    pk, sl = _PACK[pack], _SF[sf_layout]
    out = {}
    if pk & PACK_ROW:
        out["codes_row"] = torch.empty((B, R, Cc // 2), dtype=torch.uint8, device=dev)
        out["sf_row"] = torch.empty((B, lib.nvfp4_sf_bytes(R, Cc, sl)), dtype=torch.uint8, device=dev)
    if pk & PACK_COL:
        out["codes_col"] = torch.empty((B, Cc, R // 2), dtype=torch.uint8, device=dev)
        out["sf_col"] = torch.empty((B, lib.nvfp4_sf_bytes(Cc, R, sl)), dtype=torch.uint8, device=dev)
    gout = torch.empty(B, dtype=torch.float32, device=dev)
    out["global_scale"] = global_scale if global_scale is not None else gout
    a = QuantArgs(src=s3.data_ptr(), batch=B, rows=R, cols=Cc, ld=s3.stride(1),
                  batch_stride=s3.stride(0), pack=pk, sf_layout=sl,
                  global_scale_in=None if global_scale is None else global_scale.data_ptr(),
                  global_scale_out=gout.data_ptr())
    for k in ("codes_row", "sf_row", "codes_col", "sf_col"):
        if k in out:
            setattr(a, k, out[k].data_ptr())
    ws = _ws(lib.nvfp4_quantize_workspace_bytes(C.byref(a)), dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    out["workspace"] = ws
    if not batched:
        out = {k: (v[0] if k in ("codes_row", "sf_row", "codes_col", "sf_col") else v)
               for k, v in out.items()}
    return Prepared(lib.nvfp4_quantize, a, (src, s3, out, gout, global_scale), "nvfp4_quantize"), out


def nvfp4_quantize(src, pack="row", sf_layout="swizzled", global_scale=None, stream=None) -> dict:
    """bf16 [rows, cols] (or [batch, rows, cols]) -> NVFP4 packings.

    Returns codes_row/sf_row and/or codes_col/sf_col (uint8) and global_scale
    (fp32 [batch])."""
    call, out = prepare_quantize(src, pack, sf_layout, global_scale)
    call(stream)
    return out


# --------------------------------------------------------------------- GEMM --

def prepare_gemm(b_codes, b_sf, b_global_scale, N: int, K: int, *, a_codes=None, a_sf=None,
                 a_global_scale=None, a_bf16=None, M: int | None = None, out_dtype=torch.bfloat16,
                 lora=None, out=None) -> tuple[Prepared, torch.Tensor]:
    """See nvfp4_gemm; returns (Prepared call, output tensor)."""
    lib = load()
    if M is None:
        M = a_bf16.shape[0] if a_bf16 is not None else a_codes.shape[0]
    dev = b_codes.device
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype, device=dev)
    a = GemmArgs(M=M, N=N, K=K, b_codes=b_codes.data_ptr(), b_sf=b_sf.data_ptr(),
                 b_global_scale=b_global_scale.data_ptr(),
                 out_dtype=OUT_FP32 if out.dtype == torch.float32 else OUT_BF16,
                 d=out.data_ptr(), ldd=out.stride(0))
    keep = [b_codes, b_sf, b_global_scale, out, a_codes, a_sf, a_global_scale, a_bf16]
    if a_bf16 is not None:
        a.a_bf16, a.lda = a_bf16.data_ptr(), a_bf16.stride(0)
        if a_global_scale is not None:
            a.a_global_scale = a_global_scale.data_ptr()
    else:
        a.a_codes, a.a_sf = a_codes.data_ptr(), a_sf.data_ptr()
        a.a_global_scale = a_global_scale.data_ptr()
    if lora is not None:
        x = lora.get("x", a_bf16)
        a.lora_x = lora["x"].data_ptr() if "x" in lora else None
        if a_bf16 is None or "x" in lora:
            a.lda = x.stride(0)
        a.lora_a, a.lora_b = lora["a"].data_ptr(), lora["b"].data_ptr()
        a.rank, a.alpha = lora["a"].shape[0], float(lora["alpha"])
        keep += [x, lora["a"], lora["b"]]
    ws = _ws(lib.nvfp4_gemm_workspace_bytes(C.byref(a)), dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    keep.append(ws)
    call = Prepared(lib.nvfp4_gemm, a, keep, "nvfp4_gemm")
    call.workspace = ws
    return call, out


def nvfp4_gemm(b_codes, b_sf, b_global_scale, N, K, *, a_codes=None, a_sf=None,
               a_global_scale=None, a_bf16=None, out_dtype=torch.bfloat16, lora=None,
               out=None, stream=None) -> torch.Tensor:
    """D = W4A4(A, B) [+ (alpha/r) (X A_l^T) B_l^T].

    A: packed (a_codes [M,K/2], a_sf swizzled, a_global_scale [1]) or bf16
    a_bf16 [M,K] quantized in the call (a_global_scale = static scale, or None
    = dynamic).  B: b_codes [N,K/2], b_sf swizzled, b_global_scale [1].
    lora: dict(a=[r,K] bf16, b=[N,r] bf16, alpha=float[, x=[M,K] bf16])."""
    call, out = prepare_gemm(b_codes, b_sf, b_global_scale, N, K, a_codes=a_codes, a_sf=a_sf,
                             a_global_scale=a_global_scale, a_bf16=a_bf16,
                             out_dtype=out_dtype, lora=lora, out=out)
    call(stream)
    return out


# ------------------------------------------------------------------ grouped --

def prepare_grouped(expert_ids, x_bf16, w_codes, w_sf, w_global_scale, N: int, K: int,
                    num_experts: int, x_global_scale=None, lora=None, *, x_packed=None,
                    routing=None, top_k: int | None = None, out_dtype=torch.bfloat16):
    """Routing: expert_ids [T, k], or routing = (offsets [E+1], perm [T*k]) with
    top_k.  Activations: x_bf16 [T, K], or x_packed = (codes [T, K/2], linear sf
    [T, K/16]) with x_global_scale (x_bf16 still needed for a LoRA)."""
    lib = load()
    dev = w_codes.device
    if expert_ids is not None:
        T, topk = expert_ids.shape
    else:
        if routing is None or top_k is None:
            raise ValueError("routing=(offsets, perm) and top_k are needed without expert_ids")
        topk = int(top_k)
        T = routing[1].numel() // topk
    P = T * topk
    d = torch.empty((P, N), dtype=out_dtype, device=dev)
    offs = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(P, dtype=torch.int32, device=dev) if routing is None else routing[1]
    a = GroupedArgs(num_tokens=T, top_k=topk, num_experts=num_experts, N=N, K=K,
                    x_bf16=None if x_bf16 is None else x_bf16.data_ptr(),
                    x_global_scale=None if x_global_scale is None else x_global_scale.data_ptr(),
                    w_codes=w_codes.data_ptr(), w_sf=w_sf.data_ptr(),
                    w_global_scale=w_global_scale.data_ptr(), d=d.data_ptr(),
                    expert_offsets_out=offs.data_ptr(),
                    out_dtype=OUT_FP32 if out_dtype == torch.float32 else OUT_BF16)
    keep = [expert_ids, x_bf16, w_codes, w_sf, w_global_scale, x_global_scale, d, perm, offs]
    if routing is None:
        a.expert_ids, a.perm_out = expert_ids.data_ptr(), perm.data_ptr()
    else:
        a.offsets_in, a.perm_in = routing[0].data_ptr(), routing[1].data_ptr()
        keep += list(routing)
    if x_packed is not None:
        a.x_codes, a.x_sf = x_packed[0].data_ptr(), x_packed[1].data_ptr()
        keep += list(x_packed)
    if lora is not None:
        a.lora_a, a.lora_b = lora["a"].data_ptr(), lora["b"].data_ptr()
        a.rank, a.alpha = lora["a"].shape[1], float(lora["alpha"])
        keep += [lora["a"], lora["b"]]
    ws = _ws(lib.nvfp4_grouped_workspace_bytes(C.byref(a)), dev)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    keep.append(ws)
    call = Prepared(lib.nvfp4_grouped_gemm, a, keep, "nvfp4_grouped_gemm")
    call.workspace = ws
    return call, (d, perm, offs)


def nvfp4_grouped_gemm(expert_ids, x_bf16, w_codes, w_sf, w_global_scale, N, K, num_experts,
                       x_global_scale=None, lora=None, stream=None, **forms):
    """Routed-expert W4A4 GEMM.  Returns (d [T*k, N] grouped by expert,
    perm [T*k] grouped row -> pair index, offsets [E+1]).  `forms` takes
    prepare_grouped's keyword inputs (x_packed, routing + top_k, out_dtype)."""
    call, res = prepare_grouped(expert_ids, x_bf16, w_codes, w_sf, w_global_scale, N, K,
                                num_experts, x_global_scale, lora, **forms)
    call(stream)
    return res


# --------------------------------------------------------------------- LoRA --

def nvfp4_lora_epilogue(y, x, lora_a, lora_b, alpha: float, want_norm: bool = False,
                        stream=None):
    """In place: y += (alpha/r) (x lora_a^T) lora_b^T.  Returns the sum of the
    squared delta (fp32 tensor [1]) when want_norm, else None."""
    lib = load()
    M, K = x.shape
    N = y.shape[1]
    norm = torch.zeros(1, dtype=torch.float32, device=y.device) if want_norm else None
    a = LoraArgs(M=M, N=N, K=K, x=x.data_ptr(), ldx=x.stride(0), lora_a=lora_a.data_ptr(),
                 lora_b=lora_b.data_ptr(), rank=lora_a.shape[0], alpha=float(alpha),
                 y_dtype=OUT_FP32 if y.dtype == torch.float32 else OUT_BF16, y=y.data_ptr(),
                 ldy=y.stride(0), delta_sq_norm_out=None if norm is None else norm.data_ptr())
    ws = _ws(lib.nvfp4_lora_workspace_bytes(C.byref(a)), y.device)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    check(lib.nvfp4_lora_epilogue(C.byref(a), _stream(stream)), "nvfp4_lora_epilogue")
    return norm


# ----------------------------------------------------------------- backward --

def nvfp4_dequantize(codes, sf, global_scale, rows: int, cols: int, transpose: bool = False,
                     sf_layout: str = "swizzled", out=None, stream=None) -> torch.Tensor:
    """NVFP4 [rows, cols] -> bf16 [rows, cols] (or [cols, rows] with transpose)."""
    lib = load()
    if out is None:
        shape = (cols, rows) if transpose else (rows, cols)
        out = torch.empty(shape, dtype=torch.bfloat16, device=codes.device)
    a = DequantArgs(codes=codes.data_ptr(), sf=sf.data_ptr(), sf_layout=_SF[sf_layout],
                    global_scale=global_scale.data_ptr(), rows=rows, cols=cols,
                    transpose=1 if transpose else 0, out=out.data_ptr(), ldo=out.stride(0))
    check(lib.nvfp4_dequantize(C.byref(a), _stream(stream)), "nvfp4_dequantize")
    return out


def prepare_dgrad(dy, N: int, K: int, *, w=None, wcol=None, dy_global_scale=None,
                  out_dtype=torch.bfloat16, out=None) -> tuple[Prepared, torch.Tensor]:
    """dX [M, K] = dY [M, N] W [N, K].  w = (codes [N, K/2], swizzled sf, g): the
    rowwise packing, dequantized to bf16 (transposed) for a bf16 GEMM; or
    wcol = (codes [K, N/2], swizzled sf, g): the column packing, for the W4A4
    GEMM with dY quantized in the call."""
    lib = load()
    M = dy.shape[0]
    if out is None:
        out = torch.empty((M, K), dtype=out_dtype, device=dy.device)
    a = DgradArgs(M=M, N=N, K=K, dy=dy.data_ptr(), lddy=dy.stride(0),
                  out_dtype=OUT_FP32 if out.dtype == torch.float32 else OUT_BF16,
                  dx=out.data_ptr(), lddx=out.stride(0))
    keep = [dy, out, dy_global_scale]
    if w is not None:
        a.mode = DGRAD_DEQUANT_BF16
        a.w_codes, a.w_sf, a.w_global_scale = w[0].data_ptr(), w[1].data_ptr(), w[2].data_ptr()
        keep += list(w)
    else:
        a.mode = DGRAD_FP4_COLPACK
        a.wcol_codes, a.wcol_sf = wcol[0].data_ptr(), wcol[1].data_ptr()
        a.w_global_scale = wcol[2].data_ptr()
        keep += list(wcol)
    if dy_global_scale is not None:
        a.dy_global_scale = dy_global_scale.data_ptr()
    ws = _ws(lib.nvfp4_dgrad_workspace_bytes(C.byref(a)), dy.device)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    keep.append(ws)
    call = Prepared(lib.nvfp4_dgrad, a, keep, "nvfp4_dgrad")
    call.workspace = ws
    return call, out


def nvfp4_dgrad(dy, N: int, K: int, *, w=None, wcol=None, dy_global_scale=None,
                out_dtype=torch.bfloat16, out=None, stream=None) -> torch.Tensor:
    """See prepare_dgrad."""
    call, out = prepare_dgrad(dy, N, K, w=w, wcol=wcol, dy_global_scale=dy_global_scale,
                              out_dtype=out_dtype, out=out)
    call(stream)
    return out


def prepare_wgrad(dy, x, *, dy_global_scale=None, x_global_scale=None, out_dtype=torch.bfloat16,
                  out=None) -> tuple[Prepared, torch.Tensor]:
    """dW [N, K] = dY[M, N]^T X[M, K] on the FP4 datapath (both operands packed
    along M in the call)."""
    lib = load()
    M, N = dy.shape
    K = x.shape[1]
    if out is None:
        out = torch.empty((N, K), dtype=out_dtype, device=dy.device)
    a = WgradArgs(M=M, N=N, K=K, dy=dy.data_ptr(), lddy=dy.stride(0), x=x.data_ptr(),
                  ldx=x.stride(0), out_dtype=OUT_FP32 if out.dtype == torch.float32 else OUT_BF16,
                  dw=out.data_ptr(), lddw=out.stride(0))
    if dy_global_scale is not None:
        a.dy_global_scale = dy_global_scale.data_ptr()
    if x_global_scale is not None:
        a.x_global_scale = x_global_scale.data_ptr()
    keep = [dy, x, out, dy_global_scale, x_global_scale]
    ws = _ws(lib.nvfp4_wgrad_workspace_bytes(C.byref(a)), dy.device)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    keep.append(ws)
    call = Prepared(lib.nvfp4_wgrad, a, keep, "nvfp4_wgrad")
    call.workspace = ws
    return call, out


def nvfp4_wgrad(dy, x, *, dy_global_scale=None, x_global_scale=None, out_dtype=torch.bfloat16,
                out=None, stream=None) -> torch.Tensor:
    """See prepare_wgrad."""
    call, out = prepare_wgrad(dy, x, dy_global_scale=dy_global_scale,
                              x_global_scale=x_global_scale, out_dtype=out_dtype, out=out)
    call(stream)
    return out


# ------------------------------------------------------------ MoE down-proj --

def prepare_moe_down(h, perm, expert_offsets, route_weights, w_codes, w_sf, w_global_scale,
                     N: int, K: int, num_experts: int, h_global_scale=None, lora=None,
                     out=None) -> tuple[Prepared, torch.Tensor]:
    """y [T, N] = sum_j route_weights[t, j] * W4A4(h[grouped row of (t, j)], W2_e).

    h: bf16 [T*k, K] in the expert-grouped order of nvfp4_grouped_gemm's output;
    perm / expert_offsets: that call's permutation and offsets; route_weights
    fp32 [T, k]; W2 stacked codes [E, N, K/2], swizzled scales, [E] global scales."""
    lib = load()
    T, k = route_weights.shape
    if out is None:
        out = torch.empty((T, N), dtype=torch.bfloat16, device=h.device)
    a = MoeDownArgs(num_tokens=T, top_k=k, num_experts=num_experts, N=N, K=K, h=h.data_ptr(),
                    perm=perm.data_ptr(), expert_offsets=expert_offsets.data_ptr(),
                    route_weights=route_weights.data_ptr(),
                    h_global_scale=None if h_global_scale is None else h_global_scale.data_ptr(),
                    w_codes=w_codes.data_ptr(), w_sf=w_sf.data_ptr(),
                    w_global_scale=w_global_scale.data_ptr(), y=out.data_ptr())
    keep = [h, perm, expert_offsets, route_weights, h_global_scale, w_codes, w_sf, w_global_scale,
            out]
    if lora is not None:
        a.lora_a, a.lora_b = lora["a"].data_ptr(), lora["b"].data_ptr()
        a.rank, a.alpha = lora["a"].shape[1], float(lora["alpha"])
        keep += [lora["a"], lora["b"]]
    ws = _ws(lib.nvfp4_moe_down_workspace_bytes(C.byref(a)), h.device)
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    keep.append(ws)
    call = Prepared(lib.nvfp4_moe_down_combine, a, keep, "nvfp4_moe_down_combine")
    call.workspace = ws
    return call, out


def nvfp4_moe_down_combine(h, perm, expert_offsets, route_weights, w_codes, w_sf, w_global_scale,
                           N: int, K: int, num_experts: int, h_global_scale=None, lora=None,
                           out=None, stream=None) -> torch.Tensor:
    """See prepare_moe_down."""
    call, out = prepare_moe_down(h, perm, expert_offsets, route_weights, w_codes, w_sf,
                                 w_global_scale, N, K, num_experts, h_global_scale, lora, out)
    call(stream)
    return out
