"""Shared helpers of the GPU parity tests (host-side comparison only)."""
import numpy as np
import torch

from oracle import nvfp4_oracle as o


def dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bf16 tensor (same bytes)."""
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """CUDA bf16 tensor -> uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().astype(np.uint8)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got).reshape(-1)
    want = np.asarray(want).reshape(-1)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{what}: {bad.size} mismatches, first at {bad[:8]}: got {got[bad[:8]]} want {want[bad[:8]]}"


def assert_gemm_close(y_gpu: torch.Tensor, y_or: np.ndarray, S: np.ndarray, lora_term=None,
                      what="gemm"):
    """fp32 output: |Y - Y_or| <= 2e-5 S (+ LoRA bf16 term).
    bf16 output: |Y - bf16(Y_or)| <= ulp_bf16(max(|Y_or|, 2e-5 S)) (+ LoRA term)."""
    y = y_gpu.detach().float().cpu().numpy().astype(np.float64)
    extra = 0.0 if lora_term is None else lora_term
    if y_gpu.dtype == torch.float32:
        err = np.abs(y - y_or)
        tol = 2e-5 * S + extra
    else:
        ref = o.round_fp64_to_bf16(y_or)
        err = np.abs(y - ref)
        tol = o.bf16_ulp(np.maximum(np.abs(y_or), 2e-5 * S)) + extra
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (
        f"{what}: {len(bad)} of {err.size} outside tolerance; first {bad[:4].tolist()} "
        f"err {err[tuple(bad[0])]:.4g} tol {tol[tuple(bad[0])]:.4g} y {y[tuple(bad[0])]:.6g} "
        f"ref {y_or[tuple(bad[0])]:.6g}; max err/tol {np.max(err / np.maximum(tol, 1e-300)):.3g}")
    return float(np.max(err / np.maximum(tol, 1e-300)))


def lora_bf16_term(x_bits, a_bits, b_bits, alpha):
    """2^-8 (alpha/r) sum_j |T_mj| |B_nj|: the bound of rounding the scaled T to bf16."""
    _, t = o.lora_delta_fp64(x_bits, a_bits, b_bits, alpha)
    b = o.bf16_to_f32(b_bits).astype(np.float64)
    return 2.0 ** -8 * (alpha / a_bits.shape[0]) * (np.abs(t) @ np.abs(b).T)
