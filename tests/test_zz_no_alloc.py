"""nvfp4_quantize_noalloc: the quantize entry point for callers that cannot
allocate device memory (a plugin hook that only receives its input and output
pointers, or a statically planned memory layout with no slot for scratch).

Its scratch (the per-part amax words of the dynamic global scale) is an array
inside the library instead of a caller workspace.  These tests call it through
the C ABI and check its output against nvfp4_quantize's -- bit for bit, the
tolerance of every packing test -- on two calls in a row with different data
(the array keeps the previous call's contents), and that an oversized request
is rejected before any device work.  The file sorts last so that a run which
stops at the first failure has already run every other test."""
import ctypes as C

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from nvfp4_block_scaled_06_gb300._binding import (ERR_WORKSPACE, PACK_BOTH, SF_SWIZZLED,
                                                  QuantArgs)
from synth import make_case

pytestmark = pytest.mark.gpu


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def noalloc_quantize(lib, x):
    """Fill the C struct by hand (no workspace) and call the new entry point."""
    B, R, Cc = x.shape
    out = dict(
        codes_row=torch.empty((B, R, Cc // 2), dtype=torch.uint8, device="cuda"),
        sf_row=torch.empty((B, lib.nvfp4_sf_bytes(R, Cc, SF_SWIZZLED)), dtype=torch.uint8, device="cuda"),
        codes_col=torch.empty((B, Cc, R // 2), dtype=torch.uint8, device="cuda"),
        sf_col=torch.empty((B, lib.nvfp4_sf_bytes(Cc, R, SF_SWIZZLED)), dtype=torch.uint8, device="cuda"),
        global_scale=torch.empty(B, dtype=torch.float32, device="cuda"))
    a = QuantArgs(src=x.data_ptr(), batch=B, rows=R, cols=Cc, ld=x.stride(1),
                  batch_stride=x.stride(0), pack=PACK_BOTH, sf_layout=SF_SWIZZLED,
                  global_scale_out=out["global_scale"].data_ptr(),
                  codes_row=out["codes_row"].data_ptr(), sf_row=out["sf_row"].data_ptr(),
                  codes_col=out["codes_col"].data_ptr(), sf_col=out["sf_col"].data_ptr())
    st = lib.nvfp4_quantize_noalloc(C.byref(a), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.nvfp4_status_string(st)
    return out


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    lib = nv.load()
    for seed in (0, 1):                  # two calls in a row, different data
        w = make_case("quantize", E=3, N=256, K=384, seed=seed)["w"]
        x = dev(w)
        got = noalloc_quantize(lib, x)
        want = nv.nvfp4_quantize(x, pack="both", sf_layout="swizzled")
        torch.cuda.synchronize()
        for k in ("codes_row", "sf_row", "codes_col", "sf_col", "global_scale"):
            assert torch.equal(got[k], want[k]), (seed, k)


def test_noalloc_rejects_oversized_scratch_request():
    lib = nv.load()
    # 33 matrices of >= 512 rows need 33 * 512 words > the 16384 available
    a = QuantArgs(src=4096, batch=33, rows=512, cols=64, ld=64, batch_stride=512 * 64,
                  pack=1, sf_layout=1, global_scale_out=4096, codes_row=4096, sf_row=4096)
    assert lib.nvfp4_quantize_noalloc(C.byref(a), None) == ERR_WORKSPACE
