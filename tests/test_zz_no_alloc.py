"""nvfp4_quantize_noalloc: the quantize entry point for callers that cannot
allocate device memory (a plugin hook that only receives its input and output
pointers, or a statically planned memory layout with no slot for scratch).

Its scratch (the per-part amax words of the dynamic global scale) and its
device status word live in an array inside the library instead of a caller
workspace.  These tests call it through the C ABI and check its output bit
for bit against nvfp4_quantize's and against the oracle, on two calls in a row
with different data (the array keeps the previous call's contents); that an
expired wait is reported through its own status word (never through the
ignored `workspace` argument) and that the next call recovers; and that an
oversized request is rejected before any device work.  The file sorts last so
that a run which stops at the first failure has already run every other
test."""
import ctypes as C

import numpy as np
import pytest
import torch

import nvfp4_block_scaled_06_gb300 as nv
from nvfp4_block_scaled_06_gb300._binding import (ERR_TIMEOUT, ERR_WORKSPACE, PACK_BOTH,
                                                  SF_SWIZZLED, QuantArgs)
from oracle import nvfp4_oracle as o
from synth import make_case

pytestmark = pytest.mark.gpu


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def noalloc_quantize(lib, x, workspace=None):
    """Fill the C struct by hand and call the new entry point.  `workspace`
    (ignored by the call) lets a test pass a buffer that must stay untouched."""
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
    if workspace is not None:
        a.workspace = workspace.data_ptr()
        a.workspace_bytes = workspace.numel()
    st = lib.nvfp4_quantize_noalloc(C.byref(a), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.nvfp4_status_string(st)
    return out


def check_against_oracle(w_bits, got):
    for b in range(w_bits.shape[0]):
        codes, sf, g = o.quantize(w_bits[b])
        ccodes, csf, _ = o.quantize_colwise(w_bits[b])
        assert np.array_equal(got["codes_row"][b].cpu().numpy(), codes), b
        assert np.array_equal(got["sf_row"][b].cpu().numpy(), o.sf_swizzle(sf)), b
        assert np.array_equal(got["codes_col"][b].cpu().numpy(), ccodes), b
        assert np.array_equal(got["sf_col"][b].cpu().numpy(), o.sf_swizzle(csf)), b
        assert got["global_scale"][b].item() == float(g), b


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
        check_against_oracle(w, got)
    assert nv.read_device_status(None) == 0


def test_noalloc_timeout_reports_through_its_own_status_word_and_recovers():
    """A zero wait budget makes the packing kernel's first wait expire: the call
    records NVFP4_ERR_TIMEOUT in the library's own status word (read with a NULL
    workspace), leaves the `workspace` argument untouched, and the next call
    with the normal budget succeeds and matches the oracle."""
    lib = nv.load()
    w = make_case("quantize", E=2, N=128, K=256, seed=3)["w"]
    x = dev(w)
    sentinel = torch.full((4096,), 0xA5, dtype=torch.uint8, device="cuda")
    assert nv.read_device_status(None) == 0
    old = nv.set_wait_timeout_ns(0)
    try:
        noalloc_quantize(lib, x, workspace=sentinel)
        st = nv.read_device_status(None)
    finally:
        nv.set_wait_timeout_ns(old)
    assert st == ERR_TIMEOUT, st
    assert bool((sentinel == 0xA5).all()), "the ignored workspace was written"
    assert nv.read_device_status(None) == 0           # reading cleared it
    got = noalloc_quantize(lib, x, workspace=sentinel)
    assert nv.read_device_status(None) == 0
    check_against_oracle(w, got)
    assert bool((sentinel == 0xA5).all())


def test_noalloc_rejects_oversized_scratch_request():
    lib = nv.load()
    # 33 matrices of >= 512 rows need 33 * 512 words > the 16384 available
    a = QuantArgs(src=4096, batch=33, rows=512, cols=64, ld=64, batch_stride=512 * 64,
                  pack=1, sf_layout=1, global_scale_out=4096, codes_row=4096, sf_row=4096)
    assert lib.nvfp4_quantize_noalloc(C.byref(a), None) == ERR_WORKSPACE
