"""Calls from several host threads: a kernel's dynamic shared-memory limit is one
value per device for the whole process, so a smaller launch from one thread
must never lower the limit that a larger launch from another thread relies on.

The decode GEMV's shared memory grows with K (it holds the quantized X row):
a long-K call on the main thread, a short-K call on a second thread, then the
long-K call again on the main thread must all succeed and give the same
results as when run alone."""
import threading

import numpy as np
import pytest
import torch

from helpers import dev_bf16
from synth import f32_to_bf16_bits

pytestmark = pytest.mark.gpu


def _case(lib, N, K, seed):
    rng = np.random.default_rng(seed)
    w = dev_bf16(f32_to_bf16_bits((rng.standard_normal((N, K)) * 0.02).astype(np.float32)))
    x = dev_bf16(f32_to_bf16_bits(rng.standard_normal((1, K)).astype(np.float32)))
    wq = lib.nvfp4_quantize(w, pack="row", sf_layout="swizzled")
    gx = torch.tensor([16.0 / 2688.0], dtype=torch.float32, device="cuda")
    return wq, x, gx


def _gemv(lib, case, N, K):
    wq, x, gx = case
    y = lib.nvfp4_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x,
                       a_global_scale=gx, out_dtype=torch.float32)
    torch.cuda.synchronize()
    return y


def test_smaller_launch_on_another_thread_does_not_lower_the_limit(lib):
    N = 256
    long_k, short_k = 16384, 2048
    big = _case(lib, N, long_k, 1)
    small = _case(lib, N, short_k, 2)
    y_big = _gemv(lib, big, N, long_k)
    y_small_ref = _gemv(lib, small, N, short_k)
    out, err = {}, []

    def other():
        try:
            torch.cuda.set_device(0)
            out["small"] = _gemv(lib, small, N, short_k)
        except Exception as e:   # reported on the main thread
            err.append(e)

    t = threading.Thread(target=other)
    t.start()
    t.join()
    assert not err, err
    assert torch.equal(out["small"], y_small_ref)
    y_big2 = _gemv(lib, big, N, long_k)     # raised limit still in force
    assert torch.equal(y_big2, y_big)
