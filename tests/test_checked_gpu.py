"""The build with device-side index checks (NVFP4_CHECKED): caller routing
data out of range is recorded in the status word as NVFP4_ERR_DEVICE_BOUNDS
and the access skipped, never a trap; the default build drops or clamps the
same data without recording it, and valid data reads OK in both.

The checked library is built here (it is not part of the default build) and
driven from child processes, since the binding picks its library from the
environment when it is first loaded."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, "tests")
import nvfp4_block_scaled_06_gb300 as nv
from nvfp4_block_scaled_06_gb300._binding import CHECKED, OK, ERR_DEVICE_BOUNDS
from helpers import dev_bf16
from synth import make_case

c = make_case("grouped", T=64, E=8, N=256, K=256, rank=32)
E, N, K, topk, T = c["E"], c["N"], c["K"], c["topk"], c["T"]
P = T * topk
q = nv.nvfp4_quantize(dev_bf16(c["w"]), pack="row", sf_layout="swizzled")
wc, ws, wg = q["codes_row"], q["sf_row"], q["global_scale"]
x = dev_bf16(c["x"])

def status_of(ids=None, routing=None):
    call, res = nv.prepare_grouped(ids, x, wc, ws, wg, N, K, E, routing=routing,
                                   top_k=None if routing is None else topk)
    call()
    return nv.read_device_status(call.workspace), res

ids = torch.from_numpy(c["expert_ids"]).cuda()
good, (d, perm, offs) = status_of(ids)
bad_ids = ids.clone()
bad_ids[0, 0] = E + 3                      # an expert id out of range
s_ids, _ = status_of(bad_ids)
bad_offs = offs.clone()
bad_offs[3] = bad_offs[2] - 7              # a count below zero
s_offs, _ = status_of(routing=(bad_offs, perm))
bad_perm = perm.clone()
bad_perm[1] = P + 5                        # a pair index out of range
s_perm, _ = status_of(routing=(offs, bad_perm))
torch.cuda.synchronize()
print("RESULT", int(CHECKED), good, s_ids, s_offs, s_perm, ERR_DEVICE_BOUNDS, OK)
"""


def run_child(checked: bool):
    env = dict(os.environ)
    env["NVFP4_CHECKED"] = "1" if checked else "0"
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT")][-1]
    return [int(v) for v in line.split()[1:]]


@pytest.fixture(scope="module")
def checked_lib():
    r = subprocess.run([sys.executable, "-m", "nvfp4_block_scaled_06_gb300.build", "--checked"], cwd=ROOT,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout + r.stderr


def test_checked_build_records_out_of_range_routing(checked_lib):
    checked, good, s_ids, s_offs, s_perm, bounds, ok = run_child(True)
    assert checked == 1
    assert good == ok
    assert s_ids == bounds and s_offs == bounds and s_perm == bounds


def test_default_build_clamps_silently():
    checked, good, s_ids, s_offs, s_perm, bounds, ok = run_child(False)
    assert checked == 0
    assert (good, s_ids, s_offs, s_perm) == (ok, ok, ok, ok)
