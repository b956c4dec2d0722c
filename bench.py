"""Benchmark of the NVFP4 W4A4 linear layer on GB300.

Headline workload: the prefill / training QLoRA linear
  Y[8192,2048] = W4A4(X[8192,6144], W[2048,6144]) + (X A^T) B^T * 128/64,
one step = one nvfp4_gemm call from bf16 X (dynamic per-tensor amax scale,
in-call NVFP4 quantization of X, the bf16 LoRA down-projection, the tcgen05
FP4 GEMM with the fused LoRA up-projection), bf16 out.  value = FP4 TFLOP/s
(2*M*N*K per step; the LoRA's bf16 flops are not counted).

Also measured in the same run (the "secondary" object): the expert-weight
quantization sweep (32 x [2048,6144], row + column packings, GB/s), the decode
projections (q_b_proj, o_proj at M = 1, 8, 32: weight GB/s), the grouped MoE
up-projection (4096 tokens, top-8 of 256 experts, LoRA r64: TFLOP/s and GB/s),
the backward of the prefill linear (both Dgrad forms and the FP4 Wgrad) and the
MoE down-projection with the gate-weighted combine.

Timing: CUDA events on the launching stream, after >= 3 warm-up steps;
inputs rotate over buffers whose total exceeds L2, so no step reads its input
from L2.  value comes from steps with nothing recorded between the launches;
the GEMM kernel's launch durations (roofline.achieved) from a second run of
the same steps with the library's event pair around the GEMM launch.  e2e
moves every step's X in from pinned host memory and its Y back out, steps
pipelined over two buffer sets and three streams (serial_value: one after
another).  N > 1 (torchrun): every rank runs the same workload on its own GPU
(replicas; the layer has no data-path exchange on one GPU per replica); the
time is the max over ranks and value is the total over ranks.

--impl reference: the CPU oracle on this host's cores, on a bounded row sample
of the same workload, printed with the same metric and unit.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A4 GEMM FP4 TFLOP/s (prefill QLoRA linear X[8192,6144] x W[2048,6144] + LoRA r64)"
UNIT = "TFLOP/s"
PREFILL = dict(M=8192, N=2048, K=6144, rank=64, alpha=128.0)
L2_BYTES = 129 * 1024 * 1024
FP4_PER_BF16 = 13.5 / 2.25          # nominal dense fp4 : bf16 tensor ratio
# DRAM bytes (read + write) of one GEMM launch on the prefill workload, from
# one ncu capture of the current kernel; None whenever the kernel has changed
# since that capture.
GEMM_TRAFFIC_BYTES = 39.9e6    # 36.8 MB read + 3.1 MB written; Y is still in L2 when the launch ends


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, source="fallback")


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers --
def max_over_ranks(torch, ms, device, world):
    """The slowest rank's time (every rank receives it), then a barrier."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.barrier()
    return float(t)


def job_value(world, flops_per_step, ms):
    """Whole-job TFLOP/s: every rank runs the full step on its own GPU (weak
    scaling), so the job does world x the step's FLOPs per ms of the slowest."""
    return world * flops_per_step / (ms * 1e-3) / 1e12


def ev_pairs(torch, n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def arm(C, args, pr):
    """Point the library's profiling hook at an event pair (or disarm it).

    The library records the events around its kernel with cudaEventRecord;
    torch records them once first so that it accepts them in elapsed_time()
    (the library's later record on the same stream sets the timestamps)."""
    if pr is None:
        args.prof_begin = None
        args.prof_end = None
    else:
        pr[0].record()
        pr[1].record()
        args.prof_begin = C.c_void_p(pr[0].cuda_event)
        args.prof_end = C.c_void_p(pr[1].cuda_event)


def mean_ms(pairs):
    return sum(a.elapsed_time(b) for a, b in pairs) / max(1, len(pairs))


def plain_and_kernel(torch, fn, steps, warmup, prof):
    """The per-call time with nothing recorded between the calls (an event
    between two launches ends their programmatic overlap), then the main
    kernel's launch durations from a second run with the library's event pair
    around it.  Returns (ms per call, ms per call when instrumented, kernel ms)."""
    ms = time_loop(torch, fn, steps, warmup, None)
    ms_prof = time_loop(torch, fn, steps, 0, prof)
    return ms, ms_prof, mean_ms(prof)


def time_loop(torch, fn, steps, warmup, prof=None, queue_ahead=True):
    """Run fn(i) warmup + steps times; return ms/step of the timed steps.

    With queue_ahead the timed steps are enqueued behind a short GPU sleep, so
    the host has queued them before the first one starts and the GPU runs them
    back to back: short kernels (decode) are then timed without the host's
    per-call launch latency between them, as a pipelined caller would see."""
    for i in range(warmup):
        fn(i, None)
    torch.cuda.synchronize()
    if queue_ahead:
        torch.cuda._sleep(int(5e7))          # ~25 ms at 2 GHz: covers enqueueing the steps
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for i in range(steps):
        fn(warmup + i, None if prof is None else prof[i])
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / steps


# ---------------------------------------------------------- main workload --
def prefill_setup(torch, nv, device, rotate):
    from synth import torch_case
    c = torch_case("prefill", seed=0, device=device)
    M, N, K = c["M"], c["N"], c["K"]
    wq = nv.nvfp4_quantize(c["w"], pack="row", sf_layout="swizzled")
    xs = [c["x"]] + [torch.empty_like(c["x"]).copy_(c["x"].roll(i * 977, dims=0))
                     for i in range(1, rotate)]
    lora = dict(a=c["lora_a"], b=c["lora_b"], alpha=c["alpha"])
    calls = []
    out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    for x in xs:
        call, _ = nv.prepare_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K,
                                  a_bf16=x, lora=lora, out=out)
        calls.append(call)
    return c, wq, xs, calls, out


def run_main(args, torch, nv, device, rank, world):
    import ctypes as C
    M, N, K = PREFILL["M"], PREFILL["N"], PREFILL["K"]
    rotate = 4                                # 4 x 100.7 MB of X > L2
    c, wq, xs, calls, out = prefill_setup(torch, nv, device, rotate)
    prof = ev_pairs(torch, args.steps)

    def step(i, pr):
        call = calls[i % rotate]
        arm(C, call.args, pr)
        call()

    for i in range(args.warmup):
        step(i, None)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(torch.cuda.current_device()) as clk:
        # the same step, untimed, for ~0.5 s so that nvidia-smi samples the
        # clocks under this load; the timed region follows immediately
        t_end = time.perf_counter() + 0.5
        i = 0
        while time.perf_counter() < t_end:
            step(i, None)
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize()
        # the headline: K steps with nothing between the three launches
        ms = time_loop(torch, step, args.steps, 0, None)
        # the GEMM kernel's launch durations: K more steps with the library's
        # event pair around the GEMM launch (an event between two launches
        # ends their programmatic overlap, so this run is not the headline)
        ms_prof = time_loop(torch, step, args.steps, 0, prof)
    ms = max_over_ranks(torch, ms, device, world)
    gemm_ms = mean_ms(prof)
    flops = 2.0 * M * N * K
    # end to end: pinned host X in, host Y out, through the same C-ABI call
    e2e = run_e2e(args, torch, nv, device, wq, c, xs[0])
    return dict(ms=ms, ms_prof=ms_prof, gemm_ms=gemm_ms, flops=flops, clocks=clk.summary(), e2e=e2e,
                launches_per_step=3)   # LoRA-down/amax, packing, GEMM


def run_e2e(args, torch, nv, device, wq, c, x_dev):
    """End to end through the public call: every step copies its X from pinned
    host memory to the device, runs the linear, and copies Y back to pinned
    host memory.  Pipelined (the headline): two buffer sets and three streams,
    so that step i's compute overlaps the input copy of step i+1 and the output
    copy of step i-1, as a serving loop would run it; every step still moves
    all of its bytes.  Serial: the three on one stream, one step at a time."""
    M, N, K = PREFILL["M"], PREFILL["N"], PREFILL["K"]
    lora = dict(a=c["lora_a"], b=c["lora_b"], alpha=c["alpha"])
    nb = 2
    x_host = [torch.empty((M, K), dtype=torch.bfloat16, pin_memory=True) for _ in range(nb)]
    for h in x_host:
        h.copy_(x_dev.cpu())
    y_host = [torch.empty((M, N), dtype=torch.bfloat16, pin_memory=True) for _ in range(nb)]
    x_in = [torch.empty_like(x_dev) for _ in range(nb)]
    calls, ys = [], []
    for j in range(nb):
        call, y = nv.prepare_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K,
                                  a_bf16=x_in[j], lora=lora)
        calls.append(call)
        ys.append(y)

    def serial_step(i, pr):
        x_in[0].copy_(x_host[0], non_blocking=True)
        calls[0]()
        y_host[0].copy_(ys[0], non_blocking=True)

    steps = max(3, args.steps // 2)
    serial_ms = time_loop(torch, serial_step, steps, max(3, args.warmup))

    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_done, run_done, out_done = [ev() for _ in range(nb)], [ev() for _ in range(nb)], [ev() for _ in range(nb)]
    for j in range(nb):           # every buffer starts free
        for e in (run_done[j], out_done[j]):
            e.record(torch.cuda.current_stream())

    def piped_step(i):
        j = i % nb
        with torch.cuda.stream(s_in):
            s_in.wait_event(run_done[j])          # x_in[j] no longer read by step i-2
            x_in[j].copy_(x_host[j], non_blocking=True)
            in_done[j].record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(in_done[j])
            s_run.wait_event(out_done[j])         # y[j] copied out by step i-2
            calls[j](s_run)
            run_done[j].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(run_done[j])
            y_host[j].copy_(ys[j], non_blocking=True)
            out_done[j].record(s_out)

    cur = torch.cuda.current_stream()
    for i in range(max(3, args.warmup)):
        piped_step(i)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(5e7))                # the host queues the steps meanwhile
    t0.record(cur)
    for q in (s_in, s_run, s_out):
        q.wait_event(t0)
    for i in range(steps):
        piped_step(i)
    for q in (s_in, s_run, s_out):
        cur.wait_stream(q)
    t1.record(cur)
    torch.cuda.synchronize()
    piped_ms = t0.elapsed_time(t1) / steps
    return dict(ms=piped_ms, serial_ms=serial_ms, h2d=M * K * 2, d2h=M * N * 2)


# ------------------------------------------------------- secondary lines --

def run_prefill_static(torch, nv, device, steps, warmup, pk):
    """The prefill step with a static per-tensor input scale (a serving-style
    input_scale, 16/2688 for X ~ N(0,1) rows of this size) in place of the
    dynamic amax: the packing pass needs no maximum first, so the LoRA-down
    pass reads X on its own after it.  Same workload otherwise; the trade
    against the headline's dynamic scale."""
    M, N, K = PREFILL["M"], PREFILL["N"], PREFILL["K"]
    rotate = 4
    c, wq, xs, _, out = prefill_setup(torch, nv, device, rotate)
    gx = torch.tensor([16.0 / 2688.0], dtype=torch.float32, device=device)
    lora = dict(a=c["lora_a"], b=c["lora_b"], alpha=c["alpha"])
    calls = [nv.prepare_gemm(wq["codes_row"], wq["sf_row"], wq["global_scale"], N, K, a_bf16=x,
                             a_global_scale=gx, lora=lora, out=out)[0] for x in xs]

    def step(i, pr):
        calls[i % rotate]()
    ms = time_loop(torch, step, steps, warmup, None)
    flops = 2.0 * M * N * K
    del c, xs, calls
    return dict(workload="prefill QLoRA linear as the headline, X quantized with a static input scale 16/2688",
                ms=ms, tflops=flops / (ms * 1e-3) / 1e12)


def run_quantize_sweep(torch, nv, device, steps, warmup, pk):
    import ctypes as C
    from synth import torch_case
    c = torch_case("quantize", seed=0, device=device)
    E, N, K = c["E"], c["N"], c["K"]
    call, out = nv.prepare_quantize(c["w"], pack="both", sf_layout="swizzled")
    prof = ev_pairs(torch, steps)

    def step(i, pr):
        arm(C, call.args, pr)
        call()
    ms, ms_prof, kms = plain_and_kernel(torch, step, steps, warmup, prof)
    elems = E * N * K
    alg = elems * (2 + 2 * 0.5625)             # one bf16 read, two NVFP4 packings written
    del c, out
    return dict(workload="32 x W[2048,6144] bf16 -> row + column NVFP4 packings, swizzled scales, dynamic g",
                ms=ms, ms_instrumented=ms_prof, kernel_ms=kms,
                elements_per_s=elems / (ms * 1e-3), gbs=alg / (ms * 1e-3) / 1e9,
                frac_call=alg / (ms * 1e-3) / 1e9 / pk["hbm"],
                kernel_gbs=alg / (kms * 1e-3) / 1e9, algorithmic_bytes=alg,
                frac=alg / (kms * 1e-3) / 1e9 / pk["hbm"],
                note="amax pass + packing pass (2 reads of the 805 MB input); frac uses the packing kernel's time with the algorithmic one-read bytes")


def run_decode(torch, nv, device, steps, warmup, pk):
    import ctypes as C
    from synth import torch_case
    res = {}
    for name in ("decode_q_b_proj", "decode_o_proj"):
        c = torch_case(name, seed=0, device=device, M=32)
        N, K = c["N"], c["K"]
        wq0 = nv.nvfp4_quantize(c["w"], pack="row", sf_layout="swizzled")
        wbytes = N * K * 0.5625
        copies = max(2, int(3 * L2_BYTES // wbytes) + 1)        # rotate > 3x L2 of weights
        wqs = [wq0] + [{k: v.clone() for k, v in wq0.items()} for _ in range(copies - 1)]
        gx = torch.tensor([16.0 / 2688.0], dtype=torch.float32, device=device)
        for M in (1, 8, 32):
            x = c["x"][:M].contiguous()
            calls = [nv.prepare_gemm(w["codes_row"], w["sf_row"], w["global_scale"], N, K,
                                     a_bf16=x, a_global_scale=gx)[0] for w in wqs]
            prof = ev_pairs(torch, steps)

            def step(i, pr, calls=calls):
                cl = calls[i % len(calls)]
                arm(C, cl.args, pr)
                cl()
            ms, ms_prof, kms = plain_and_kernel(torch, step, steps, warmup, prof)
            alg = wbytes + M * K * 2 + M * N * 2
            res[f"{name[7:]}_M{M}"] = dict(
                ms=ms, ms_instrumented=ms_prof, kernel_ms=kms,
                weight_gbs=wbytes / (ms * 1e-3) / 1e9, frac_call=alg / (ms * 1e-3) / 1e9 / pk["hbm"],
                kernel_gbs=alg / (kms * 1e-3) / 1e9, frac=alg / (kms * 1e-3) / 1e9 / pk["hbm"],
                path="cuda-core GEMV" if M <= 4 else "tcgen05 GEMM, weights as the 128-row operand")
        del wqs, c
        torch.cuda.empty_cache()
    return res


def run_grouped(torch, nv, device, steps, warmup, pk, experts=None):
    import ctypes as C
    from synth import torch_case
    c = torch_case("grouped", seed=0, device=device, **({"E": experts} if experts else {}))
    E, N, K, T, topk = c["E"], c["N"], c["K"], c["T"], c["topk"]
    wq = nv.nvfp4_quantize(c["w"], pack="row", sf_layout="swizzled")
    del c["w"]
    torch.cuda.empty_cache()
    lora = dict(a=c["lora_a"], b=c["lora_b"], alpha=c["alpha"])
    call, (d, perm, offs) = nv.prepare_grouped(c["expert_ids"], c["x"], wq["codes_row"],
                                               wq["sf_row"], wq["global_scale"], N, K, E,
                                               lora=lora)
    prof = ev_pairs(torch, steps)

    def step(i, pr):
        arm(C, call.args, pr)
        call()
    ms, ms_prof, kms = plain_and_kernel(torch, step, steps, warmup, prof)
    counts = torch.bincount(c["expert_ids"].reshape(-1).long(), minlength=E).cpu()
    active = int((counts > 0).sum())
    P = T * topk
    flops = 2.0 * P * N * K
    wbytes = active * N * K * 0.5625
    lbytes = active * (c["rank"] * K + N * c["rank"]) * 2
    alg = wbytes + lbytes + T * K * 2 + P * N * 2
    return dict(workload=f"{T} tokens x top-{topk} of {E} experts W_e[{N},{K}] + LoRA r{c['rank']}",
                ms=ms, ms_instrumented=ms_prof, tflops=flops / (ms * 1e-3) / 1e12, kernel_ms=kms,
                kernel_tflops=flops / (kms * 1e-3) / 1e12, gbs=alg / (ms * 1e-3) / 1e9,
                kernel_gbs=alg / (kms * 1e-3) / 1e9, active_experts=active,
                max_rows=int(counts.max()), hbm_frac=alg / (kms * 1e-3) / 1e9 / pk["hbm"],
                tensor_frac=flops / (kms * 1e-3) / 1e12 / (pk["bf16"] * FP4_PER_BF16))


def run_dgrad(torch, nv, device, steps, warmup, pk):
    """dX = dY W for the prefill linear's backward, both ways the pages weigh:
    dequantize the rowwise packing to bf16 (transposed) + bf16 GEMM, or the
    column packing + W4A4 GEMM with dY quantized in the call."""
    import ctypes as C
    from synth import torch_case
    c = torch_case("dgrad", seed=0, device=device)
    M, N, K = c["M"], c["N"], c["K"]
    q = nv.nvfp4_quantize(c["w"], pack="both", sf_layout="swizzled")
    flops = 2.0 * M * N * K
    out = {}
    for name, kw in (("dequant_bf16", dict(w=(q["codes_row"][0], q["sf_row"][0], q["global_scale"]))),
                     ("fp4_colpack", dict(wcol=(q["codes_col"][0], q["sf_col"][0], q["global_scale"])))):
        call, dx = nv.prepare_dgrad(c["dy"], N, K, **kw)
        prof = ev_pairs(torch, steps)

        def step(i, pr, call=call):
            arm(C, call.args, pr)
            call()
        ms, ms_prof, kms = plain_and_kernel(torch, step, steps, warmup, prof)
        peak = pk["bf16"] * (1.0 if name == "dequant_bf16" else FP4_PER_BF16)
        out[name] = dict(ms=ms, ms_instrumented=ms_prof, tflops=flops / (ms * 1e-3) / 1e12, gemm_ms=kms,
                         gemm_tflops=flops / (kms * 1e-3) / 1e12,
                         gemm_frac=flops / (kms * 1e-3) / 1e12 / peak,
                         pre_ms=ms - kms)
    # the weight-gradient product on the FP4 datapath: dW[N,K] = dY^T X, both packed along M
    x = torch_case("prefill", seed=1, device=device)["x"]
    call, dw = nv.prepare_wgrad(c["dy"], x)
    prof = ev_pairs(torch, steps)

    def wstep(i, pr):
        arm(C, call.args, pr)
        call()
    ms, ms_prof, kms = plain_and_kernel(torch, wstep, steps, warmup, prof)
    out["wgrad_fp4"] = dict(ms=ms, ms_instrumented=ms_prof, tflops=flops / (ms * 1e-3) / 1e12, gemm_ms=kms,
                            gemm_tflops=flops / (kms * 1e-3) / 1e12,
                            gemm_frac=flops / (kms * 1e-3) / 1e12 / (pk["bf16"] * FP4_PER_BF16),
                            pre_ms=ms - kms)
    out["workload"] = (f"dX[{M},{K}] = dY[{M},{N}] W[{N},{K}] and dW[{N},{K}] = dY^T X[{M},{K}] "
                       f"(prefill linear backward), bf16 out")
    out["note"] = ("pre_ms = dequantization (bf16 mode) or the in-call quantizations (fp4 modes); "
                   "gemm_frac against the burst bf16 / 6x bf16 peak")
    return out


def run_moe_down(torch, nv, device, steps, warmup, pk, experts=None):
    """The routed experts' down-projection W2_e[6144,2048] + gate-weighted combine
    for 4096 tokens x top-8 (the grouped up-projection's successor)."""
    import ctypes as C
    from synth import torch_case
    c = torch_case("moe_down", seed=0, device=device, **({"E": experts} if experts else {}))
    E, N, K, T, k = c["E"], c["N"], c["K"], c["T"], c["topk"]
    wq = nv.nvfp4_quantize(c["w"], pack="row", sf_layout="swizzled")
    del c["w"]
    torch.cuda.empty_cache()
    flat = c["expert_ids"].reshape(-1).long()
    perm = torch.sort(flat, stable=True).indices.to(torch.int32)
    counts = torch.bincount(flat, minlength=E)
    offsets = torch.zeros(E + 1, dtype=torch.int32, device=device)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    lora = dict(a=c["lora_a"], b=c["lora_b"], alpha=c["alpha"])
    call, y = nv.prepare_moe_down(c["h"], perm, offsets, c["route_weights"], wq["codes_row"],
                                  wq["sf_row"], wq["global_scale"], N, K, E, lora=lora)
    prof = ev_pairs(torch, steps)

    def step(i, pr):
        arm(C, call.args, pr)
        call()
    ms, ms_prof, kms = plain_and_kernel(torch, step, steps, warmup, prof)
    active = int((counts > 0).sum())
    P = T * k
    flops = 2.0 * P * N * K
    wbytes = active * N * K * 0.5625
    return dict(workload=f"{T} tokens x top-{k}: down-projection of {E} experts W2_e[{N},{K}] + LoRA "
                         f"r{c['rank']} + gate-weighted combine -> y[{T},{N}]",
                ms=ms, ms_instrumented=ms_prof, tflops=flops / (ms * 1e-3) / 1e12, gemm_ms=kms,
                gemm_tflops=flops / (kms * 1e-3) / 1e12,
                gemm_weight_gbs=wbytes / (kms * 1e-3) / 1e9, active_experts=active)


# ----------------------------------------------------------- CPU baseline --
CPU_ROWS = 256          # rows of X per oracle step (both CPU legs)


class OracleStep:
    """The oracle on the headline workload, as the GPU arm runs it: W is
    quantized once outside the timed region; one step quantizes `rows` rows of
    X (dynamic scale) and forms their W4A4 product + LoRA in fp64.  Both CPU
    legs (cpu_baseline and --impl reference) time exactly this step, so their
    rates measure the same work per row."""

    def __init__(self, rows: int = CPU_ROWS):
        from oracle import nvfp4_oracle as o
        from synth import make_case
        self.o = o
        c = make_case("prefill", M=rows)
        self.c = c
        self.rows = rows
        self.wq = o.quantize(c["w"])
        self.lora = (c["lora_a"], c["lora_b"], PREFILL["alpha"])
        self.flops = 2.0 * rows * PREFILL["N"] * PREFILL["K"]

    def __call__(self):
        xq = self.o.quantize(self.c["x"])
        return self.o.linear_fp64(xq, self.wq, self.c["x"], self.lora)


def timed_oracle_steps(step, n):
    """Run n oracle steps; return (seconds per step, average busy cores)."""
    c0, t0 = time.process_time(), time.perf_counter()
    for _ in range(n):
        step()
    dt = time.perf_counter() - t0
    return dt / n, (time.process_time() - c0) / dt


def cpu_baseline(budget_s: float = 12.0):
    """The oracle timed on this host's cores for about `budget_s` seconds of
    steps (a bounded sample of the headline workload).  The oracle is numpy:
    its elementwise steps run on one thread, its fp64 matmul on the BLAS
    threads; `cores` is the CPU time the process used divided by the wall time
    (the average number of busy cores)."""
    step = OracleStep()
    step()                                   # warm-up (and first-touch of W)
    one, _ = timed_oracle_steps(step, 1)
    n = max(1, int(budget_s / max(one, 1e-3)))
    sec, busy = timed_oracle_steps(step, n)
    return dict(value=step.flops / sec / 1e12, unit=UNIT, cores=round(busy, 1), kind="oracle",
                host_cores=os.cpu_count(),
                sample=f"{n} steps of {step.rows} rows of X [of 8192] through quantize + dequantized "
                       f"fp64 W4A4 product + LoRA, W quantized once outside the timing (as the GPU "
                       f"arm); {sec * n:.1f} s, {busy:.1f} cores busy on average of {os.cpu_count()}",
                rows_per_step=step.rows, seconds=sec * n)


def reference_arm(args):
    """--impl reference: the oracle (there is no reference code: the pages hold
    none) on the host cores, each step the same bounded sample that
    cpu_baseline times."""
    step = OracleStep()
    for _ in range(args.warmup):
        step()
    sec, busy = timed_oracle_steps(step, args.steps)
    ms = 1e3 * sec
    v = step.flops / sec / 1e12
    line = dict(impl="reference", metric=METRIC, value=v, unit=UNIT, n_gpus=args.gpus,
                steps=args.steps, warmup=args.warmup, ms_per_step=ms, higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=dict(workload="prefill QLoRA linear (X[8192,6144] bf16, NVFP4 W[2048,6144], "
                                     "LoRA r64), CPU oracle on a row sample per step",
                            M=PREFILL["M"], M_sample=step.rows, N=PREFILL["N"], K=PREFILL["K"],
                            rank=64),
                cpu_baseline=dict(value=v, unit=UNIT, cores=round(busy, 1), kind="oracle",
                                  sample=f"{step.rows} rows of X per step, W quantized once before "
                                         f"the timed steps"),
                e2e=dict(value=v, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line))


# ------------------------------------------------------------------- main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--only-main", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--only", choices=["quantize", "decode", "grouped", "dgrad", "moe_down", "prefill_static"],
                    help="run just this secondary workload (for profiling) and print its numbers")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--experts", type=int, default=None,
                    help="with --only grouped/moe_down: number of routed experts (default: the "
                         "workload's 256; fewer keep an ncu capture to a few GB on the device)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        if rank == 0:
            os.environ.setdefault("OMP_NUM_THREADS", "1")
            reference_arm(args)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    import nvfp4_block_scaled_06_gb300 as nv
    nv.load()
    pk = peaks()

    if args.only:
        fn = dict(quantize=run_quantize_sweep, decode=run_decode, grouped=run_grouped,
                  dgrad=run_dgrad, moe_down=run_moe_down, prefill_static=run_prefill_static)[args.only]
        kw = {"experts": args.experts} if args.only in ("grouped", "moe_down") and args.experts else {}
        res = fn(torch, nv, device, args.steps, args.warmup, pk, **kw)
        if rank == 0:
            print(json.dumps({"only": args.only, "steps": args.steps, "warmup": args.warmup, **res}))
        return

    main_res = run_main(args, torch, nv, device, rank, world)
    sec = {}
    if not args.only_main:
        steps2 = max(10, min(args.steps, 30))
        sec["prefill_static_scale"] = run_prefill_static(torch, nv, device, steps2, max(3, args.warmup), pk)
        torch.cuda.empty_cache()
        sec["quantize"] = run_quantize_sweep(torch, nv, device, steps2, max(3, args.warmup), pk)
        torch.cuda.empty_cache()
        sec["decode"] = run_decode(torch, nv, device, steps2, max(3, args.warmup), pk)
        torch.cuda.empty_cache()
        sec["grouped"] = run_grouped(torch, nv, device, steps2, max(3, args.warmup), pk)
        torch.cuda.empty_cache()
        sec["dgrad"] = run_dgrad(torch, nv, device, steps2, max(3, args.warmup), pk)
        torch.cuda.empty_cache()
        sec["moe_down"] = run_moe_down(torch, nv, device, steps2, max(3, args.warmup), pk)
        torch.cuda.empty_cache()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    ms = main_res["ms"]
    value = job_value(world, main_res["flops"], ms)
    # the GEMM launches are timed over a few ms of steps: the burst bf16 figure
    fp4_peak = pk["bf16"] * FP4_PER_BF16
    gemm_tflops = main_res["flops"] / (main_res["gemm_ms"] * 1e-3) / 1e12
    e2e = main_res["e2e"]
    line = dict(
        metric=METRIC, value=value, unit=UNIT, n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="e2m1xe2m1->f32 (bf16 LoRA, bf16 out)", data="synthetic",
        config=dict(workload="prefill QLoRA linear: X[8192,6144] bf16 ~N(0,1) -> NVFP4 (dynamic amax), "
                             "frozen NVFP4 W[2048,6144] ~N(0,0.02), LoRA A[64,6144] B[2048,64] ~N(0,0.01), "
                             "alpha 128, Y bf16",
                    M=PREFILL["M"], N=PREFILL["N"], K=PREFILL["K"], rank=64, alpha=128.0,
                    l2="X rotates over 4 buffers (403 MB > 129 MB L2)",
                    parallelism=f"replicas x{world}"),
        roofline=dict(bound="tensor", kernel="k_gemm_fp4_pair", achieved=gemm_tflops,
                      peak=fp4_peak, unit="TFLOP/s", frac=gemm_tflops / fp4_peak,
                      traffic=GEMM_TRAFFIC_BYTES,
                      traffic_note=("dram__bytes_read.sum + dram__bytes_write.sum per launch, one ncu "
                                    "capture of this kernel on this workload (M8192 N2048 K6144, "
                                    "cold L2); algorithmic bytes 70.3 MB" if GEMM_TRAFFIC_BYTES else
                                    "null: no ncu capture of the kernel as it stands; algorithmic "
                                    "bytes 70.3 MB"),
                      peak_note=f"{pk['source']} bf16 burst {pk['bf16']} TFLOP/s x 6 "
                                f"(nominal fp4:bf16), of {pk['source']}",
                      timing_note="CUDA events around each GEMM launch in a second run of the same "
                                  f"{args.steps} steps ({main_res['ms_prof']:.4f} ms/step with the events)"),
        e2e=dict(value=job_value(world, main_res["flops"], e2e["ms"]), unit=UNIT,
                 h2d_bytes_per_step=e2e["h2d"], d2h_bytes_per_step=e2e["d2h"],
                 overlap="steps pipelined: the input copy of step i+1 and the output copy of "
                         "step i-1 run during step i (two buffer sets, three streams)",
                 serial_value=job_value(world, main_res["flops"], e2e["serial_ms"])),
        gpu_launches=main_res["launches_per_step"] * args.steps,
        clocks=main_res["clocks"],
        secondary=sec,
    )
    if not args.no_cpu:
        cb = cpu_baseline()
        cb.pop("seconds", None)
        line["cpu_baseline"] = cb
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
