"""Benchmark of the EXL3 trellis-quantized linear on one GB300.

Workload of a step: the dense decode sweep k = 5120, n in {5120, 17408,
25600}, K = 4, M = 1 (three fused GEMV launches, fp16 out).  `value` is the
aggregate algorithmic HBM traffic of those linears (packed weights + x + y +
suh + svh) per second, with inputs resident on the device.  Three copies of
the weights rotate between steps (3 x 123 MB > 2 x L2), so no step reads
another's weights from L2.

Extra objects on the same JSON line: `roofline` (the GEMV kernel against the
measured HBM copy bandwidth), `cpu_baseline` (the CPU oracle on a bounded
sample), `e2e` (the same metric through the C ABI with host buffers: each
step copies x in from pinned host memory with exl3_copy_in and the linears
write y straight into pinned host memory; copy-engine transfers beside it),
`prefill` (M = 4096 TFLOP/s), `configs` (every decode and small-M shape),
`other` (MoE, fused shards, row-invariant mode) and `clocks`.

    python bench.py [--gpus 1] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import exl3_synth as synth  # noqa: E402

METRIC = "EXL3 trellis GEMV HBM GB/s (M=1) & GEMM TFLOPS (M=4096), % of roofline"


def _world() -> int:
    """Ranks of the job (torchrun sets WORLD_SIZE; 1 without it)."""
    return int(os.environ.get("WORLD_SIZE", "1"))


def _barrier():
    """All ranks meet here when the job runs replicas under torchrun."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_replicas(out: dict, dist, device) -> dict:
    """The whole-job line of N replicas: every rank's algorithmic bytes over
    the slowest rank's step time (max over ranks); n_gpus = world size."""
    import torch
    t = torch.tensor([out["ms_per_step"]], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ws = dist.get_world_size()
    step_bytes = out["value"] * 1e9 * out["ms_per_step"] * 1e-3      # this rank's bytes per step
    res = dict(out)
    res["ms_per_step"] = float(t.item())
    res["value"] = round(step_bytes * ws / (res["ms_per_step"] * 1e-3) / 1e9, 1)
    res["n_gpus"] = ws
    return res
WORKLOAD = "dense decode GEMV sweep k=5120 n={5120,17408,25600} K=4 M=1 mul1, fp16 out"
FALLBACK_HBM_GBS = 6800.0
# The mul1 decode's ceiling at K = 4 on this chip (ubench/pipes.cu, bench.py
# --only pipes): hash + byte sum + accumulate share one 64-lane pipe, ~26
# weights per clock per SM = 26 * 152 * 2.07 GHz * 0.5 B = 4.09 TB/s, 0.60 of
# the measured 6767 GB/s copy rate.
DECODE_CEILING_FRAC_K4 = 0.60
FALLBACK_BF16_TFLOPS = 1900.0

# dram bytes (read + write) per launch from an ncu capture of gemv_m1_kernel<4>
# at k=5120 n=25600, with the hash of the kernel's sources at capture time; a
# changed kernel source makes the recorded traffic stale (reported as null).
TRAFFIC = {"files": ["trellis_quantized_gb300/csrc/gemv.cu", "trellis_quantized_gb300/csrc/gemv_core.cuh",
                     "trellis_quantized_gb300/csrc/exl3_common.cuh"],
           "sha1": "f2e2cc0efb10200a5f71703c019acfcba9b7827f", "bytes_per_launch": 65670400,
           "workload": "k5120 n25600 K4 M1"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        # burst figure: the prefill GEMM is timed alone (a graph of back-to-back calls)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def linear_bytes(case) -> int:
    return case.trellis.nbytes + case.x.nbytes + case.suh.nbytes + case.svh.nbytes + case.M * case.n * 2


def files_sha1(rels):
    h = hashlib.sha1()
    for rel in rels:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- ours

def run_ours(args):
    import torch
    import trellis_quantized_gb300 as tq

    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                     else np.ascontiguousarray(a)).cuda()
    cases = [synth.config2(n, 1) for n in synth.CONFIG2_N]
    copies = 3
    dcases = []
    for c in cases:
        base_t = dev(c.trellis)
        ts = [base_t] + [base_t.clone() for _ in range(copies - 1)]
        ws = tq.workspace(tq.exl3_linear_workspace_size(1, c.k, c.n, c.K))
        wsc = torch.zeros_like(ws)
        dcases.append(dict(case=c, x=dev(c.x), t=ts, suh=dev(c.suh), svh=dev(c.svh),
                           y=torch.empty((1, c.n), dtype=torch.float16, device="cuda"), ws=wsc))
    L = tq.lib()

    def launch(d, copy):
        c = d["case"]
        rc = L.exl3_linear(d["x"].data_ptr(), 1, c.k, c.n, d["t"][copy].data_ptr(), d["suh"].data_ptr(),
                           d["svh"].data_ptr(), c.K, tq.EXL3_CB_MUL1, d["y"].data_ptr(), tq.EXL3_OUT_F16,
                           d["ws"].data_ptr(), d["ws"].numel(), torch.cuda.current_stream().cuda_stream)
        if rc:
            raise tq.Exl3Error(rc, L.exl3_last_error().decode())

    step_bytes = sum(linear_bytes(d["case"]) for d in dcases)
    for d in dcases:
        tq.exl3_workspace_clear(d["ws"])
    for i in range(args.warmup):
        for d in dcases:
            launch(d, i % copies)
    torch.cuda.synchronize()

    # One step = the three linears, captured as a CUDA graph per weight copy,
    # so the timed region measures the device and not Python launch overhead.
    # With weight prefetch (the default) each linear is a programmatic
    # dependent launch that streams its weights while the previous one ends.
    # Steps are captured `chunk` at a time, one graph per starting weight
    # copy, so that the copies keep rotating from one replay to the next.
    prefetch = not args.no_prefetch
    tq.exl3_set_weight_prefetch(prefetch)
    chunk = 10 if args.steps >= 10 else 1
    graphs = []
    for cp in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for j in range(chunk):
                for d in dcases:
                    launch(d, (cp + j) % copies)
        graphs.append(g)
    single = []
    for cp in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for d in dcases:
                launch(d, cp)
        single.append(g)
    # Per-kernel duration for the roofline: 30 launches of the largest linear
    # in one graph, launched as in the step (programmatic dependent launches
    # when weight_prefetch), and the same 30 launched plainly for reference.
    big = len(dcases) - 1
    reps_k = 30
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk):
        for i in range(reps_k):
            launch(dcases[big], i % copies)
    tq.exl3_set_weight_prefetch(False)
    gkp = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gkp):
        for i in range(reps_k):
            launch(dcases[big], i % copies)
    tq.exl3_set_weight_prefetch(prefetch)
    for i in range(args.warmup):
        single[i % copies].replay()
    graphs[0].replay()
    gk.replay()
    gkp.replay()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        _barrier()
        t_start.record(stream)
        done = 0
        while done + chunk <= args.steps:
            graphs[done % copies].replay()
            done += chunk
        while done < args.steps:
            single[done % copies].replay()
            done += 1
        t_end.record(stream)
        torch.cuda.synchronize()
        _barrier()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        kreps = 20
        k0.record(stream)
        for _ in range(kreps):
            gk.replay()
        k1.record(stream)
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for _ in range(kreps):
            gkp.replay()
        p1.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.2)
    total_ms = t_start.elapsed_time(t_end)
    ms_per_step = total_ms / args.steps
    value = step_bytes / (ms_per_step * 1e-3) / 1e9

    hbm, bf16, src = peaks()
    big_bytes = linear_bytes(dcases[big]["case"])
    kern_ms = k0.elapsed_time(k1) / (kreps * reps_k)
    plain_ms = p0.elapsed_time(p1) / (kreps * reps_k)
    achieved = big_bytes / (kern_ms * 1e-3) / 1e9
    traffic = None
    if TRAFFIC["sha1"] and TRAFFIC["sha1"] == files_sha1(TRAFFIC["files"]):
        traffic = TRAFFIC["bytes_per_launch"]
    roofline = {"bound": "hbm", "kernel": "gemv_m1_kernel<K=4> (k=5120 n=25600)", "achieved": round(achieved, 1),
                "peak": hbm, "peak_source": src, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                "traffic": traffic, "kernel_us": round(kern_ms * 1e3, 2),
                "algorithmic_bytes_per_launch": big_bytes,
                "kernel_us_plain_launches": round(plain_ms * 1e3, 2),
                "frac_plain_launches": round(big_bytes / (plain_ms * 1e-3) / 1e9 / hbm, 4),
                "decode_ceiling_frac": DECODE_CEILING_FRAC_K4,
                "timing": "CUDA events around 20 replays of a graph of 30 launches (3 rotating weight copies), "
                          "launched as in the step (programmatic dependent launches when weight_prefetch); "
                          "kernel_us_plain_launches: the same without overlap between launches"}

    # e2e: the step's inputs (the three linears' x, packed in one pinned host
    # buffer) go host -> device through exl3_copy_in (SM loads over
    # NVLink-C2C, chained to the linears by programmatic dependent launch),
    # the linears run through the C ABI on views of the device copy and write
    # their y straight into one pinned host buffer; the transfers both ways
    # are inside the timed region.  The same step with copy-engine transfers
    # (one packed copy each way) is measured beside it.
    kx = [d["case"].k for d in dcases]
    ny = [d["case"].n for d in dcases]
    hx = torch.from_numpy(np.concatenate([d["case"].x.reshape(-1) for d in dcases]).view(np.int16)).pin_memory()
    hy = torch.empty(sum(ny), dtype=torch.float16).pin_memory()
    dx = torch.empty(hx.shape, dtype=hx.dtype, device="cuda")
    dy = torch.empty(sum(ny), dtype=torch.float16, device="cuda")
    xo = np.cumsum([0] + kx) * 2
    yo = np.cumsum([0] + ny) * 2
    hx_bytes = hx.numel() * hx.element_size()
    hy_bytes = hy.numel() * hy.element_size()

    def launch_e2e(j, copy, yp):
        d, c = dcases[j], dcases[j]["case"]
        rc = L.exl3_linear(dx.data_ptr() + int(xo[j]), 1, c.k, c.n, d["t"][copy].data_ptr(), d["suh"].data_ptr(),
                           d["svh"].data_ptr(), c.K, tq.EXL3_CB_MUL1, yp + int(yo[j]), tq.EXL3_OUT_F16,
                           d["ws"].data_ptr(), d["ws"].numel(), torch.cuda.current_stream().cuda_stream)
        if rc:
            raise tq.Exl3Error(rc, L.exl3_last_error().decode())

    def e2e_step(i):
        rc = L.exl3_copy_in(hx.data_ptr(), dx.data_ptr(), hx_bytes, torch.cuda.current_stream().cuda_stream)
        if rc:
            raise tq.Exl3Error(rc, L.exl3_last_error().decode())
        for j in range(len(dcases)):
            launch_e2e(j, i % copies, hy.data_ptr())

    def e2e_step_ce(i):
        dx.copy_(hx, non_blocking=True)
        for j in range(len(dcases)):
            launch_e2e(j, i % copies, dy.data_ptr())
        hy.copy_(dy, non_blocking=True)

    e2e_steps = max(10, args.steps // 4)
    e2e_steps -= e2e_steps % chunk
    stream = torch.cuda.current_stream()
    ref_y = [dcases[j]["y"].cpu() for j in range(len(dcases))]

    def check_hy(what):
        for j in range(len(dcases)):   # the packed path computes what the per-linear path did
            got = hy[int(yo[j]) // 2:int(yo[j + 1]) // 2].view(1, -1)
            assert torch.equal(got, ref_y[j]), f"e2e ({what}) output differs"

    def timed_e2e(fn):
        hy.zero_()
        for i in range(3):
            fn(i)
        torch.cuda.synchronize()
        check_hy("eager")
        # eager: one C-ABI call per copy and linear from Python each step
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        eager_ms = e0.elapsed_time(e1) / e2e_steps
        # as a decode loop runs it: the same calls and copies captured in CUDA
        # graphs (`chunk` steps per graph, one graph per starting weight copy)
        egraphs = []
        for cp in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for jj in range(chunk):
                    fn(cp + jj)
            egraphs.append(g)
        hy.zero_()
        for g in egraphs:
            g.replay()
        torch.cuda.synchronize()
        check_hy("graph")
        e0.record(stream)
        done = 0
        while done < e2e_steps:
            egraphs[(done // chunk) % copies].replay()
            done += chunk
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / e2e_steps, eager_ms

    e2e_ms, eager_ms = timed_e2e(e2e_step)
    ce_ms, ce_eager_ms = timed_e2e(e2e_step_ce)
    gbs = lambda ms: round(step_bytes / (ms * 1e-3) / 1e9, 1)
    e2e = {"value": gbs(e2e_ms), "unit": "GB/s",
           "h2d_bytes_per_step": int(hx_bytes),
           "d2h_bytes_per_step": int(hy_bytes),
           "ms_per_step": round(e2e_ms, 5),
           "eager": {"value": gbs(eager_ms), "ms_per_step": round(eager_ms, 5)},
           "copy_engine": {"value": gbs(ce_ms), "ms_per_step": round(ce_ms, 5),
                           "eager": {"value": gbs(ce_eager_ms), "ms_per_step": round(ce_eager_ms, 5)}},
           "timing": "per step: the step's x (pinned host, packed) copied to the device by exl3_copy_in "
                     "(SM loads over NVLink-C2C, a programmatic dependent launch), the three linears through "
                     "the C ABI writing their y straight into pinned host memory; all inside the timed region, "
                     "in stream order; captured in CUDA graphs of 10 steps as a decode loop runs them "
                     "(eager: the same calls issued from Python every step; copy_engine: one packed "
                     "cudaMemcpyAsync each way instead)"}

    prefill = bench_prefill(args, bf16, src) if not args.skip_prefill else None
    extras = bench_extras() if not args.skip_prefill else None
    configs = bench_configs() if not args.skip_prefill else None
    for d in dcases:
        assert tq.exl3_check_device_error(d["ws"]) == 0

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u16 trellis -> f32 accumulate, f16 out",
        "data": "synthetic (seeded PCG64: uniform trellis, +-1 suh/svh, x ~ N(0,1) fp16)",
        "config": {"workload": WORKLOAD, "K": 4, "k": 5120, "n": list(synth.CONFIG2_N), "M": 1,
                   "l2": "3 rotating weight copies (369 MB > 2x L2), no flush",
                   "weight_prefetch": prefetch,
                   "parallelism": "single GPU; replicas only"},
        "gpu_launches": int(args.steps * len(dcases)),
        "step": "the three M=1 linears (one GEMV kernel each; programmatic dependent launches when "
                "weight_prefetch), captured 10 steps per CUDA graph",
        "roofline": roofline, "e2e": e2e, "clocks": clk.summary(), "prefill": prefill, "configs": configs,
        "other": extras,
    }
    if not args.skip_cpu and _world() == 1:   # the oracle baseline: rank 0 of a one-GPU run only
        out["cpu_baseline"] = cpu_baseline(args)
    return out


def bench_prefill(args, bf16_peak, src):
    """M = 4096, k = 5120, n = 17408, K = 4 (fp16 path): TFLOP/s of the whole call."""
    import torch
    import trellis_quantized_gb300 as tq
    c = synth.config4()
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                     else np.ascontiguousarray(a)).cuda()
    x, t, suh, svh = dev(c.x), dev(c.trellis), dev(c.suh), dev(c.svh)
    ws = tq.workspace(tq.exl3_linear_workspace_size(c.M, c.k, c.n, c.K))
    y = torch.empty((c.M, c.n), dtype=torch.float16, device="cuda")
    for _ in range(3):
        tq.exl3_linear(x, t, suh, svh, 4, y=y, workspace_buf=ws)
    torch.cuda.synchronize()
    reps = 10
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        tq.exl3_linear(x, t, suh, svh, 4, y=y, workspace_buf=ws)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    flops = 2.0 * c.M * c.k * c.n
    tf = flops / (ms * 1e-3) / 1e12
    # int8 variant: same shapes, q_x/q_w integer-exact on the f16 tensor path
    ws8 = tq.workspace(tq.exl3_linear_int8_workspace_size(c.M, c.k, c.n, c.K))
    for _ in range(3):
        tq.exl3_linear_int8(x, t, suh, svh, 4, y=y, workspace_buf=ws8)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        tq.exl3_linear_int8(x, t, suh, svh, 4, y=y, workspace_buf=ws8)
    b.record()
    torch.cuda.synchronize()
    ms8 = a.elapsed_time(b) / reps
    tf8 = flops / (ms8 * 1e-3) / 1e12
    return {"workload": "M=4096 k=5120 n=17408 K=4 fp16 out", "ms": round(ms, 4), "tflops": round(tf, 1),
            "peak_tflops": bf16_peak, "peak_source": src + " bf16 burst (fp16 dense rate = bf16)", "frac": round(tf / bf16_peak, 4),
            "path": "input RHT + transposed reconstruct + tcgen05/TMEM GEMM with fused output RHT",
            "int8": {"ms": round(ms8, 4), "tops": round(tf8, 1), "frac_of_f16_peak": round(tf8 / bf16_peak, 4),
                     "path": "quantise + q_w reconstruct + exact int32 on tcgen05 kind::f16 (no kind::i8 on sm_103a)"}}


def _timed(fn, reps=10, warm=3):
    """Device time per call: the call is captured in a CUDA graph of `reps`
    back-to-back calls, replayed and timed with CUDA events."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(3):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (3 * reps)


L2_BYTES = 129 * 2 ** 20       # GB300 L2; rotated weight copies exceed 2x this
ROTATE_BYTES = 2 * L2_BYTES + 8 * 2 ** 20


def _copies_for(nbytes: int, minimum: int = 3) -> int:
    """Weight copies to rotate so that together they exceed twice the L2."""
    return max(minimum, -(-ROTATE_BYTES // max(nbytes, 1)))


def _timed_rotating(calls, rounds=4, warm=2):
    """Device time per call of a list of closures (one per weight copy, so
    that consecutive calls read different copies): `rounds` passes over the
    list captured in one CUDA graph, replayed and timed with CUDA events."""
    import torch
    for _ in range(warm):
        for f in calls:
            f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(rounds):
            for f in calls:
                f()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(2):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (2 * rounds * len(calls))


def _linear_line(case, ms, hbm):
    gb = linear_bytes(case) / (ms * 1e-3) / 1e9
    return {"us": round(ms * 1e3, 2), "GBs": round(gb, 1), "frac": round(gb / hbm, 4),
            "tflops": round(2.0 * case.M * case.k * case.n / (ms * 1e-3) / 1e12, 2)}


def bench_configs(which=("1", "2", "3")):
    """Every linear workload, each call timed on weight copies that rotate
    through more than twice the L2 (so the weights come from HBM), M = 1
    with weight prefetch on as in a decode loop:
      config1  k=2048 n=512 K=4 M=1 (a latency figure: 0.5 MB of weights)
      config2  k=5120, n in {5120, 17408, 25600}, K=4, M in {1, 4, 16}, fp16 and fp32 out
      config3  k=n=4096, K=2..8, M in {1, 8, 64} (fp16 out; int8 variant at M=64)"""
    import torch
    import trellis_quantized_gb300 as tq
    hbm = peaks()[0]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                     else np.ascontiguousarray(a)).cuda()
    prev = tq.exl3_set_weight_prefetch(True)
    out = {}

    def run(case, out_dtype=tq.EXL3_OUT_F16, int8=False):
        x, suh, svh = dev(case.x), dev(case.suh), dev(case.svh)
        base = dev(case.trellis)
        ts = [base] + [base.clone() for _ in range(_copies_for(base.numel() * 2) - 1)]
        if int8:
            ws = tq.workspace(tq.exl3_linear_int8_workspace_size(case.M, case.k, case.n, case.K))
        else:
            ws = tq.workspace(tq.exl3_linear_workspace_size(case.M, case.k, case.n, case.K))
        y = torch.empty((case.M, case.n), dtype=torch.float32 if out_dtype == tq.EXL3_OUT_F32 else torch.float16,
                        device="cuda")
        if int8:
            calls = [lambda t=t: tq.exl3_linear_int8(x, t, suh, svh, case.K, y=y, workspace_buf=ws) for t in ts]
        else:
            calls = [lambda t=t: tq.exl3_linear(x, t, suh, svh, case.K, out_dtype=out_dtype, y=y, workspace_buf=ws)
                     for t in ts]
        ms = _timed_rotating(calls, rounds=2 if case.M > 16 else 4)
        assert tq.exl3_check_device_error(ws) == 0
        del ts, ws, y
        return ms

    try:
        if "1" in which:
            c = synth.config1()
            out["config1_k2048_n512_K4_M1"] = dict(_linear_line(c, run(c), hbm),
                                                   note="0.5 MB of weights: a latency figure (launch-bound)")
        if "2" in which:
            for n in synth.CONFIG2_N:
                for M in synth.CONFIG2_M:
                    c = synth.config2(n, M)
                    for od, tag in ((tq.EXL3_OUT_F16, "f16"), (tq.EXL3_OUT_F32, "f32")):
                        out[f"config2_k5120_n{n}_K4_M{M}_{tag}"] = _linear_line(c, run(c, od), hbm)
        if "3" in which:
            for K in synth.CONFIG3_K:
                for M in synth.CONFIG3_M:
                    c = synth.config3(K, M)
                    out[f"config3_k4096_n4096_K{K}_M{M}"] = _linear_line(c, run(c), hbm)
                c = synth.config3(K, 64)
                out[f"config3_k4096_n4096_K{K}_M64_int8"] = _linear_line(c, run(c, int8=True), hbm)
    finally:
        tq.exl3_set_weight_prefetch(prev)
    return {"per_call": out, "peak_GBs": hbm,
            "timing": "CUDA graph of back-to-back calls over weight copies rotating through > 2x L2; "
                      "GB/s = packed trellis + x + suh + svh + y bytes per call"}


MOE_T = (1, 16, 32, 64, 128, 4096)


def bench_extras(only=None, moe_tokens=None):
    """Small-M linears (config 2 shapes) and the grouped MoE (config 5) per call."""
    import torch
    import trellis_quantized_gb300 as tq
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                     else np.ascontiguousarray(a)).cuda()
    # fused shards: gate and up of the dense family (2 x k=5120 -> n=17408,
    # K=4) at M = 1, as one grouped-GEMV launch and as two linears; two
    # copies of the weights (178 MB, more than L2) alternate; weight
    # prefetch on, as in a decode loop
    shards = {}
    if only in (None, "small"):
        cs = [synth.linear_case(2, 80 + i, 1, 5120, 17408, 4) for i in range(4)]
        x = dev(cs[0].x)
        copies = []
        for j in (0, 2):
            copies.append((dev(np.stack([cs[j].trellis, cs[j + 1].trellis])), dev(np.stack([cs[j].suh, cs[j + 1].suh])),
                           dev(np.stack([cs[j].svh, cs[j + 1].svh]))))
        ys = torch.empty((2, 1, 17408), dtype=torch.float16, device="cuda")
        ws = tq.workspace(max(tq.exl3_linear_shards_workspace_size(1, 5120, 17408, 4, 2),
                              tq.exl3_linear_workspace_size(1, 5120, 17408, 4)))
        prev = tq.exl3_set_weight_prefetch(True)
        try:
            turn = [0]

            def fused():
                t, su, sv = copies[turn[0] % 2]
                turn[0] += 1
                tq.exl3_linear_shards(x, t, su, sv, 4, y=ys, workspace_buf=ws)

            def separate():
                t, su, sv = copies[turn[0] % 2]
                turn[0] += 1
                for i in range(2):
                    tq.exl3_linear(x, t[i], su[i], sv[i], 4, y=ys[i], workspace_buf=ws)

            one = _timed(fused)
            two = _timed(separate)
        finally:
            tq.exl3_set_weight_prefetch(prev)
        gb = 2 * linear_bytes(cs[0]) / 1e9
        shards = {"one_launch": {"ms": round(one, 4), "GBs": round(gb / (one * 1e-3), 1)},
                  "two_linears": {"ms": round(two, 4), "GBs": round(gb / (two * 1e-3), 1)}}
        del copies, x, ys
    # shards of different widths at M = 1, one launch against one linear
    # each, weight prefetch on: q, k, v of grouped-query attention (k=5120,
    # n = 5120 + 1024 + 1024, 8 weight copies = 147 MB) and the three
    # linears of the decode sweep (n = 5120 + 17408 + 25600, 3 copies =
    # 369 MB), both more than L2
    var = {}
    if only in (None, "small"):
        for name, widths, ncopy in (("qkv_gqa_k5120_n5120+1024+1024", (5120, 1024, 1024), 8),
                                    ("sweep_k5120_n5120+17408+25600", (5120, 17408, 25600), 3)):
            cs = [[synth.linear_case(2, 60 + 10 * j + i, 1, 5120, n, 4) for i, n in enumerate(widths)]
                  for j in range(ncopy)]
            x = dev(cs[0][0].x)
            copies = [(dev(np.concatenate([c.trellis.reshape(-1) for c in cc])), dev(np.stack([c.suh for c in cc])),
                       dev(np.concatenate([c.svh for c in cc])), [dev(c.trellis) for c in cc]) for cc in cs]
            yv = torch.empty(sum(widths), dtype=torch.float16, device="cuda")
            ws = tq.workspace(tq.exl3_linear_shards_var_workspace_size(1, 5120, widths, 4))
            prev = tq.exl3_set_weight_prefetch(True)
            try:
                turn = [0]

                def fused():
                    t, su, sv, _ = copies[turn[0] % ncopy]
                    turn[0] += 1
                    tq.exl3_linear_shards_var(x, t, su, sv, widths, 4, y=yv, workspace_buf=ws)

                def separate():
                    _, su, sv, ts = copies[turn[0] % ncopy]
                    turn[0] += 1
                    off = 0
                    for i, n in enumerate(widths):
                        tq.exl3_linear(x, ts[i], su[i], sv[off:off + n], 4, y=yv[off:off + n].view(1, n),
                                       workspace_buf=ws)
                        off += n

                one = _timed(fused, reps=ncopy * 2)
                sep = _timed(separate, reps=ncopy * 2)
            finally:
                tq.exl3_set_weight_prefetch(prev)
            gb = sum(linear_bytes(c) for c in cs[0]) / 1e9
            var[name] = {"one_launch": {"ms": round(one, 4), "GBs": round(gb / (one * 1e-3), 1)},
                         "one_linear_each": {"ms": round(sep, 4), "GBs": round(gb / (sep * 1e-3), 1)}}
            del copies, x, yv
    # the row-invariant mode (every M through the 32-token-wide fused
    # kernel, 32 rows at a time): its cost against the default paths
    inv = {}
    if only in (None, "small"):
        prev = tq.exl3_set_row_invariant(True)
        try:
            for i, M in enumerate((1, 16, 4096)):
                c = synth.linear_case(2, 90 + i, M, 5120, 17408, 4)
                x, t, suh, svh = dev(c.x), dev(c.trellis), dev(c.suh), dev(c.svh)
                ws = tq.workspace(tq.exl3_linear_workspace_size(M, c.k, c.n, c.K))
                y = torch.empty((M, c.n), dtype=torch.float16, device="cuda")
                ms = _timed(lambda: tq.exl3_linear(x, t, suh, svh, 4, y=y, workspace_buf=ws), reps=3 if M > 128 else 10)
                inv[f"M{M}"] = {"ms": round(ms, 4), "tflops": round(2.0 * M * c.k * c.n / (ms * 1e-3) / 1e12, 2)}
                del x, ws, y
        finally:
            tq.exl3_set_row_invariant(prev)
    # grouped experts over the whole 302 MB arena; few-token calls rotate
    # through several routing draws so that consecutive calls hit different
    # experts (the weights they read come from HBM, not from the L2)
    moe = {}
    for T in ((moe_tokens or MOE_T) if only in (None, "moe") else ()):
        c = synth.config5(T) if T in synth.CONFIG5_T else synth.moe_case(5, 10 + T, T,
                                                                           name=f"E256 top8 h2048 i512 K3 T{T}")
        d = dict(x=dev(c.x), t13=dev(c.w13.trellis), s13=dev(c.w13.suh),
                 v13=dev(c.w13.svh), t2=dev(c.w2.trellis), s2=dev(c.w2.suh), v2=dev(c.w2.svh))
        w13 = tq.expert_proj(d["t13"], d["s13"], d["v13"], c.K)
        w2 = tq.expert_proj(d["t2"], d["s2"], d["v2"], c.K)
        # between two calls with the same routing, more than 2x L2 of expert
        # weights goes through (T <= 4: 32 draws of about 9.4 MB per token)
        nr = 32 if T <= 4 else (16 if T <= 64 else (4 if T <= 128 else 1))
        routes = [(c.ids, c.weights)] + [synth.routing(synth.rng_for(5, 1000 + 10 * T + r), T, c.E, c.topk)
                                         for r in range(nr - 1)]
        rd = [(dev(i), dev(w)) for i, w in routes]
        ws = tq.workspace(tq.exl3_moe_workspace_size(T, c.topk, c.E, w13, w2))
        y = torch.empty((T, c.hidden), dtype=torch.float16, device="cuda")
        calls = [lambda i=i, w=w: tq.exl3_moe_grouped(d["x"], i, w, w13, w2, c.E, y=y, workspace_buf=ws)
                 for i, w in rd]
        ms = _timed_rotating(calls, rounds=max(1, 6 // nr)) if nr > 1 else _timed(calls[0], reps=3)
        assert tq.exl3_check_device_error(ws) == 0
        used = np.mean([len(np.unique(i)) for i, _ in routes])
        per_expert = (c.w13.trellis.nbytes + c.w2.trellis.nbytes) // c.E
        flops = 2.0 * T * c.topk * (2 * c.hidden * c.inter + c.inter * c.hidden)
        hbm = peaks()[0]
        gbs = used * per_expert / (ms * 1e-3) / 1e9
        moe[f"T{T}"] = {"ms": round(ms, 4), "experts_hit": round(float(used), 1),
                        "unique_weight_GBs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                        "tflops": round(flops / (ms * 1e-3) / 1e12, 2), "routings_rotated": nr}
        del d, rd, ws
    # per-expert widths: the same shape with experts 0-127 at K = 3 and
    # 128-255 at K = 4 (down the other way round), two runs per projection
    mixed = {}
    for T in ((moe_tokens or (1, 128)) if only in (None, "moe") else ()):
        K13, K2 = [3] * 128 + [4] * 128, [4] * 128 + [3] * 128
        c = synth.mixed_moe_case(59, 10 + T, T, K13, K2)
        d = dict(x=dev(c.x), ids=dev(c.ids), w=dev(c.weights), t13=dev(c.w13.trellis), s13=dev(c.w13.suh),
                 v13=dev(c.w13.svh), t2=dev(c.w2.trellis), s2=dev(c.w2.suh), v2=dev(c.w2.svh))
        w13 = tq.expert_proj_mixed(d["t13"], d["s13"], d["v13"], K13, c.hidden, c.inter)
        w2 = tq.expert_proj_mixed(d["t2"], d["s2"], d["v2"], K2, c.inter, c.hidden)
        ws = tq.workspace(tq.exl3_moe_mixed_workspace_size(T, c.topk, c.E, w13, w2))
        y = torch.empty((T, c.hidden), dtype=torch.float16, device="cuda")
        nr = 32 if T <= 4 else (4 if T <= 128 else 1)   # routings rotated, as for one width
        routes = [(c.ids, c.weights)] + [synth.routing(synth.rng_for(59, 1000 + 10 * T + r), T, c.E, c.topk)
                                         for r in range(nr - 1)]
        rd = [(dev(i), dev(w)) for i, w in routes]
        calls = [lambda i=i, w=w: tq.exl3_moe_grouped_mixed(d["x"], i, w, w13, w2, c.E, y=y, workspace_buf=ws)
                 for i, w in rd]
        ms = _timed_rotating(calls, rounds=max(1, 6 // nr)) if nr > 1 else _timed(calls[0], reps=3)
        assert tq.exl3_check_device_error(ws) == 0
        words13 = [2 * (c.hidden // 16) * (c.inter // 16) * 16 * K for K in K13]
        words2 = [(c.inter // 16) * (c.hidden // 16) * 16 * K for K in K2]
        ubytes = np.mean([2 * sum(words13[e] + words2[e] for e in np.unique(i)) for i, _ in routes])
        used = np.mean([len(np.unique(i)) for i, _ in routes])
        mixed[f"T{T}"] = {"ms": round(ms, 4), "experts_hit": round(float(used), 1),
                          "unique_weight_GBs": round(ubytes / (ms * 1e-3) / 1e9, 1), "routings_rotated": nr}
        del d
    return {"shards_gate_up_k5120_n17408x2_M1": shards, "shards_var_M1": var,
            "row_invariant_k5120_n17408": inv, "moe_E256_top8_h2048_i512_K3": moe,
            "moe_mixed_E256_top8_h2048_i512_K3K4": mixed,
            "note": "MoE: device remap + gather/RHT + two grouped tcgen05 kernels decoding the experts' trellis "
                    "on the fly + fixed-order combine (expert tiles of 32/128/160/256 rows by routed rows per "
                    "expert); up to 32 routed rows, or up to 1.25 per expert: one grouped M=1 GEMV launch per "
                    "projection + combine. Mixed widths: the tile kernels once per run of equal width (two runs "
                    "here); up to 32 routed rows, or up to one per expert, one grouped GEMV launch per "
                    "projection over all widths"}


# ---------------------------------------------------------------- pipe ceilings

# (mix id, name, chains per thread, lane-instructions per chain-iteration by
# class (an ffma2 is one instruction of two FMAs), weights per chain-iteration)
PIPE_MIXES = [
    (0, "imad", 8, {"imad": 1}, 0), (1, "dp4a", 8, {"dp4a": 1}, 0),
    (2, "imad+dp4a", 8, {"imad": 1, "dp4a": 1}, 0),
    (3, "fhfma", 8, {"fhfma": 1}, 0), (4, "ffma2", 8, {"ffma2": 1}, 0), (5, "ffma", 8, {"ffma": 1}, 0),
    (6, "decode_fhfma", 8, {"imad": 1, "dp4a": 1, "fhfma": 1}, 1),
    (7, "decode_ffma2", 8, {"imad": 1, "dp4a": 1, "ffma2": 0.5}, 1),
    (8, "alu", 8, {"alu": 1}, 0),
    (9, "decode_k4_ffma2", 1, {"alu": 13, "imad": 8, "dp4a": 8, "ffma2": 4}, 8),
    (10, "decode_k4_fhfma", 1, {"alu": 13, "imad": 8, "dp4a": 8, "fhfma": 8}, 8),
    (11, "hmma_m16n8k16", 1, {"hmma_warp_inst": 8 / 32}, 0),
    (12, "decode_k4_hmma", 1, {"alu": 26, "imad": 16, "dp4a": 16, "hmma_warp_inst": 4 / 32}, 16),
    (13, "decode_ffma", 8, {"imad": 1, "dp4a": 1, "ffma": 1}, 1),
    (14, "decode_k4_ffma", 1, {"alu": 13, "imad": 8, "dp4a": 8, "ffma": 8}, 8),
]


def bench_pipes(iters=20000):
    """Instruction throughput per SM clock (lane-operations, or decoded
    weights, per clock per SM) of the decode's instruction classes, measured
    with clock64 in one 1024-thread CTA per SM; see ubench/pipes.cu."""
    import ctypes

    import torch
    from trellis_quantized_gb300 import _build
    L = ctypes.CDLL(_build.build_ubench())
    L.exl3_ubench_pipes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                    ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cyc = torch.zeros(sms, dtype=torch.int64, device="cuda")
    sink = torch.zeros(1024, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    res = {}
    for mix, name, chains, ops, wpc in PIPE_MIXES:
        for rep in range(2):   # the first run warms up
            rc = L.exl3_ubench_pipes(mix, sms, iters, cyc.data_ptr(), sink.data_ptr(), ctypes.c_void_p(stream))
            assert rc == 0, f"ubench mix {mix}: cuda error {rc}"
            torch.cuda.synchronize()
        cycles = float(cyc.double().median().item())
        units = 1024.0 * iters * chains / cycles   # chain-iterations per clock per SM
        r = {k: round(v * units, 2) for k, v in ops.items()}
        if wpc:
            r["weights_per_clk"] = round(wpc * units, 2)
        res[name] = r
    return {"sms": sms, "per_sm_per_clock": res,
            "method": "one 1024-thread CTA per SM, 8 independent chains per thread, clock64 cycles (median CTA)"}


# ---------------------------------------------------------- single calls

def one_linear(M, n, calls=5):
    """exl3_linear on the dense decode family (k = 5120, K = 4, config-2
    inputs at M rows and n columns), `calls` times: the case a profiler
    captures one launch of (no timing)."""
    import torch
    import trellis_quantized_gb300 as tq
    c = synth.linear_case(2, 900 + M, M, 5120, n, 4)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                     else np.ascontiguousarray(a)).cuda()
    x, t, suh, svh = dev(c.x), dev(c.trellis), dev(c.suh), dev(c.svh)
    for _ in range(calls):
        y = tq.exl3_linear(x, t, suh, svh, 4)
    torch.cuda.synchronize()
    return {"case": f"k5120 n{n} K4 M{M}", "calls": calls, "y_shape": list(y.shape)}


def one_moe(T, calls=3, mixed=False):
    """exl3_moe_grouped on the MoE workload (256 experts, top-8, hidden
    2048, inter 512, K = 3) at T tokens, `calls` times (no timing); with
    `mixed`, exl3_moe_grouped_mixed with experts 0-127 at K = 3 and 128-255 at
    K = 4 for gate+up (down the other way round)."""
    import torch
    import trellis_quantized_gb300 as tq
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                                     else np.ascontiguousarray(a)).cuda()
    if mixed:
        K13, K2 = [3] * 128 + [4] * 128, [4] * 128 + [3] * 128
        c = synth.mixed_moe_case(59, 10 + T, T, K13, K2)
        d = {k: dev(v) for k, v in dict(x=c.x, ids=c.ids, w=c.weights, t13=c.w13.trellis, s13=c.w13.suh,
                                         v13=c.w13.svh, t2=c.w2.trellis, s2=c.w2.suh, v2=c.w2.svh).items()}
        w13 = tq.expert_proj_mixed(d["t13"], d["s13"], d["v13"], K13, c.hidden, c.inter)
        w2 = tq.expert_proj_mixed(d["t2"], d["s2"], d["v2"], K2, c.inter, c.hidden)
        for _ in range(calls):
            y = tq.exl3_moe_grouped_mixed(d["x"], d["ids"], d["w"], w13, w2, c.E)
        torch.cuda.synchronize()
        return {"case": f"E256 top8 h2048 i512 K3/K4 T{T}", "calls": calls, "y_shape": list(y.shape)}
    c = synth.config5(T) if T in synth.CONFIG5_T else synth.moe_case(5, 10 + T, T)
    d = {k: dev(v) for k, v in dict(x=c.x, ids=c.ids, w=c.weights, t13=c.w13.trellis, s13=c.w13.suh,
                                     v13=c.w13.svh, t2=c.w2.trellis, s2=c.w2.suh, v2=c.w2.svh).items()}
    w13 = tq.expert_proj(d["t13"], d["s13"], d["v13"], c.K)
    w2 = tq.expert_proj(d["t2"], d["s2"], d["v2"], c.K)
    for _ in range(calls):
        y = tq.exl3_moe_grouped(d["x"], d["ids"], d["w"], w13, w2, c.E)
    torch.cuda.synchronize()
    return {"case": f"E256 top8 h2048 i512 K3 T{T}", "calls": calls, "y_shape": list(y.shape)}


# ---------------------------------------------------------------- dense peaks

def bench_peaks():
    """Dense tensor-core peaks for the prefill fractions, measured the way
    the driver measures bf16: torch.matmul of 8192^3 (2 N^3 flop), best of
    10 (burst) and back to back for about 4 s (sustained); fp16 and bf16 on
    cuBLAS, and int8 through torch._int_mm (s8 x s8 -> s32) for context."""
    import torch
    N = 8192
    out = {}
    for name, dt in (("fp16", torch.float16), ("bf16", torch.bfloat16), ("int8", torch.int8)):
        if dt == torch.int8:
            a = torch.randint(-127, 128, (N, N), dtype=dt, device="cuda")
            b = torch.randint(-127, 128, (N, N), dtype=dt, device="cuda").t().contiguous().t()
            mm = lambda: torch._int_mm(a, b)
        else:
            a = torch.randn(N, N, dtype=dt, device="cuda")
            b = torch.randn(N, N, dtype=dt, device="cuda")
            mm = lambda: torch.matmul(a, b)
        try:
            for _ in range(3):
                mm()
            torch.cuda.synchronize()
        except Exception as e:   # an unsupported int8 layout or kernel: report, do not guess
            out[name] = {"error": str(e).splitlines()[0][:200]}
            continue
        best = float("inf")
        for _ in range(10):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            mm()
            e.record()
            torch.cuda.synchronize()
            best = min(best, s.elapsed_time(e))
        reps = max(1, int(4000.0 / best))
        with ClockSampler(torch.cuda.current_device()) as clk:
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(reps):
                mm()
            e.record()
            torch.cuda.synchronize()
        sus = s.elapsed_time(e) / reps
        flop = 2.0 * N ** 3
        unit = "TOP/s" if dt == torch.int8 else "TFLOP/s"
        out[name] = {"burst": round(flop / (best * 1e-3) / 1e12, 1), "sustained": round(flop / (sus * 1e-3) / 1e12, 1),
                     "unit": unit, "clocks": clk.summary()}
        del a, b
    return {"N": N, "peaks": out, "method": "torch.matmul / torch._int_mm of N^3, CUDA events; burst = best of 10, "
                                            "sustained = mean of back-to-back calls over ~4 s"}


# ------------------------------------------------------------------------- oracle

CPU_SAMPLE_S = 10.0   # seconds of oracle work in the bench's cpu_baseline


def cpu_baseline(args):
    """The CPU oracle, as it stands, on a bounded sample of the workload: the
    sweep's three M = 1 linears (decode + float64 contraction + transforms),
    repeated whole until at least CPU_SAMPLE_S seconds have passed."""
    import oracle
    oracle.build()
    cases = [synth.config2(n, 1) for n in synth.CONFIG2_N]
    oracle.linear(cases[0].x[:1, :128], cases[0].trellis[:8, :8], cases[0].suh[:128], cases[0].svh[:128], 4)  # load
    step_bytes = sum(linear_bytes(c) for c in cases)
    reps = 0
    t0 = time.perf_counter()
    while True:
        for c in cases:
            oracle.linear(c.x, c.trellis, c.suh, c.svh, 4)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= CPU_SAMPLE_S:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": round(step_bytes * reps / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} repetitions of the step's three k=5120 K=4 M=1 linears (n = 5120, 17408, 25600; "
                      f"{step_bytes} algorithmic bytes each) in {dt:.1f} s"}


def run_reference(args):
    """--impl reference: the CPU oracle timed as the reference arm."""
    import oracle
    oracle.build()
    c = synth.config2(5120, 1)
    for _ in range(args.warmup):
        oracle.linear(c.x[:1, :128], c.trellis[:8, :8], c.suh[:128], c.svh[:128], 4)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.linear(c.x, c.trellis, c.suh, c.svh, 4)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = linear_bytes(c) / dt / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded PCG64)",
            "config": {"workload": WORKLOAD + " (each step: the n=5120 linear, a bounded sample)", "K": 4,
                       "k": 5120, "n": [5120], "M": 1, "parallelism": "CPU oracle"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "one k=5120 n=5120 K=4 M=1 linear per step"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-prefill", action="store_true")
    ap.add_argument("--no-prefetch", action="store_true",
                    help="launch the step's linears plainly (no weight prefetch across launches)")
    ap.add_argument("--only", choices=["small", "moe", "prefill", "pipes", "peaks", "configs", "linear", "moecall"],
                    default=None,
                    help="run one extra section alone and print its JSON (for profiling)")
    ap.add_argument("--configs", nargs="*", default=["1", "2", "3"], help="workloads of --only configs")
    ap.add_argument("--m", type=int, default=16, help="rows of --only linear")
    ap.add_argument("--n", type=int, default=17408, help="columns of --only linear")
    ap.add_argument("--t", type=int, default=128, help="tokens of --only moecall")
    ap.add_argument("--mixed", action="store_true", help="--only moecall with two expert widths")
    ap.add_argument("--moe-tokens", type=int, nargs="*", default=None,
                    help="token counts of the MoE section (default: all of the MoE workload's)")
    args = ap.parse_args()
    if args.only:
        import torch
        if args.only == "prefill":
            print(json.dumps(bench_prefill(args, *peaks()[1:])))
        elif args.only == "pipes":
            print(json.dumps(bench_pipes()))
        elif args.only == "peaks":
            print(json.dumps(bench_peaks()))
        elif args.only == "configs":
            print(json.dumps(bench_configs(tuple(args.configs))))
        elif args.only == "linear":
            print(json.dumps(one_linear(args.m, args.n)))
        elif args.only == "moecall":
            print(json.dumps(one_moe(args.t, mixed=args.mixed)))
        else:
            print(json.dumps(bench_extras(args.only, args.moe_tokens)))
        return
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if args.steps > 20:
            args.steps = 3
        if rank == 0:
            print(json.dumps(run_reference(args)))
        return
    if args.gpus > 1 or int(os.environ.get("WORLD_SIZE", "1")) > 1:
        # replicas only: every rank runs the same single-GPU workload
        import torch
        import torch.distributed as dist
        local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        out = aggregate_replicas(run_ours(args), dist, "cuda")
        if rank == 0:
            print(json.dumps(out))
        dist.destroy_process_group()
        return
    print(json.dumps(run_ours(args)))


if __name__ == "__main__":
    main()
