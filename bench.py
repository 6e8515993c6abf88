"""Benchmark of the differential-attention forward on GB300 (one JSON line).

A step is one DIFF V1 layer forward of the selected workload: lambda_init and
the lambda re-parameterisation (one warp), then the fused forward (two
softmax maps, their lambda-weighted difference times V, the per-head RMSNorm
with (1 - lambda_init)) on inputs already resident in HBM.  For the DIFF V2
workload a step is the V2 forward.  The default workload is the largest one
that fits one GPU (B1 H12 n65536 d128, causal: 4.0e13 FLOP a step);
``--config`` selects another, and the line's ``configs`` object reports every
workload measured in the same run.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--config C]
       python bench.py --impl reference ...   (the fp64 CPU oracle, timed on
       the host cores on a bounded sample of the same workload)
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "diff-attn fwd TFLOP/s (bf16) and % of GB300 dense tensor peak; tokens/s"
DEFAULT_CONFIG = 4
FLUSH_BYTES = 512 << 20  # > 129 MB L2


def flops(w) -> float:
    """Algorithmic FLOPs of one forward: V1 12 n^2 d per (b, h), V2 4 n^2 d per query head; x1/2 causal."""
    if w.kind == "v1":
        f = 12.0 * w.n * w.n * w.d * w.B * w.H
    else:
        f = 4.0 * w.n * w.n * w.d * w.B * w.Hq
    return f / 2 if w.causal else f


def hbm_bytes(w) -> float:
    """Algorithmic HBM bytes: every input read once, the output written once."""
    e = 4 if w.dtype == "f32" else 2
    if w.kind == "v1":
        return float(w.B * w.H * w.n * w.d * 8 * e)  # q1 q2 k1 k2 (4d) + v (2d) + out (2d)
    return float(w.B * w.n * w.d * (w.Hq + 2 * w.Hkv + w.Hq // 2) * e)


# DRAM traffic of the dominant kernel per launch (dram__bytes_read.sum +
# dram__bytes_write.sum) from one ncu --set full capture of each workload
# (cold-cache replay; summaries under profiles/).  A figure holds only for the
# kernel it was taken from: it is keyed to the hash of that kernel's source
# files and reported while the hash still matches, null otherwise.
KERNEL_FILES = {
    "v1-bf16-B4H16-n2048-d64": ['onepass.cuh', 'onepass_inst.cuh', 'k_onepass_v1_d64.cu', 'params.h', 'ptx.cuh', 'status.cuh', 'bounds.cuh', 'api.cu'],
    "v1-bf16-B2H12-n4096-d128": ['twopass.cuh', 'twopass_inst.cuh', 'k_twopass_v1_d128.cu', 'params.h', 'ptx.cuh', 'status.cuh', 'bounds.cuh', 'api.cu'],
    "v1-bf16-B1H12-n65536-d128": ['twopass.cuh', 'twopass_inst.cuh', 'k_twopass_v1_d128.cu', 'params.h', 'ptx.cuh', 'status.cuh', 'bounds.cuh', 'api.cu'],
    "v2-bf16-B8Hq32Hkv16-n8192-d128": ['onepass.cuh', 'onepass_inst.cuh', 'k_onepass_v2_d128.cu', 'params.h', 'ptx.cuh', 'status.cuh', 'bounds.cuh', 'api.cu'],
}
NCU_TRAFFIC = {  # workload: (source hash of its kernel, bytes per launch: dram__bytes_read.sum + dram__bytes_write.sum)
    "v1-bf16-B4H16-n2048-d64": ("eda8ec60b9e91f7f", 139291648 + 12816640),
    "v1-bf16-B2H12-n4096-d128": ("a645e087502723ac", 152373248 + 30054400),
    "v1-bf16-B1H12-n65536-d128": ("a645e087502723ac", 1761939968 + 405562368),
    "v2-bf16-B8Hq32Hkv16-n8192-d128": ("ae8a8492959243df", 1073912832 + 254664704),
}


def kernel_sources_hash(workload: str) -> str:
    """Hash of the source files of the kernel that runs `workload`."""
    import hashlib
    d = os.path.join(ROOT, "differential_attention_03_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(KERNEL_FILES.get(workload, [])):
        h.update(f.encode())
        with open(os.path.join(d, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    if workload not in NCU_TRAFFIC:
        return None
    digest, nbytes = NCU_TRAFFIC[workload]
    return nbytes if kernel_sources_hash(workload) == digest else None


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """Polls nvidia-smi from a thread while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index: int, period_s: float = 0.05):
        import threading
        self.index = index
        self.period = period_s
        self.rows = []
        self.stop_evt = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.error = None

    def _run(self):
        while not self.stop_evt.is_set():
            try:
                out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                      "--format=csv,noheader,nounits"], capture_output=True, text=True,
                                     timeout=10).stdout
                stamp = time.perf_counter()
                for line in out.splitlines():
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 7:
                        self.rows.append((stamp, parts))
            except Exception as e:  # noqa: BLE001
                self.error = str(e)
                return
            self.stop_evt.wait(self.period)

    def start(self):
        self.thread.start()

    def stop(self, window=None):
        """Summary of the samples taken inside `window` = (t0, t1) (perf_counter seconds), the
        timed region; of every sample if none fell inside it."""
        self.stop_evt.set()
        self.thread.join(timeout=15)
        rows = self.rows
        scope = "whole run"
        if window is not None:
            inside = [r for r in rows if window[0] <= r[0] <= window[1]]
            if inside:
                rows, scope = inside, "timed region"
        sm, mx, reasons = [], [], set()
        for _, parts in rows:
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.error or "no samples"], "samples": 0}
        loaded = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "scope": scope}


# --------------------------------------------------------------------------- our path
def make_step(w, x, da):
    """Returns (step(), kernel-only call, output) for workload w on device tensors x."""
    import torch
    if w.kind == "v1":
        lam = torch.empty(1, device=x["q1"].device, dtype=torch.float32)
        out = torch.empty(x["v"].shape, device=x["v"].device, dtype=x["v"].dtype)

        def lam_call():
            lin = da.lambda_init(w.layer)
            da.lambda_reparam(x["lq1"], x["lk1"], x["lq2"], x["lk2"], lin, out=lam)

        def fwd_call():
            da.diffattn_forward(x["q1"], x["q2"], x["k1"], x["k2"], x["v"], lam, da.lambda_init(w.layer),
                                gamma=x["gamma"], causal=w.causal, out=out)
        return lam_call, fwd_call, out
    out = torch.empty((w.B, w.n, w.Hq // 2, w.d), device=x["q"].device, dtype=x["q"].dtype)

    def fwd_call():
        da.diffattn_v2_forward(x["q"], x["k"], x["v"], x["lam_logits"], causal=w.causal, out=out)
    return (lambda: None), fwd_call, out


def flush_l2(flush):
    """Evict L2 before a timed call: write the 512 MB buffer, then read it back, so that L2 ends up
    holding clean lines of the buffer.  (A write alone leaves ~129 MB of dirty lines whose
    write-backs the next call would pay for while it evicts them: 12-21 us on a 0.27 ms decode.)"""
    flush.zero_()
    flush.sum()


def time_device(w, x, da, steps, warmup, flush, dist=None):
    """Device timing with CUDA events on the launching stream; L2 flushed between steps."""
    import torch
    lam_call, fwd_call, out = make_step(w, x, da)
    stream = torch.cuda.current_stream()
    h0 = time.perf_counter()
    for _ in range(warmup):
        flush_l2(flush)
        lam_call()
        fwd_call()
    host_per_step = (time.perf_counter() - h0) / warmup
    da.device_status()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    c0 = da.launch_count()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    # Hold the stream in a device-side sleep (outside the events) long enough for
    # the host to enqueue every timed step, so that the events see device time
    # only, not gaps while Python marshals the next call.
    torch.cuda._sleep(int(min(2e9, 3.0e9 * host_per_step * steps + 2e6)))
    t0 = time.perf_counter()  # the device sleep above belongs to the timed region's clock window
    for k in range(steps):
        flush_l2(flush)
        ev[k][0].record(stream)
        lam_call()
        ev[k][1].record(stream)
        fwd_call()
        ev[k][2].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    launches = da.launch_count() - c0
    if dist is not None:
        dist.barrier()
    da.device_status()
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    kern_ms = [b.elapsed_time(c) for a, b, c in ev]
    return {"step_ms": sum(step_ms) / steps, "kernel_ms": sum(kern_ms) / steps,
            "kernel_ms_median": statistics.median(kern_ms), "wall_s": wall, "launches": launches, "out": out,
            "window": (t0, t0 + wall)}


def time_e2e(w, x, da, steps):
    """End to end through the C ABI with host buffers.

    V1: diffattn_forward_host takes the step's inputs in page-locked host
    memory and returns the output there (copies in, forward and copies out
    pipelined over batch or token chunks inside the library); lambda and gamma are
    layer parameters resident on the device.  V2: the inputs are copied in
    and the output back around diffattn_v2_forward.  Every step includes the
    copies of its inputs and output.
    """
    import torch
    stream = torch.cuda.current_stream()
    if w.kind == "v1":
        names = ("q1", "q2", "k1", "k2", "v")
        host = {k: x[k].cpu().pin_memory() for k in names}
        lam = torch.empty(1, device=x["q1"].device, dtype=torch.float32)
        lin = da.lambda_init(w.layer)
        out_host = torch.empty(x["v"].shape, dtype=x["v"].dtype).pin_memory()
        ws = torch.empty(da.forward_host_workspace_bytes(x["q1"].dtype, w.B, w.H, w.n, w.d), dtype=torch.uint8,
                         device=x["q1"].device)

        def one():
            da.lambda_reparam(x["lq1"], x["lk1"], x["lq2"], x["lk2"], lin, out=lam)
            da.diffattn_forward_host(host["q1"], host["q2"], host["k1"], host["k2"], host["v"], lam, lin,
                                     gamma=x["gamma"], causal=w.causal, out=out_host, workspace=ws)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()
    else:
        host = {k: t.cpu().pin_memory() for k, t in x.items()}
        dev = {k: torch.empty_like(t) for k, t in x.items()}
        _, fwd_call, out = make_step(w, dev, da)
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()

        def one():
            for k in host:
                dev[k].copy_(host[k], non_blocking=True)
            fwd_call()
            out_host.copy_(out, non_blocking=True)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out.numel() * out.element_size()

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


DECODE_WORKLOADS = [  # (name, B, H or (Hq, Hkv), n, d, key cache): one new token per sequence over n cached tokens
    ("v1-decode-bf16-B8H16-n32768-d64", 8, 16, 32768, 64, "bf16"),
    ("v1-decode-bf16-B8H8-n32768-d128", 8, 8, 32768, 128, "bf16"),
    ("v2-decode-bf16-B8Hq32Hkv16-n32768-d128", 8, (32, 16), 32768, 128, "bf16"),
    # one sequence, long cache: the pairs are split over clusters through the workspace
    ("v1-decode-bf16-B1H16-n131072-d64-workspace", 1, 16, 131072, 64, "bf16"),
    # FP8 (e4m3) key caches, bf16 values
    ("v1-decode-fp8k-B8H16-n32768-d64", 8, 16, 32768, 64, "e4m3"),
    ("v1-decode-fp8k-B8H8-n32768-d128", 8, 8, 32768, 128, "e4m3"),
    ("v2-decode-fp8k-B8Hq32Hkv16-n32768-d128", 8, (32, 16), 32768, 128, "e4m3"),
]


def time_decode(da, flush, B, H, n, d, keys="bf16", runs=20):
    """DIFF decode step over a key/value cache: median CUDA-event time (L2 flushed), HBM GB/s.

    keys "e4m3": the key caches hold FP8 codes (1 byte an element) with one scale per tensor.
    """
    import torch
    g = torch.Generator(device="cuda").manual_seed(1000 + n + d)

    def rnd(*shape):
        return torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    if isinstance(H, tuple):  # DIFF V2: (Hq, Hkv)
        Hq, Hkv = H
        q, k, v = rnd(B, Hq, d), rnd(B, n, Hkv, d), rnd(B, n, Hkv, d)
        lg = torch.randn((B, Hq // 2), generator=g, device="cuda")
        out = torch.empty((B, Hq // 2, d), device="cuda", dtype=torch.bfloat16)
        kb = 1 if keys == "e4m3" else 2  # bytes of a key element
        nbytes_kv = B * n * Hkv * d * (kb + 2) + B * (Hq + Hq // 2) * d * 2  # K and V once; q in, out

        ws = torch.empty(da.v2_decode_workspace_bytes(B, Hq, d), dtype=torch.uint8, device="cuda")
        if keys == "e4m3":
            k8 = (k.float() * (448.0 / 6.0)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
            del k

            def call():
                da.diffattn_v2_decode_fp8k(q, k8, 6.0 / 448.0, v, lg, out=out, workspace=ws)
        else:
            def call():
                da.diffattn_v2_decode(q, k, v, lg, out=out, workspace=ws)
    else:
        q1, q2 = rnd(B, H, d), rnd(B, H, d)
        k1, k2, v = rnd(B, n, H, d), rnd(B, n, H, d), rnd(B, n, H, 2 * d)
        lam = torch.tensor([0.3], device="cuda")
        gamma = torch.ones(2 * d, device="cuda")
        out = torch.empty((B, H, 2 * d), device="cuda", dtype=torch.bfloat16)
        kb = 1 if keys == "e4m3" else 2  # bytes of a key element
        nbytes_kv = B * H * n * d * (2 * kb + 4) + B * H * 4 * d * 2  # K1, K2, V read once; q in, out

        ws = torch.empty(da.decode_workspace_bytes(B, H, d), dtype=torch.uint8, device="cuda")
        if keys == "e4m3":
            k1, k2 = ((t.float() * (448.0 / 6.0)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
                      for t in (k1, k2))

            def call():
                da.diffattn_decode_fp8k(q1, q2, k1, k2, 6.0 / 448.0, 6.0 / 448.0, v, lam, 0.2, gamma=gamma,
                                        out=out, workspace=ws)
        else:
            def call():
                da.diffattn_decode(q1, q2, k1, k2, v, lam, 0.2, gamma=gamma, out=out, workspace=ws)
    for _ in range(3):
        call()
    da.device_status()
    ts = []
    for _ in range(runs):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    da.device_status()
    ms = statistics.median(ts)
    torch.cuda.empty_cache()
    return ms, nbytes_kv


def cpu_baseline(w, x, budget_s=12.0):
    """The fp64 oracle as it stands, on a bounded sample of the same workload.

    Units (one (batch, head) for V1, one (batch, head pair) for V2) are taken in
    order, each with all its query rows in 128-row blocks (heaviest causal
    blocks first), until the time budget is spent; the value is the
    algorithmic causal FLOPs of the rows done divided by the time taken.
    """
    import numpy as np
    import oracle
    cores = len(os.sched_getaffinity(0))
    n = w.n
    order = list(range(0, n, 128))[::-1]
    rows_done, units_done, fl = 0, 0, 0.0
    t0 = time.perf_counter()
    units = [(b, u) for b in range(w.B) for u in range(w.H if w.kind == "v1" else w.Hq // 2)]
    for b, u in units:
        if w.kind == "v1":
            xs = {k: (t[b:b + 1, :, u:u + 1] if t.dim() == 4 else t).cpu() for k, t in x.items()}
            lin = oracle.lambda_init(w.layer)
            lam = oracle.lambda_reparam(xs["lq1"], xs["lk1"], xs["lq2"], xs["lk2"], lin)
            arrs = {k: oracle.diffattn_oracle._f64(xs[k]) for k in ("q1", "q2", "k1", "k2", "v")}
        else:
            kvh = (2 * u) // (w.Hq // w.Hkv)
            xs = {"q": x["q"][b:b + 1, :, 2 * u:2 * u + 2].cpu(), "k": x["k"][b:b + 1, :, kvh:kvh + 1].cpu(),
                  "v": x["v"][b:b + 1, :, kvh:kvh + 1].cpu()}
            arrs = {k: oracle.diffattn_oracle._f64(t) for k, t in xs.items()}
            lg = np.broadcast_to(x["lam_logits"][u:u + 1].cpu().double().numpy(), (1, n, 1))
        for s in order:
            rows = np.arange(s, min(s + 128, n))
            if w.kind == "v1":
                oracle.diff_attn_v1(arrs["q1"], arrs["q2"], arrs["k1"], arrs["k2"], arrs["v"], lam, lin,
                                    xs["gamma"], 1e-5, w.causal, rows)
                per = 12.0 * w.d
            else:
                oracle.diff_attn_v2(arrs["q"], arrs["k"], arrs["v"], lg, w.causal, rows=rows)
                per = 8.0 * w.d
            rows_done += rows.size
            fl += float(sum(per * ((r + 1) if w.causal else n) for r in rows))
            if time.perf_counter() - t0 > budget_s:
                break
        units_done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    unit = "head pair" if w.kind == "v2" else "head"
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows_done} query rows over {units_done} (batch, {unit}) units of {len(units)}, "
                      f"heaviest 128-row blocks first, {dt:.1f} s; algorithmic causal FLOPs of those rows",
            "seconds": dt}


def run_ours(args):
    import torch
    import torch.distributed as tdist
    from differential_attention_03_gb300 import binding as da, build
    from differential_attention_03_gb300.inputs import WORKLOADS, make_v1, make_v2, shrink
    from differential_attention_03_gb300.sharding import weak_scaling_seed

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    if rank == 0:
        build.build()
    if dist is not None:
        dist.barrier()
    da.lib()
    peaks = read_peaks()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)

    def inputs(w):
        w = shrink(w, seed=weak_scaling_seed(w.seed, rank))
        return make_v1(w, "cuda") if w.kind == "v1" else make_v2(w, "cuda")

    w = WORKLOADS[args.config]
    if args.kernel_only:
        # The forward of the workload alone (for profilers): warm-up and timed
        # steps, nothing else launched; one short JSON line.
        x = inputs(w)
        res = time_device(w, x, da, args.steps, args.warmup, flush, dist)
        if rank == 0:
            print(json.dumps({"workload": w.name, "kernel_ms": round(res["kernel_ms"], 4),
                              "tflops": round(flops(w) / (res["kernel_ms"] * 1e-3) / 1e12, 2),
                              "steps": args.steps, "warmup": args.warmup}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    sampler = ClockSampler(local)
    sampler.start()  # polls from before the warm-up to the end of the timed steps
    x = inputs(w)
    res = time_device(w, x, da, args.steps, args.warmup, flush, dist)
    clocks = sampler.stop(res["window"])
    step_ms = torch.tensor([res["step_ms"], res["kernel_ms"]], device="cuda", dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(step_ms, op=tdist.ReduceOp.MAX)
    step_ms, kern_ms = float(step_ms[0]), float(step_ms[1])
    f = flops(w)
    value = world * f / (step_ms * 1e-3) / 1e12
    e2e_ms, h2d, d2h = time_e2e(w, x, da, max(3, min(args.steps, 10)))
    e2e_t = torch.tensor([e2e_ms], device="cuda", dtype=torch.float64)
    if dist is not None:
        dist.all_reduce(e2e_t, op=tdist.ReduceOp.MAX)
    e2e_value = world * f / (float(e2e_t[0]) * 1e-3) / 1e12

    kernel_tflops = f / (kern_ms * 1e-3) / 1e12
    if w.dtype == "bf16":
        roof = {"bound": "tensor", "achieved": round(kernel_tflops, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(kernel_tflops / peaks["bf16_tflops"], 4),
                "frac_of_sustained": (round(kernel_tflops / peaks["bf16_tflops_sustained"], 4)
                                      if peaks.get("bf16_tflops_sustained") else None),
                "traffic": ncu_traffic(w.name), "traffic_unit": "bytes per launch (ncu, cold-cache replay)",
                "algorithmic_bytes": hbm_bytes(w), "peak_source": peaks["source"] + " (burst bf16 dense)"}
    else:
        gbs = hbm_bytes(w) / (kern_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(gbs, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": ncu_traffic(w.name),
                "traffic_unit": "bytes per launch (ncu, cold-cache replay)", "algorithmic_bytes": hbm_bytes(w),
                "peak_source": peaks["source"]}

    configs = {}
    if rank == 0 and world == 1 and not args.no_all_configs:
        for cid, wc in WORKLOADS.items():
            xc = x if cid == args.config else inputs(wc)
            r = time_device(wc, xc, da, max(5, min(args.steps, 20)), 3, flush)
            fc = flops(wc)
            tf = fc / (r["kernel_ms"] * 1e-3) / 1e12
            configs[wc.name] = {
                "kernel_ms": round(r["kernel_ms"], 4), "step_ms": round(r["step_ms"], 4),
                "tflops": round(tf, 2), "pct_peak": round(100 * tf / peaks["bf16_tflops"], 2),
                "tokens_per_s": round(wc.B * wc.n / (r["step_ms"] * 1e-3), 1),
                "hbm_gbs": round(hbm_bytes(wc) / (r["kernel_ms"] * 1e-3) / 1e9, 1)}
            if cid != args.config:
                del xc
            torch.cuda.empty_cache()

    decode, backward, layer, fp8, graphs = {}, {}, {}, {}, {}
    if rank == 0 and world == 1 and not args.no_all_configs:
        decode = decode_results(da, flush, peaks)
        graphs = graph_results(da)
        backward = backward_results(da, flush, (clocks or {}).get("sm_mhz") or 2070, peaks)
        layer = layer_results(da, flush, peaks)
        fp8 = fp8_results(da, flush, peaks, inputs)

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1) inputs, shapes of the workload)",
        "config": {"workload": w.name, "global_batch": w.B * world, "seq_len": w.n,
                   "heads": w.H or w.Hq, "head_dim": w.d, "causal": w.causal,
                   "parallelism": f"dp{world} (batch split, no collective)",
                   "l2": "flushed between timed steps (512 MB written, then read back)"},
        "tokens_per_s": round(world * w.B * w.n / (step_ms * 1e-3), 1),
        "pct_of_peak": round(100 * kernel_tflops / peaks["bf16_tflops"], 2) if w.dtype == "bf16" else None,
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(float(e2e_t[0]), 4)},
        "gpu_launches": res["launches"],
        "roofline": roof,
        "clocks": clocks,
    }
    if configs:
        line["configs"] = configs
    if decode:
        line["decode"] = decode
    if backward:
        line["backward"] = backward
    if layer:
        line["layer"] = layer
    if fp8:
        line["fp8"] = fp8
    if graphs:
        line["graphs"] = graphs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(w, x)
        cb.pop("seconds", None)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def run_reference(args):
    """The oracle as it stands, on the host cores, same workload/metric/unit (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import torch
    from differential_attention_03_gb300.inputs import WORKLOADS, make_v1, make_v2
    w = WORKLOADS[args.config]
    x = make_v1(w, "cpu") if w.kind == "v1" else make_v2(w, "cpu")
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(w, x, budget_s=min(per_step, 2.0))
    vals, secs, last = [], [], None
    for _ in range(args.steps):
        last = cpu_baseline(w, x, budget_s=per_step)
        vals.append(last["value"])
        secs.append(last["seconds"])
    v = statistics.mean(vals)
    f_step = flops(w)
    # A whole step of the workload would take the oracle far longer than the
    # run: each timed step is a bounded sample, and ms_per_step is the time a
    # full step would take at the sample's rate (extrapolated, not measured).
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": f_step / (v * 1e12) * 1e3,
            "ms_per_step_kind": "extrapolated (full-workload FLOPs / the sampled rate)",
            "ms_per_sampled_step": round(1e3 * statistics.mean(secs), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) inputs, shapes of the workload)",
            "config": {"workload": w.name, "global_batch": w.B, "seq_len": w.n, "heads": w.H or w.Hq,
                       "head_dim": w.d, "causal": w.causal, "parallelism": "host cores"},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"] + "; each step one such bounded sample"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    del torch
    print(json.dumps(line), flush=True)


BACKWARD_WORKLOADS = [  # (name, B, H or (Hq, Hkv), n, d, dtype): DIFF V1 / V2 backward, causal
    ("v1-bwd-bf16-B4H16-n2048-d64", 4, 16, 2048, 64, "bf16"),
    ("v2-bwd-bf16-B2Hq32Hkv16-n2048-d128", 2, (32, 16), 2048, 128, "bf16"),
    # from a training forward's saved statistics (no second forward inside the backward)
    ("v1-bwd-saved-bf16-B4H16-n2048-d64", 4, 16, 2048, 64, "bf16-saved"),
    ("v2-bwd-saved-bf16-B2Hq32Hkv16-n2048-d128", 2, (32, 16), 2048, 128, "bf16-saved"),
    # one training step of the layer's operator: training forward + backward from its statistics
    ("v1-train-step-bf16-B4H16-n2048-d64", 4, 16, 2048, 64, "bf16-train"),
    ("v2-train-step-bf16-B2Hq32Hkv16-n2048-d128", 2, (32, 16), 2048, 128, "bf16-train"),
    ("v1-bwd-f32-B4H16-n2048-d64", 4, 16, 2048, 64, "f32"),
    ("v1-bwd-f32-B1H1-n128-d64", 1, 1, 128, 64, "f32"),
    ("v2-bwd-f32-B2Hq32Hkv16-n2048-d128", 2, (32, 16), 2048, 128, "f32"),
]
# fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 flops x the SM clock (MHz).
FP32_LANES = 152 * 128


def backward_flops(B, H, n, d):
    """Algorithmic FLOPs of the backward per visible (query, key) pair, causal: n (n + 1) / 2 pairs.

    V1 (H heads): 20 d a pair: 2 d each for the two score recomputations, 4 d for
    dO . v (value width 2d), 4 d for dV, 2 d each for dQ_1, dQ_2, dK_1, dK_2.
    V2 (H = (Hq, Hkv), Hq / 2 head pairs): 16 d a pair and head pair: the same
    terms with a value width of d.
    """
    pairs = n * (n + 1) // 2
    if isinstance(H, tuple):
        return B * (H[0] // 2) * pairs * 16 * d
    return B * H * pairs * 20 * d


def train_step_flops(B, H, n, d):
    """A training step of the operator: the forward (V1 12 d a visible pair per head, V2 8 d a pair per
    head pair) plus the backward's algorithmic FLOPs (backward_flops)."""
    pairs = n * (n + 1) // 2
    fwd = B * (H[0] // 2) * pairs * 8 * d if isinstance(H, tuple) else B * H * pairs * 12 * d
    return fwd + backward_flops(B, H, n, d)


def time_backward(da, flush, B, H, n, d, dtype="f32", runs=10):
    """DIFF V1 / V2 backward: median CUDA-event time, L2 flushed.  fp32 inputs run on the CUDA cores,
    bf16 inputs on the tensor cores (statistics pass, dK/dV/dQ kernel, reductions; fp32 gradients).
    "bf16-saved": the backward from a training forward's saved statistics (the forward runs once,
    untimed); "bf16-train": the training forward and that backward, both timed."""
    import torch
    g = torch.Generator(device="cuda").manual_seed(3000 + n + d)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16

    def rnd(*shape):
        return torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(tdt)
    if isinstance(H, tuple):  # DIFF V2: (Hq, Hkv), one logit per pair
        Hq, Hkv = H
        q, k, v, dy = rnd(B, n, Hq, d), rnd(B, n, Hkv, d), rnd(B, n, Hkv, d), rnd(B, n, Hq // 2, d)
        lg = torch.randn(Hq // 2, generator=g, device="cuda")
        ws = torch.empty(da.v2_backward_workspace_bytes(B, Hq, n, d), dtype=torch.uint8, device="cuda")
        if dtype in ("f32", "bf16"):
            def call():
                da.diffattn_v2_backward(q, k, v, lg, dy, workspace=ws)
        else:
            y = torch.empty((B, n, Hq // 2, d), device="cuda", dtype=torch.bfloat16)
            _, saved = da.diffattn_v2_forward_train(q, k, v, lg, out=y)

            def call():
                if dtype == "bf16-train":
                    da.diffattn_v2_forward_train(q, k, v, lg, out=y, saved=saved)
                da.diffattn_v2_backward_saved(q, k, v, lg, dy, saved, workspace=ws)
    else:
        q1, q2, k1, k2 = (rnd(B, n, H, d) for _ in range(4))
        v, dy = rnd(B, n, H, 2 * d), rnd(B, n, H, 2 * d)
        gamma = torch.ones(2 * d, device="cuda")
        lam = torch.tensor([0.3], device="cuda")
        ws = torch.empty(da.backward_workspace_bytes(B, H, n, d), dtype=torch.uint8, device="cuda")
        if dtype in ("f32", "bf16"):
            def call():
                da.diffattn_backward(q1, q2, k1, k2, v, lam, 0.2, dy, gamma=gamma, workspace=ws)
        else:
            y = torch.empty((B, n, H, 2 * d), device="cuda", dtype=torch.bfloat16)
            _, saved = da.diffattn_forward_train(q1, q2, k1, k2, v, lam, 0.2, gamma=gamma, out=y)

            def call():
                if dtype == "bf16-train":
                    da.diffattn_forward_train(q1, q2, k1, k2, v, lam, 0.2, gamma=gamma, out=y, saved=saved)
                da.diffattn_backward_saved(q1, q2, k1, k2, v, lam, 0.2, dy, saved, gamma=gamma, workspace=ws)
    for _ in range(3):
        call()
    da.device_status()
    ts = []
    for _ in range(runs):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    da.device_status()
    torch.cuda.empty_cache()
    return statistics.median(ts)


def backward_results(da, flush, sm_mhz, peaks=None, only=None):
    out = {}
    peaks = peaks or read_peaks()
    peak32 = 2 * FP32_LANES * sm_mhz * 1e6 / 1e12
    for name, B, H, n, d, dtype in BACKWARD_WORKLOADS:
        if only and name not in only:
            continue
        ms = time_backward(da, flush, B, H, n, d, dtype)
        fl = train_step_flops(B, H, n, d) if dtype == "bf16-train" else backward_flops(B, H, n, d)
        tf = fl / (ms * 1e-3) / 1e12
        if dtype != "f32":
            out[name] = {"ms": round(ms, 4), "tflops": round(tf, 2), "bound": "tensor",
                         "peak_tflops": peaks["bf16_tflops"], "peak": "measured burst bf16 dense",
                         "frac": round(tf / peaks["bf16_tflops"], 4), "tokens_per_s": round(B * n / (ms * 1e-3), 1)}
        else:
            out[name] = {"ms": round(ms, 4), "tflops": round(tf, 3), "bound": "alu",
                         "peak_tflops": round(peak32, 1), "peak": f"fp32 FMA: {FP32_LANES} lanes x 2 x {sm_mhz} MHz",
                         "frac": round(tf / peak32, 4), "tokens_per_s": round(B * n / (ms * 1e-3), 1)}
    return out


LAYER_WORKLOADS = [  # (name, kind, B, n, D, H or (Hq, Hkv), d): attention layers around the operator, causal
    ("v1-layer-bf16-B2-n4096-D3072-H12-d128", "v1", 2, 4096, 3072, 12, 128),
    ("v2-layer-bf16-B2-n8192-D2048-Hq32Hkv16-d128", "v2", 2, 8192, 2048, (32, 16), 128),
]
PROJECTION_WORKLOADS = [  # (name, M, N, K): c = a w^T alone
    ("projection-bf16-8192x8192x8192", 8192, 8192, 8192),
    ("projection-bf16-8192x9216x3072", 8192, 9216, 3072),
]


GRAPH_DECODE = ("v1-decode-bf16-B1H16-n4096-d64-x8-layers", 1, 16, 4096, 64, 8)  # name, B, H, n, d, layers


def graph_results(da):
    """A decode step short enough to be bound by launches: one new token over eight layers' caches
    (B1 H16 n4096 d64, 33.5 MB of keys and values a layer), eight library calls per token.  Timed
    back to back (CUDA events around 50 tokens) as eager calls through the binding and as one CUDA-graph
    replay of the same eight calls; the caches (268 MB) exceed L2, so no flush is needed."""
    import torch
    name, B, H, n, d, layers = GRAPH_DECODE
    g = torch.Generator(device="cuda").manual_seed(77)

    def rnd(*shape):
        return torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    cache = [(rnd(B, n, H, d), rnd(B, n, H, d), rnd(B, n, H, 2 * d)) for _ in range(layers)]
    qs = [(rnd(B, H, d), rnd(B, H, d)) for _ in range(layers)]
    lam = torch.tensor([0.3], device="cuda")
    ws = torch.empty(da.decode_workspace_bytes(B, H, d), dtype=torch.uint8, device="cuda")
    outs = [torch.empty((B, H, 2 * d), device="cuda", dtype=torch.bfloat16) for _ in range(layers)]

    def token():
        for i in range(layers):
            k1, k2, v = cache[i]
            da.diffattn_decode(qs[i][0], qs[i][1], k1, k2, v, lam, 0.2, out=outs[i], workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            token()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    da.device_status()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        token()

    def timed(fn, tokens=50):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(tokens):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (tokens * layers)  # us per decode call
    eager = statistics.median(timed(token) for _ in range(3))
    replay = statistics.median(timed(graph.replay) for _ in range(3))
    da.device_status()
    nbytes = B * H * n * d * 8 + B * H * 4 * d * 2  # K1, K2, V once; q in, out
    del graph
    torch.cuda.empty_cache()
    return {name: {"eager_us_per_call": round(eager, 2), "graph_us_per_call": round(replay, 2),
                   "speedup": round(eager / replay, 2),
                   "graph_tb_s": round(nbytes / (replay * 1e-6) / 1e12, 3),
                   "calls_per_token": layers}}


def fp8_results(da, flush, peaks, inputs):
    """The V1 and V2 forwards with e4m3 queries and keys (one scale per tensor, amax / 448) on the
    tensor-core workloads (d = 64 and d = 128): TFLOP/s (the same algorithmic FLOPs as bf16) against the
    measured burst bf16 peak."""
    import torch
    from differential_attention_03_gb300.inputs import WORKLOADS
    out = {}
    for wid in (2, 3, 4, 5):
        w = WORKLOADS[wid]
        x = inputs(w)
        if w.kind == "v2":
            cq_sc = [float(x[k].float().abs().max()) / 448.0 for k in ("q", "k")]
            cq, ck = ((x[k].float() / sc).to(torch.float8_e4m3fn) for k, sc in zip(("q", "k"), cq_sc))
            y = torch.empty((w.B, w.n, w.Hq // 2, w.d), device="cuda", dtype=torch.bfloat16)

            def call2():
                da.diffattn_v2_forward_fp8qk(cq, ck, cq_sc, x["v"], x["lam_logits"], causal=w.causal, out=y)
            ms = _median_ms(call2, flush, runs=10)
            da.device_status()
            tf = flops(w) / (ms * 1e-3) / 1e12
            out["fp8qk-" + w.name] = {"ms": round(ms, 4), "tflops": round(tf, 2),
                                      "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                                      "tokens_per_s": round(w.B * w.n / (ms * 1e-3), 1)}
            del cq, ck, x, y
            torch.cuda.empty_cache()
            continue
        codes, scales = [], []
        for k in ("q1", "q2", "k1", "k2"):
            sc = float(x[k].float().abs().max()) / 448.0
            codes.append((x[k].float() / sc).to(torch.float8_e4m3fn))
            scales.append(sc)
            del x[k]
        lin = da.lambda_init(w.layer)
        lam = da.lambda_reparam(x["lq1"], x["lk1"], x["lq2"], x["lk2"], lin)
        y = torch.empty(x["v"].shape, device="cuda", dtype=torch.bfloat16)

        def call():
            da.diffattn_forward_fp8qk(*codes, scales, x["v"], lam, lin, gamma=x["gamma"], causal=w.causal, out=y)
        ms = _median_ms(call, flush, runs=5 if wid == 4 else 10)
        da.device_status()
        tf = flops(w) / (ms * 1e-3) / 1e12
        out["fp8qk-" + w.name] = {"ms": round(ms, 4), "tflops": round(tf, 2),
                                  "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                                  "tokens_per_s": round(w.B * w.n / (ms * 1e-3), 1)}
        del codes, x, y
        torch.cuda.empty_cache()
    return out


def layer_flops(kind, B, n, D, H, d):
    """Algorithmic FLOPs of one layer forward: the two projections (2 M K N each) plus the operator
    (V1 12 n^2 d per (b, h), V2 4 n^2 d per query head; halved for causal)."""
    M = B * n
    if kind == "v1":
        return 2.0 * M * D * 6 * H * d + 6.0 * n * n * d * B * H + 2.0 * M * 2 * H * d * D
    Hq, Hkv = H
    G = Hq // 2
    return 2.0 * M * D * ((Hq + 2 * Hkv) * d + G) + 2.0 * n * n * d * B * Hq + 2.0 * M * G * d * D


def _median_ms(call, flush, runs=10):
    import torch
    for _ in range(3):
        call()
    ts = []
    for _ in range(runs):
        flush_l2(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def layer_results(da, flush, peaks, only=None):
    """Attention layers (projections, operator, W^O) and the projection GEMM alone: TFLOP/s against the
    measured burst bf16 peak."""
    import torch
    out = {}
    g = torch.Generator(device="cuda").manual_seed(4242)

    def rnd(*shape, scale=1.0):
        return (scale * torch.randn(shape, generator=g, device="cuda")).to(torch.bfloat16)
    for name, kind, B, n, D, H, d in LAYER_WORKLOADS:
        if only and name not in only:
            continue
        x = rnd(B, n, D)
        if kind == "v1":
            w_qkv, w_o = rnd(6 * H * d, D, scale=D ** -0.5), rnd(D, 2 * H * d, scale=(2 * H * d) ** -0.5)
            lv = [0.1 * torch.randn(d, generator=g, device="cuda") for _ in range(4)]
            ws = torch.empty(da.layer_workspace_bytes(B, n, H, d), dtype=torch.uint8, device="cuda")
            y = torch.empty((B, n, D), device="cuda", dtype=torch.bfloat16)

            def call():
                da.layer_forward(x, w_qkv, w_o, *lv, 0.7, H, out=y, workspace=ws)
        else:
            Hq, Hkv = H
            w = rnd((Hq + 2 * Hkv) * d + Hq // 2, D, scale=D ** -0.5)
            w_o = rnd(D, Hq // 2 * d, scale=(Hq // 2 * d) ** -0.5)
            ws = torch.empty(da.v2_layer_workspace_bytes(B, n, Hq, Hkv, d), dtype=torch.uint8, device="cuda")
            y = torch.empty((B, n, D), device="cuda", dtype=torch.bfloat16)

            def call():
                da.v2_layer_forward(x, w, w_o, Hq, Hkv, out=y, workspace=ws)
        ms = _median_ms(call, flush)
        da.device_status()
        tf = layer_flops(kind, B, n, D, H, d) / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "tflops": round(tf, 2), "frac": round(tf / peaks["bf16_tflops"], 4),
                     "tokens_per_s": round(B * n / (ms * 1e-3), 1), "bound": "tensor"}
        del x, ws, y
        torch.cuda.empty_cache()
    for name, M, N, K in PROJECTION_WORKLOADS:
        if only and name not in only:
            continue
        a, w = rnd(M, K), rnd(N, K)
        c = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
        ms = _median_ms(lambda: da.projection(a, w, out=c), flush)
        da.device_status()
        tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        out[name] = {"ms": round(ms, 4), "tflops": round(tf, 2), "frac": round(tf / peaks["bf16_tflops"], 4),
                     "bound": "tensor"}
        del a, w, c
        torch.cuda.empty_cache()
    return out


def decode_results(da, flush, peaks, only=None):
    out = {}
    for name, B, H, n, d, keys in DECODE_WORKLOADS:
        if only and name not in only:
            continue
        ms, nb = time_decode(da, flush, B, H, n, d, keys)
        gbs = nb / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 1), "hbm_gbs": round(gbs, 1), "bound": "hbm",
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "peak_gbs": peaks["hbm_gbs"],
                     "algorithmic_bytes": nb, "tokens_per_s": round(B / (ms * 1e-3), 1)}
    return out


def run_backward_only(only=None):
    import torch
    from differential_attention_03_gb300 import binding as da, build
    build.build()
    da.lib()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    print(json.dumps({"backward": backward_results(da, flush, 2070, None, only)}), flush=True)


def run_layer_only(only=None):
    import torch
    from differential_attention_03_gb300 import binding as da, build
    build.build()
    da.lib()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    from differential_attention_03_gb300.inputs import make_v1, make_v2
    peaks = read_peaks()
    line = {"layer": layer_results(da, flush, peaks, only)}
    if not only:
        line["fp8"] = fp8_results(da, flush, peaks,
                                  lambda w: make_v1(w, "cuda") if w.kind == "v1" else make_v2(w, "cuda"))
    print(json.dumps(line), flush=True)


def run_decode_only(only=None):
    import torch
    from differential_attention_03_gb300 import binding as da, build
    build.build()
    da.lib()
    flush = torch.empty(FLUSH_BYTES // 4, device="cuda", dtype=torch.float32)
    print(json.dumps({"decode": decode_results(da, flush, read_peaks(), only), "graphs": graph_results(da)}),
          flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-all-configs", action="store_true")
    ap.add_argument("--kernel-only", action="store_true",
                    help="time only the workload's forward (warm-up + timed steps) and print a short line; "
                         "the command the ncu captures run")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode workloads (one JSON line with the 'decode' object)")
    ap.add_argument("--layer-only", action="store_true",
                    help="time only the attention layers, the projection GEMM and the FP8 forward (one JSON line)")
    ap.add_argument("--workload", action="append", default=None,
                    help="with --decode-only / --backward-only / --layer-only: time only the named workload(s)")
    ap.add_argument("--backward-only", action="store_true",
                    help="time only the fp32 backward workloads (one JSON line with the 'backward' object)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        # One process per GPU: N > 1 needs a launcher (torch.distributed.run) that
        # starts N ranks; timing one GPU under --gpus N would misreport the job.
        sys.stderr.write(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one process per GPU, "
                         f"e.g. python -m torch.distributed.run --nproc-per-node {args.gpus} "
                         f"--master-addr 127.0.0.1 bench.py --gpus {args.gpus}\n")
        return 2
    if args.impl == "reference":
        run_reference(args)
    elif args.decode_only:
        run_decode_only(args.workload)
    elif args.backward_only:
        run_backward_only(args.workload)
    elif args.layer_only:
        run_layer_only(args.workload)
    else:
        run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
