"""Benchmark of the fused contraction + activation + reduction library.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload B] [--impl reference]

A "step" is one call of the fused operator on one batch of the workload
(default: conv3x3 + erf-GELU + global average pool, x (128, 8, 256, 256) fp32,
Cout 64 -- the Conv2d->GELU->pool page's full problem), inputs resident in
HBM.  Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own
shard of images on its own GPU (no collective on the data path); the timed
region is bracketed by a barrier + synchronize and the max over ranks is used.

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of the same workload per step (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import fc_inputs  # noqa: E402

TF32_OVER_BF16 = 1.1 / 2.25   # nominal dense TF32 : BF16 tensor ratio of the part
METRIC = "fused-op TFLOP/s, ms/call and % of roofline (conv3x3+act(+pool), GEMM+LSE)"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# Per-element cost of the conv epilogue's activation (and its pool accumulate or store scaling),
# from the instruction sequences in csrc/fc_act.cuh: FMA-pipe results (each paired-FP32
# instruction yields one result per element; 128 results per clock per SM) and SFU cycles per
# SM (ex2.approx 32 lanes per clock, rcp.approx 16; microbenchmarked on this GB300).
#   erf-GELU: 5 Horner FMAs, z + |z|, the final FMA, the accumulate; one exponential
#   tanh-GELU: 3 for the exponent, 1 + e, the product, the accumulate; one exponential, one reciprocal
#   Mish: 4 arithmetic (the scaled exponent, v, h, z - z / h), the accumulate; one exponential, one
#   reciprocal; Mish twice: 8 + 1, two of each
EPILOGUE_COST = {"gelu": (8, 1 / 32), "gelu_tanh": (6, 1 / 32 + 1 / 16), "mish": (5, 1 / 32 + 1 / 16),
                 "mish_mish": (9, 2 * (1 / 32 + 1 / 16))}
FMA_RESULTS_PER_CLK_SM = 128


def epilogue_roofline(wl, call_ms, sm_count, sm_mhz):
    """The conv epilogue's own floor: every one of the N x Cout x OH x OW contraction outputs takes
    one activation evaluation on the FMA pipe and the special-function units, a rate that the tensor
    roofline does not see (it binds workload B, whose contraction is short).  Peak = SMs x clock /
    the busier unit's cycles per element."""
    elems = wl.N * wl.Cout * wl.OH * wl.OW
    fma, sfu = EPILOGUE_COST[wl.act]
    cycles = max(fma / FMA_RESULTS_PER_CLK_SM, sfu)
    peak = sm_count * sm_mhz * 1e6 / cycles / 1e9
    achieved = elems / (call_ms * 1e-3) / 1e9
    return {"bound": "alu", "unit": "Gelem/s", "achieved": achieved, "peak": peak, "frac": achieved / peak,
            "peak_source": f"{'FMA pipe' if fma / FMA_RESULTS_PER_CLK_SM >= sfu else 'SFU'}: {fma} FMA-pipe results "
                           f"(128 / clk / SM) and {sfu:.4f} SFU cycles per element x {sm_count} SMs x "
                           f"{sm_mhz:.0f} MHz (median SM clock in the timed region)",
            "elements": elems}


def tf32_peak(pk):
    """TF32 dense peak: the larger of the nominal-ratio figure (measured BF16 x 1.1/2.25) and the
    TF32 library GEMM measured in this run (pk["tf32_measured_tflops"], when present)."""
    nominal = pk["bf16_tflops"] * TF32_OVER_BF16
    measured = pk.get("tf32_measured_tflops")
    if measured and measured > nominal:
        return measured, f"tf32 = measured library TF32 GEMM {measured:.1f} TFLOP/s ({pk['tf32_how']})"
    return nominal, f"tf32 = bf16 burst ({pk['source']}) x nominal 1.1/2.25" + \
        (f"; measured TF32 GEMM {measured:.1f} TFLOP/s is lower" if measured else "")


def tensor_peak(wl, pk):
    bf16 = pk["bf16_tflops"]
    if getattr(wl, "dtype", "f32") == "bf16":
        return bf16, f"bf16 burst ({pk['source']})"
    tf32, note = tf32_peak(pk)
    if getattr(wl, "precision", "tf32") == "3xtf32":
        # three TF32 products per term: the contraction's flops take three times the TF32 tensor time
        return tf32 / 3.0, f"3xtf32 = tf32 / 3, {note}"
    return tf32, note


def measure_tf32_gemm(torch, device, n=8192, reps=10):
    """Peak measurement only (not the operator's path): best time of an fp32 n^3 library matmul
    with TF32 tensor-core math enabled, CUDA events around each call; returns TFLOP/s."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        a = torch.randn(n, n, device=device)
        b = torch.randn(n, n, device=device)
        for _ in range(3):
            torch.matmul(a, b)
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ profile summary (ncu traffic)

# Translation units with host code only (stream and copy orchestration): they cannot change
# what a kernel reads or writes, so they are left out of the kernel-source hash.
HOST_ONLY_SOURCES = ("fc_host.cu",)


def kernel_sources_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gemm_activation_reduction_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in HOST_ONLY_SOURCES:
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def traffic_profile_name(workload_key):
    """The committed DRAM-traffic summary of a workload's dominant kernel: <kernel>_<workload>_dram_traffic.md."""
    wl = fc_inputs.WORKLOADS[workload_key]
    kernel = "linear_lse" if isinstance(wl, fc_inputs.LinearWorkload) else "conv3x3_fused"
    return f"{kernel}_{wl.name}_dram_traffic.md"


def profiled_traffic(workload_key):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    or None when that summary was taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", traffic_profile_name(workload_key))
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_b = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", text)
    if not m_b or not m_h or m_h.group(1) != kernel_sources_hash():
        return None
    return float(m_b.group(1))


# ------------------------------------------------------------------ GPU arm

def _dev(torch, a, device):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


L2_BYTES = 129e6


def epilogue_call(fc, torch, wl, inputs, device):
    """One call of an epilogue workload; with several input tensors (copies of one input), call
    i reads inputs[i % len(inputs)]."""
    if wl.kind == "act_map":
        out = torch.empty(wl.shape, dtype=torch.float32, device=device)
    elif wl.kind == "act_mean":
        out = torch.empty(wl.shape[:-2], dtype=torch.float32, device=device)
    else:
        out = torch.empty((wl.shape[0], 1), dtype=torch.float32, device=device)
    count = [0]

    def call():
        v = inputs[count[0] % len(inputs)]
        count[0] += 1
        if wl.kind == "act_map":
            fc.fc_act_map(v, act=wl.act, out=out)
        elif wl.kind == "act_mean":
            fc.fc_act_mean(v, act=wl.act, out=out)
        else:
            fc.fc_scale_clamp_lse_mish(v, 2.0, -10.0, 10.0, out=out)
    return call, out


def rotation_copies(nbytes, l2_bytes=L2_BYTES):
    """Input copies whose total is at least twice the L2, so that a call rotating over them finds
    its input evicted since its last use (1 when one input is that large already)."""
    return max(1, -(-int(2 * l2_bytes) // int(nbytes)))


def make_call(fc, torch, key, d, device):
    wl = fc_inputs.WORKLOADS[key]
    if isinstance(wl, fc_inputs.EpilogueWorkload):
        call, out = epilogue_call(fc, torch, wl, [_dev(torch, d["v"], device)], device)
        return call, 1, out
    if isinstance(wl, fc_inputs.LinearWorkload):
        x, W, b = (_dev(torch, d[k], device) for k in ("x", "W", "b"))
        out = torch.empty((wl.M, 1), dtype=torch.float32, device=device)
        split = wl.dtype != "bf16" and wl.precision == "3xtf32"
        ldt = fc.FC_BF16 if wl.dtype == "bf16" else (fc.FC_F32_3XTF32 if split else fc.FC_F32)
        ws = torch.empty(fc.fc_workspace_bytes("linear_lse_mish", wl.M, wl.K, 1, 1, wl.Nout, ldt), dtype=torch.uint8,
                         device=device)
        prec = None if wl.dtype == "bf16" else wl.precision

        def call():
            fc.fc_linear_lse_mish(x, W, b, wl.scale, wl.clamp_lo, wl.clamp_hi, out=out, workspace=ws, precision=prec)
        return call, 4 if split else 2, out
    x, w, b = (_dev(torch, d[k], device) for k in ("x", "w", "b"))
    nhwc = wl.layout == "nhwc"
    if nhwc:
        # x stored [N][H][W][Cin], passed as the channels_last view of logical shape [N, Cin, H, W]
        x = _dev(torch, np.ascontiguousarray(np.transpose(d["x"], (0, 2, 3, 1))), device).permute(0, 3, 1, 2)
    dt = fc.FC_BF16 if wl.dtype == "bf16" else (fc.FC_F32_3XTF32 if wl.precision == "3xtf32" else fc.FC_F32)
    prec = None if wl.dtype == "bf16" else wl.precision
    op = "conv3x3_act_pool" if wl.pool else "conv3x3_act"
    shape = (wl.N, wl.Cout) if wl.pool else (wl.N, wl.Cout, wl.OH, wl.OW)
    out = torch.empty(shape, dtype=torch.float32, device=device,
                      memory_format=torch.channels_last if (nhwc and not wl.pool) else torch.contiguous_format)
    ws = torch.empty(max(1, fc.load().fc_workspace_bytes_ex(fc.OPS[op], wl.N, wl.Cin, wl.H, wl.W, wl.Cout, wl.pad,
                                                             fc.FC_NHWC if nhwc else fc.FC_NCHW, dt)),
                     dtype=torch.uint8, device=device)
    f = fc.fc_conv3x3_act_pool if wl.pool else fc.fc_conv3x3_act

    def call():
        f(x, w, b, act=wl.act, out=out, workspace=ws, precision=prec, pad=wl.pad)
    return call, (3 if wl.pool else 2), out


def time_graph(torch, call, reps, replays=5, warm_s=0.1):
    """ms per call: `reps` calls captured once in a CUDA graph, the graph replayed `replays`
    times between CUDA events on the current stream; the median replay / reps.  Before the timed
    replays the graph is replayed for `warm_s` seconds, so that a few-microsecond kernel is not
    timed while the SM clock is still rising from idle."""
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            call()
    g.replay()
    torch.cuda.synchronize()
    t_end = time.perf_counter() + warm_s
    while time.perf_counter() < t_end:
        for _ in range(10):
            g.replay()
        torch.cuda.synchronize()
    times = []
    for _ in range(replays):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) / reps)
    return statistics.median(times)


def time_cold(torch, call, reps=10, flush_bytes=512 << 20):
    """Median ms of `reps` calls, each preceded by a write of a `flush_bytes` scratch buffer (more
    than 4x the L2), with the CUDA events placed after the write: the inputs come from HBM."""
    scratch = torch.empty(flush_bytes // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    call()
    torch.cuda.synchronize()
    times = []
    for i in range(reps):
        scratch.fill_(float(i))
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    del scratch
    return statistics.median(times)


def max_over_ranks(torch, value, dist, device):
    """The maximum of a per-rank float over all ranks (a job's time is its slowest rank's);
    `device` is where the collective's tensor lives (cuda for NCCL, cpu for gloo)."""
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seeds(rank):
    """Weak scaling: rank r owns its own shard (batch) of the workload, drawn with its own x seed
    (weights and bias are shared)."""
    return (fc_inputs.SEED_X + 1000 * rank, fc_inputs.SEED_W, fc_inputs.SEED_B)


def r4(v):
    """v to 4 significant digits (keeps the JSON line short)."""
    return None if v is None else float(f"{v:.4g}")


def job_tflops(flops_per_call, world, ms_per_call):
    """Whole-job throughput: every rank's calls over the slowest rank's time per call."""
    return flops_per_call * world / (ms_per_call * 1e-3) / 1e12


def time_device(torch, call, steps, warmup, dist=None):
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    evs[0].record(stream)
    for i in range(steps):
        call()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    total = evs[0].elapsed_time(evs[-1])
    if dist is not None:
        total = max_over_ranks(torch, total, dist, "cuda")
        dist.barrier()
    torch.cuda.synchronize()
    return total, per


def time_e2e(fc, torch, key, d, device, steps, warmup, chunks=8):
    """Same operator through the public API with pinned-host inputs: H2D of the
    inputs, the call, and D2H of the result inside the timed region.  The conv
    operators use their host-buffer entry points (the batch copied in `chunks`
    slices, each slice's copy overlapped with the previous slice's kernels); the
    Linear chain copies its operands, calls the device-buffer entry point and
    reads the result back."""
    wl = fc_inputs.WORKLOADS[key]
    if not isinstance(wl, fc_inputs.LinearWorkload):
        return time_e2e_conv_host(fc, torch, wl, d, device, steps, warmup, chunks)
    names = ("x", "W", "b") if isinstance(wl, fc_inputs.LinearWorkload) else ("x", "w", "b")
    host = []
    nhwc = getattr(wl, "layout", "nchw") == "nhwc"
    for k in names:
        a = d[k]
        if nhwc and k == "x":
            a = np.ascontiguousarray(np.transpose(a, (0, 2, 3, 1)))
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a))
        host.append(t.pin_memory())
    h2d = sum(t.numel() * t.element_size() for t in host)
    bf16 = getattr(wl, "dtype", "f32") == "bf16"

    def step():
        dev = [t.to(device, non_blocking=True) for t in host]
        if bf16:
            dev = [t.view(torch.bfloat16) for t in dev]
        if nhwc:
            dev[0] = dev[0].permute(0, 3, 1, 2)
        if isinstance(wl, fc_inputs.LinearWorkload):
            y = fc.fc_linear_lse_mish(*dev, wl.scale, wl.clamp_lo, wl.clamp_hi,
                                      precision=None if bf16 else wl.precision)
        elif wl.pool:
            y = fc.fc_conv3x3_act_pool(*dev, act=wl.act, precision=None if bf16 else wl.precision, pad=wl.pad)
        else:
            y = fc.fc_conv3x3_act(*dev, act=wl.act, precision=None if bf16 else wl.precision, pad=wl.pad)
        return y.to("cpu", non_blocking=False)

    for _ in range(warmup):
        y = step()
    d2h = y.numel() * y.element_size()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    return (time.perf_counter() - t0) * 1e3 / steps, h2d, d2h


def time_e2e_conv_host(fc, torch, wl, d, device, steps, warmup, chunks):
    nhwc = getattr(wl, "layout", "nchw") == "nhwc"
    host = {}
    for k in ("x", "w", "b"):
        a = d[k]
        if nhwc and k == "x":
            a = np.ascontiguousarray(np.transpose(a, (0, 2, 3, 1)))
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else np.ascontiguousarray(a)).pin_memory()
        host[k] = t.view(torch.bfloat16) if a.dtype == np.uint16 else t
    if nhwc:
        host["x"] = host["x"].permute(0, 3, 1, 2)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    bf16 = getattr(wl, "dtype", "f32") == "bf16"
    op = "conv3x3_act_pool" if wl.pool else "conv3x3_act"
    fn = fc.fc_conv3x3_act_pool_host if wl.pool else fc.fc_conv3x3_act_host
    dt = fc.FC_BF16 if bf16 else (fc.FC_F32_3XTF32 if wl.precision == "3xtf32" else fc.FC_F32)
    with torch.cuda.device(device):
        nb = fc.fc_host_staging_bytes(op, wl.N, wl.Cin, wl.H, wl.W, wl.Cout, pad=wl.pad,
                                      layout="nhwc" if nhwc else "nchw", dtype=dt, chunks=chunks)
        staging = torch.empty(nb, dtype=torch.uint8, device=device)
        kw = dict(act=wl.act, precision=None if bf16 else wl.precision, pad=wl.pad, chunks=chunks,
                  staging=staging, device=device)
        y = fn(host["x"], host["w"], host["b"], **kw)
        for _ in range(warmup):
            fn(host["x"], host["w"], host["b"], out=y, **kw)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            fn(host["x"], host["w"], host["b"], out=y, **kw)
        torch.cuda.synchronize()
        ms = (time.perf_counter() - t0) * 1e3 / steps
    return ms, h2d, y.numel() * y.element_size()


def oracle_sample(key, budget_s=12.0):
    """The oracle on a bounded sample of the workload: returns (flops done, seconds, sample text, threads)."""
    import oracle
    wl = fc_inputs.WORKLOADS[key]
    d = fc_inputs.workload_inputs(key)
    threads = oracle.threads()
    if isinstance(wl, fc_inputs.LinearWorkload):
        unit_flops = 2.0 * wl.K * wl.Nout        # one row
        run = lambda idx: oracle.linear_lse_mish(d["x"], d["W"], d["b"], wl.scale, wl.clamp_lo, wl.clamp_hi,
                                                 rows=idx)
        total_units, what = wl.M, "rows"
    elif wl.pool:
        unit_flops = 2.0 * wl.OH * wl.OW * wl.Cin * 9   # one (n, co) pooled output
        run = lambda idx: oracle.conv3x3_act_pool_at(d["x32"], d["w32"], d["b32"], idx, wl.act, pad=wl.pad)
        total_units, what = wl.N * wl.Cout, "(image, channel) pooled outputs"
    else:
        unit_flops = 2.0 * wl.Cin * 9                    # one output element
        run = lambda idx: oracle.conv3x3_act_at(d["x32"], d["w32"], d["b32"], idx, wl.act, pad=wl.pad)
        total_units, what = wl.N * wl.Cout * wl.OH * wl.OW, "output elements"
    n = min(total_units, max(threads, 4))
    t0 = time.perf_counter()
    run(np.arange(n))
    dt = time.perf_counter() - t0
    n2 = int(min(total_units, max(n, n * budget_s / max(dt, 1e-6))))
    n2 = max(threads, (n2 // threads) * threads) if n2 >= threads else n2
    t0 = time.perf_counter()
    run(np.arange(n2))
    dt2 = time.perf_counter() - t0
    return (unit_flops * n2, dt2, f"first {n2} of {total_units} {what} of workload {key}", threads, run, unit_flops,
            total_units)


def oracle_tiny_times(threads):
    """Wall time of the oracle on the whole tiny workload (2, 8, 32, 32) -> 64 channels, on one
    core and on `threads` cores (best of 3 each)."""
    import oracle
    wl = fc_inputs.WORKLOADS["A"]
    d = fc_inputs.workload_inputs("A")
    out = {}
    for n in (1, threads):
        oracle.set_threads(n)
        best = float("inf")
        for _ in range(3):
            t0 = time.perf_counter()
            oracle.conv3x3_act_pool(d["x32"], d["w32"], d["b32"], wl.act)
            best = min(best, time.perf_counter() - t0)
        out[f"{n}_core" if n == 1 else f"{n}_cores"] = best
    oracle.set_threads(threads)
    return out


def reference_arm(args):
    """--impl reference: the fp64 oracle on the host cores, K timed steps of a bounded sample."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    key = args.workload
    wl = fc_inputs.WORKLOADS[key]
    oracle.build()
    flops_cal, dt_cal, _, threads, run, unit_flops, total_units = oracle_sample(key, budget_s=0.5)
    per_unit = dt_cal / (flops_cal / unit_flops)
    # size each step so that warmup + steps fit in about two minutes
    steps, warmup = args.steps or 5, max(args.warmup, 3)
    per_step_s = max(0.05, min(10.0, 60.0 / (steps + warmup)))
    n = min(total_units, max(1, int(per_step_s / max(per_unit, 1e-9))))
    idx = np.arange(n)
    for _ in range(warmup):
        run(idx)
    t0 = time.perf_counter()
    for _ in range(steps):
        run(idx)
    sec = (time.perf_counter() - t0) / steps
    value = unit_flops * n / sec / 1e12
    sample = f"first {n} units of workload {key} per step ({unit_flops:.3e} flop each)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "sample_per_step": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def gpu_arm(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl")
        dist = tdist
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    import gemm_activation_reduction_gb300 as fc
    fc.load()
    key = args.workload
    wl = fc_inputs.WORKLOADS[key]
    seeds = rank_seeds(rank)
    if isinstance(wl, fc_inputs.LinearWorkload):
        d = fc_inputs.linear_inputs(wl.M, wl.K, wl.Nout, seeds=seeds, dtype=wl.dtype)
    else:
        d = fc_inputs.conv_inputs(wl.N, wl.Cin, wl.H, wl.W, wl.Cout, wl.dtype, seeds=seeds)
    call, launches_per_call, out = make_call(fc, torch, key, d, device)

    warmup = max(3, args.warmup)
    # auto-size the timed region to ~2 s of device time unless --steps is given
    if args.steps:
        steps = args.steps
    else:
        _, per = time_device(torch, call, 5, 2)
        steps = int(min(5000, max(20, 2000.0 / max(statistics.median(per), 1e-3))))

    sampler = ClockSampler(local)
    sampler.start()
    total_ms, per = time_device(torch, call, steps, warmup, dist)
    clocks = sampler.stop()
    status = fc.fc_device_status(clear=True)
    if status != fc.FC_OK:
        raise RuntimeError(f"device status after the timed region: {fc.fc_status_string(status)}")

    ms = total_ms / steps
    flops = wl.flops()
    value = job_tflops(flops, world, ms)
    pk = peaks()
    if not args.no_tf32_peak:
        try:
            pk["tf32_measured_tflops"] = measure_tf32_gemm(torch, device)
            pk["tf32_how"] = "torch.matmul fp32 8192^3 with TF32 math, best of 10 in this run"
        except Exception as e:  # the line still prints; the nominal figure is used
            pk["tf32_how"] = f"failed: {e}"
    cold_ms = time_cold(torch, call) if world == 1 else None
    peak, peak_note = tensor_peak(wl, pk)
    kernel_ms = statistics.mean(per)
    achieved = flops / (kernel_ms * 1e-3) / 1e12

    e2e_ms = h2d = d2h = e2e_value = None
    if not args.no_e2e:
        e2e_ms, h2d, d2h = time_e2e(fc, torch, key, d, device, steps=max(3, min(20, steps // 10)), warmup=2,
                                    chunks=args.e2e_chunks)
        e2e_ms = max_over_ranks(torch, e2e_ms, dist, "cuda")
        e2e_value = job_tflops(flops, world, e2e_ms)

    if rank != 0:
        return 0
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": profiled_traffic(key),
                "peak_source": peak_note,
                "duration_source": "CUDA events around each call on its stream (relayout + fused kernel"
                                   + (" + combine" if launches_per_call == 3 else "") + ")"}
    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    sm_mhz = float((clocks or {}).get("sm_mhz") or (clocks or {}).get("sm_max_mhz") or 2070.0)
    epi = None if isinstance(wl, (fc_inputs.LinearWorkload, fc_inputs.EpilogueWorkload)) else \
        epilogue_roofline(wl, kernel_ms, sm_count, sm_mhz)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        try:
            fl, sec, sample, threads, _, _, _ = oracle_sample(key)
            cpu = {"value": fl / sec / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": sample, "seconds": sec, "tiny_workload_seconds": oracle_tiny_times(threads)}
        except Exception as e:  # the line still prints; the failure is recorded
            cpu = {"value": None, "unit": "TFLOP/s", "cores": None, "kind": "oracle", "sample": f"failed: {e}"}
    cfg = {"workload": wl.name, "l2": "inputs larger than L2" if wl.compulsory_bytes() > L2_BYTES else
           "inputs smaller than L2 (timed back to back)",
           "compulsory_bytes": wl.compulsory_bytes(), "flops_per_step": flops,
           "roofline_ms": max(flops / (peak * 1e12), wl.compulsory_bytes() / (pk["hbm_gbs"] * 1e9)) * 1e3,
           "parallelism": f"shard-by-batch x{world}" if world > 1 else "single GPU"}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": ms, "ms_median": statistics.median(per), "ms_best": min(per),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if getattr(wl, "dtype", "f32") == "bf16" else "tf32",
            "data": "synthetic (seeded N(0,1) inputs, U(+-1/sqrt(fan_in)) weights)", "config": cfg,
            "roofline": roofline, "epilogue_roofline": epi, "cpu_baseline": cpu,
            "e2e": None if args.no_e2e else
            {"value": e2e_value, "unit": "TFLOP/s", "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
             "d2h_bytes_per_step": d2h,
             "api": "linear: H2D + fc_linear_lse_mish + D2H" if isinstance(wl, fc_inputs.LinearWorkload)
             else f"{'fc_conv3x3_act_pool_host' if wl.pool else 'fc_conv3x3_act_host'}"
                  f" (pinned host buffers, {args.e2e_chunks} overlapped slices)"},
            "gpu_launches": steps * launches_per_call, "clocks": clocks,
            "pct_of_roofline": 100.0 * cfg["roofline_ms"] / ms,
            "cold_l2": {"ms_median": cold_ms, "warm_ms_median": statistics.median(per),
                        "how": "each of 10 calls after a 512 MB scratch write, events after the write"}
            if cold_ms is not None else None,
            "tf32_peak_tflops": {"measured_gemm": pk.get("tf32_measured_tflops"),
                                 "nominal": pk["bf16_tflops"] * TF32_OVER_BF16, "used": tf32_peak(pk)[0]}}
    if not args.no_others and world == 1:
        others = {}
        for k in args.others.split(","):
            if not k or k == key:
                continue
            owl = fc_inputs.WORKLOADS[k]
            od = fc_inputs.workload_inputs(k)
            ocall, _, oout = make_call(fc, torch, k, od, device)
            if isinstance(owl, fc_inputs.EpilogueWorkload):
                # short kernels: 20 calls captured in a CUDA graph and replayed, so that host-side
                # enqueue time (Python, ctypes) stays out of the device time
                oms = time_graph(torch, ocall, 20)
            else:
                ot, oper = time_device(torch, ocall, 20, 3)
                oms = ot / 20
            if isinstance(owl, fc_inputs.EpilogueWorkload):
                # HBM-bound: the roofline is one pass over the compulsory bytes.  An input smaller
                # than the L2 would be read from the L2 by back-to-back calls, so there the timed
                # calls rotate over copies of it (twice the L2 in total) and the L2-resident time
                # is reported beside
                rl = owl.compulsory_bytes() / (pk["hbm_gbs"] * 1e9) * 1e3
                ncopy = rotation_copies(owl.compulsory_bytes())
                l2_ms = None
                if ncopy > 1:
                    v0 = _dev(torch, od["v"], device)
                    rcall, _ = epilogue_call(fc, torch, owl, [v0] + [v0.clone() for _ in range(ncopy - 1)], device)
                    l2_ms, oms = oms, time_graph(torch, rcall, 20)
                    del v0, rcall
                others[k] = {"workload": owl.name, "ms_per_call": r4(oms),
                             "gbs": r4(owl.compulsory_bytes() / (oms * 1e-3) / 1e9), "bound": "hbm",
                             "roofline_ms": r4(rl), "pct_of_roofline": r4(100.0 * rl / oms)}
                if l2_ms is not None:
                    others[k]["inputs"] = f"rotated over {ncopy} copies ({ncopy * owl.compulsory_bytes() / 1e6:.0f} MB)"
                    others[k]["ms_l2_resident"] = r4(l2_ms)
            else:
                opeak, _ = tensor_peak(owl, pk)
                rl = max(owl.flops() / (opeak * 1e12), owl.compulsory_bytes() / (pk["hbm_gbs"] * 1e9)) * 1e3
                others[k] = {"workload": owl.name, "ms_per_call": r4(oms),
                             "tflops": r4(owl.flops() / (oms * 1e-3) / 1e12),
                             "roofline_ms": r4(rl), "pct_of_roofline": r4(100.0 * rl / oms),
                             "ms_cold_l2": r4(time_cold(torch, ocall))}
                if isinstance(owl, fc_inputs.ConvWorkload):
                    others[k]["epilogue_frac"] = r4(epilogue_roofline(owl, oms, sm_count, sm_mhz)["frac"])
            del od, ocall, oout
            torch.cuda.empty_cache()
        line["other_workloads"] = others
        # the five configurations of the problem statements, compact and last on the line (so that a
        # record that keeps only the line's end still shows each): ms per call and % of roofline
        summ = {key: [r4(ms), r4(line["pct_of_roofline"])]}
        for k in ("A", "B", "C", "D", "E"):
            if k in others:
                summ[k] = [others[k]["ms_per_call"], others[k]["pct_of_roofline"]]
        line["configs_ms_pct"] = {k: summ[k] for k in ("A", "B", "C", "D", "E") if k in summ}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (default: about 2 s of device time)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="B",
                    choices=sorted(k for k, w in fc_inputs.WORKLOADS.items()
                                   if not isinstance(w, fc_inputs.EpilogueWorkload)))
    ap.add_argument("--impl", default="fc", choices=["fc", "reference"])
    ap.add_argument("--others", default="Bt,Cb,Db,D3,B3,C3,Bp,Cp,Cn,Cbn,Bn,En,K1e,K2e,K3e,A,C,D,E",
                    help="other workloads timed briefly into other_workloads")
    ap.add_argument("--no-others", action="store_true")
    ap.add_argument("--e2e-chunks", type=int, default=8,
                    help="slices of the batch whose host copies overlap the kernels in the end-to-end timing")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end leg (for launch lists of the device-resident calls alone)")
    ap.add_argument("--no-tf32-peak", action="store_true", help="skip the TF32 library GEMM peak measurement")
    args = ap.parse_args()
    if args.impl == "reference":
        return reference_arm(args)
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
