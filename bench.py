"""Benchmark of the gated delta rule forward on GB300.

One step = one chunked prefill of the whole workload through the C ABI
(lr_fwd_chunked): every row of the hot path (staging, log-decay, masked
scores, delta couplings, UT/WY pseudo-values, output, state carry).  The
default workload is the long gated-delta prefill: B=2, H=16, T=16384,
dk=dv=128, bf16 q/k/v/o, fp32 state, chunk 64.  Its inputs (545 MB) are larger
than L2, so no flush is needed between steps.  The other prefill workloads --
RetNet retention (B=4, H=8, T=2048; its inputs fit in L2, so L2 is flushed
before every timed call) and the Mamba-2-style gate (B=8, H=16, T=4096) --
are measured the same way under their own keys, each with its roofline,
tensor, end-to-end and oracle lines.  "decode" times 1000 consecutive decode
steps (lr_step) over 512 sequences x 32 heads.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload (independent sequences, no data exchange): weak scaling.
"""
from __future__ import annotations

import argparse
import csv
import dataclasses
import io
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

DEFAULT_WORKLOAD = "gdn_prefill_bf16"
DECODE_WORKLOAD = "gdn_decode_bf16"
DIAG_WORKLOAD = "gla_bf16"
MLSTM_WORKLOAD = "mlstm_bf16"
GEN_DELTA_WORKLOAD = "rwkv7_bf16"
# the other prefill workloads measured beside the headline, each with its own lines
CONFIG_WORKLOADS = ("retnet_bf16", "mamba2_gate_bf16")
METRIC = "chunked fwd tokens/s"
UNIT = "tokens/s"


# DRAM traffic per lr_fwd_chunked call (prep + scan launches) from one ncu
# capture of each kernel (dram__bytes_read.sum + dram__bytes_write.sum), tied
# to the kernel source it was taken on: reported only while that source is
# unchanged.
TRAFFIC_SOURCES = ("gated_delta_rule_fwd_gb300/csrc/chunked_tc.cu",
                   "gated_delta_rule_fwd_gb300/csrc/scan_tc.cuh",
                   "gated_delta_rule_fwd_gb300/csrc/tc_common.cuh")
TRAFFIC = {
    "gdn_prefill_bf16": {"bytes": 272.936448e6 + 289.770496e6 + 750.092032e6 + 118.885376e6,
                         "sha256": "fdb5480613b20bc288441e97f04ca6e27aa906d3ce6ad8aebdf633b2e2b9c158"},
}

def kernel_source_sha256():
    import hashlib
    h = hashlib.sha256()
    for rel in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(w):
    t = TRAFFIC.get(w.name)
    if t is None or t["sha256"] != kernel_source_sha256():
        return None
    return t["bytes"]


# --------------------------------------------------------------- work counts

def head_token_bytes(w):
    """Algorithmic bytes per head-token: q, k, v, o once each, alpha and beta
    where the mode reads them."""
    es = 2 if w.dtype == "bf16" else 4
    b = es * (2 * w.dk + 2 * w.dv)
    if w.mode in (workloads.DECAY, workloads.GATED_DELTA):
        b += 4
    if w.mode == workloads.DIAG_DECAY:   # one gate per key channel
        b += 4 * w.dk
    if w.mode in (workloads.DELTA, workloads.GATED_DELTA):
        b += 4
    return b


def chunk_bytes(w):
    """Algorithmic bytes of one chunked call: per head-token bytes plus S0 read
    (when given) and S_T written once."""
    heads = w.B * w.H
    state = heads * w.dv * w.dk * 4
    return heads * w.T * head_token_bytes(w) + state * (2 if w.s0_std > 0 else 1)


def chunk_flops(w):
    """Chunk-form tensor flops (dense C x C tiles counted in full, UT inverse
    excluded): 2C(3dk+2dv)+6dk*dv per head-token with delta,
    2C(dk+dv)+4dk*dv without (the diagonal gate's four 64 x 16 sub-block
    score products add up to one C x C product)."""
    C = w.chunk
    if w.mode in (workloads.DELTA, workloads.GATED_DELTA):
        per = 2 * C * (3 * w.dk + 2 * w.dv) + 6 * w.dk * w.dv
    else:
        per = 2 * C * (w.dk + w.dv) + 4 * w.dk * w.dv
    return w.B * w.H * w.T * per


def recurrent_flops(w):
    """Recurrent-form count: three d_k x d_v products per head-token."""
    return w.B * w.H * w.T * 6 * w.dk * w.dv


def decode_step_bytes(w):
    """State read + written once, plus q, k, v, o and alpha, beta."""
    nh = w.B * w.H
    es = 2 if w.dtype == "bf16" else 4
    return nh * (2 * w.dv * w.dk * 4 + es * (2 * w.dk + 2 * w.dv) + 8)


# ------------------------------------------------------------------- helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock/throttle samples, kept for a [t0, t1] wall window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(f"/tmp/lr_clocks_{os.getpid()}.csv", "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.out.name) as f:
            for r in csv.reader(io.StringIO(f.read())):
                if len(r) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + r[0].strip().split(".")[1]) if "." in r[0] else 0.0
                    rows.append((ts + frac, [x.strip() for x in r]))
                except ValueError:
                    continue
        os.unlink(self.out.name)
        inside = [x for t, x in rows if t0 - 0.05 <= t <= t1 + 0.05] or [x for _, x in rows]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(x[2]) for x in inside if x[2].replace(".", "").isdigit()]
        mx = [float(x[3]) for x in inside if x[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for x in inside for i in range(4) if x[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(inside),
                "power_w_max": max((float(x[4]) for x in inside
                                    if x[4].replace(".", "").isdigit()), default=None)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, rank, ws, local
    return None, 0, 1, 0


def barrier(dist, device):
    if dist is not None:
        dist.barrier(device_ids=[device.index] if device.type == "cuda" else None)


def max_over_ranks(dist, x, device):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ oracle timing

def host_cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def time_oracle(w, budget_s=15.0, max_heads=None):
    """The fp64 oracle, as it stands, on a bounded sample of the workload:
    whole sequences of the first n heads of batch 0, n sized for about
    ``budget_s`` of CPU work.  Returns (tokens/s scaled to the workload, info)."""
    import oracle
    x = workloads.draw(w.gen, 1, w.H, w.T, w.dk, w.dv, w.seed, w.torch_dtype, w.s0_std)
    cores = host_cores()

    def run(nh, threads):
        sl = lambda t: None if t is None else t[:, :nh].contiguous()
        t0 = time.perf_counter()
        oracle.recurrent(w.mode, sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["alpha"]), sl(x["beta"]),
                         sl(x["S0"]), threads=threads)
        return time.perf_counter() - t0

    one = run(1, 1)                                    # one head, one thread
    # about budget_s seconds of single-core work, spread over the host cores
    n = max(1, min(w.H if max_heads is None else max_heads, int(budget_s / max(one, 1e-6))))
    threads = min(n, cores)
    wall = run(n, threads)
    head_tokens_per_s = n * w.T / wall
    tokens_per_s = head_tokens_per_s / w.H             # a token carries H heads
    info = {"value": tokens_per_s, "unit": UNIT, "cores": threads, "host_cores": cores,
            "kind": "oracle",
            "sample": f"{n} of {w.B * w.H} (batch, head) sequences, all T={w.T} tokens each, "
                      f"fp64 C recurrence on {threads} threads ({cores} host cores); "
                      f"{n * w.T} head-tokens in {wall:.2f} s wall "
                      f"({one:.2f} s for one sequence on one core)"}
    return tokens_per_s, info


def l2_note(w, dev, flush):
    """Input bytes of one call against the device's L2, and what the timing did."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    es = 2 if w.dtype == "bf16" else 4
    heads = w.B * w.H
    inputs = heads * w.T * es * (2 * w.dk + w.dv) + heads * w.T * 4 * 2
    if w.s0_std > 0:
        inputs += heads * w.dv * w.dk * 4
    how = (f"L2 flushed before every timed call (a {2 * l2 >> 20} MB write outside the timed "
           "events)" if flush else "no flush between calls")
    rel = "<" if inputs < l2 else ">"
    return f"inputs {inputs / 1e6:.1f} MB {rel} {l2 / 1e6:.1f} MB L2; {how}", inputs


class Flusher:
    """Writes a buffer of twice the L2 size, evicting whatever L2 held."""

    def __init__(self, dev):
        n = 2 * torch.cuda.get_device_properties(dev).L2_cache_size
        self.buf = torch.empty(n // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.buf.fill_(1)


def time_calls(step, stream, steps, dist, dev, flush=None):
    """Mean ms per call over ``steps`` calls, CUDA events on ``stream``, max
    over ranks.  With ``flush``: L2 is flushed before every call, outside the
    timed events, and each call is timed on its own."""
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
    else:
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            with torch.cuda.stream(stream):
                flush()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = sum(a.elapsed_time(b) for a, b in evs)
    return max_over_ranks(dist, ms, dev) / steps


def e2e_chunked(lr, w, x, dev, dist, stream, ws, steps):
    """End to end through the public API: every step copies its inputs from
    pinned host memory to the device, calls lr_fwd_chunked and copies o and
    S_T back to pinned host memory.  Steps are pipelined over streams
    (uploads, calls, downloads) with two device buffer sets, so the uploads of
    step i+1 and the downloads of step i-1 overlap the call of step i.
    Returns (tokens/s over all ranks, h2d bytes, d2h bytes)."""
    world = dist.get_world_size() if dist else 1
    hx = {n: (t.pin_memory() if t is not None else None) for n, t in x.items()}
    used = {n for n, t in hx.items()
            if t is not None and not (n == "alpha" and w.mode in (workloads.LINEAR, workloads.DELTA))
            and not (n == "beta" and w.mode in (workloads.LINEAR, workloads.DECAY,
                                                 workloads.DIAG_DECAY))}
    oshape, sshape = (w.B, w.H, w.T, w.dv), (w.B, w.H, w.dv, w.dk)
    ho = [torch.empty(oshape, dtype=w.torch_dtype).pin_memory() for _ in range(2)]
    hs = [torch.empty(sshape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(hx[n].numel() * hx[n].element_size() for n in used)
    d2h = ho[0].numel() * ho[0].element_size() + hs[0].numel() * hs[0].element_size()
    dx = [{n: (torch.empty_like(hx[n], device=dev) if n in used else None) for n in hx}
          for _ in range(2)]
    do_ = [torch.empty(oshape, dtype=w.torch_dtype, device=dev) for _ in range(2)]
    ds_ = [torch.empty(sshape, dtype=torch.float32, device=dev) for _ in range(2)]
    s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    up_done = [torch.cuda.Event() for _ in range(2)]
    call_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    started = [False, False]

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(s_up):
            if started[b]:
                s_up.wait_event(call_done[b])  # the call of step i-2 has read these inputs
            for n in used:
                dx[b][n].copy_(hx[n], non_blocking=True)
            up_done[b].record(s_up)
        stream.wait_event(up_done[b])
        if started[b]:
            stream.wait_event(down_done[b])    # outputs of step i-2 copied out
        d = dx[b]
        lr.lr_fwd_chunked(d["q"], d["k"], d["v"], d["alpha"], d["beta"], d["S0"], mode=w.mode,
                          chunk=w.chunk, o=do_[b], S_T=ds_[b], workspace=ws, stream=stream)
        call_done[b].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(call_done[b])
            ho[b].copy_(do_[b], non_blocking=True)
            hs[b].copy_(ds_[b], non_blocking=True)
            down_done[b].record(s_down)
        started[b] = True

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_up)
    for i in range(steps):
        e2e_step(i)
    s_down.wait_stream(s_up)
    s_down.wait_stream(stream)
    e1.record(s_down)
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    return w.B * w.T * world * steps / (e_ms / 1e3), h2d, d2h


def work_lines(w, ms_per_call, peaks, traffic=None):
    """roofline (HBM, algorithmic bytes) and tensor (chunk-form flops) objects
    for one lr_fwd_chunked call of ``w`` taking ``ms_per_call``."""
    s = ms_per_call / 1e3
    nbytes, nflops = chunk_bytes(w), chunk_flops(w)
    gbs, tf = nbytes / s / 1e9, nflops / s / 1e12
    roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": gbs / peaks["hbm_gbs"], "traffic": traffic,
            "peak_source": peaks["source"] + " burst copy", "algorithmic_bytes_per_launch": nbytes}
    tensor = {"achieved_tflops": tf, "peak_tflops": peaks["bf16_tflops"],
              "frac_of_bf16_peak": tf / peaks["bf16_tflops"], "flops_per_launch": nflops,
              "count": "chunk-form MMA flops", "recurrent_flops_per_launch": recurrent_flops(w),
              "achieved_tflops_recurrent_count": recurrent_flops(w) / s / 1e12}
    return roof, tensor


def mode_name(w):
    return ["linear", "decay", "delta", "gated_delta", "diag_decay"][w.mode]


def bench_config(lr, w, args, dist, dev, peaks, rank, world):
    """One of the other prefill workloads (RetNet retention, Mamba-2-style
    gate), measured like the headline: device-resident calls (with an L2
    flush before every call when the inputs fit in L2, and back to back),
    its roofline and tensor lines, the end-to-end number and the oracle on
    the host cores."""
    x = workloads.draw_workload(w)
    xd = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype, device=dev)
    st = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, lr.workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.torch_dtype, w.mode,
                                              w.chunk)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        lr.lr_fwd_chunked(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                          mode=w.mode, chunk=w.chunk, o=o, S_T=st, workspace=ws, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    steps = max(3, min(args.steps, 100))
    note, inputs = l2_note(w, dev, flush=False)
    fits = inputs < torch.cuda.get_device_properties(dev).L2_cache_size
    ms_b2b = time_calls(step, stream, steps, dist, dev)
    ms_fl = time_calls(step, stream, steps, dist, dev, flush=Flusher(dev)) if fits else None
    ms = ms_fl if fits else ms_b2b
    roof, tensor = work_lines(w, ms, peaks)
    e2e_v, h2d, d2h = e2e_chunked(lr, w, x, dev, dist, stream, ws, max(3, min(args.steps, 20)))
    out = {"workload": w.name, "entry_point": "lr_fwd_chunked", "metric": METRIC,
           "value": w.B * w.T * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
           "steps": steps, "higher_is_better": True, "dtype": w.dtype,
           "config": {"workload": w.name, "mode": mode_name(w), "B": w.B, "H": w.H, "T": w.T,
                      "dk": w.dk, "dv": w.dv, "chunk": w.chunk, "state": "fp32",
                      "l2": l2_note(w, dev, flush=fits)[0]},
           "ms_per_step_back_to_back": ms_b2b, "roofline": roof, "tensor": tensor,
           "e2e": {"value": e2e_v, "unit": UNIT, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h},
           "gpu_launches": steps * 2}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = time_oracle(w, budget_s=min(args.cpu_budget, 8.0))[1]
    return out


def run_ours(args, dist, rank, world, local):
    import gated_delta_rule_fwd_gb300 as lr
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    peaks = load_peaks()

    x = workloads.draw_workload(w)
    xd = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype, device=dev)
    st = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ws = torch.empty(max(1, lr.workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.torch_dtype, w.mode,
                                              w.chunk)), dtype=torch.uint8, device=dev)

    def step():
        lr.lr_fwd_chunked(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                          mode=w.mode, chunk=w.chunk, o=o, S_T=st, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    note, inputs = l2_note(w, dev, flush=False)
    fits = inputs < torch.cuda.get_device_properties(dev).L2_cache_size
    flush = Flusher(dev) if fits else None

    # the timed region: exactly K steps (with an L2 flush before each when the
    # inputs would fit in L2); then the same steps repeated for at least a
    # second, so the clock sampler sees the GPU under this load
    clocks = ClockSampler(dev.index)
    clocks.start()
    time.sleep(0.3)
    wall0 = time.time()
    ms_per_step = time_calls(step, stream, args.steps, dist, dev, flush=flush)
    sustained_steps, t_end = 0, time.time() + 1.0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    while time.time() < t_end or sustained_steps < args.steps:
        for _ in range(args.steps):
            step()
        sustained_steps += args.steps
        torch.cuda.synchronize(dev)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    barrier(dist, dev)
    clocks.stop()
    sustained_ms = max_over_ranks(dist, e0.elapsed_time(e1), dev) / sustained_steps

    tokens = w.B * w.T * world
    value = tokens / (ms_per_step / 1e3)
    roof, tensor = work_lines(w, ms_per_step, peaks,
                              args.traffic if args.traffic is not None else measured_traffic(w))
    e2e_value, h2d, d2h = e2e_chunked(lr, w, x, dev, dist, stream, ws, max(3, min(args.steps, 20)))

    extra = {}
    if not args.no_configs:
        for name in CONFIG_WORKLOADS:
            if name != w.name:
                extra[name] = bench_config(lr, workloads.WORKLOADS[name], args, dist, dev, peaks,
                                           rank, world)
    if not args.no_decode:
        extra["decode"] = run_decode(lr, dev, dist, peaks, args)
    if not args.no_fused and w.gen in workloads.FUSED_FLAGS:
        extra["fused"] = run_fused(lr, dev, dist, args, w, ms_per_step)
    if not args.no_fused and not args.no_decode:
        extra["fused_decode"] = run_decode(lr, dev, dist, peaks, args, fused=True)
    if not args.no_diag and not args.only_gen_delta and w.name != DIAG_WORKLOAD:
        extra["diag"] = run_diag(lr, dev, dist, args, peaks)
    if not args.no_diag and not args.only_gen_delta:
        extra["mlstm"] = run_mlstm(lr, dev, dist, args, peaks)
    if not args.no_diag:
        extra["gen_delta"] = run_gen_delta(lr, dev, dist, args, peaks)

    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        _, cpu = time_oracle(w, budget_s=args.cpu_budget)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded; shapes and distributions of the workload)",
        "config": {"workload": w.name, "mode": mode_name(w),
                   "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
                   "state": "fp32", "global_batch": w.B * world, "seq_len": w.T,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": l2_note(w, dev, flush=fits)[0]},
        "roofline": roof,
        "tensor": tensor,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": max(3, min(args.steps, 20)),
                "pipelined": "uploads, calls and downloads on three streams, two buffer sets"},
        # lr_fwd_chunked launches its per-block pass and its scan for bf16, one kernel for fp32
        "gpu_launches": args.steps * (2 if w.dtype == "bf16" else 1),
        "clocks": clocks.summary(wall0, wall1),
        "sustained": {"ms_per_step": sustained_ms, "steps": sustained_steps,
                      "note": "the timed steps repeated back to back for at least 1 s after the "
                              "timed region; clocks are sampled over both"},
        "cpu_baseline": cpu,
    }
    out.update(extra)
    return out


def run_gen_delta(lr, dev, dist, args, peaks):
    """The generalised delta rule (RWKV-7 reading) through
    lr_fwd_chunked_gen_delta: three launches, the per-block pass over 32-token
    blocks (decays on the CUDA cores, the four score matrices by one tcgen05
    product, the triangular solve), the coupling of consecutive blocks (one
    tcgen05 product per block) and the tensor-core scan with values stacked on
    pseudo-values.  Algorithmic bytes: q, kw, v, o at bf16, w, kappa, a at fp32
    per head-token, the state read and written."""
    w = workloads.WORKLOADS[GEN_DELTA_WORKLOAD]
    if args.gen_delta_batch:  # a smaller case of the same shape per sequence (profiling)
        w = dataclasses.replace(w, B=args.gen_delta_batch)
    x = workloads.draw_gen_delta(w.B, w.H, w.T, w.dk, w.dv, seed=w.seed, dtype=w.torch_dtype,
                                 state=True)
    xd = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype, device=dev)
    st = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, lr.gen_delta_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.torch_dtype)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(3, min(args.steps, 100))

    def step():
        lr.lr_fwd_chunked_gen_delta(xd["q"], xd["kw"], xd["v"], xd["w"], xd["kappa"], xd["a"],
                                    xd["S0"], o=o, S_T=st, workspace=ws, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(dist, e0.elapsed_time(e1), dev) / steps
    world = dist.get_world_size() if dist else 1
    heads = w.B * w.H
    nbytes = heads * w.T * (2 * (2 * w.dk + 2 * w.dv) + 12 * w.dk) + 2 * heads * w.dv * w.dk * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": w.name, "entry_point": "lr_fwd_chunked_gen_delta", "B": w.B, "H": w.H,
            "T": w.T, "dk": w.dk, "dv": w.dv, "value": w.B * w.T * world / (ms / 1e3),
            "unit": UNIT, "ms_per_step": ms, "steps": steps, "algorithmic_bytes_per_launch": nbytes,
            "achieved_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "gpu_launches": 3 * steps,
            "workspace_bytes": ws.numel(),
            "path": "per-block pass (tcgen05 scores, fp32 solve) + tcgen05 coupling + tcgen05 "
                    "scan (bf16 operands, fp32 state)"}


def run_mlstm(lr, dev, dist, args, peaks):
    """The mLSTM workload through lr_fwd_chunked_mlstm (five launches: the
    stabiliser, the per-block pass, the scan, the normaliser, the division),
    timed like the headline.  Algorithmic bytes: q, k, v, h at bf16 and the two
    gates per head-token, plus the final state."""
    w = workloads.WORKLOADS[MLSTM_WORKLOAD]
    x = workloads.draw_mlstm(w.B, w.H, w.T, w.dk, w.dv, seed=w.seed, dtype=w.torch_dtype)
    xd = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    ws = torch.empty(max(1, lr.mlstm_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.torch_dtype)),
                     dtype=torch.uint8, device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    h = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype, device=dev)
    CT = torch.empty((w.B, w.H, w.dv, w.dk), **f32)
    nT = torch.empty((w.B, w.H, w.dk), **f32)
    mT = torch.empty((w.B, w.H), **f32)
    stream = torch.cuda.current_stream(dev)
    steps = max(3, min(args.steps, 100))

    def step():
        lr.lr_fwd_chunked_mlstm(xd["q"], xd["k"], xd["v"], xd["fgate"], xd["igate"], h=h, C_T=CT,
                                n_T=nT, m_T=mT, workspace=ws, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(dist, e0.elapsed_time(e1), dev) / steps
    world = dist.get_world_size() if dist else 1
    heads = w.B * w.H
    nbytes = heads * w.T * (2 * (2 * w.dk + 2 * w.dv) + 8) + heads * (w.dv * w.dk + w.dk + 1) * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": w.name, "entry_point": "lr_fwd_chunked_mlstm", "B": w.B, "H": w.H,
            "T": w.T, "dk": w.dk, "dv": w.dv, "value": w.B * w.T * world / (ms / 1e3),
            "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "algorithmic_bytes_per_launch": nbytes, "achieved_gbs": gbs,
            "frac_hbm": gbs / peaks["hbm_gbs"], "gpu_launches": steps * 5}


def run_diag(lr, dev, dist, args, peaks):
    """The diagonal-gate (GLA) workload through lr_fwd_chunked, timed like the
    headline, with its HBM roofline (algorithmic bytes include alpha, one fp32
    gate per key channel and token)."""
    w = workloads.WORKLOADS[DIAG_WORKLOAD]
    x = workloads.draw_workload(w)
    xd = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype, device=dev)
    st = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, lr.workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.torch_dtype, w.mode,
                                              w.chunk)), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(3, min(args.steps, 100))

    def step():
        lr.lr_fwd_chunked(xd["q"], xd["k"], xd["v"], xd["alpha"], None, xd["S0"], mode=w.mode,
                          chunk=w.chunk, o=o, S_T=st, workspace=ws, stream=stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(dist, e0.elapsed_time(e1), dev) / steps
    world = dist.get_world_size() if dist else 1
    gbs = chunk_bytes(w) / (ms / 1e3) / 1e9
    return {"workload": w.name, "mode": "diag_decay", "entry_point": "lr_fwd_chunked",
            "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
            "value": w.B * w.T * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "steps": steps, "algorithmic_bytes_per_launch": chunk_bytes(w),
            "achieved_gbs": gbs, "frac_hbm": gbs / peaks["hbm_gbs"],
            "achieved_tflops": chunk_flops(w) / (ms / 1e3) / 1e12,
            "gpu_launches": steps * 2}


def run_fused(lr, dev, dist, args, w, plain_ms):
    """The same workload through lr_fwd_chunked_fused from pre-activation
    inputs (the maps of the workload's layer in the kernels), timed like the
    headline, with and without the output RMSNorm pass."""
    flags_all = workloads.FUSED_FLAGS[w.gen]
    x = workloads.draw_pre(w.gen, w.B, w.H, w.T, w.dk, w.dv, w.seed, w.torch_dtype, w.s0_std)
    if w.gen == "mamba2":
        x["q"] = (x["q"].float() / w.dk ** 0.5).to(w.torch_dtype)
        x["k"] = (x["k"].float() / w.dk ** 0.5).to(w.torch_dtype)
    xd = {n: (t.to(dev) if t is not None else None) for n, t in x.items()}
    o = torch.empty((w.B, w.H, w.T, w.dv), dtype=w.torch_dtype, device=dev)
    st = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, lr.fused_workspace_size(w.B, w.H, w.T, w.dk, w.dv, w.torch_dtype,
                                                    w.mode, flags_all, w.chunk)),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    steps = max(3, min(args.steps, 50))
    res = {}
    for name, flags in (("maps", flags_all & ~workloads.FUSE_O_RMSNORM), ("maps_and_norm", flags_all)):
        def step():
            lr.lr_fwd_chunked_fused(xd["q"], xd["k"], xd["v"], xd["alpha"], xd["beta"], xd["S0"],
                                    mode=w.mode, flags=flags, alpha_scale=xd["alpha_scale"],
                                    norm_weight=xd["norm_weight"], chunk=w.chunk, o=o, S_T=st,
                                    workspace=ws, stream=stream)
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        res[name] = max_over_ranks(dist, e0.elapsed_time(e1), dev) / steps
    world = dist.get_world_size() if dist else 1
    ms = res["maps_and_norm"]
    return {"workload": w.name, "entry_point": "lr_fwd_chunked_fused", "flags": flags_all,
            "maps": "SiLU+L2 q,k; sigmoid beta; sigmoid alpha; output RMSNorm" if w.gen == "gdn"
                    else "softplus alpha gate (c = 0.1); output RMSNorm",
            "value": w.B * w.T * world / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "ms_per_step_without_norm": res["maps"], "ms_per_step_plain": plain_ms,
            "steps": steps,
            # bf16: per-block pass + scan (which applies the norm); fp32: the
            # chunked kernel + the norm pass
            "gpu_launches": steps * 2}


def run_decode(lr, dev, dist, peaks, args, fused=False):
    """1000 consecutive decode steps (fresh inputs per step, drawn beforehand
    on the device), timed as a whole after 10 warm-up steps on a scratch
    copy of the state.  With ``fused``: pre-activation inputs through
    lr_step_fused with the gated-delta layer's maps (200 steps)."""
    w = workloads.WORKLOADS[DECODE_WORKLOAD]
    g = torch.Generator(dev)
    S = workloads.draw_decode_state(w, dev, g)
    steps = w.steps if args.decode_steps is None else max(1, args.decode_steps)
    if fused:
        steps = min(steps, 200)
        inputs = [workloads.draw_decode_step_pre(w, s, dev, g) for s in range(steps)]
        wn = (0.5 + torch.rand((w.dv,), generator=g, device=dev)).float()
        flags = workloads.FUSED_FLAGS["gdn"]
    else:
        inputs = [workloads.draw_decode_step(w, s, dev, g) for s in range(steps)]
    o = torch.empty((w.B, w.H, w.dv), dtype=w.torch_dtype, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(i, state):
        if fused:
            lr.lr_step_fused(i["q"], i["k"], i["v"], i["alpha"], i["beta"], state, mode=w.mode,
                             flags=flags, norm_weight=wn, o=o, stream=stream)
        else:
            lr.lr_step(i["q"], i["k"], i["v"], i["alpha"], i["beta"], state, mode=w.mode, o=o,
                       stream=stream)

    scratch = S.clone()
    for s in range(min(10, steps)):
        call(inputs[s], scratch)
    del scratch
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in inputs:
        call(i, S)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(dist, e0.elapsed_time(e1), dev)
    per = ms / steps / 1e3
    gbs = decode_step_bytes(w) / per / 1e9
    return {"workload": w.name, "entry_point": "lr_step_fused (all maps)" if fused else "lr_step",
            "metric": "decode step state GB/s", "value": gbs, "unit": "GB/s",
            "frac_hbm": gbs / peaks["hbm_gbs"], "peak_gbs": peaks["hbm_gbs"],
            "us_per_step": per * 1e6, "steps": steps, "tokens_per_s": w.B / per,
            "bytes_per_step": decode_step_bytes(w), "gpu_launches": steps,
            "N": w.B, "H": w.H, "dk": w.dk, "dv": w.dv}


def run_reference(args, rank):
    """The oracle on the host cores, as the reference arm: each step is the
    fp64 recurrence over a bounded sample of the workload."""
    if rank != 0:
        return None
    w = workloads.WORKLOADS[args.workload]
    import oracle
    x = workloads.draw(w.gen, 1, w.H, w.T, w.dk, w.dv, w.seed, w.torch_dtype, w.s0_std)
    cores = host_cores()
    nh = min(w.H, cores)
    T = min(w.T, args.ref_tokens)
    def sl(name, t):
        if t is None:
            return None
        if name == "S0":
            return t[:, :nh].contiguous()
        return t[:, :nh, :T].contiguous()

    xs = {n: sl(n, t) for n, t in x.items()}

    def step():
        oracle.recurrent(w.mode, xs["q"], xs["k"], xs["v"], xs["alpha"], xs["beta"], xs["S0"],
                         threads=nh)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = nh * T * args.steps / dt / w.H
    sample = (f"{nh} of {w.B * w.H} (batch, head) sequences x first {T} of {w.T} tokens per step, "
              f"fp64 C recurrence, {nh} threads")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the workload)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                       "chunk": w.chunk},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nh, "host_cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    # the lr_fwd_chunked workloads (the mLSTM and RWKV-7 ones have
                    # their own legs: --no-* flags select them)
                    choices=[k for k, v in workloads.WORKLOADS.items()
                             if k != DECODE_WORKLOAD and v.gen not in ("mlstm", "gd")])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the RetNet and Mamba-2-style prefill workloads")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="decode steps to time (default: the workload's 1000)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fused", action="store_true",
                    help="skip the fused entry points' timings (prefill and decode)")
    ap.add_argument("--no-diag", action="store_true",
                    help="skip the diagonal-gate (GLA) and mLSTM workloads' timings")
    ap.add_argument("--only-gen-delta", action="store_true",
                    help="of the extra workloads time only the RWKV-7 one")
    ap.add_argument("--gen-delta-batch", type=int, default=None,
                    help="batch of the RWKV-7 workload (default: its own; for profiling)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of single-core oracle work in the cpu_baseline sample")
    ap.add_argument("--ref-tokens", type=int, default=2048,
                    help="tokens per sequence in each reference-arm step")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    dist, rank, world, local = dist_setup()
    if args.impl == "reference":
        out = run_reference(args, rank)
    else:
        out = run_ours(args, dist, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
