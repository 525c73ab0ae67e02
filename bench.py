"""Benchmark of the retention hot path on B300.

Headline: chunkwise-forward tokens/s (B*N sequence positions per second, all
heads included) on the 7B-shaped workload B=8, H=16, N=8192, d_k=256,
d_v=512, chunk=128 (the largest single-GPU workload), bf16 q/k/v/out with
fp32 accumulation and state.  One step = one retention_chunkwise call over
one batch; inputs are resident in HBM and L2 is flushed between timed steps,
outside the timed events: a 512 MiB write, then a 512 MiB read, so that
neither the inputs nor the flush's own dirty lines (whose write-back would
land inside the timed call) remain in L2.

Also reported on the same line:
  e2e         the headline metric through host buffers: one
              retention_chunkwise_host call per step on pinned host q/k/v
              (copies in, kernels, out and state copied back, pipelined over
              slabs of batch rows inside the call).
  roofline    algorithmic bytes of one retention_chunkwise call (Q,K,V read,
              out and final state written) over its CUDA-event duration,
              against the measured HBM copy bandwidth; the tensor fraction
              (algorithmic flops over the measured bf16 peak) beside it.
  cpu_baseline  the fp64 CPU oracle (chunkwise form, same chunk) on the host
              cores, timed on one batch row of the workload (all its heads)
              and scaled to the whole batch.
  mid, long   the mid (B=4,H=8,N=2048,d_k=d_v=128,C=64) and long-context
              (B=1,H=16,N=16384,d_k=128,d_v=256,C=128) chunkwise runs, each
              with its own roofline and e2e.
  decode      the recurrent decode step on 64 sequences x 16 heads, d_k=128,
              d_v=256, fp32 state (128 MiB > L2): 1024 sequential steps
              captured in one CUDA graph; steps/s and HBM roofline.
  groupnorm, rotate, mid_groupnorm_fused, mid_rotated, mid_backward,
  7b_backward, mid_parallel, long_parallel   the other kernels.

`--impl reference` times the fp64 CPU oracle alone on the same workload and
metric (one batch row of the 7B-shaped workload per step, scaled to the
batch) and prints its own line.
`--only {mid,long,7b,decode,groupnorm,rotate,backward,backward_long,backward_7b,parallel,parallel_long,rotated,e2e}`
runs one workload alone and prints its timing
(used to give ncu a small, single-workload command).
Under torchrun each rank runs its own replica (independent batches, no
collective on the data path); value = all ranks' tokens / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MID = dict(name="mid", B=4, H=8, N=2048, dk=128, dv=128, chunk=64)
LONG = dict(name="long", B=1, H=16, N=16384, dk=128, dv=256, chunk=128)
B7 = dict(name="7b", B=8, H=16, N=8192, dk=256, dv=512, chunk=128)
DECODE = dict(name="decode", T=1024, B=64, H=16, dk=128, dv=256)
METRIC = "retention tokens/s (chunkwise fwd, 1 B300) + decode steps/s; % of roofline"
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Run between timed steps: writes a buffer larger than the 126 MB L2, then
    reads another one, so that the timed call finds neither its inputs in L2
    nor the flush's own dirty lines still waiting to be written back to DRAM."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.acc += self.r.sum()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, "fallback"


def chunk_bytes(w) -> int:
    """Algorithmic HBM bytes of one chunkwise call: Q,K,V read, out written (bf16), S written (fp32)."""
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    return B * H * N * (2 * dk + dv) * 2 + B * H * N * dv * 2 + B * H * dk * dv * 4


def chunk_flops(w) -> int:
    """Algorithmic flops of one chunkwise call (causal part only)."""
    B, H, N, dk, dv, C = w["B"], w["H"], w["N"], w["dk"], w["dv"], w["chunk"]
    return B * H * N * ((dk + dv) * (C + 1) + 4 * dk * dv)


def decode_bytes(w) -> int:
    """Algorithmic HBM bytes of one decode step: S read+write (fp32), q,k,v read, out written (bf16)."""
    B, H, dk, dv = w["B"], w["H"], w["dk"], w["dv"]
    return B * H * (8 * dk * dv + 2 * (2 * dk + dv) + 2 * dv)


# The source files of the kernels each workload's traffic was captured on.
TRAFFIC_SOURCE = {"decode_step": ("simt.cu",), "groupnorm": ("groupnorm.cu",), "rotate": ("rotate.cu",),
                  "mid_parallel": ("parallel_tc.cu",), "long_parallel": ("parallel_tc.cu",),
                  "mid_backward": ("bwd_tc.cu", "chunk_tc.cu")}


def kernel_sha(workload: str = "mid") -> str:
    """sha256[:16] of the kernel source (of the concatenated sources where a call runs kernels of several files)."""
    h = hashlib.sha256()
    for name in TRAFFIC_SOURCE.get(workload, ("chunk_tc.cu",)):
        with open(os.path.join(ROOT, "linear_attention_sequence_02_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per call from the committed ncu summary, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_sha(workload)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == sha and parts[1] == workload:
                return int(parts[2])
    return None


class ClockSampler:
    """SM clock and throttle reasons sampled during a region.

    In-process NVML polling every millisecond (so even a region of a few
    milliseconds gets several samples); if NVML is unavailable, nvidia-smi
    every 200 ms.
    """

    REASONS = (("hw_slowdown", "nvmlClocksEventReasonHwSlowdown"),
               ("hw_thermal_slowdown", "nvmlClocksEventReasonHwThermalSlowdown"),
               ("sw_thermal_slowdown", "nvmlClocksEventReasonSwThermalSlowdown"),
               ("sw_power_cap", "nvmlClocksEventReasonSwPowerCap"))
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []  # (sm_mhz, max_mhz, set of reasons)
        self._stop = threading.Event()
        self._t = None
        self.proc = None
        self.source = None

    def __enter__(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            mx = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
            reasons = getattr(pynvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(pynvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            masks = [(name, getattr(pynvml, attr, getattr(pynvml, attr.replace("Event", "Throttle"), 0)))
                     for name, attr in self.REASONS]

            def poll():
                while not self._stop.is_set():
                    sm = pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM)
                    r = reasons(h)
                    self.samples.append((float(sm), float(mx), {n for n, m in masks if r & m}))
                    time.sleep(0.001)

            self.source = "nvml 1 ms"
            self._t = threading.Thread(target=poll, daemon=True)
            self._t.start()
            return self
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi 200 ms"

            def read():
                names = [n for n, _ in self.REASONS]
                for line in self.proc.stdout:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) < 6:
                        continue
                    try:
                        self.samples.append((float(parts[0]), float(parts[1]),
                                             {n for n, v in zip(names, parts[2:6]) if v.lower() == "active"}))
                    except ValueError:
                        continue

            self._t = threading.Thread(target=read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self._t:
            self._t.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        reasons = set()
        for _, _, r in self.samples:
            reasons |= r
        return {"sm_mhz": statistics.median(x[0] for x in self.samples),
                "sm_max_mhz": max(x[1] for x in self.samples),
                "reasons": sorted(reasons), "samples": len(self.samples), "source": self.source}


def dist_setup(backend: str | None = None):
    """Rendezvous of the replicas (N > 1).  The backend is `backend`, else the
    BENCH_DIST_BACKEND variable, else nccl when CUDA is present and gloo
    otherwise; max_over_ranks then keeps its tensor on the matching device."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = backend or os.environ.get("BENCH_DIST_BACKEND") or (
            "nccl" if torch.cuda.is_available() else "gloo")
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput of weak-scaled replicas: the units all ranks
    processed divided by the slowest rank's time."""
    return units_per_rank * world / max_seconds


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    if dist.get_backend() == "gloo":
        device = torch.device("cpu")  # gloo reduces host tensors
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# our arm

def time_chunkwise(w, steps, warmup, dev, flush, seed=0, norm=False):
    """Per-call device times (ms) of retention_chunkwise (with norm: of
    retention_chunkwise_groupnorm, the GroupNorm fused in), L2 flushed between calls.

    The call (state-only pre-pass, main pass launched with programmatic
    dependent launch, stream-ordered scratch) is captured once in a CUDA graph
    and each timed step replays it, so host-side launch work stays outside the
    device-timed region.  Falls back to eager calls if capture is refused.
    """
    from linear_attention_sequence_02_b300 import binding, inputs
    B, H, N, dk, dv, C = w["B"], w["H"], w["N"], w["dk"], w["dv"], w["chunk"]
    q, k, v = (x.to(dev) for x in inputs.qkv(B, H, N, dk, dv, seed, torch.bfloat16))
    g = binding.gamma_schedule(H).to(dev)
    st = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if norm:
        out = torch.empty(B, N, H, dv, dtype=torch.bfloat16, device=dev)
        gw = torch.Generator().manual_seed(seed + 1)
        wt, bs = torch.randn(H * dv, generator=gw).to(dev), torch.randn(H * dv, generator=gw).to(dev)

        def call(s=None):
            binding.retention_chunkwise_groupnorm(q, k, v, g, C, wt, bs, 1e-6, out=out, state_out=st, stream=s)
    else:
        out = torch.empty(B, H, N, dv, dtype=torch.bfloat16, device=dev)

        def call(s=None):
            binding.retention_chunkwise(q, k, v, g, C, out=out, state_out=st, stream=s)
    for _ in range(max(1, warmup)):
        flush()
        call()
    torch.cuda.synchronize(dev)
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call(torch.cuda.current_stream(dev))
        for _ in range(warmup):
            flush()
            graph.replay()
        torch.cuda.synchronize(dev)
    except Exception:
        graph = None
        torch.cuda.synchronize(dev)

    def run():
        if graph is not None:
            graph.replay()
        else:
            call()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize(dev)
    times = [a.elapsed_time(b) for a, b in evs]
    launches = binding.chunkwise_launches(B, H, N, dk, dv, C) * steps
    how = "cuda graph replay" if graph is not None else "eager calls"
    del graph, q, k, v, out, st
    return times, launches, how


def time_e2e(w, steps, warmup, dev, seed=0):
    """Headline metric through host buffers: retention_chunkwise_host on pinned
    q, k, v (host-to-device copies, the kernels and the device-to-host copies
    of out and state, slab by slab on the library's pipeline streams), timed
    with CUDA events on the calling stream around whole calls.  The device
    buffer is allocated once, before the timed region."""
    from linear_attention_sequence_02_b300 import binding, inputs
    B, H, N, dk, dv, C = w["B"], w["H"], w["N"], w["dk"], w["dv"], w["chunk"]
    qh, kh, vh = (x.pin_memory() for x in inputs.qkv(B, H, N, dk, dv, seed, torch.bfloat16))
    oh = torch.empty(B, H, N, dv, dtype=torch.bfloat16).pin_memory()
    sh = torch.empty(B, H, dk, dv, dtype=torch.float32).pin_memory()
    g = binding.gamma_schedule(H).to(dev)
    buf = torch.empty(binding.chunkwise_host_buffer_size(B, H, N, dk, dv, C), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def one():
        binding.retention_chunkwise_host(qh, kh, vh, g, C, out=oh, state_out=sh, buffer=buf, stream=stream)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        one()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / steps
    h2d = sum(x.numel() * x.element_size() for x in (qh, kh, vh))
    d2h = oh.numel() * oh.element_size() + sh.numel() * sh.element_size()
    return ms, h2d, d2h


def time_decode(w, reps, dev, seed=0):
    """ms per step of 1024 retention_step launches captured in one CUDA graph."""
    from linear_attention_sequence_02_b300 import binding, inputs
    T, B, H, dk, dv = w["T"], w["B"], w["H"], w["dk"], w["dv"]
    q, k, v = (x.to(dev) for x in inputs.decode_steps(T, B, H, dk, dv, seed))
    state = inputs.decode_state(B, H, dk, dv, seed).to(dev)
    outs = torch.empty(T, B, H, dv, dtype=torch.bfloat16, device=dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        for t in range(3):  # warm-up outside capture
            binding.retention_step(q[t], k[t], v[t], state, out=outs[t], stream=side)
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream(dev)
        for t in range(T):
            binding.retention_step(q[t], k[t], v[t], state, out=outs[t], stream=cap)
    stream = torch.cuda.current_stream(dev)
    graph.replay()  # warm-up replay
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        graph.replay()
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b) / T)
    del graph, q, k, v, outs, state
    return times


GROUPNORM = dict(name="groupnorm", B=4, H=8, N=2048, dv=128)  # the mid workload's output


def time_groupnorm(w, reps, dev, flush, seed=0):
    """ms per retention_groupnorm call on a [B,H,N,dv] bf16 input, L2 flushed first."""
    from linear_attention_sequence_02_b300 import binding
    B, H, N, dv = w["B"], w["H"], w["N"], w["dv"]
    g = torch.Generator().manual_seed(seed)
    r = torch.randn(B, H, N, dv, generator=g).to(torch.bfloat16).to(dev)
    wt = torch.randn(H * dv, generator=g).to(dev)
    bs = torch.randn(H * dv, generator=g).to(dev)
    y = torch.empty(B, N, H, dv, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        binding.retention_groupnorm(r, wt, bs, 1e-6, out=y)
    times = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.retention_groupnorm(r, wt, bs, 1e-6, out=y)
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    return times


ROTATE = dict(name="rotate", B=4, H=8, N=2048, d=128)  # the mid workload's queries


def time_rotate(w, reps, dev, flush, seed=0):
    """ms per retention_rotate call on a [B,H,N,d] bf16 input, L2 flushed first."""
    from linear_attention_sequence_02_b300 import binding
    B, H, N, d = w["B"], w["H"], w["N"], w["d"]
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).to(dev)
    th = torch.tensor([10000.0 ** (-2.0 * j / d) for j in range(d // 2)], dtype=torch.float32, device=dev)
    y = torch.empty_like(x)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        binding.retention_rotate(x, th, 0, out=y)
    times = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.retention_rotate(x, th, 0, out=y)
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    return times


def backward_chunk(w) -> int:
    """The chunk length the gradient call's forwards use (128 from N = 4096 on)."""
    return 128 if w["N"] >= 4096 else 64


def backward_flops(w) -> int:
    """Algorithmic flops of one gradient call: three chunkwise forwards (dq,
    and dk and dv walked from the last token), each (C+1)(dk+dv) + 4 dk dv per
    head-token, causal part only."""
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    C = backward_chunk(w)
    return 3 * B * H * N * ((C + 1) * (dk + dv) + 4 * dk * dv)


def backward_bytes(w) -> int:
    """Algorithmic HBM bytes of one gradient call without states: q, k, v and
    dout read, dq, dk, dv written (bf16)."""
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    return B * H * N * 2 * (2 * (2 * dk + dv) + dv)


def time_backward(w, reps, dev, flush, seed=0):
    """Per-call device times (ms) of retention_backward (no starting state, no
    final-state gradient: the usual training case), L2 flushed before each
    call.  The call is captured once in a CUDA graph and replayed, so the
    host-side work of its launches stays outside the timed region (eager calls
    if capture is refused)."""
    from linear_attention_sequence_02_b300 import binding
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    g = torch.Generator().manual_seed(seed)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).to(dev) for d in (dk, dk, dv, dv))
    gam = binding.gamma_schedule(H).to(dev)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), None)
    stream = torch.cuda.current_stream(dev)

    def call(s=None):
        binding.retention_backward(q, k, v, gam, do, want_dstate_in=False, grads=grads, stream=s)
    for _ in range(3):
        call()
    torch.cuda.synchronize(dev)
    graph = None
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call(torch.cuda.current_stream(dev))
        graph.replay()
        torch.cuda.synchronize(dev)
    except Exception:
        graph = None
        torch.cuda.synchronize(dev)
    times = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if graph is not None:
            graph.replay()
        else:
            call()
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    return times


def time_rotated(w, reps, dev, flush, seed=0):
    """ms per call of the chunkwise forward of rotated q and k: the fused call
    (retention_chunkwise_rotated) and the separate path (retention_rotate on
    q, on k, then retention_chunkwise), each captured in a CUDA graph and
    replayed with L2 flushed before each call."""
    from linear_attention_sequence_02_b300 import binding, inputs
    B, H, N, dk, dv, C = w["B"], w["H"], w["N"], w["dk"], w["dv"], w["chunk"]
    q, k, v = (x.to(dev) for x in inputs.qkv(B, H, N, dk, dv, seed, torch.bfloat16))
    g = binding.gamma_schedule(H).to(dev)
    th = torch.tensor([10000.0 ** (-2.0 * j / dk) for j in range(dk // 2)], dtype=torch.float32, device=dev)
    out = torch.empty(B, H, N, dv, dtype=torch.bfloat16, device=dev)
    st = torch.empty(B, H, dk, dv, dtype=torch.float32, device=dev)
    rq, rk = torch.empty_like(q), torch.empty_like(k)
    stream = torch.cuda.current_stream(dev)

    def fused(s=None):
        binding.retention_chunkwise_rotated(q, k, v, g, th, 0, C, out=out, state_out=st, stream=s)

    def separate(s=None):
        binding.retention_rotate(q, th, 0, out=rq, stream=s)
        binding.retention_rotate(k, th, 0, out=rk, stream=s)
        binding.retention_chunkwise(rq, rk, v, g, C, out=out, state_out=st, stream=s)
    res = {}
    for name, fn in (("fused", fused), ("separate", separate)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn(torch.cuda.current_stream(dev))
        graph.replay()
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(reps):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
        del graph
    return res


def parallel_flops(w) -> int:
    """Algorithmic flops of the parallel form (causal part only): per head,
    sum over n of (n+1) scores and (n+1) weighted value rows, N(N+1)(dk+dv)."""
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    return B * H * N * (N + 1) * (dk + dv)


def time_parallel(w, reps, dev, flush, seed=0):
    """ms per retention_parallel call (tensor cores), L2 flushed before each call."""
    from linear_attention_sequence_02_b300 import binding, inputs
    B, H, N, dk, dv = w["B"], w["H"], w["N"], w["dk"], w["dv"]
    q, k, v = (x.to(dev) for x in inputs.qkv(B, H, N, dk, dv, seed, torch.bfloat16))
    g = binding.gamma_schedule(H).to(dev)
    out = torch.empty(B, H, N, dv, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        binding.retention_parallel(q, k, v, g, out=out)
    times = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        binding.retention_parallel(q, k, v, g, out=out)
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    return times


def parallel_entry(w, reps, dev, flush, tflops):
    t = statistics.median(time_parallel(w, reps, dev, flush)) / 1e3
    fl = parallel_flops(w)
    return {"tokens_per_s": round(w["B"] * w["N"] / t, 1), "ms_per_call": round(t * 1e3, 5),
            "config": {k: w[k] for k in ("B", "H", "N", "dk", "dv")} | {
                "workload": f"{w['name']} retention parallel form (O(N^2), tensor cores)",
                "l2": "flushed before each call (512 MiB write, then 512 MiB read)"},
            "roofline": {"bound": "tensor", "achieved": round(fl / t / 1e12, 1), "peak": tflops, "unit": "TFLOP/s",
                         "frac": round(fl / t / 1e12 / tflops, 4), "traffic": recorded_traffic(w["name"] + "_parallel"),
                         "algorithmic_flops_per_call": fl},
            "gpu_launches": 1}


def oracle_sample(w, seed=0):
    """One batch row of workload `w` (all H heads) as fp64 arrays for the oracle."""
    from linear_attention_sequence_02_b300 import binding, inputs
    H, N, dk, dv = w["H"], w["N"], w["dk"], w["dv"]
    q, k, v = inputs.qkv(1, H, N, dk, dv, seed, torch.bfloat16)
    g = binding.gamma_schedule(H).double().numpy()
    return tuple(x.double().numpy() for x in (q, k, v)) + (g,)


def cpu_baseline_chunkwise(w, min_seconds=10.0, max_passes=30):
    """fp64 oracle (chunkwise form, same chunk) on one batch row of the
    workload (all its heads), repeated for >= min_seconds; tokens/s of the
    whole batch = B*N / (B * seconds per row)."""
    import oracle
    B, H, N, dk, dv, C = w["B"], w["H"], w["N"], w["dk"], w["dv"], w["chunk"]
    qd, kd, vd, g = oracle_sample(w)
    orc = oracle.default()
    passes, t0 = 0, time.perf_counter()
    while passes < max_passes and (time.perf_counter() - t0) < min_seconds:
        orc.chunkwise(qd, kd, vd, g, C)
        passes += 1
    dt = (time.perf_counter() - t0) / passes
    return {"value": round(N / dt, 1), "unit": "tokens/s", "cores": orc.threads(), "kind": "oracle",
            "sample": f"one batch row of the {w['name']} workload (H={H},N={N},dk={dk},dv={dv},chunk={C}, "
                      f"all {H} heads) per pass, {passes} fp64 passes of {dt:.3f} s; scaled to B={B} rows"}


def chunkwise_entry(w, steps, warmup, dev, flush, hbm, tflops, peak_kind, rank=0):
    """Device-timed chunkwise call on workload `w`: per-call times, rate, roofline."""
    times, launches, how = time_chunkwise(w, steps, warmup, dev, flush, seed=rank)
    avg_s = sum(times) / len(times) / 1e3
    achieved = chunk_bytes(w) / avg_s / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": recorded_traffic(w["name"]),
                "peak_kind": peak_kind, "kernel": "retention_chunkwise call (every launch of one call)",
                "algorithmic_bytes_per_call": chunk_bytes(w),
                "tensor_flops_frac": round(chunk_flops(w) / avg_s / 1e12 / tflops, 4)}
    cfg = {k: w[k] for k in ("B", "H", "N", "dk", "dv", "chunk")}
    return times, launches, how, roofline, cfg


def e2e_entry(w, steps, warmup, dev, world=1, rank=0):
    e2e_ms, h2d, d2h = time_e2e(w, steps, warmup, dev, seed=rank)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    return {"value": round(whole_job_rate(w["B"] * w["N"], world, e2e_ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "call": "retention_chunkwise_host (pinned host buffers)"}


def run_ours(args):
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from linear_attention_sequence_02_b300 import binding
    binding.lib()
    hbm, tflops, peak_kind = peaks()
    flush = L2Flush(dev)

    # ---- headline: 7B-shaped chunkwise, device-timed ----
    w = B7
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        times, launches, how, roofline, cfg = chunkwise_entry(w, args.steps, args.warmup, dev, flush, hbm, tflops,
                                                              peak_kind, rank)
    torch.cuda.synchronize(dev)
    barrier(world)
    total_ms = max_over_ranks(sum(times), world, dev)
    ms = total_ms / args.steps
    value = whole_job_rate(w["B"] * w["N"] * args.steps, world, total_ms / 1e3)

    # ---- e2e through host buffers ----
    e2e = e2e_entry(w, max(3, args.steps // 4), 3, dev, world, rank)

    extra = {}
    if not args.quick:
        # ---- the other chunkwise workloads ----
        for wl in (MID, LONG):
            t, n, h, rf, c = chunkwise_entry(wl, args.steps, 3, dev, flush, hbm, tflops, peak_kind, rank)
            a_s = statistics.median(t) / 1e3
            extra[wl["name"]] = {
                "tokens_per_s": round(wl["B"] * wl["N"] / a_s, 1), "ms_per_call": round(a_s * 1e3, 5),
                "config": c | {"l2": "flushed between timed calls (512 MiB write, then 512 MiB read)", "timing": h},
                "roofline": rf, "e2e": e2e_entry(wl, max(3, args.steps // 2), 3, dev, world, rank),
                "gpu_launches": n}
        # ---- decode step ----
        dt = time_decode(DECODE, 3, dev)
        step_ms = statistics.median(dt)
        bytes_step = decode_bytes(DECODE)
        extra["decode"] = {
            "steps_per_s": round(1e3 / step_ms, 1),
            "tokens_per_s": round(DECODE["B"] * 1e3 / step_ms, 1),
            "ms_per_step": round(step_ms, 5),
            "config": {"batch": DECODE["B"], "H": DECODE["H"], "dk": DECODE["dk"], "dv": DECODE["dv"],
                       "steps": DECODE["T"], "graph": "1024 launches in one CUDA graph",
                       "l2": "fp32 state 128 MiB > L2"},
            "roofline": {"bound": "hbm", "achieved": round(bytes_step / (step_ms / 1e3) / 1e9, 1),
                         "peak": hbm, "unit": "GB/s",
                         "frac": round(bytes_step / (step_ms / 1e3) / 1e9 / hbm, 4),
                         "traffic": recorded_traffic("decode_step")},
            "gpu_launches": DECODE["T"] * 3,
        }
        gw = GROUPNORM
        gt = statistics.median(time_groupnorm(gw, 20, dev, flush)) / 1e3
        rows = gw["B"] * gw["H"] * gw["N"]
        gbytes = 4 * gw["dv"] * rows  # bf16 row read + bf16 row written
        extra["groupnorm"] = {
            "rows_per_s": round(rows / gt, 1), "ms_per_call": round(gt * 1e3, 5),
            "config": {k: gw[k] for k in ("B", "H", "N", "dv")} | {"l2": "flushed before each call (512 MiB write, then 512 MiB read)",
                                                                   "timing": "CUDA events per call"},
            "roofline": {"bound": "hbm", "achieved": round(gbytes / gt / 1e9, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(gbytes / gt / 1e9 / hbm, 4), "traffic": recorded_traffic("groupnorm")},
            "gpu_launches": 1}
        rw = ROTATE
        rt = statistics.median(time_rotate(rw, 20, dev, flush)) / 1e3
        rrows = rw["B"] * rw["H"] * rw["N"]
        rbytes = 4 * rw["d"] * rrows  # bf16 row read + bf16 row written
        extra["rotate"] = {
            "rows_per_s": round(rrows / rt, 1), "ms_per_call": round(rt * 1e3, 5),
            "config": {k: rw[k] for k in ("B", "H", "N", "d")} | {"l2": "flushed before each call (512 MiB write, then 512 MiB read)",
                                                                  "timing": "CUDA events per call"},
            "roofline": {"bound": "hbm", "achieved": round(rbytes / rt / 1e9, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(rbytes / rt / 1e9 / hbm, 4), "traffic": recorded_traffic("rotate")},
            "gpu_launches": 1}
        # chunkwise with the GroupNorm fused into its epilogue, on the mid workload
        mid_ms = extra["mid"]["ms_per_call"]
        tf, nf, _ = time_chunkwise(MID, args.steps, 3, dev, flush, norm=True)
        f_s = statistics.median(tf) / 1e3
        extra["mid_groupnorm_fused"] = {
            "tokens_per_s": round(MID["B"] * MID["N"] / f_s, 1), "ms_per_call": round(f_s * 1e3, 5),
            "separate_ms": round(mid_ms + gt * 1e3, 5),
            "config": {"workload": "mid retention chunkwise fwd + GroupNorm over each head (fused epilogue)",
                       "out_layout": "[B, N, H, dv]"},
            "gpu_launches": nf}
        # the chunkwise forward of rotated q and k: rotation fused, against separate passes
        rr = time_rotated(MID, args.steps, dev, flush)
        extra["mid_rotated"] = {
            "tokens_per_s": round(MID["B"] * MID["N"] / (rr["fused"] / 1e3), 1), "ms_per_call": round(rr["fused"], 5),
            "separate_ms": round(rr["separate"], 5),
            "config": {"workload": "mid retention chunkwise fwd of rotated q, k (rotation fused in the kernels)",
                       "separate": "retention_rotate on q and on k, then retention_chunkwise",
                       "timing": "CUDA graph replay, L2 flushed before each call"},
            "gpu_launches": binding.chunkwise_launches(MID["B"], MID["H"], MID["N"], MID["dk"], MID["dv"],
                                                       MID["chunk"])}
        # the parallel form (tensor cores) on the mid and long workloads
        extra["mid_parallel"] = parallel_entry(MID, 10, dev, flush, tflops)
        extra["long_parallel"] = parallel_entry(LONG, 5, dev, flush, tflops)
        # gradients of the mid workload (tensor cores: three chunkwise forwards)
        bt = statistics.median(time_backward(MID, 10, dev, flush)) / 1e3
        bbytes = backward_bytes(MID)
        extra["mid_backward"] = {
            "tokens_per_s": round(MID["B"] * MID["N"] / bt, 1), "ms_per_call": round(bt * 1e3, 5),
            "config": {"workload": "mid retention gradients (dq, dk, dv), no states", "B": MID["B"], "H": MID["H"],
                       "N": MID["N"], "dk": MID["dk"], "dv": MID["dv"], "chunk": backward_chunk(MID),
                       "l2": "flushed before each call (512 MiB write, then 512 MiB read)",
                       "timing": "CUDA graph replay of the call"},
            "roofline": {"bound": "hbm", "achieved": round(bbytes / bt / 1e9, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(bbytes / bt / 1e9 / hbm, 4), "traffic": recorded_traffic("mid_backward"),
                         "algorithmic_bytes_per_call": bbytes,
                         "tensor_flops_frac": round(backward_flops(MID) / bt / 1e12 / tflops, 4)},
            "gpu_launches": binding.backward_launches(MID["B"], MID["H"], MID["N"], MID["dk"], MID["dv"])}
        # gradients of the 7B-shaped workload (512-wide queries in the dq and dk forwards)
        bt7 = statistics.median(time_backward(B7, 5, dev, flush)) / 1e3
        b7bytes = backward_bytes(B7)
        extra["7b_backward"] = {
            "tokens_per_s": round(B7["B"] * B7["N"] / bt7, 1), "ms_per_call": round(bt7 * 1e3, 5),
            "config": {"workload": "7B-shaped retention gradients (dq, dk, dv), no states", "B": B7["B"], "H": B7["H"],
                       "N": B7["N"], "dk": B7["dk"], "dv": B7["dv"], "chunk": backward_chunk(B7),
                       "l2": "flushed before each call (512 MiB write, then 512 MiB read)",
                       "timing": "CUDA graph replay of the call"},
            "roofline": {"bound": "tensor", "achieved": round(backward_flops(B7) / bt7 / 1e12, 1), "peak": tflops,
                         "unit": "TFLOP/s", "frac": round(backward_flops(B7) / bt7 / 1e12 / tflops, 4),
                         "traffic": None, "algorithmic_flops_per_call": backward_flops(B7),
                         "hbm_frac": round(b7bytes / bt7 / 1e9 / hbm, 4)},
            "gpu_launches": binding.backward_launches(B7["B"], B7["H"], B7["N"], B7["dk"], B7["dv"])}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded iid N(0,1) q,k,v)",
        "config": {"workload": "7B-shaped retention chunkwise fwd", **cfg, "global_batch": w["B"] * world,
                   "seq_len": w["N"], "parallelism": f"replicas x{world} (independent batches)",
                   "l2": "flushed between timed steps (512 MiB write, then 512 MiB read); inputs 3.2 GB > L2",
                   "timing": how},
        "roofline": roofline, "e2e": e2e, "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    line.update(extra)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_chunkwise(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the fp64 CPU oracle

def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    w = B7
    B, H, N, dk, dv, C = w["B"], w["H"], w["N"], w["dk"], w["dv"], w["chunk"]
    qd, kd, vd, g = oracle_sample(w)
    orc = oracle.default()
    for _ in range(args.warmup):
        orc.chunkwise(qd, kd, vd, g, C)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.chunkwise(qd, kd, vd, g, C)
    row_s = (time.perf_counter() - t0) / args.steps
    full_s = row_s * B  # the whole batch is B such rows
    value = B * N / full_s
    sample = (f"one batch row of the 7B-shaped workload per step (all {H} heads, N={N}), fp64 chunkwise "
              f"form, chunk {C}; scaled to the B={B} rows of the workload")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(full_s * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded iid N(0,1) q,k,v)",
            "config": {"workload": "7B-shaped retention chunkwise fwd", "B": B, "H": H, "N": N, "dk": dk,
                       "dv": dv, "chunk": C, "global_batch": B, "seq_len": N,
                       "parallelism": "host cores (OpenMP over heads)"},
            "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": orc.threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_only(args):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    if args.only == "decode":
        t = time_decode(DECODE, args.steps, dev)
        print(json.dumps({"only": "decode", "ms_per_step": statistics.median(t)}))
        return
    flush = L2Flush(dev)
    if args.only in ("backward", "backward_long", "backward_7b"):
        wl = dict({"backward": MID, "backward_long": LONG, "backward_7b": B7}[args.only])
        if args.batch:
            wl["B"] = args.batch
        t = time_backward(wl, args.steps, dev, flush)
        print(json.dumps({"only": args.only, "ms_per_call": statistics.median(t), "launches": args.steps,
                          "tokens_per_s": round(wl["B"] * wl["N"] / (statistics.median(t) / 1e3), 1)}))
        return
    if args.only == "e2e":
        for wl in (B7, MID):
            print(json.dumps({"only": "e2e", "w": wl["name"], **e2e_entry(wl, args.steps, args.warmup, dev)}))
        return
    if args.only == "rotated":
        r = time_rotated(MID, args.steps, dev, flush)
        print(json.dumps({"only": "rotated", "fused_ms": r["fused"], "separate_ms": r["separate"]}))
        return
    if args.only in ("parallel", "parallel_long"):
        wl = MID if args.only == "parallel" else LONG
        t = time_parallel(wl, args.steps, dev, flush)
        print(json.dumps({"only": args.only, "ms_per_call": statistics.median(t), "launches": args.steps,
                          "tflops": round(parallel_flops(wl) / (statistics.median(t) / 1e3) / 1e12, 1)}))
        return
    if args.only in ("groupnorm", "rotate"):
        fn, wl = (time_groupnorm, GROUPNORM) if args.only == "groupnorm" else (time_rotate, ROTATE)
        t = fn(wl, args.steps, dev, flush)
        print(json.dumps({"only": args.only, "ms_per_call": statistics.median(t), "launches": args.steps}))
        return
    w = dict({"mid": MID, "long": LONG, "7b": B7}[args.only])
    if args.batch:
        w["B"] = args.batch  # a smaller case of the same shape (e.g. for an ncu capture)
    t, n, how = time_chunkwise(w, args.steps, args.warmup, dev, flush)
    print(json.dumps({"only": args.only, "B": w["B"], "ms_per_call": statistics.median(t), "launches": n,
                      "timing": how}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="with --only: batch rows instead of the workload's")
    ap.add_argument("--only", choices=["mid", "long", "7b", "decode", "groupnorm", "rotate", "backward", "backward_long",
                                       "backward_7b", "parallel", "parallel_long", "rotated", "e2e"], default=None)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.only:
        run_only(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
