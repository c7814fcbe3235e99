"""Benchmark of the tile-pipelined AllGather+GEMM and GEMM+ReduceScatter on one GB300.

One step = one fused AllGather+GEMM call (W=8 logical ranks, shards 1024x8192 bf16, B 8192x3584)
followed by one fused GEMM+ReduceScatter call (W=8, A_r 8192x3584, B_r 3584x8192, bf16 output
shards 1024x8192), i.e. every step of the hot path: chunk producer, flag-gated rank-swizzled
tcgen05 GEMM, and the rank-ordered reduction. Inputs are seeded synthetic data (workloads.py).

Prints ONE JSON line (rank 0). ``value`` is whole-job TFLOP/s with inputs resident in HBM; ``e2e``
repeats the step through the same C-ABI calls with pinned host inputs copied in and outputs copied
back inside the timed region. ``roofline`` is for the dominant kernel (the GEMM+ReduceScatter
launch), timed with CUDA events on its stream inside the timed region. ``cpu_baseline`` times the
CPU oracle on a bounded sample of the same workload (rank 0, N=1 only).

``--impl reference`` times the CPU oracle itself (the reference arm of this repository: the pages
ship no runnable reference code) on a bounded sample of the same workload per step.

Multi-GPU: launched under torchrun, every rank runs an independent replica of the step on its own
GPU (weak scaling; the logical ranks of each replica live in that GPU's memory, so there is no
data-path collective); the timed region is bracketed by a barrier and the maximum over ranks is
reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "AG-GEMM & GEMM-RS TFLOP/s (1 GB300), % tensor peak, overlap efficiency"
WORKLOAD = ("AG-GEMM W=8 bf16 (8 shards 1024x8192, B 8192x3584, C 8192x3584, chunk 128) + "
            "GEMM-RS W=8 bf16 (A_r 8192x3584, B_r 3584x8192, out 8 shards 1024x8192)")
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


# A timed region shorter than this runs at the clocks of a burst (the power cap has not ramped in);
# longer ones are compared with the sustained (seconds-long, power-capped) bf16 peak.
SUSTAINED_AFTER_S = 1.0


def bf16_peak(pk: dict, kind: str, region_s: float):
    """(peak TFLOP/s, description) for a kernel timed inside a region of region_s seconds: the
    burst figure for regions under SUSTAINED_AFTER_S, the sustained one for longer regions."""
    if region_s < SUSTAINED_AFTER_S or "bf16_tflops_sustained" not in pk:
        return float(pk.get("bf16_tflops", FALLBACK["bf16_tflops"])), \
            f"{kind} bf16 dense, burst (timed region {region_s:.3f} s < {SUSTAINED_AFTER_S:.0f} s)"
    return float(pk["bf16_tflops_sustained"]), \
        f"{kind} bf16 dense, sustained (timed region {region_s:.3f} s >= {SUSTAINED_AFTER_S:.0f} s)"


FUSED_KERNEL_SOURCES = ["tdx_api.cu", "tdx_internal.h", "tdx_kernel.cuh", "tdx_kernel_bf16.cu",
                        "tdx_kernel_fp8.cu", "tdx_ptx.cuh"]


def code_tokens(text: str) -> str:
    """C/C++/CUDA source with its comments removed and whitespace runs collapsed to one space
    (string and character literals kept as written), so that editing a comment or the layout does
    not change what identifies the code."""
    out = []
    i, n = 0, len(text)
    while i < n:
        c = text[i]
        if c == "/" and i + 1 < n and text[i + 1] == "/":
            j = text.find("\n", i)
            i = n if j < 0 else j
            out.append(" ")
        elif c == "/" and i + 1 < n and text[i + 1] == "*":
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """sha256 over the code (comments and layout excluded) of the fused GEMM kernel and its host
    launch code: identifies the kernel an ncu capture measured."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "comm_overlapped_gemm_gb300", "csrc")
    for name in FUSED_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + code_tokens(f.read()).encode())
    return h.hexdigest()


def kernel_traffic():
    """DRAM bytes (read + written) per GEMM-RS W=8 launch from the committed ncu summary, or None
    when the kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", "tdx_fused_rs_w8_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_sha256") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


def reduce_max(x: float, world: int, device=None) -> float:
    """Maximum of x over all ranks (the job's time is its slowest rank's); identity at world 1."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_step: float, steps: int, world: int, ms_max: float) -> float:
    """Units all ranks processed (weak scaling: every rank runs the same step) over the slowest
    rank's time."""
    return world * flops_per_step * steps / (ms_max * 1e-3) / 1e12


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


class ClockSampler:
    """nvidia-smi sampled every 100 ms during the timed region."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        import tempfile
        self.path = os.path.join(os.environ.get("TDX_CLOCKS_DIR") or tempfile.gettempdir(),
                                 f"tdx_clocks_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(self.path), exist_ok=True)
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------------- CPU oracle arm
def oracle_sample(ag_inp, rs_inp, frac_rows: int = 8):
    """The oracle on a bounded sample of the step: rows of rank 0's shard of C (1/8 of the AG
    output) and output shard 0 of the GEMM-RS (1/8 of its rows). Returns (flops, seconds)."""
    from oracle import reference as R
    t0 = time.perf_counter()
    wl = ag_inp.wl
    rows = np.arange(wl.W * wl.M // frac_rows)
    R.ag_gemm_rows(ag_inp.a, ag_inp.b[0], rows, "bf16")
    f_ag = 2.0 * len(rows) * wl.K * wl.N
    wr = rs_inp.wl
    rrows = np.arange(wr.M // frac_rows)
    R.gemm_rs_rows(rs_inp.a, rs_inp.b, rrows, "bf16")
    f_rs = 2.0 * wr.W * len(rrows) * wr.K * wr.N
    return f_ag + f_rs, time.perf_counter() - t0


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    import workloads as wls
    ag = wls.make_inputs(wls.WORKLOADS["ag_w8"])
    rs = wls.make_inputs(wls.WORKLOADS["rs_w8"])
    for _ in range(args.warmup):
        oracle_sample(ag, rs, frac_rows=128)
    flops = 0.0
    secs = 0.0
    for _ in range(args.steps):
        f, s = oracle_sample(ag, rs, frac_rows=128)
        flops += f
        secs += s
    v = flops / secs / 1e12
    sample = "per step: rows 0..63 of the AG-GEMM output (1/128) and rows 0..63 of the GEMM-RS sum (1/128), fp64 numpy"
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, workloads.py)",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------------- GPU arm
class Step:
    """Device buffers and the two C-ABI calls of one step."""

    def __init__(self, tdx, torch, ag_inp, rs_inp, dev):
        self.tdx, self.torch = tdx, torch
        t = torch

        def d(a):
            return t.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)

        wa, wr = ag_inp.wl, rs_inp.wl
        self.wa, self.wr = wa, wr
        self.shards = [d(a) for a in ag_inp.a]
        self.B = d(ag_inp.b[0])
        self.C = t.empty((wa.W * wa.M, wa.N), dtype=t.bfloat16, device=dev)
        self.A = [d(a) for a in rs_inp.a]
        self.Bs = [d(b) for b in rs_inp.b]
        self.out = [t.empty((wr.M // wr.W, wr.N), dtype=t.bfloat16, device=dev) for _ in range(wr.W)]
        self.ws_ag = t.empty(1, dtype=t.uint8, device=dev)
        self.ws_rs = t.empty(1, dtype=t.uint8, device=dev)
        self.size_workspaces({})
        self.epoch = 0

    def size_workspaces(self, extra, ops=("ag", "rs")):
        """(Re)allocate the two workspaces, those named in `ops` for the tiling options in `extra`."""
        tdx, t, wa, wr = self.tdx, self.torch, self.wa, self.wr
        dev = self.ws_ag.device
        ea = extra if "ag" in ops else {}
        er = extra if "rs" in ops else {}
        self.ws_ag = t.empty(tdx.tdx_workspace_size(tdx.OP_AG, wa.W, wa.M, wa.K, wa.N, tdx.TDX_BF16,
                                                    tdx.make_opts(chunk_rows=wa.chunk_rows, **ea)),
                             dtype=t.uint8, device=dev)
        self.ws_rs = t.empty(tdx.tdx_workspace_size(tdx.OP_RS, wr.W, wr.M, wr.K, wr.N, tdx.TDX_BF16,
                                                    tdx.make_opts(**er)), dtype=t.uint8, device=dev)
        tdx.check(tdx.tdx_workspace_init(self.ws_ag))
        tdx.check(tdx.tdx_workspace_init(self.ws_rs))

    extra: dict = {}

    def ag(self, mode=0, producer=0, epoch=None):
        self.epoch += 1
        o = self.tdx.make_opts(epoch=self.epoch if epoch is None else epoch, mode=mode, producer=producer,
                               chunk_rows=self.wa.chunk_rows, **self.extra)
        wa = self.wa
        return self.tdx.tdx_ag_gemm(self.shards, self.B, self.C, self.ws_ag, wa.W, wa.M, wa.K, wa.N,
                                    self.tdx.TDX_BF16, o)

    def rs(self, mode=0, epoch=None):
        self.epoch += 1
        o = self.tdx.make_opts(epoch=self.epoch if epoch is None else epoch, mode=mode, **self.extra)
        wr = self.wr
        return self.tdx.tdx_gemm_rs(self.A, self.Bs, self.out, self.ws_rs, wr.W, wr.M, wr.K, wr.N,
                                    self.tdx.TDX_BF16, o)

    def status(self):
        for ws in (self.ws_ag, self.ws_rs):
            st, detail = self.tdx.tdx_read_device_status(ws)
            if st != 0:
                raise RuntimeError(f"device status {self.tdx.tdx_status_string(st)} {detail}")


def time_interleaved(torch, fns: dict, reps: int) -> dict:
    """Median per-call CUDA-event time (ms) of each fn in `fns`, the calls taken in turn (a, b, c,
    a, b, c, ...), so that every variant runs under the same clock and power state; a variant timed
    in a block of its own would see the power cap ramp in differently."""
    s = torch.cuda.current_stream()
    ts = {k: [] for k in fns}
    for _ in range(reps):
        for k, fn in fns.items():
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
            fn()
            e1.record(s)
            e1.synchronize()
            ts[k].append(e0.elapsed_time(e1))
    return {k: statistics.median(v) for k, v in ts.items()}


def time_mode(torch, fn, reps: int):
    """Median of per-call CUDA-event times of fn() on the current stream (ms)."""
    s = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        fn()
        e1.record(s)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def ag_case(tdx, torch, wl, dev, integer=False):
    """Device buffers + a timed call for one AllGather workload (extra configurations)."""
    import workloads as wls
    inp = wls.make_inputs(wl, integer=integer)
    view = np.int16 if wl.dtype == "bf16" else np.uint8
    # the ranks' shards at one stride in one buffer, as a symmetric heap places them
    stacked = torch.from_numpy(np.ascontiguousarray(np.stack(inp.a)).view(view)).to(dev)
    shards = [stacked[r] for r in range(wl.W)]
    B = torch.from_numpy(np.ascontiguousarray(inp.b[0]).view(view)).to(dev)
    C = torch.empty((wl.W * wl.M, wl.N), dtype=torch.bfloat16, device=dev)
    dt = tdx.TDX_BF16 if wl.dtype == "bf16" else tdx.TDX_FP8_E4M3
    kw = dict(chunk_rows=wl.chunk_rows)
    if wl.dtype == "e4m3":
        kw.update(scale_a=inp.scale_a, scale_b=inp.scale_b[0])
    ws = torch.empty(tdx.tdx_workspace_size(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, dt, tdx.make_opts(**kw)),
                     dtype=torch.uint8, device=dev)
    tdx.check(tdx.tdx_workspace_init(ws))
    state = {"epoch": 0}

    def call(mode=0, producer=0, epoch=None):
        state["epoch"] += 1
        o = tdx.make_opts(epoch=state["epoch"] if epoch is None else epoch, mode=mode, producer=producer, **kw)
        tdx.check(tdx.tdx_ag_gemm(shards, B, C, ws, wl.W, wl.M, wl.K, wl.N, dt, o))

    def status():
        st, d = tdx.tdx_read_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {tdx.tdx_status_string(st)} {d}")
    status.reset = lambda: tdx.check(tdx.tdx_workspace_init(ws))
    return call, status


def rs_case(tdx, torch, wl, dev, **kw):
    """Device buffers + a timed call for one bf16 ReduceScatter workload; ``kw`` are extra options."""
    import workloads as wls
    inp = wls.make_inputs(wl)
    A = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev) for a in inp.a]
    Bs = [torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev) for b in inp.b]
    out = [torch.empty((wl.M // wl.W, wl.N), dtype=torch.bfloat16, device=dev) for _ in range(wl.W)]
    ws = torch.empty(tdx.tdx_workspace_size(tdx.OP_RS, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, tdx.make_opts(**kw)),
                     dtype=torch.uint8, device=dev)
    tdx.check(tdx.tdx_workspace_init(ws))
    state = {"epoch": 0}

    def call(mode=0, epoch=None):
        state["epoch"] += 1
        o = tdx.make_opts(epoch=state["epoch"] if epoch is None else epoch, mode=mode, **kw)
        tdx.check(tdx.tdx_gemm_rs(A, Bs, out, ws, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))

    def status():
        st, d = tdx.tdx_read_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {tdx.tdx_status_string(st)} {d}")
    status.reset = lambda: tdx.check(tdx.tdx_workspace_init(ws))
    return call, status


def moe_case(tdx, torch, wl, dev, **extra):
    """Device buffers + a timed call for one MoE dispatch + grouped GEMM workload; ``extra`` are
    tdx_opts fields (tiling)."""
    import workloads as wls
    inp = wls.make_inputs(wl)
    view = np.int16 if wl.dtype == "bf16" else np.uint8
    dt = tdx.TDX_BF16 if wl.dtype == "bf16" else tdx.TDX_FP8_E4M3
    kw = dict(extra) if wl.dtype == "bf16" else dict(extra, scale_a=inp.scale_a, scale_b=inp.scale_b)
    X = [torch.from_numpy(np.ascontiguousarray(a).view(view)).to(dev) for a in inp.a]
    route = [torch.from_numpy(np.ascontiguousarray(r)).to(dev) for r in inp.route]
    B = torch.from_numpy(np.ascontiguousarray(inp.b[0]).view(view)).to(dev)
    Y = torch.empty((wl.M_total, wl.N), dtype=torch.bfloat16, device=dev)
    dest = torch.empty((wl.W, wl.M, wl.topk), dtype=torch.int32, device=dev)
    ws = torch.empty(tdx.tdx_moe_workspace_size(wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk, dt, tdx.make_opts(**kw)),
                     dtype=torch.uint8, device=dev)
    tdx.check(tdx.tdx_workspace_init(ws))
    state = {"epoch": 0}

    def call(mode=0, epoch=None):
        state["epoch"] += 1
        o = tdx.make_opts(epoch=state["epoch"] if epoch is None else epoch, mode=mode, **kw)
        tdx.check(tdx.tdx_moe_dispatch_gemm(X, route, B, Y, dest, None, ws, wl.W, wl.M, wl.K, wl.N, wl.E,
                                            wl.topk, dt, o))

    def status():
        st, d = tdx.tdx_read_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {tdx.tdx_status_string(st)} {d}")
    status.reset = lambda: tdx.check(tdx.tdx_workspace_init(ws))
    return call, status


def combine_case(tdx, torch, wl, dev, **extra):
    """Device buffers + a timed call for one MoE grouped GEMM + combine workload; ``extra`` are
    tdx_opts fields (tiling)."""
    import workloads as wls
    inp = wls.make_inputs(wl)
    Hd = torch.from_numpy(np.ascontiguousarray(inp.a[0]).view(np.int16)).to(dev)
    route = [torch.from_numpy(np.ascontiguousarray(r)).to(dev) for r in inp.route]
    gates = [torch.from_numpy(np.ascontiguousarray(g)).to(dev) for g in inp.gates]
    B = torch.from_numpy(np.ascontiguousarray(inp.b[0]).view(np.int16)).to(dev)
    out = [torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device=dev) for _ in range(wl.W)]
    ws = torch.empty(tdx.tdx_moe_combine_workspace_size(wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk, tdx.TDX_BF16,
                                                        tdx.make_opts(**extra)),
                     dtype=torch.uint8, device=dev)
    tdx.check(tdx.tdx_workspace_init(ws))
    state = {"epoch": 0}

    def call(mode=0, epoch=None):
        state["epoch"] += 1
        o = tdx.make_opts(epoch=state["epoch"] if epoch is None else epoch, mode=mode, **extra)
        tdx.check(tdx.tdx_moe_gemm_combine(Hd, route, B, gates, out, ws, wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk,
                                           tdx.TDX_BF16, o))

    def status():
        st, d = tdx.tdx_read_device_status(ws)
        if st != 0:
            raise RuntimeError(f"device status {tdx.tdx_status_string(st)} {d}")
    status.reset = lambda: tdx.check(tdx.tdx_workspace_init(ws))
    return call, status


def graph_time_us(torch, fn, reps: int = 50, reset=None):
    """GPU time per call (us) of fn captured in a CUDA graph of `reps` back-to-back calls (no host
    submission cost inside the timed region); None if the call cannot be captured. fn makes its
    call with device-kept epochs (nothing cleared between calls); `reset` re-initialises the
    workspace first, since the eager calls before used host epochs."""
    try:
        if reset is not None:
            reset()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(3):
                fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        return 1e3 * e0.elapsed_time(e1) / reps
    except Exception as exc:  # capture not supported for this call
        print(f"graph capture failed: {exc}", file=sys.stderr)
        return None


def extra_configs(tdx, torch, dev, peak_bf16, hbm_gbs, reps=20):
    """The other configurations, timed alone (median of CUDA-event times, warm; the fused / GEMM
    alone / movement alone modes of one configuration interleaved call by call, so that all three
    run under the same clock and power state): e4m3 AllGather and ReduceScatter, GEMM+AllReduce,
    bf16 partials, the MoE dispatch and combine, and the small-M latency cases."""
    import workloads as wls
    W = wls.WORKLOADS
    res = {}
    call, status = ag_case(tdx, torch, W["ag_fp8_w8"], dev)
    for _ in range(3):
        call()
    t = time_interleaved(torch, {"f": call, "g": lambda: call(mode=1), "m": lambda: call(mode=2)}, reps)
    f, g, m = t["f"], t["g"], t["m"]
    status()
    tf = W["ag_fp8_w8"].flops / (f * 1e-3) / 1e12
    res["ag_fp8_w8"] = {"ms_fused": f, "ms_gemm_only": g, "ms_move_only": m, "overlap_efficiency": max(g, m) / f,
                        "tflops": tf, "peak_fp8_tflops": 2 * peak_bf16, "frac_of_peak": tf / (2 * peak_bf16)}
    del call, status
    wl = W["rs_fp8_w8"]
    inp = wls.make_inputs(wl)
    A = [torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in inp.a]
    Bs = [torch.from_numpy(np.ascontiguousarray(x)).to(dev) for x in inp.b]
    out = [torch.empty((wl.M // wl.W, wl.N), dtype=torch.bfloat16, device=dev) for _ in range(wl.W)]
    ws = torch.empty(tdx.tdx_workspace_size(tdx.OP_RS, wl.W, wl.M, wl.K, wl.N, tdx.TDX_FP8_E4M3),
                     dtype=torch.uint8, device=dev)
    tdx.check(tdx.tdx_workspace_init(ws))
    ep = {"e": 0}

    def rs8(mode=0):
        ep["e"] += 1
        o = tdx.make_opts(epoch=ep["e"], mode=mode, scale_a=inp.scale_a, scale_b=inp.scale_b)
        tdx.check(tdx.tdx_gemm_rs(A, Bs, out, ws, wl.W, wl.M, wl.K, wl.N, tdx.TDX_FP8_E4M3, o))
    for _ in range(3):
        rs8()
    f = time_mode(torch, rs8, reps)
    st8, d8 = tdx.tdx_read_device_status(ws)
    if st8 != 0:
        raise RuntimeError(f"device status {tdx.tdx_status_string(st8)} {d8}")
    tf = wl.flops / (f * 1e-3) / 1e12
    res["rs_fp8_w8"] = {"ms_fused": f, "tflops": tf, "peak_fp8_tflops": 2 * peak_bf16, "frac_of_peak": tf / (2 * peak_bf16)}
    del A, Bs, out, ws
    # GEMM+AllReduce: the ReduceScatter's fold writes each reduced tile into all W full outputs
    wl = W["ar_w8"]
    inp = wls.make_inputs(wl)
    A = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev) for a in inp.a]
    Bs = [torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev) for x in inp.b]
    out = [torch.empty((wl.M, wl.N), dtype=torch.bfloat16, device=dev) for _ in range(wl.W)]
    ws = torch.empty(tdx.tdx_workspace_size(tdx.OP_AR, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16),
                     dtype=torch.uint8, device=dev)
    tdx.check(tdx.tdx_workspace_init(ws))

    def ar(mode=0):
        ep["e"] += 1
        o = tdx.make_opts(epoch=ep["e"], mode=mode)
        tdx.check(tdx.tdx_gemm_ar(A, Bs, out, ws, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))
    for _ in range(3):
        ar()
    f = time_mode(torch, ar, reps)
    st, d = tdx.tdx_read_device_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {tdx.tdx_status_string(st)} {d}")
    tf = wl.flops / (f * 1e-3) / 1e12
    res["ar_w8"] = {"ms_fused": f, "tflops": tf, "frac_of_peak": tf / peak_bf16,
                    "output_bytes": wl.W * wl.M * wl.N * 2}
    del A, Bs, out, ws
    # ReduceScatter with bf16 partials (slotted fold of rounded partials: half the slot bytes)
    call, status = rs_case(tdx, torch, W["rs_w8"], dev, bf16_partials=1)
    for _ in range(3):
        call()
    f = time_mode(torch, call, reps)
    status()
    tf = W["rs_w8"].flops / (f * 1e-3) / 1e12
    res["rs_w8_bf16_partials"] = {"ms_fused": f, "tflops": tf, "frac_of_peak": tf / peak_bf16}
    del call, status
    # MoE AllToAll dispatch + grouped GEMM: fused, GEMM alone (receive buffer already filled), dispatch alone
    wl = W["moe_w8"]
    call, status = moe_case(tdx, torch, wl, dev)
    for _ in range(3):
        call()
    t = time_interleaved(torch, {"f": call, "g": lambda: call(mode=1), "m": lambda: call(mode=2)}, reps)
    f, g, m = t["f"], t["g"], t["m"]
    status()
    tf = wl.flops / (f * 1e-3) / 1e12
    moved = 2 * wl.M_total * wl.K * 2                       # dispatched rows read + written
    res["moe_w8"] = {"ms_fused": f, "ms_gemm_only": g, "ms_move_only": m, "overlap_efficiency": max(g, m) / f,
                     "tflops": tf, "frac_of_peak": tf / peak_bf16, "dispatch_bytes": moved,
                     "dispatch_gbs_alone": moved / (m * 1e-3) / 1e9}
    del call, status
    # the same in e4m3 (tokens and expert weights quantised per tensor; dispatch moves half the bytes)
    wl = W["moe_fp8_w8"]
    call, status = moe_case(tdx, torch, wl, dev)
    for _ in range(3):
        call()
    t = time_interleaved(torch, {"f": call, "g": lambda: call(mode=1), "m": lambda: call(mode=2)}, reps)
    f, g, m = t["f"], t["g"], t["m"]
    status()
    tf = wl.flops / (f * 1e-3) / 1e12
    res["moe_fp8_w8"] = {"ms_fused": f, "ms_gemm_only": g, "ms_move_only": m, "overlap_efficiency": max(g, m) / f,
                         "tflops": tf, "peak_fp8_tflops": 2 * peak_bf16, "frac_of_peak": tf / (2 * peak_bf16)}
    del call, status
    wl = W["moe_fp8_w8_decode"]
    call, status = moe_case(tdx, torch, wl, dev)
    for _ in range(5):
        call()
    f = time_mode(torch, call, reps)
    m = time_mode(torch, lambda: call(mode=2), reps)
    gus = graph_time_us(torch, lambda: call(epoch=tdx.TDX_EPOCH_DEVICE), reset=status.reset)
    status()
    byt = wl.E * wl.K * wl.N + 2 * wl.M_total * wl.K + wl.M_total * wl.N * 2   # weights, dispatch r+w, Y
    t_us = gus or 1e3 * f
    res["moe_fp8_w8_decode"] = {"us_call": 1e3 * f, "us_gpu_graph": gus, "us_dispatch_alone": 1e3 * m,
                                "algorithmic_bytes": byt, "hbm_frac": byt / (t_us * 1e-6) / 1e9 / hbm_gbs}
    del call, status
    # MoE grouped GEMM + combine: fused, GEMM alone (expert outputs only), combine alone
    wl = W["moe_combine_w8"]
    call, status = combine_case(tdx, torch, wl, dev)
    for _ in range(3):
        call()
    t = time_interleaved(torch, {"f": call, "g": lambda: call(mode=1), "m": lambda: call(mode=2)}, reps)
    f, g, m = t["f"], t["g"], t["m"]
    status()
    tf = wl.flops / (f * 1e-3) / 1e12
    res["moe_combine_w8"] = {"ms_fused": f, "ms_gemm_only": g, "ms_move_only": m,
                             "overlap_efficiency": max(g, m) / f, "tflops": tf, "frac_of_peak": tf / peak_bf16}
    del call, status
    wl = W["moe_w8_decode"]
    call, status = moe_case(tdx, torch, wl, dev)
    for _ in range(5):
        call()
    f = time_mode(torch, call, reps)
    gus = graph_time_us(torch, lambda: call(epoch=tdx.TDX_EPOCH_DEVICE), reset=status.reset)
    status()
    byt = wl.E * wl.K * wl.N * 2 + 2 * wl.M_total * wl.K * 2 + wl.M_total * wl.N * 2   # weights, dispatch r+w, Y
    t_us = gus or 1e3 * f
    res["moe_w8_decode"] = {"us_call": 1e3 * f, "us_gpu_graph": gus, "algorithmic_bytes": byt,
                            "tflops": wl.flops / (t_us * 1e-6) / 1e12,
                            "hbm_frac": byt / (t_us * 1e-6) / 1e9 / hbm_gbs}
    del call, status
    call, status = ag_case(tdx, torch, W["ag_small"], dev)
    for _ in range(5):
        call()
    f = time_mode(torch, call, reps)
    gus = graph_time_us(torch, lambda: call(epoch=tdx.TDX_EPOCH_DEVICE), reset=status.reset)
    status()
    wl = W["ag_small"]
    byt = wl.W * wl.M * wl.K * 2 * 2 + wl.K * wl.N * 2 + wl.W * wl.M * wl.N * 2   # move r+w, B, C
    res["ag_small"] = {"us_call": 1e3 * f, "us_gpu_graph": gus, "algorithmic_bytes": byt,
                       "tflops": wl.flops / ((gus or 1e3 * f) * 1e-6) / 1e12,
                       "hbm_frac": byt / ((gus or 1e3 * f) * 1e-6) / 1e9 / hbm_gbs}
    del call, status
    call, status = rs_case(tdx, torch, W["rs_small"], dev)
    for _ in range(5):
        call()
    f = time_mode(torch, call, reps)
    gus = graph_time_us(torch, lambda: call(epoch=tdx.TDX_EPOCH_DEVICE), reset=status.reset)
    status()
    wl = W["rs_small"]
    byt = wl.W * (wl.M * wl.K + wl.K * wl.N) * 2 + wl.M * wl.N * 2
    res["rs_small"] = {"us_call": 1e3 * f, "us_gpu_graph": gus, "algorithmic_bytes": byt,
                       "tflops": wl.flops / ((gus or 1e3 * f) * 1e-6) / 1e12,
                       "hbm_frac": byt / ((gus or 1e3 * f) * 1e-6) / 1e9 / hbm_gbs}
    return res


def run_gpu(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import comm_overlapped_gemm_gb300 as tdx
    import workloads as wls

    ag_inp = wls.make_inputs(wls.WORKLOADS["ag_w8"])
    rs_inp = wls.make_inputs(wls.WORKLOADS["rs_w8"])
    st = Step(tdx, torch, ag_inp, rs_inp, dev)
    fl_ag = wls.WORKLOADS["ag_w8"].flops
    fl_rs = wls.WORKLOADS["rs_w8"].flops
    fl_step = fl_ag + fl_rs
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warm-up
    for _ in range(args.warmup):
        tdx.check(st.ag())
        tdx.check(st.rs())
    torch.cuda.synchronize()
    st.status()

    # timed region: K steps, per-launch events for the dominant kernel (GEMM-RS) on its stream
    ev_rs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ev_ag = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    launches = 0
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_begin.record(stream)
        for i in range(args.steps):
            ev_ag[i][0].record(stream)
            tdx.check(st.ag())
            ev_ag[i][1].record(stream)
            ev_rs[i][0].record(stream)
            tdx.check(st.rs())
            ev_rs[i][1].record(stream)
            launches += 2
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = reduce_max(t_begin.elapsed_time(t_end), world, dev)
    st.status()
    ms_rs = statistics.mean(a.elapsed_time(b) for a, b in ev_rs)
    ms_ag = statistics.mean(a.elapsed_time(b) for a, b in ev_ag)
    value = whole_job_tflops(fl_step, args.steps, world, ms_total)

    # overlap efficiency: fused vs GEMM-alone and movement-alone of the same kernel
    reps = max(5, min(20, args.steps))
    with ClockSampler(local) as clk_modes:
        t = time_interleaved(torch, {"f": lambda: tdx.check(st.ag(tdx.TDX_FUSED)),
                                     "g": lambda: tdx.check(st.ag(tdx.TDX_GEMM_ONLY)),
                                     "m": lambda: tdx.check(st.ag(tdx.TDX_MOVE_ONLY))}, 2 * reps)
        t_ag_f, t_ag_g, t_ag_m = t["f"], t["g"], t["m"]
        t = time_interleaved(torch, {"f": lambda: tdx.check(st.rs(tdx.TDX_FUSED)),
                                     "g": lambda: tdx.check(st.rs(tdx.TDX_GEMM_ONLY)),
                                     "m": lambda: tdx.check(st.rs(tdx.TDX_MOVE_ONLY))}, reps)
        t_rs_f, t_rs_g, t_rs_m = t["f"], t["g"], t["m"]
    st.status()

    # stall-on-flag: one traced fused AllGather call; the kernel's trace holds, per CTA, the TMA
    # issuer's total time spent waiting for chunk flags and the number of tiles that waited
    wa = st.wa
    plan_ag = tdx.tdx_plan_info(tdx.OP_AG, wa.W, wa.M, wa.K, wa.N, tdx.TDX_BF16, tdx.make_opts(chunk_rows=wa.chunk_rows))
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    items_ag = plan_ag["L"] * plan_ag["T"]
    # the layout depends on the grid actually launched (at most one CTA per SM): size for any of them
    chunks_ag = wa.W * plan_ag["n_chunks"]
    trace = torch.zeros(max(tdx.tdx_trace_size(g, items_ag, chunks_ag) // 4 for g in range(2, n_sm + 1)),
                        dtype=torch.int32,
                        device=dev)
    saved = st.extra
    st.extra = dict(saved, trace=trace)
    tdx.check(st.ag())
    st.extra = saved
    torch.cuda.synchronize()
    st.status()
    tr = trace.cpu().numpy().view(np.uint32)
    g_ag = int(tr[0])
    per_cta = tr[4:4 + 12 * g_ag].reshape(g_ag, 12).astype(np.float64)
    flag_wait = {"mean_us": float(per_cta[:, 0].mean() / 1e3), "max_us": float(per_cta[:, 0].max() / 1e3),
                 "tiles_that_waited_per_cta": float(per_cta[:, 1].mean())}

    # end to end through the same C-ABI calls with pinned host buffers, double-buffered: step i+1's
    # inputs go host -> device on four copy streams (several copy engines) while step i computes on
    # the other device buffer set; every step's results come back to pinned host memory
    h_shards = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory() for a in ag_inp.a]
    h_B = torch.from_numpy(np.ascontiguousarray(ag_inp.b[0]).view(np.int16)).pin_memory()
    h_A = [torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory() for a in rs_inp.a]
    h_Bs = [torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).pin_memory() for b in rs_inp.b]
    h_C = torch.empty(st.C.shape, dtype=torch.bfloat16).pin_memory()
    h_out = [torch.empty(o.shape, dtype=torch.bfloat16).pin_memory() for o in st.out]
    h2d = sum(t.numel() * 2 for t in h_shards + [h_B] + h_A + h_Bs)
    d2h = h_C.numel() * 2 + sum(o.numel() * 2 for o in h_out)

    sets = [st, Step(tdx, torch, ag_inp, rs_inp, dev)]
    n_copy = 4
    copy_streams = [torch.cuda.Stream(device=dev) for _ in range(n_copy)]
    d2h_stream = torch.cuda.Stream(device=dev)
    plans = []
    for sd in sets:
        # the step's uploads, spread over the copy streams by bytes (largest first)
        pairs = list(zip(sd.shards, h_shards)) + [(sd.B, h_B)] + list(zip(sd.A, h_A)) + list(zip(sd.Bs, h_Bs))
        pairs.sort(key=lambda dh: -dh[1].numel())
        lanes, load = [[] for _ in range(n_copy)], [0] * n_copy
        for dst, src in pairs:
            k = load.index(min(load))
            lanes[k].append((dst, src))
            load[k] += src.numel()
        plans.append(lanes)
    in_free = [stream.record_event(), stream.record_event()]    # set's inputs no longer read
    out_free = [stream.record_event(), stream.record_event()]   # set's outputs read back

    def e2e_step(i):
        b = i % 2
        sd = sets[b]
        ups = []
        for cs, lane in zip(copy_streams, plans[b]):
            cs.wait_event(in_free[b])
            with torch.cuda.stream(cs):
                for dst, src in lane:
                    dst.copy_(src, non_blocking=True)
            ups.append(cs.record_event())
        for e in ups:
            stream.wait_event(e)
        stream.wait_event(out_free[b])
        tdx.check(sd.ag())
        tdx.check(sd.rs())
        in_free[b] = stream.record_event()
        d2h_stream.wait_event(in_free[b])
        with torch.cuda.stream(d2h_stream):
            h_C.copy_(sd.C, non_blocking=True)
            for h, d in zip(h_out, sd.out):
                h.copy_(d, non_blocking=True)
        out_free[b] = d2h_stream.record_event()

    e2e_steps = max(3, min(args.steps, 20))
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    for cs in copy_streams + [d2h_stream]:
        cs.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_stream(d2h_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = reduce_max(e0.elapsed_time(e1) / e2e_steps, world, dev)
    for sd in sets:
        sd.status()
    # the e2e outputs are the step's results: every element read back equals the resident run's
    if not torch.equal(h_C, st.C.cpu()) or not all(torch.equal(h, d.cpu()) for h, d in zip(h_out, st.out)):
        raise RuntimeError("end-to-end outputs differ from the resident run")
    del sets

    pk, pk_kind = peaks()
    peak_tf, peak_src = bf16_peak(pk, pk_kind, ms_total * 1e-3)
    achieved = fl_rs / (ms_rs * 1e-3) / 1e12
    traffic = kernel_traffic()

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded numpy PCG64, workloads.py)",
        "config": {"workload": WORKLOAD, "logical_ranks": 8,
                   "l2": "no flush; every step reads inputs larger than L2 (184 MiB AG + 896 MiB RS)",
                   "parallelism": f"replicas x{world} (each GPU runs W=8 logical ranks)"},
        "roofline": {"kernel": "tdx_fused_kernel<256,bf16> (GEMM+ReduceScatter W=8)", "bound": "tensor",
                     "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s", "frac": achieved / peak_tf,
                     "peak_source": peak_src, "traffic": traffic,
                     "algorithmic_flops_per_launch": fl_rs},
        "e2e": {"value": world * fl_step / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "device": {"name": torch.cuda.get_device_name(dev),
                   "sms": torch.cuda.get_device_properties(dev).multi_processor_count},
    }
    if not args.no_extra:
        line["configs"] = extra_configs(tdx, torch, dev, float(pk.get("bf16_tflops", FALLBACK["bf16_tflops"])),
                                        float(pk.get("hbm_gbs", FALLBACK["hbm_gbs"])))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        f, s = oracle_sample(ag_inp, rs_inp, frac_rows=8)
        line["cpu_baseline"] = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": "rows 0..1023 of the AG-GEMM output and rows 0..1023 of the GEMM-RS "
                                          "sum (1/8 of each), fp64 numpy", "seconds": s}
    # the headline per-kernel numbers go last, so that the end of the line carries them
    line["ag_gemm"] = {"tflops": fl_ag / (ms_ag * 1e-3) / 1e12, "ms": ms_ag, "frac_of_peak": fl_ag / (ms_ag * 1e-3) / 1e12 / peak_tf,
                       "ms_fused": t_ag_f, "ms_gemm_only": t_ag_g, "ms_move_only": t_ag_m,
                       "overlap_efficiency": max(t_ag_g, t_ag_m) / t_ag_f,
                       "stall_on_flag_us_per_cta": {"mean": flag_wait["mean_us"], "max": flag_wait["max_us"]}}
    line["gemm_rs"] = {"tflops": achieved, "ms": ms_rs, "frac_of_peak": achieved / peak_tf,
                       "ms_fused": t_rs_f, "ms_gemm_only": t_rs_g, "ms_move_only": t_rs_m,
                       "overlap_efficiency": max(t_rs_g, t_rs_m) / t_rs_f,
                       "modes_timed": "interleaved fused / GEMM alone / movement alone, median",
                       "modes_clocks": clk_modes.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


PHASES = ["entry", "setup", "first_item_loaded", "first_item_mma", "mma_done", "items_done", "epilogue_done"]


def trace_phase_summary(tr: np.ndarray) -> dict:
    """Median and maximum over CTAs (us from the earliest kernel entry) of each phase stamp of a
    traced call (12 statistics words per CTA; stamps a CTA did not record are left out)."""
    g = int(tr[0])
    stv = tr[4:4 + 12 * g].reshape(g, 12).astype(np.int64)
    t0 = stv[:, 4].min()
    out = {}
    for k, name in enumerate(PHASES):
        col = stv[:, 4 + k]
        v = ((col[col != 0] - t0) % (1 << 32)) / 1e3
        out[name] = [round(float(np.median(v)), 2), round(float(np.max(v)), 2)] if len(v) else None
    return out


def run_case(args):
    """One op on a given shape (profiling helper): --case ag|rs --shape W,M,K,N."""
    import torch
    import comm_overlapped_gemm_gb300 as tdx
    import workloads as wls
    W, M, K, N = (int(x) for x in args.shape.split(","))
    dev = torch.device("cuda", 0)
    name = "ag_w8" if args.case == "ag" else "rs_w8"
    inp = wls.make_inputs(wls.with_shape(wls.WORKLOADS[name], W=W, M=M, K=K, N=N, chunk_rows=min(128, M)))
    ai = inp if args.case == "ag" else wls.make_inputs(wls.with_shape(wls.WORKLOADS["ag_w8"], W=1, M=128, K=64, N=64))
    ri = inp if args.case == "rs" else wls.make_inputs(wls.with_shape(wls.WORKLOADS["rs_w8"], W=1, M=128, K=64, N=64))
    st = Step(tdx, torch, ai, ri, dev)
    extra = {}
    for kv in filter(None, args.opts.split(",")):
        k, v = kv.split("=")
        extra[k] = int(v)
    st.extra = extra
    st.size_workspaces(extra, ops=(args.case,))
    mode = {"fused": tdx.TDX_FUSED, "gemm": tdx.TDX_GEMM_ONLY, "move": tdx.TDX_MOVE_ONLY}[args.mode]
    base = st.ag if args.case == "ag" else st.rs
    fn = lambda epoch=None: base(mode=mode, epoch=epoch)
    for _ in range(args.warmup + args.steps):
        tdx.check(fn())
    torch.cuda.synchronize()
    st.status()
    ms = time_mode(torch, lambda: tdx.check(fn()), 5)
    fl = inp.wl.flops
    gus_clear = graph_time_us(torch, lambda: fn(epoch=0))
    ws = st.ws_ag if args.case == "ag" else st.ws_rs
    gus = graph_time_us(torch, lambda: fn(epoch=tdx.TDX_EPOCH_DEVICE),
                        reset=lambda: tdx.check(tdx.tdx_workspace_init(ws)))
    plan = tdx.tdx_plan_info(tdx.OP_AG if args.case == "ag" else tdx.OP_RS, W, M, K, N, tdx.TDX_BF16,
                             tdx.make_opts(chunk_rows=min(128, M), **extra) if args.case == "ag" else tdx.make_opts(**extra))
    # one traced call: per-CTA phase stamps (median / max over CTAs, us from the first CTA's entry)
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    items = plan["L"] * plan["T"]
    chunks = W * plan["n_chunks"] if args.case == "ag" else 0
    trace = torch.zeros(max(tdx.tdx_trace_size(g, items, chunks) // 4 for g in range(1, n_sm + 1)),
                        dtype=torch.int32, device=dev)
    tdx.check(tdx.tdx_workspace_init(ws))
    saved = st.extra
    st.extra = dict(saved, trace=trace)
    tdx.check(fn(epoch=0))
    st.extra = saved
    torch.cuda.synchronize()
    st.status()
    tr = trace.cpu().numpy().view(np.uint32)
    g = int(tr[0])
    phases = trace_phase_summary(tr)
    print(json.dumps({"case": args.case, "shape": [W, M, K, N], "mode": args.mode, "opts": extra, "ms": ms,
                      "us_gpu_graph": gus,
                      "us_gpu_graph_clearing": gus_clear, "tflops": fl / (ms * 1e-3) / 1e12,
                      "phases_us_median_max": phases,
                      "plan": {k: plan[k] for k in ("BN", "L", "T", "reduce_mode", "cluster", "coop_fold")}}))
    return 0


def run_moe_case(args):
    """One MoE op on a given shape (profiling helper): --case moe|moe_combine --shape W,T,K,N,E,topk
    (moe: K = hidden, N = expert width; moe_combine: K = expert width, N = hidden) --mode."""
    import torch
    import comm_overlapped_gemm_gb300 as tdx
    import workloads as wls
    W, T, K, N, E, k = (int(x) for x in args.shape.split(","))
    name = "moe_w8" if args.case == "moe" else "moe_combine_w8"
    if args.case == "moe" and args.dtype == "e4m3":
        name = "moe_fp8_w8"
    wl = wls.with_shape(wls.WORKLOADS[name], W=W, M=T, K=K, N=N, E=E, topk=k)
    dev = torch.device("cuda", 0)
    extra = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in filter(None, args.opts.split(","))}
    if args.case == "moe":
        call, status = moe_case(tdx, torch, wl, dev, **extra)
    else:
        call, status = combine_case(tdx, torch, wl, dev, **extra)
    mode = {"fused": 0, "gemm": 1, "move": 2}[args.mode]
    for _ in range(args.warmup + args.steps):
        call(mode=mode)
    torch.cuda.synchronize()
    status()
    ms = time_mode(torch, lambda: call(mode=mode), 5)
    print(json.dumps({"case": args.case, "shape": [W, T, K, N, E, k], "dtype": args.dtype, "opts": extra,
                      "mode": args.mode, "ms": ms,
                      "tflops": wl.flops / (ms * 1e-3) / 1e12}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="tdx", choices=["tdx", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the extra configurations")
    ap.add_argument("--case", choices=["ag", "rs", "moe", "moe_combine"], default=None)
    ap.add_argument("--mode", choices=["fused", "gemm", "move"], default="fused", help="--case only: which part runs")
    ap.add_argument("--shape", default="8,1024,8192,3584")
    ap.add_argument("--dtype", choices=["bf16", "e4m3"], default="bf16", help="--case moe only")
    ap.add_argument("--opts", default="", help="--case only: tdx_opts fields, e.g. block_n=256,split_k=4")
    ap.add_argument("--source-hash", action="store_true", help="print the kernel source hash and exit")
    args = ap.parse_args()
    if args.warmup < 3 and args.case is None:
        ap.error("--warmup must be >= 3")
    if args.source_hash:
        print(kernel_source_hash())
        return 0
    if args.impl == "reference":
        return run_reference(args)
    if args.case in ("moe", "moe_combine"):
        return run_moe_case(args)
    if args.case is not None:
        return run_case(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
