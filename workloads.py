"""Seeded synthetic workloads for tile-pipelined AllGather+GEMM and GEMM+ReduceScatter.

This module only *draws* inputs: shapes, seeds, value distributions and the casts that turn
the draws into the bytes a kernel consumes (bf16 by round-to-nearest-even, e4m3 by per-tensor
scaling and round-to-nearest-even with saturation). It holds none of the arithmetic of the
method itself (no gathering, no GEMM, no reduction, no output rounding), so both the CUDA path
(tests, bench) and the CPU oracle can take their inputs from here without sharing any code.

The pages describe the overlapped AllGather-plus-GEMM and GEMM-plus-ReduceScatter kernels only
qualitatively ("The first move was to expose the overlap", cronfeed.work article on
Triton-distributed/DITRON); they print no shapes. The shapes below are the workloads this
library is measured on: logical ranks W, per-rank shard sizes and value distributions.

Seeds: numpy PCG64 with ``seed = 20260 + 100 * config_index + r`` for the rank-r tensor and
``+ 50`` on top of that for the rank-r B tensor (B of an AllGather config uses ``r = 0``).
Values are drawn in fp32 and cast with torch on the CPU.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One synthetic configuration.

    ``op`` is ``"ag"`` (AllGather+GEMM: W shards of M_local x K, B is K x N, C is (W*M_local) x N),
    ``"rs"`` (GEMM+ReduceScatter: W pairs A_r (M x K), B_r (K x N); the output is split into
    W row shards of (M/W) x N), ``"ar"`` (GEMM+AllReduce: inputs as ``"rs"``, every rank
    receives the full M x N sum), ``"moe"`` (AllToAll dispatch + grouped GEMM: rank s holds M
    tokens X_s (M x K) routed to ``topk`` of E experts, expert weights E x K x N) or
    ``"moe_combine"`` (grouped GEMM + AllToAll combine: the dispatched rows (W*M*topk x K) times
    expert weights E x K x N, summed back per token with the gates).
    """

    name: str
    index: int
    op: str
    W: int
    M: int            # ag: M_local (rows per shard); rs, ar: M (rows of every A_r)
    K: int
    N: int
    dtype: str        # "bf16" or "e4m3"
    out_dtype: str    # "bf16" or "fp32"
    chunk_rows: int   # AllGather chunk (rows); ignored for rs
    a_dist: tuple = ("normal", 1.0)
    b_dist: tuple = ("normal", 0.02)
    note: str = ""
    E: int = 0        # moe: experts (a multiple of W)
    topk: int = 0     # moe: experts per token

    @property
    def M_total(self) -> int:
        if self.op in ("moe", "moe_combine"):
            return self.W * self.M * self.topk
        return self.W * self.M if self.op == "ag" else self.M

    @property
    def flops(self) -> float:
        """Algorithmic FLOP of one call: 2*M*N*K summed over the GEMMs the op defines (moe: one
        GEMM row per routed token-expert pair)."""
        if self.op in ("moe", "moe_combine"):
            return 2.0 * self.M_total * self.N * self.K
        return 2.0 * self.W * self.M * self.N * self.K


WORKLOADS = {
    "ag_tiny": Workload("ag_tiny", 0, "ag", W=2, M=64, K=128, N=256, dtype="bf16", out_dtype="fp32",
                        chunk_rows=32, a_dist=("uniform", 1.0), b_dist=("uniform", 1.0),
                        note="W=2, shard 64x128, B 128x256, C fp32, chunk 32 rows"),
    "ag_w8": Workload("ag_w8", 1, "ag", W=8, M=1024, K=8192, N=3584, dtype="bf16", out_dtype="bf16",
                      chunk_rows=128, note="W=8, shard 1024x8192 N(0,1), B 8192x3584 N(0,0.02)"),
    "rs_w8": Workload("rs_w8", 2, "rs", W=8, M=8192, K=3584, N=8192, dtype="bf16", out_dtype="bf16",
                      chunk_rows=0, note="W=8, A_r 8192x3584 N(0,1), B_r 3584x8192 N(0,0.02)"),
    "ag_fp8_w8": Workload("ag_fp8_w8", 3, "ag", W=8, M=2048, K=8192, N=8192, dtype="e4m3",
                          out_dtype="bf16", chunk_rows=128, b_dist=("normal", 1.0),
                          note="W=8, shard 2048x8192 e4m3, B 8192x8192 e4m3, per-tensor scales"),
    "rs_fp8_w8": Workload("rs_fp8_w8", 6, "rs", W=8, M=8192, K=3584, N=8192, dtype="e4m3", out_dtype="bf16",
                          chunk_rows=0, b_dist=("normal", 1.0),
                          note="W=8, A_r 8192x3584 e4m3, B_r 3584x8192 e4m3, per-tensor scales, bf16 shards"),
    "ar_w8": Workload("ar_w8", 7, "ar", W=8, M=8192, K=3584, N=8192, dtype="bf16", out_dtype="bf16",
                      chunk_rows=0, note="W=8, A_r 8192x3584 N(0,1), B_r 3584x8192 N(0,0.02), full sum on every rank"),
    "moe_w8": Workload("moe_w8", 8, "moe", W=8, M=4096, K=7168, N=2048, dtype="bf16", out_dtype="bf16",
                       chunk_rows=128, E=64, topk=8,
                       note="W=8, 4096 tokens/rank of 7168, top-8 of 64 experts (8 per rank), expert weights "
                            "7168x2048 N(0,0.02); 262144 dispatched rows"),
    "moe_w8_decode": Workload("moe_w8_decode", 9, "moe", W=8, M=128, K=7168, N=2048, dtype="bf16",
                              out_dtype="bf16", chunk_rows=128, E=64, topk=8,
                              note="W=8, 128 tokens/rank, top-8 of 64 experts; 8192 dispatched rows"),
    "moe_combine_w8": Workload("moe_combine_w8", 10, "moe_combine", W=8, M=4096, K=2048, N=7168, dtype="bf16",
                               out_dtype="bf16", chunk_rows=128, E=64, topk=8,
                               note="W=8, 262144 dispatched rows of 2048, expert weights 2048x7168, combined "
                                    "back to 4096x7168 per rank with top-8 gates"),
    "moe_fp8_w8": Workload("moe_fp8_w8", 11, "moe", W=8, M=4096, K=7168, N=2048, dtype="e4m3", out_dtype="bf16",
                           chunk_rows=128, E=64, topk=8, b_dist=("normal", 1.0),
                           note="moe_w8 in e4m3: tokens and expert weights quantised per tensor (per rank, per expert)"),
    "moe_fp8_w8_decode": Workload("moe_fp8_w8_decode", 12, "moe", W=8, M=128, K=7168, N=2048, dtype="e4m3",
                                  out_dtype="bf16", chunk_rows=128, E=64, topk=8, b_dist=("normal", 1.0),
                                  note="128 e4m3 tokens per rank (the AllToAll size the pages quote), top-8 of 64"),
    "ag_small": Workload("ag_small", 4, "ag", W=8, M=16, K=8192, N=1024, dtype="bf16",
                         out_dtype="bf16", chunk_rows=16,
                         note="small-M latency: shard 16x8192, B 8192x1024, chunk 16"),
    "rs_small": Workload("rs_small", 5, "rs", W=8, M=128, K=1024, N=8192, dtype="bf16",
                         out_dtype="bf16", chunk_rows=0,
                         note="small-M latency: A_r 128x1024, B_r 1024x8192, shards 16x8192"),
}


def seed_for(wl: Workload, rank: int, is_b: bool) -> int:
    return 20260 + 100 * wl.index + rank + (50 if is_b else 0)


def route_seed_for(wl: Workload, rank: int) -> int:
    """Seed of rank ``rank``'s routing scores (moe). Expert e's weights use
    ``20260 + 100*index + 50 + 1000*(e + 1)``."""
    return 20260 + 100 * wl.index + 25 + rank


def _draw(rng: np.random.Generator, shape, dist, integer: bool) -> np.ndarray:
    if integer:
        return rng.integers(-4, 5, size=shape).astype(np.float32)
    kind, scale = dist
    if kind == "normal":
        return rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)
    if kind == "uniform":
        return rng.uniform(-scale, scale, size=shape).astype(np.float32)
    raise ValueError(kind)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round to nearest even, torch's CPU cast); returns uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def quantize_e4m3(x: np.ndarray):
    """Per-tensor e4m3 quantisation of an fp32 draw: scale = amax/448 (1 if amax is 0),
    code = e4m3(x/scale) by torch's round-to-nearest-even cast (|x/scale| <= 448 by
    construction, so nothing saturates beyond the largest finite code). Returns (uint8 codes,
    fp32 scale)."""
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    scale = np.float32(amax / 448.0) if amax > 0 else np.float32(1.0)
    y = torch.from_numpy(np.ascontiguousarray(x / scale, dtype=np.float32))
    y = torch.clamp(y, -448.0, 448.0).to(torch.float8_e4m3fn)
    return y.view(torch.uint8).numpy(), float(scale)


@dataclass
class Inputs:
    """Host-side inputs of one workload as the bytes the kernels take.

    ag: ``a[r]`` is shard r (M_local x K), ``b[0]`` is B (K x N).
    rs: ``a[r]`` is A_r (M x K), ``b[r]`` is B_r (K x N).
    bf16 tensors are uint16 bit patterns, e4m3 tensors uint8 codes; ``scale_a[r]``/``scale_b[r]``
    are the per-tensor dequantisation scales (1.0 for bf16 or integer mode).
    moe: ``a[s]`` X_s (M x K) for "moe" / the dispatched rows (W*M*topk x K, one array) for
    "moe_combine"; ``b[0]`` the E x K x N expert weights; ``route[s]`` int32 (M x topk) expert ids
    and ``gates[s]`` fp32 (M x topk) gate weights of rank s's tokens.
    """

    wl: Workload
    integer: bool
    a: list = field(default_factory=list)
    b: list = field(default_factory=list)
    scale_a: list = field(default_factory=list)
    scale_b: list = field(default_factory=list)
    route: list = field(default_factory=list)
    gates: list = field(default_factory=list)


def make_inputs(wl: Workload, integer: bool = False, shape_override: dict | None = None) -> Inputs:
    """Draw the seeded inputs of ``wl``.

    ``integer=True`` draws uniform integers in [-4, 4] (exact in bf16 and e4m3, scales 1) for the
    bit-exact check. ``shape_override`` replaces W/M/K/N (a smaller case with the same recipe).
    """
    if shape_override:
        wl = Workload(**{**wl.__dict__, **shape_override})
    if wl.op in ("moe", "moe_combine"):
        return _make_moe_inputs(wl, integer)
    out = Inputs(wl=wl, integer=integer)
    nb = 1 if wl.op == "ag" else wl.W
    for r in range(wl.W):
        rng = np.random.Generator(np.random.PCG64(seed_for(wl, r, False)))
        x = _draw(rng, (wl.M, wl.K), wl.a_dist, integer)
        if wl.dtype == "bf16":
            out.a.append(to_bf16_bits(x)); out.scale_a.append(1.0)
        elif integer:
            y = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            out.a.append(y); out.scale_a.append(1.0)
        else:
            q, s = quantize_e4m3(x); out.a.append(q); out.scale_a.append(s)
    for r in range(nb):
        rng = np.random.Generator(np.random.PCG64(seed_for(wl, r, True)))
        x = _draw(rng, (wl.K, wl.N), wl.b_dist, integer)
        if wl.dtype == "bf16":
            out.b.append(to_bf16_bits(x)); out.scale_b.append(1.0)
        elif integer:
            y = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            out.b.append(y); out.scale_b.append(1.0)
        else:
            q, s = quantize_e4m3(x); out.b.append(q); out.scale_b.append(s)
    return out


def with_shape(wl: Workload, **kw) -> Workload:
    """A copy of ``wl`` with some of W/M/K/N/chunk_rows replaced (same seeds and recipe)."""
    return Workload(**{**wl.__dict__, **kw})


def make_routing(wl: Workload, integer: bool = False):
    """Seeded top-k routing of every rank's tokens: each token draws E standard-normal scores (a
    stand-in for router logits) and picks the ``topk`` largest (descending score; ties cannot occur
    with continuous draws). Gates are the softmax of the chosen scores (fp32), or in integer mode
    powers of two drawn from {1/4, 1/2, 1, 2} (exact products). Returns (route, gates): lists of W
    arrays (M x topk), int32 and fp32."""
    route, gates = [], []
    for s in range(wl.W):
        rng = np.random.Generator(np.random.PCG64(route_seed_for(wl, s)))
        scores = rng.standard_normal(size=(wl.M, wl.E), dtype=np.float32)
        idx = np.argsort(-scores, axis=1, kind="stable")[:, :wl.topk].astype(np.int32)
        top = np.take_along_axis(scores, idx, axis=1).astype(np.float64)
        if integer:
            g = (2.0 ** rng.integers(-2, 2, size=idx.shape)).astype(np.float32)
        else:
            ex = np.exp(top - top.max(axis=1, keepdims=True))
            g = (ex / ex.sum(axis=1, keepdims=True)).astype(np.float32)
        route.append(np.ascontiguousarray(idx))
        gates.append(np.ascontiguousarray(g))
    return route, gates


def _cast(x: np.ndarray, dtype: str, integer: bool):
    if dtype == "bf16":
        return to_bf16_bits(x), 1.0
    if integer:
        return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy(), 1.0
    return quantize_e4m3(x)


def _make_moe_inputs(wl: Workload, integer: bool) -> Inputs:
    out = Inputs(wl=wl, integer=integer)
    out.route, out.gates = make_routing(wl, integer)
    if wl.op == "moe":
        for s in range(wl.W):
            rng = np.random.Generator(np.random.PCG64(seed_for(wl, s, False)))
            q, sc = _cast(_draw(rng, (wl.M, wl.K), wl.a_dist, integer), wl.dtype, integer)
            out.a.append(q); out.scale_a.append(sc)
    else:
        rng = np.random.Generator(np.random.PCG64(seed_for(wl, 0, False)))
        q, sc = _cast(_draw(rng, (wl.M_total, wl.K), wl.a_dist, integer), wl.dtype, integer)
        out.a.append(q); out.scale_a.append(sc)
    dt = np.uint16 if wl.dtype == "bf16" else np.uint8
    b = np.empty((wl.E, wl.K, wl.N), dtype=dt)
    for e in range(wl.E):
        rng = np.random.Generator(np.random.PCG64(20260 + 100 * wl.index + 50 + 1000 * (e + 1)))
        q, sc = _cast(_draw(rng, (wl.K, wl.N), wl.b_dist, integer), wl.dtype, integer)
        b[e] = q
        out.scale_b.append(sc)
    out.b.append(b)
    return out
