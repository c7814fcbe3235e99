"""Helpers for the GPU tests: move workloads.py inputs to the device, call the C ABI through the
Python binding, bring outputs back as numpy, and compare them with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import reference as R

TOL = {"bf16": 1e-2, "e4m3": 4e-2}


def dev_bits(a: np.ndarray) -> torch.Tensor:
    """uint16 (bf16 bits) or uint8 (e4m3 codes) host array -> device tensor with the same bytes."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def workspace(op, W, Mx, K, N, dtype, opts=None) -> torch.Tensor:
    n = tdx.tdx_workspace_size(op, W, Mx, K, N, dtype, opts)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    tdx.check(tdx.tdx_workspace_init(ws), "init")
    return ws


def shard_layout(shards, layout: str):
    """Place the shards in device memory: "separate" (one allocation each), "stacked" (one buffer,
    rank r at r times the shard size: one stride), "scattered" (one buffer, uneven gaps between
    shards) or "reversed" (one buffer, rank r at (W-1-r) times the shard size)."""
    if layout == "separate" or not shards:
        return shards
    W = len(shards)
    nb = shards[0].numel() * shards[0].element_size()
    if layout == "stacked":
        offs = [r * nb for r in range(W)]
    elif layout == "reversed":
        offs = [(W - 1 - r) * nb for r in range(W)]
    elif layout == "scattered":
        offs, o = [], 0
        for r in range(W):
            offs.append(o)
            o += nb + 256 * (1 + r % 3)
    else:
        raise ValueError(layout)
    buf = torch.zeros(max(offs) + nb, dtype=torch.uint8, device="cuda")
    out = []
    for r, t in enumerate(shards):
        v = buf[offs[r]:offs[r] + nb].view(t.dtype).view(t.shape)
        v.copy_(t)
        out.append(v)
    return out


def dtype_code(name: str) -> int:
    return tdx.TDX_BF16 if name == "bf16" else tdx.TDX_FP8_E4M3


class AGCase:
    """Device buffers of one AllGather+GEMM problem."""

    def __init__(self, inp, out_dtype="bf16", opts=None, layout="separate"):
        wl = inp.wl
        self.inp, self.wl = inp, wl
        self.W, self.M_local, self.K, self.N = wl.W, wl.M, wl.K, wl.N
        self.dt = dtype_code(wl.dtype)
        self.shards = shard_layout([dev_bits(a) for a in inp.a], layout)
        self.B = dev_bits(inp.b[0])
        tdt = torch.float32 if out_dtype == "fp32" else torch.bfloat16
        self.C = torch.full((wl.W * wl.M, wl.N), float("nan"), dtype=tdt, device="cuda")
        self.out_dtype = out_dtype
        self.opts = opts
        self.ws = workspace(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, self.dt, opts)

    def run(self, opts=None):
        o = opts if opts is not None else self.opts
        return tdx.tdx_ag_gemm(self.shards, self.B, self.C, self.ws, self.W, self.M_local, self.K, self.N,
                               self.dt, o)

    def result(self) -> np.ndarray:
        torch.cuda.synchronize()
        if self.out_dtype == "fp32":
            return self.C.cpu().numpy().astype(np.float64)
        return R.decode_bf16(host_bits(self.C))

    def result_bits(self) -> np.ndarray:
        torch.cuda.synchronize()
        return host_bits(self.C)

    def oracle(self, rows=None):
        i = self.inp
        sa = i.scale_a if self.wl.dtype == "e4m3" else None
        sb = i.scale_b[0] if self.wl.dtype == "e4m3" else None
        if rows is None:
            return R.ag_gemm(i.a, i.b[0], self.wl.dtype, sa, sb)
        return R.ag_gemm_rows(i.a, i.b[0], rows, self.wl.dtype, sa, sb)


class RSCase:
    def __init__(self, inp, opts=None):
        wl = inp.wl
        self.inp, self.wl = inp, wl
        self.W, self.M, self.K, self.N = wl.W, wl.M, wl.K, wl.N
        self.dt = dtype_code(wl.dtype)
        self.A = [dev_bits(a) for a in inp.a]
        self.B = [dev_bits(b) for b in inp.b]
        self.out = [torch.full((wl.M // wl.W, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
                    for _ in range(wl.W)]
        self.opts = opts
        self.ws = workspace(tdx.OP_RS, wl.W, wl.M, wl.K, wl.N, self.dt, opts)

    def run(self, opts=None):
        o = opts if opts is not None else self.opts
        return tdx.tdx_gemm_rs(self.A, self.B, self.out, self.ws, self.W, self.M, self.K, self.N,
                               self.dt, o)

    def result_bits(self) -> np.ndarray:
        torch.cuda.synchronize()
        return np.concatenate([host_bits(o) for o in self.out])

    def result(self) -> np.ndarray:
        return R.decode_bf16(self.result_bits())

    def oracle(self, rows=None, partials="fp32"):
        i, dt = self.inp, self.wl.dtype
        sa = i.scale_a if dt == "e4m3" else None
        sb = i.scale_b if dt == "e4m3" else None
        if rows is None:
            return np.concatenate(R.gemm_rs(i.a, i.b, dt, sa, sb, partials=partials))
        return R.gemm_rs_rows(i.a, i.b, rows, dt, sa, sb, partials=partials)


class ARCase:
    """Device buffers of one GEMM+AllReduce problem: W full M x N outputs."""

    def __init__(self, inp, opts=None):
        wl = inp.wl
        self.inp, self.wl = inp, wl
        self.W, self.M, self.K, self.N = wl.W, wl.M, wl.K, wl.N
        self.dt = dtype_code(wl.dtype)
        self.A = [dev_bits(a) for a in inp.a]
        self.B = [dev_bits(b) for b in inp.b]
        self.out = [torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
                    for _ in range(wl.W)]
        self.opts = opts
        self.ws = workspace(tdx.OP_AR, wl.W, wl.M, wl.K, wl.N, self.dt, opts)

    def run(self, opts=None):
        o = opts if opts is not None else self.opts
        return tdx.tdx_gemm_ar(self.A, self.B, self.out, self.ws, self.W, self.M, self.K, self.N,
                               self.dt, o)

    def result_bits(self, rank: int) -> np.ndarray:
        torch.cuda.synchronize()
        return host_bits(self.out[rank])

    def oracle(self, rows=None, partials="fp32"):
        i, dt = self.inp, self.wl.dtype
        sa = i.scale_a if dt == "e4m3" else None
        sb = i.scale_b if dt == "e4m3" else None
        if rows is None:
            return R.gemm_ar(i.a, i.b, dt, sa, sb, partials=partials)[0]
        return R.gemm_rs_rows(i.a, i.b, rows, dt, sa, sb, partials=partials)


def assert_bit_exact(got_bits: np.ndarray, oracle_fp64: np.ndarray, out_dtype: str):
    want = R.round_out(oracle_fp64, out_dtype)
    if out_dtype == "fp32":
        got_bits = np.asarray(got_bits, dtype=np.float32)
        bad = np.argwhere(got_bits != want)
    else:
        bad = np.argwhere(got_bits != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[:5].tolist()}"


def assert_within_tol(got: np.ndarray, oracle_fp64: np.ndarray, dtype: str):
    assert np.all(np.isfinite(got)), "non-finite output"
    scale = float(np.max(np.abs(oracle_fp64)))
    err = float(np.max(np.abs(got - oracle_fp64)))
    assert err <= TOL[dtype] * scale, f"max err {err:.4g} > {TOL[dtype]} * {scale:.4g}"
    return err / scale if scale else 0.0


def sample_rows(M: int, chunk: int, extra_stride: int = 97) -> np.ndarray:
    """First, second and last row of every chunk (and of every 128-row tile), plus a stride."""
    rows = set()
    for c0 in range(0, M, chunk):
        rows.update({c0, c0 + 1, min(c0 + chunk, M) - 1})
    for t0 in range(0, M, 128):
        rows.update({t0, min(t0 + 128, M) - 1, min(t0 + 77, M - 1)})
    rows.update(range(0, M, extra_stride))
    return np.array(sorted(rows), dtype=np.int64)


class MoECase:
    """Device buffers of one AllToAll dispatch + grouped GEMM problem."""

    def __init__(self, inp, opts=None, offsets=True):
        wl = inp.wl
        self.inp, self.wl = inp, wl
        self.W, self.T, self.H, self.F, self.E, self.k = wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk
        self.dt = dtype_code(wl.dtype)
        self.X = [dev_bits(a) for a in inp.a]
        self.route = [torch.from_numpy(np.ascontiguousarray(r)).cuda() for r in inp.route]
        self.B = dev_bits(inp.b[0])
        rows = wl.M_total
        self.Y = torch.full((rows, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        self.dest = torch.full((wl.W, wl.M, wl.topk), -7, dtype=torch.int32, device="cuda")
        self.offsets = torch.full((wl.E + 1,), -7, dtype=torch.int32, device="cuda") if offsets else None
        self.opts = opts
        n = tdx.tdx_moe_workspace_size(wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk, self.dt, opts)
        self.ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        tdx.check(tdx.tdx_workspace_init(self.ws), "init")

    def run(self, opts=None):
        o = opts if opts is not None else self.opts
        return tdx.tdx_moe_dispatch_gemm(self.X, self.route, self.B, self.Y, self.dest, self.offsets, self.ws,
                                         self.W, self.T, self.H, self.F, self.E, self.k, self.dt, o)

    def result_bits(self) -> np.ndarray:
        torch.cuda.synchronize()
        return host_bits(self.Y)

    def plan(self, opts=None):
        return tdx.tdx_moe_plan_info(self.W, self.T, self.H, self.F, self.E, self.k, self.dt,
                                     opts if opts is not None else self.opts)


class CombineCase:
    """Device buffers of one grouped GEMM + AllToAll combine problem (workload op "moe_combine":
    M tokens per rank, K = expert input width F, N = hidden width H)."""

    def __init__(self, inp, opts=None):
        wl = inp.wl
        self.inp, self.wl = inp, wl
        self.W, self.T, self.F, self.H, self.E, self.k = wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk
        self.Hd = dev_bits(inp.a[0])
        self.route = [torch.from_numpy(np.ascontiguousarray(r)).cuda() for r in inp.route]
        self.gates = [torch.from_numpy(np.ascontiguousarray(g)).cuda() for g in inp.gates]
        self.B = dev_bits(inp.b[0])
        self.out = [torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(wl.W)]
        self.opts = opts
        n = tdx.tdx_moe_combine_workspace_size(wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk, tdx.TDX_BF16, opts)
        self.ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        tdx.check(tdx.tdx_workspace_init(self.ws), "init")

    def run(self, opts=None):
        o = opts if opts is not None else self.opts
        return tdx.tdx_moe_gemm_combine(self.Hd, self.route, self.B, self.gates, self.out, self.ws, self.W, self.T,
                                        self.F, self.H, self.E, self.k, tdx.TDX_BF16, o)

    def result_bits(self) -> np.ndarray:
        torch.cuda.synchronize()
        return np.stack([host_bits(o) for o in self.out])

    def plan(self, opts=None):
        return tdx.tdx_moe_combine_plan_info(self.W, self.T, self.F, self.H, self.E, self.k, tdx.TDX_BF16,
                                             opts if opts is not None else self.opts)

    def z_bits(self) -> np.ndarray:
        pl = self.plan()
        rows = pl["total_rows"]
        torch.cuda.synchronize()
        z = self.ws[pl["off_R"]:pl["off_R"] + rows * self.H * 2].view(torch.int16).cpu().numpy().view(np.uint16)
        return z.reshape(rows, self.H)


# ------------------------------------------------------------------ trace decoding (tdx_trace_size)
STAT_WORDS = 12   # statistics words per CTA
PHASES = ["entry", "setup", "first_item_loaded", "first_item_mma", "mma_done", "items_done", "epilogue_done"]


def trace_phases(tr: np.ndarray, grid: int) -> np.ndarray:
    """Per CTA (grid x 7, ns) the phase stamps of PHASES relative to the earliest kernel entry of
    the grid; stamps a CTA did not record (0) stay 0."""
    st = tr[4:4 + STAT_WORDS * grid].reshape(grid, STAT_WORDS).astype(np.int64)
    t0 = st[:, 4].min()
    cols = [np.where(st[:, c] == 0, 0, (st[:, c] - t0) % (1 << 32)) for c in range(4, 11)]
    return np.stack(cols, axis=1)

def trace_items(tr: np.ndarray, grid: int, chunks: int, cl: int = 1) -> dict:
    """Work items a traced call took: {(item index in the cluster-wide sequence, CTA rank in its
    pair): (chain element, tile id)}. CTA b of a grid of pairs (cl = 2) is CTA b % 2 of pair b // 2,
    and pair q takes items q, q + grid/2, ...; single CTAs (cl = 1) take b, b + grid, ..."""
    items = int(tr[1])
    per = (items + grid - 1) // grid
    base = 4 + STAT_WORDS * grid + 1 + chunks
    ncl = grid // cl
    out = {}
    for b in range(grid):
        cid, crank = divmod(b, cl)
        mine = list(range(cid, items // cl, ncl))
        assert int(tr[4 + STAT_WORDS * b + 3]) == len(mine), (b, int(tr[4 + STAT_WORDS * b + 3]), len(mine))
        for k, it in enumerate(mine):
            w = int(tr[base + b * per + k])
            out[(it, crank)] = (w >> 24, w & 0xFFFFFF)
    return out


def trace_releases(tr: np.ndarray, grid: int, chunks: int) -> list:
    """Flag indices of the chunks a traced call released, in release order."""
    base = 4 + STAT_WORDS * grid
    n = int(tr[base])
    assert n == chunks, (n, chunks)
    return [int(x) for x in tr[base + 1:base + 1 + n]]


def check_each_item_once(taken: dict, L: int, T: int):
    got = sorted(taken.values())
    assert got == [(c, t) for c in range(L) for t in range(T)], "some (element, tile) missing or repeated"


def check_ag_consumer_order(taken: dict, L: int, tiles_n: int, W: int, M_local: int, self_rank: int):
    """For every K split c, the first rows of the tiles taken, in item order, visit the ranks in the
    oracle's arrival order (own shard first, then self+1, self+2, ...)."""
    for c in range(L):
        seq = sorted((it, crank, t) for (it, crank), (cc, t) in taken.items() if cc == c)
        rows, last = [], None
        for it, _, t in seq:
            if it != last:     # the two CTAs of a pair share an item: its first row is the lower tile's
                rows.append(min((tt // tiles_n) * 128 for i2, _, tt in seq if i2 == it))
                last = it
        assert R.ag_consumer_order_ok(rows, W, M_local, self_rank), rows[:16]


def check_rs_fold_order(taken: dict, W: int, T: int):
    """For every output tile, the ranks' items come in the oracle's fold order 0, 1, ..., W-1."""
    by_tile = {}
    for (it, _), (r, t) in taken.items():
        by_tile.setdefault(t, []).append((it, r))
    assert len(by_tile) == T
    for t, lst in by_tile.items():
        assert [r for _, r in sorted(lst)] == R.rs_fold_order(W), (t, sorted(lst))
