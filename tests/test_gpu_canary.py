"""Out-of-bounds writes, checked with guard regions (compute-sanitizer is not available here).

Every output and workspace of a call is carved out of a larger device buffer whose bytes before and
after it hold a fixed pattern; after ragged-shape calls (partial M and N tiles, tiles spanning
ranks, K splits, 512-column tiles, the grid-wide fold, MoE tiles cut at expert boundaries) the
pattern must be intact, and the outputs must still match the oracle.
"""
import numpy as np
import pytest
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import moe as MO
from oracle import reference as R
import workloads as wls
from gpu_util import assert_bit_exact, dev_bits, host_bits

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side; keeps the 256-byte alignment workspaces need
PATTERN = 0xA5


class Guarded:
    """A device tensor of `shape`/`dtype` with GUARD pattern bytes before and after it."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.n = n
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(*shape)
        if fill is not None:
            self.t.fill_(fill)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def guarded_ws(nbytes):
    g = Guarded((nbytes,), torch.uint8)
    tdx.check(tdx.tdx_workspace_init(g.t))
    return g


def opts(**kw):
    return tdx.make_opts(timeout_ns=500_000_000, **kw)


@pytest.mark.parametrize("shape,variant", [
    (dict(W=3, M=96, K=320, N=200, chunk_rows=32), {}),
    (dict(W=3, M=96, K=320, N=200, chunk_rows=32), dict(split_k=3, block_n=128, reduce_mode=2)),
    (dict(W=5, M=64, K=1024, N=72, chunk_rows=16), dict(split_k=4, reduce_mode=3, num_sms=6)),
    (dict(W=2, M=384, K=512, N=1344, chunk_rows=128), dict(cluster=3, block_n=512)),
    (dict(W=8, M=16, K=2048, N=200, chunk_rows=16), {}),
])
def test_ag_writes_stay_in_bounds(shape, variant):
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], **shape)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(chunk_rows=shape["chunk_rows"], **variant)
    shards = [dev_bits(a) for a in inp.a]
    B = dev_bits(inp.b[0])
    C = Guarded((wl.W * wl.M, wl.N), torch.bfloat16, float("nan"))
    ws = guarded_ws(tdx.tdx_workspace_size(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))
    for _ in range(2):
        tdx.check(tdx.tdx_ag_gemm(shards, B, C.t, ws.t, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))
    st, d = tdx.tdx_read_device_status(ws.t)
    assert st == tdx.TDX_OK, d
    assert C.intact() and ws.intact()
    assert_bit_exact(host_bits(C.t), R.ag_gemm(inp.a, inp.b[0], "bf16"), "bf16")


@pytest.mark.parametrize("shape,variant", [
    (dict(W=3, M=384, K=200, N=136), {}),
    (dict(W=4, M=200, K=64, N=264), dict(reduce_mode=1, block_n=128)),
    (dict(W=4, M=512, K=256, N=520), dict(reduce_mode=3, num_sms=7)),
    (dict(W=3, M=768, K=256, N=1344), dict(cluster=3, block_n=512, reduce_mode=1)),
    (dict(W=4, M=512, K=256, N=520), dict(bf16_partials=1)),
])
def test_rs_writes_stay_in_bounds(shape, variant):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], **shape)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(**variant)
    A = [dev_bits(a) for a in inp.a]
    Bs = [dev_bits(b) for b in inp.b]
    outs = [Guarded((wl.M // wl.W, wl.N), torch.bfloat16, float("nan")) for _ in range(wl.W)]
    ws = guarded_ws(tdx.tdx_workspace_size(tdx.OP_RS, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))
    for _ in range(2):
        tdx.check(tdx.tdx_gemm_rs(A, Bs, [g.t for g in outs], ws.t, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))
    st, d = tdx.tdx_read_device_status(ws.t)
    assert st == tdx.TDX_OK, d
    assert all(g.intact() for g in outs) and ws.intact()
    partials = "bf16" if variant.get("bf16_partials") else "fp32"
    want = np.concatenate(R.gemm_rs(inp.a, inp.b, "bf16", partials=partials))
    assert_bit_exact(np.concatenate([host_bits(g.t) for g in outs]), want, "bf16")


def test_ar_writes_stay_in_bounds():
    wl = wls.with_shape(wls.WORKLOADS["ar_w8"], W=4, M=200, K=136, N=264)
    inp = wls.make_inputs(wl, integer=True)
    o = opts()
    A = [dev_bits(a) for a in inp.a]
    Bs = [dev_bits(b) for b in inp.b]
    outs = [Guarded((wl.M, wl.N), torch.bfloat16, float("nan")) for _ in range(wl.W)]
    ws = guarded_ws(tdx.tdx_workspace_size(tdx.OP_AR, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))
    tdx.check(tdx.tdx_gemm_ar(A, Bs, [g.t for g in outs], ws.t, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o))
    st, d = tdx.tdx_read_device_status(ws.t)
    assert st == tdx.TDX_OK, d
    assert all(g.intact() for g in outs) and ws.intact()
    want = R.gemm_ar(inp.a, inp.b)[0]
    for g in outs:
        assert_bit_exact(host_bits(g.t), want, "bf16")


@pytest.mark.parametrize("shape,variant", [
    (dict(W=3, M=70, K=200, N=136, E=6, topk=3), {}),
    (dict(W=4, M=300, K=512, N=1344, E=8, topk=3), dict(cluster=3, block_n=512)),
])
def test_moe_writes_stay_in_bounds(shape, variant):
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], **shape)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(**variant)
    X = [dev_bits(a) for a in inp.a]
    route = [torch.from_numpy(np.ascontiguousarray(r)).cuda() for r in inp.route]
    B = dev_bits(inp.b[0])
    Y = Guarded((wl.M_total, wl.N), torch.bfloat16, float("nan"))
    dest = Guarded((wl.W, wl.M, wl.topk), torch.int32, -7)
    offs = Guarded((wl.E + 1,), torch.int32, -7)
    ws = guarded_ws(tdx.tdx_moe_workspace_size(wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk, tdx.TDX_BF16, o))
    tdx.check(tdx.tdx_moe_dispatch_gemm(X, route, B, Y.t, dest.t, offs.t, ws.t, wl.W, wl.M, wl.K, wl.N, wl.E,
                                        wl.topk, tdx.TDX_BF16, o))
    st, d = tdx.tdx_read_device_status(ws.t)
    assert st == tdx.TDX_OK, d
    assert Y.intact() and dest.intact() and offs.intact() and ws.intact()
    want, _ = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E)
    assert_bit_exact(host_bits(Y.t), want, "bf16")


def test_combine_writes_stay_in_bounds():
    wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], W=3, M=70, K=136, N=200, E=6, topk=3)
    inp = wls.make_inputs(wl, integer=True)
    o = opts()
    Hd = dev_bits(inp.a[0])
    route = [torch.from_numpy(np.ascontiguousarray(r)).cuda() for r in inp.route]
    gates = [torch.from_numpy(np.ascontiguousarray(g)).cuda() for g in inp.gates]
    B = dev_bits(inp.b[0])
    outs = [Guarded((wl.M, wl.N), torch.bfloat16, float("nan")) for _ in range(wl.W)]
    ws = guarded_ws(tdx.tdx_moe_combine_workspace_size(wl.W, wl.M, wl.K, wl.N, wl.E, wl.topk, tdx.TDX_BF16, o))
    tdx.check(tdx.tdx_moe_gemm_combine(Hd, route, B, gates, [g.t for g in outs], ws.t, wl.W, wl.M, wl.K, wl.N,
                                       wl.E, wl.topk, tdx.TDX_BF16, o))
    st, d = tdx.tdx_read_device_status(ws.t)
    assert st == tdx.TDX_OK, d
    assert all(g.intact() for g in outs) and ws.intact()
    want = np.stack(MO.moe_gemm_combine(inp.a[0], inp.route, inp.b[0], inp.gates, wl.E, z_dtype="bf16"))
    assert_bit_exact(np.stack([host_bits(g.t) for g in outs]), want, "bf16")
