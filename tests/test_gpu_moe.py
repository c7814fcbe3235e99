"""AllToAll dispatch + grouped GEMM of a mixture-of-experts layer on the GPU through the C ABI,
against the CPU oracle: the routing layout (row of every token slot, expert offsets) is compared
exactly, the expert outputs bit-exactly on integer inputs and within the bf16 tolerance on random
ones; the receive buffer, chunk flags and tile table left in the workspace are checked as well."""
import numpy as np
import pytest
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import moe as MO
from oracle import reference as R
import workloads as wls
from gpu_util import MoECase, assert_bit_exact, assert_within_tol

pytestmark = pytest.mark.gpu

TMO = int(5e8)


def opts(**kw):
    return tdx.make_opts(timeout_ns=TMO, **kw)


def status_ok(case):
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_OK, (tdx.tdx_status_string(st), detail)


def check_layout(case, lay):
    counts, offsets, dest, _ = lay
    torch.cuda.synchronize()
    got = case.dest.cpu().numpy()
    for s in range(case.W):
        assert np.array_equal(got[s], dest[s])
    if case.offsets is not None:
        assert np.array_equal(case.offsets.cpu().numpy(), offsets)


SHAPES = [
    dict(W=2, M=5, K=64, N=128, E=4, topk=2),          # a handful of rows, every tile partial
    dict(W=3, M=70, K=200, N=136, E=6, topk=3),        # ragged K and N
    dict(W=8, M=128, K=256, N=512, E=64, topk=8),      # 128 tokens per rank, 8 experts per rank
    dict(W=1, M=300, K=128, N=256, E=3, topk=1),
    dict(W=4, M=257, K=64, N=64, E=8, topk=2),         # experts with several tiles and a tail
    dict(W=16, M=17, K=64, N=192, E=32, topk=4),
    dict(W=4, M=33, K=128, N=256, E=16, topk=16),      # the most slots a token may have: every expert
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("integer", [True, False])
def test_moe_small_shapes(shape, integer):
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    want, lay = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E)
    for bn, cl in ((0, 0), (64, 0), (256, 1), (256, 3)):
        case = MoECase(inp, opts=opts(block_n=bn, cluster=cl))
        tdx.check(case.run(), f"moe {shape} bn={bn} cluster={cl}")
        status_ok(case)
        check_layout(case, lay)
        if integer:
            assert_bit_exact(case.result_bits(), want, "bf16")
        else:
            assert_within_tol(R.decode_bf16(case.result_bits()), want, "bf16")


def test_moe_workspace_bookkeeping():
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], W=4, M=100, K=256, N=256, E=8, topk=2)
    inp = wls.make_inputs(wl, integer=True)
    case = MoECase(inp, opts=opts(epoch=5))
    tdx.check(case.run())
    status_ok(case)
    _, lay = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E)
    counts, offsets, dest, src = lay
    pl = case.plan()
    ws = case.ws
    rows = pl["total_rows"]
    # the receive buffer holds every dispatched token row, bit for bit
    R_ = ws[pl["off_R"]:pl["off_R"] + rows * wl.K * 2].view(torch.int16).cpu().numpy().view(np.uint16)
    R_ = R_.reshape(rows, wl.K)
    for r in range(rows):
        s, t = src[r]
        assert np.array_equal(R_[r], inp.a[s][t])
    # every chunk flag holds the epoch; the tile table lists each expert's 128-row tiles
    fl = ws[pl["off_chunk_flags"]:pl["off_chunk_flags"] + 4 * pl["n_chunks"]].view(torch.int32).cpu().numpy()
    assert np.array_equal(fl.astype(np.uint32), R.expected_flags(pl["n_chunks"], 5))
    nt = ws[pl["off_ntiles"]:pl["off_ntiles"] + 8].view(torch.int32).cpu().numpy()
    tiles = ws[pl["off_tiles"]:pl["off_tiles"] + 16 * int(nt[0])].view(torch.int32).cpu().numpy().reshape(-1, 4)
    want_tiles = [(int(offsets[e]) + 128 * i, int(offsets[e + 1]), e, 0)
                  for e in range(wl.E) for i in range((int(offsets[e + 1] - offsets[e]) + 127) // 128)]
    assert nt[1] == 0 and [tuple(x) for x in tiles.tolist()] == want_tiles
    srcw = ws[pl["off_src"]:pl["off_src"] + 4 * rows].view(torch.int32).cpu().numpy()
    assert [tuple(divmod(int(v), wl.M)) for v in srcw] == src


def test_moe_modes_and_epochs():
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], W=4, M=128, K=512, N=256, E=16, topk=4)
    inp = wls.make_inputs(wl, integer=True)
    want, _ = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E)
    case = MoECase(inp, opts=opts())
    # dispatch alone, then the grouped GEMM alone on the filled receive buffer
    tdx.check(case.run(opts(mode=tdx.TDX_MOVE_ONLY, epoch=1)))
    tdx.check(case.run(opts(mode=tdx.TDX_GEMM_ONLY, epoch=2)))
    status_ok(case)
    assert_bit_exact(case.result_bits(), want, "bf16")
    for ep in (3, 4):
        case.Y.fill_(float("nan"))
        tdx.check(case.run(opts(epoch=ep, perturb_seed=ep)))
        status_ok(case)
        assert_bit_exact(case.result_bits(), want, "bf16")


def test_moe_device_epochs_and_release_trace():
    # epochs kept in the workspace across calls (modes included), and the dispatch's chunk
    # releases recorded in the trace: every 128-row chunk of the receive buffer exactly once
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], W=4, M=128, K=512, N=256, E=16, topk=4)
    inp = wls.make_inputs(wl, integer=True)
    want, _ = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E)
    o = opts(epoch=tdx.TDX_EPOCH_DEVICE)
    case = MoECase(inp, opts=o)
    tdx.check(case.run(opts(mode=tdx.TDX_MOVE_ONLY, epoch=tdx.TDX_EPOCH_DEVICE)))
    tdx.check(case.run(opts(mode=tdx.TDX_GEMM_ONLY, epoch=tdx.TDX_EPOCH_DEVICE)))
    status_ok(case)
    assert_bit_exact(case.result_bits(), want, "bf16")
    plan = case.plan()
    grid = 24
    chunks = plan["n_chunks"]
    trace = torch.zeros(tdx.tdx_trace_size(grid, plan["max_tiles"] * plan["tiles_n"], chunks) // 4,
                        dtype=torch.int32, device="cuda")
    for call in range(2):
        case.Y.fill_(float("nan"))
        trace.zero_()
        tdx.check(case.run(opts(epoch=tdx.TDX_EPOCH_DEVICE, num_sms=grid, trace=trace, perturb_seed=call + 1)))
        status_ok(case)
        assert_bit_exact(case.result_bits(), want, "bf16")
        tr = trace.cpu().numpy().astype(np.uint32)
        n = int(tr[4 + 12 * grid])
        assert n == chunks and sorted(tr[4 + 12 * grid + 1:4 + 12 * grid + 1 + n].tolist()) == list(range(chunks))
    assert int(case.ws[64:68].view(torch.int32).item()) == 4


def test_moe_invalid_expert_id_is_reported_not_run():
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], W=2, M=16, K=64, N=64, E=4, topk=2)
    inp = wls.make_inputs(wl, integer=True)
    inp.route[1] = inp.route[1].copy()
    inp.route[1][3, 1] = 9
    case = MoECase(inp, opts=opts())
    tdx.check(case.run())
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_ERR_INVALID_ARG and detail[1] == 5 and detail[4] == 9
    assert bool(torch.isnan(case.Y.float()).all())         # nothing was computed


def test_moe_degenerate_sizes():
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], W=2, M=8, K=64, N=64, E=4, topk=2)
    inp = wls.make_inputs(wl, integer=True)
    _, lay = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E)
    case = MoECase(inp, opts=opts())
    # H = 0: the layout is still produced and every expert output is zero
    tdx.check(tdx.tdx_moe_dispatch_gemm(case.X, case.route, case.B, case.Y, case.dest, case.offsets, case.ws,
                                        2, 8, 0, 64, 4, 2, tdx.TDX_BF16, opts()))
    check_layout(case, lay)
    assert int(torch.count_nonzero(case.Y)) == 0
    # T = 0: no rows; the expert offsets are all zero
    tdx.check(tdx.tdx_moe_dispatch_gemm(case.X, case.route, case.B, case.Y, case.dest, case.offsets, case.ws,
                                        2, 0, 64, 64, 4, 2, tdx.TDX_BF16, opts()))
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(case.offsets)) == 0
    status_ok(case)


def test_moe_full_size_sampled_and_deterministic():
    wl = wls.WORKLOADS["moe_w8"]
    inp = wls.make_inputs(wl, integer=False)
    case = MoECase(inp, opts=opts())
    tdx.check(case.run())
    status_ok(case)
    counts, offsets, dest, src = MO.moe_layout(inp.route, wl.E)
    check_layout(case, (counts, offsets, dest, src))
    first = case.result_bits()
    # first, second and last row of every expert, plus a stride
    rows = set(range(0, wl.M_total, 4099))
    for e in range(wl.E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            rows.update({a, min(a + 1, b - 1), b - 1, min(a + 127, b - 1), min(a + 128, b - 1)})
    rows = np.array(sorted(rows))
    want = MO.moe_dispatch_gemm_rows(inp.a, inp.route, inp.b[0], wl.E, rows)
    assert_within_tol(R.decode_bf16(first[rows]), want, "bf16")
    case.Y.fill_(float("nan"))
    tdx.check(case.run(opts(perturb_seed=17)))
    status_ok(case)
    assert np.array_equal(case.result_bits(), first)


def test_moe_pairs_match_single_ctas_bitwise():
    wl = wls.with_shape(wls.WORKLOADS["moe_w8"], W=4, M=300, K=512, N=512, E=8, topk=2)
    inp = wls.make_inputs(wl, integer=False)
    bits = []
    for cl in (1, 3):
        case = MoECase(inp, opts=opts(block_n=256, cluster=cl, perturb_seed=3))
        assert case.plan()["cluster"] == cl
        tdx.check(case.run())
        status_ok(case)
        bits.append(case.result_bits())
    assert np.array_equal(bits[0], bits[1])


@pytest.mark.parametrize("shape", [dict(W=2, M=5, K=128, N=128, E=4, topk=2),
                                   dict(W=8, M=128, K=512, N=512, E=64, topk=8),
                                   dict(W=4, M=300, K=256, N=384, E=8, topk=2)])
@pytest.mark.parametrize("integer", [True, False])
def test_moe_e4m3(shape, integer):
    wl = wls.with_shape(wls.WORKLOADS["moe_fp8_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    want, lay = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E, "e4m3", inp.scale_a, inp.scale_b)
    for bn, cl in ((0, 0), (256, 1), (256, 3)):
        case = MoECase(inp, opts=opts(block_n=bn, cluster=cl, scale_a=inp.scale_a, scale_b=inp.scale_b))
        tdx.check(case.run(), f"moe e4m3 {shape} bn={bn} cluster={cl}")
        status_ok(case)
        check_layout(case, lay)
        if integer:
            assert_bit_exact(case.result_bits(), want, "bf16")
        else:
            assert_within_tol(R.decode_bf16(case.result_bits()), want, "e4m3")


def test_moe_e4m3_full_size_sampled():
    wl = wls.WORKLOADS["moe_fp8_w8"]
    inp = wls.make_inputs(wl, integer=False)
    case = MoECase(inp, opts=opts(scale_a=inp.scale_a, scale_b=inp.scale_b))
    tdx.check(case.run())
    status_ok(case)
    _, offsets, _, _ = MO.moe_layout(inp.route, wl.E)
    rows = set(range(0, wl.M_total, 8191))
    for e in range(0, wl.E, 7):
        a, b = int(offsets[e]), int(offsets[e + 1])
        rows.update({a, b - 1, min(a + 128, b - 1)})
    rows = np.array(sorted(rows))
    want = MO.moe_dispatch_gemm_rows(inp.a, inp.route, inp.b[0], wl.E, rows, "e4m3", inp.scale_a, inp.scale_b)
    assert_within_tol(R.decode_bf16(case.result_bits()[rows]), want, "e4m3")


def _skewed(inp, experts):
    """Every token of every rank routed to the same `experts` (one slot each)."""
    for s in range(len(inp.route)):
        r = np.empty_like(inp.route[s])
        r[:] = np.asarray(experts, dtype=np.int32)[None, :]
        inp.route[s] = r
    return inp


@pytest.mark.parametrize("case_name", ["mostly_empty", "skewed"])
@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_moe_empty_and_skewed_experts(case_name, dtype):
    base = "moe_w8" if dtype == "bf16" else "moe_fp8_w8"
    if case_name == "mostly_empty":
        wl = wls.with_shape(wls.WORKLOADS[base], W=2, M=3, K=128, N=256, E=64, topk=2)   # 12 rows, 64 experts
        inp = wls.make_inputs(wl, integer=True)
    else:
        wl = wls.with_shape(wls.WORKLOADS[base], W=4, M=660, K=128, N=256, E=8, topk=2)  # all to experts 1 and 6: 21 tiles each
        inp = _skewed(wls.make_inputs(wl, integer=True), [6, 1])
    sa = inp.scale_a if dtype == "e4m3" else None
    sb = inp.scale_b if dtype == "e4m3" else None
    want, lay = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E, dtype, sa, sb)
    kw = dict(scale_a=sa, scale_b=sb) if dtype == "e4m3" else {}
    for bn, cl in ((0, 0), (256, 3)):
        case = MoECase(inp, opts=opts(block_n=bn, cluster=cl, **kw))
        tdx.check(case.run())
        status_ok(case)
        check_layout(case, lay)
        assert_bit_exact(case.result_bits(), want, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "e4m3"])
def test_moe_wide_tiles_match_256(dtype):
    # 512-column tiles on 2-SM pairs for the dispatch's grouped GEMM: the same bits as 256 columns
    # (the K accumulation is the same), exact on integers; ragged F (1344 = 2.6 tiles of 512)
    name = "moe_w8" if dtype == "bf16" else "moe_fp8_w8"
    wl = wls.with_shape(wls.WORKLOADS[name], W=4, M=300, K=512, N=1344, E=8, topk=3)
    for integer in (True, False):
        inp = wls.make_inputs(wl, integer=integer)
        kw = dict(scale_a=inp.scale_a, scale_b=inp.scale_b) if dtype == "e4m3" else {}
        want, _ = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E, dtype=dtype,
                                       scale_x=kw.get("scale_a"), scale_b=kw.get("scale_b"))
        bits = []
        for bn in (512, 256):
            case = MoECase(inp, opts=opts(block_n=bn, cluster=3, **kw))
            assert case.plan()["BN"] == bn and case.plan()["cluster"] == 3
            tdx.check(case.run())
            status_ok(case)
            bits.append(case.result_bits())
            if integer:
                assert_bit_exact(bits[-1], want, "bf16")
            else:
                assert_within_tol(R.decode_bf16(bits[-1]), want, dtype)
        assert np.array_equal(bits[0], bits[1])
