"""GEMM+ReduceScatter on the GPU through the C ABI against the CPU oracle, plus run-to-run
bit-identity of the rank-ordered reduction under injected timing perturbation."""
import numpy as np
import pytest
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import reference as R
import workloads as wls
from gpu_util import (RSCase, assert_bit_exact, assert_within_tol, check_each_item_once, check_rs_fold_order,
                      sample_rows, trace_items)

pytestmark = pytest.mark.gpu

TMO = int(5e8)


def opts(**kw):
    return tdx.make_opts(timeout_ns=TMO, **kw)


def status_ok(case):
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_OK, (tdx.tdx_status_string(st), detail)


@pytest.mark.parametrize("shape", [
    dict(W=2, M=256, K=256, N=512),
    dict(W=3, M=384, K=200, N=136),     # ragged K and N, shard = 128 rows
    dict(W=4, M=200, K=64, N=264),      # shards of 50 rows: tiles span shards
    dict(W=1, M=128, K=128, N=256),
    dict(W=16, M=256, K=64, N=64),
])
@pytest.mark.parametrize("integer", [True, False])
def test_rs_small_shapes(shape, integer):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    for bn, rm in ((0, 0), (128, 1), (256, 2)):
        case = RSCase(inp, opts=opts(block_n=bn, reduce_mode=rm))
        tdx.check(case.run(), f"rs {shape} bn={bn} reduce_mode={rm}")
        status_ok(case)
        if integer:
            assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
        else:
            assert_within_tol(case.result(), case.oracle(), "bf16")


@pytest.mark.parametrize("integer", [True, False])
def test_rs_full_size_full_output(integer):
    # the headline shape, every element of the W output shards against the full fp64 oracle
    wl = wls.WORKLOADS["rs_w8"]
    inp = wls.make_inputs(wl, integer=integer)
    case = RSCase(inp, opts=opts())
    tdx.check(case.run())
    status_ok(case)
    got = case.result_bits()
    want = case.oracle()
    assert want.shape == got.shape == (wl.M, wl.N)
    if integer:
        assert_bit_exact(got, want, "bf16")
    else:
        assert_within_tol(R.decode_bf16(got), want, "bf16")
    if not integer:
        # run-to-run bit identity, with and without injected delays
        first = case.result_bits()
        for seed in (0, 1234):
            for o in case.out:
                o.fill_(float("nan"))
            tdx.check(case.run(opts(perturb_seed=seed)))
            assert np.array_equal(case.result_bits(), first)
        status_ok(case)


@pytest.mark.parametrize("integer", [True, False])
def test_rs_small_m_full_output(integer):
    wl = wls.WORKLOADS["rs_small"]
    inp = wls.make_inputs(wl, integer=integer)
    case = RSCase(inp, opts=opts())
    tdx.check(case.run())
    status_ok(case)
    if integer:
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    else:
        assert_within_tol(case.result(), case.oracle(), "bf16")


def test_rs_chain_flags_trace_and_order():
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], W=4, M=512, K=256, N=512)
    inp = wls.make_inputs(wl, integer=False)
    grid = 8
    o = opts(num_sms=grid, reduce_mode=1)
    plan = tdx.tdx_plan_info(tdx.OP_RS, 4, 512, 256, 512, tdx.TDX_BF16, o)
    assert plan["reduce_mode"] == 1
    items = plan["L"] * plan["T"]
    trace = torch.zeros(tdx.tdx_trace_size(grid, items, 0) // 4, dtype=torch.int32, device="cuda")
    case = RSCase(inp, opts=opts(num_sms=grid, trace=trace, epoch=3, reduce_mode=1))
    tdx.check(case.run())
    status_ok(case)
    assert_within_tol(case.result(), case.oracle(), "bf16")
    n = (plan["L"] - 1) * plan["T"]
    f = case.ws[plan["off_chain_flags"]:plan["off_chain_flags"] + 4 * n].view(torch.int32).cpu().numpy()
    assert np.array_equal(f.astype(np.uint32), R.expected_flags(n, 3))
    tr = trace.cpu().numpy().astype(np.uint32)
    taken = trace_items(tr, grid, 0)
    check_each_item_once(taken, plan["L"], plan["T"])
    check_rs_fold_order(taken, 4, plan["T"])
    # the running sum of ranks 0..W-2 left in the workspace is the left fold of the partials:
    # with fp32 partials it matches the oracle's fp64 sum of ranks 0..W-2 to fp32 accuracy
    S = case.ws[plan["off_S"]:plan["off_S"] + 4 * plan["T"] * 128 * plan["BN"]].view(torch.float32).cpu().numpy()
    full3 = R.gemm_rs_rows(inp.a[:3], inp.b[:3], np.arange(512), "bf16")   # ranks 0..2 summed
    BN = plan["BN"]
    for (mt, nt) in [(0, 0), (3, 1)]:
        tile = mt * plan["tiles_n"] + nt
        T = S[tile * 128 * BN:(tile + 1) * 128 * BN]
        # layout: ((cc*8 + j)*128 + i)*4 + t  ->  element (i, 32*cc + 4*j + t)
        T = T.reshape(BN // 32, 8, 128, 4).transpose(2, 0, 1, 3).reshape(128, BN)
        want = full3[mt * 128:(mt + 1) * 128, nt * BN:(nt + 1) * BN]
        assert np.max(np.abs(T - want)) <= 1e-5 * np.max(np.abs(want))


@pytest.mark.parametrize("variant", [dict(), dict(reduce_mode=2), dict(cluster=3, block_n=256)])
def test_rs_modes_run(variant):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], W=4, M=512, K=256, N=512)
    inp = wls.make_inputs(wl, integer=True)
    case = RSCase(inp, opts=opts(**variant))
    # GEMM alone: every rank's partial computed, only rank W-1's stored into the output
    tdx.check(case.run(opts(mode=tdx.TDX_GEMM_ONLY, **variant)))
    status_ok(case)
    last = np.concatenate(R.gemm_rs(inp.a[3:], inp.b[3:], "bf16"))
    assert_bit_exact(case.result_bits(), last, "bf16")
    for mode in (tdx.TDX_MOVE_ONLY, tdx.TDX_FUSED):
        tdx.check(case.run(opts(mode=mode, **variant)))
        status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")


def test_rs_degenerate_k_zero():
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    outs = [torch.full((64, 128), 2.0, dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    tdx.check(tdx.tdx_gemm_rs([dummy] * 2, [dummy] * 2, outs, ws, 2, 128, 0, 128, tdx.TDX_BF16, opts()))
    torch.cuda.synchronize()
    assert all(int(torch.count_nonzero(o)) == 0 for o in outs)


@pytest.mark.parametrize("shape", [dict(W=8, M=1024, K=512, N=1024), dict(W=3, M=384, K=200, N=136)])
def test_rs_chained_and_slotted_give_identical_bits(shape):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], **shape)
    inp = wls.make_inputs(wl, integer=False)
    outs = []
    for rm in (1, 2):
        case = RSCase(inp, opts=opts(reduce_mode=rm, perturb_seed=99))
        tdx.check(case.run())
        status_ok(case)
        outs.append(case.result_bits())
        assert_within_tol(case.result(), case.oracle(), "bf16")
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("shape,grid", [(dict(W=8, M=128, K=1024, N=8192), 0),     # the small-M shape
                                        (dict(W=4, M=512, K=256, N=512), 7),       # several waves
                                        (dict(W=3, M=384, K=200, N=136), 5),       # ragged K and N
                                        (dict(W=16, M=256, K=64, N=64), 3),
                                        (dict(W=4, M=128, K=320, N=2048), 8),      # one M-tile, four waves
                                        (dict(W=3, M=126, K=200, N=1000), 6)])     # ragged M, K, N
@pytest.mark.parametrize("integer", [True, False])
def test_rs_grid_fold(shape, grid, integer):
    # every CTA stores its partials, meets the others at a grid barrier, then folds 1/grid of all
    # tiles: the same bits as the chained running sum, bit-exact on integers
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    o = opts(reduce_mode=3, num_sms=grid, epoch=2)
    plan = tdx.tdx_plan_info(tdx.OP_RS, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o)
    assert plan["coop_fold"] == 2
    case = RSCase(inp, opts=o)
    tdx.check(case.run())
    status_ok(case)
    if integer:
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    else:
        assert_within_tol(case.result(), case.oracle(), "bf16")
    first = case.result_bits()
    # counters reset: a second call (next epoch, injected delays) gives the same bits
    for x in case.out:
        x.fill_(float("nan"))
    tdx.check(case.run(opts(reduce_mode=3, num_sms=grid, epoch=3, perturb_seed=11)))
    status_ok(case)
    assert np.array_equal(case.result_bits(), first)
    n = 2
    bar = case.ws[plan["off_tile_cnt"]:plan["off_tile_cnt"] + 4 * (2 * plan["T"] + n)].view(torch.int32).cpu().numpy()
    assert not bar.any()
    chained = RSCase(inp, opts=opts(reduce_mode=1))
    tdx.check(chained.run())
    status_ok(chained)
    assert np.array_equal(chained.result_bits(), first)


@pytest.mark.parametrize("rm", [1, 2, 3])
def test_rs_device_epochs_in_a_graph(rm):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], W=4, M=512, K=256, N=512)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(reduce_mode=rm, epoch=tdx.TDX_EPOCH_DEVICE)
    case = RSCase(inp, opts=o)
    want = R.round_out(case.oracle(), "bf16")
    tdx.check(case.run())
    status_ok(case)
    assert np.array_equal(case.result_bits(), want)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            tdx.check(tdx.tdx_gemm_rs(case.A, case.B, case.out, case.ws, 4, 512, 256, 512, tdx.TDX_BF16, o, stream=s))
    torch.cuda.synchronize()
    for _ in range(2):
        for x in case.out:
            x.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(case.result_bits(), want)
    status_ok(case)
    assert int(case.ws[64:68].view(torch.int32).item()) == 1 + 3 * 2


def test_rs_slotted_bookkeeping():
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], W=4, M=512, K=256, N=512)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(reduce_mode=2, epoch=7)
    plan = tdx.tdx_plan_info(tdx.OP_RS, 4, 512, 256, 512, tdx.TDX_BF16, o)
    assert plan["reduce_mode"] == 2
    case = RSCase(inp, opts=o)
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    # every tile's arrival counter is back to zero for the next call
    T = plan["T"]
    cnt = case.ws[plan["off_tile_cnt"]:plan["off_tile_cnt"] + 4 * T].view(torch.int32).cpu().numpy()
    assert not cnt.any()
    # slot r of a tile holds rank r's partial A_r @ B_r (fp32, exact on integers)
    BN = plan["BN"]
    S = case.ws[plan["off_S"]:plan["off_S"] + 4 * 4 * T * 128 * BN].view(torch.float32).cpu().numpy()
    for r in range(4):
        P = R.gemm_rs_rows([inp.a[r]], [inp.b[r]], np.arange(512), "bf16")
        for (mt, nt) in [(0, 0), (2, 3)]:
            tile = mt * plan["tiles_n"] + nt
            blk = S[(r * T + tile) * 128 * BN:(r * T + tile + 1) * 128 * BN]
            blk = blk.reshape(BN // 32, 8, 128, 4).transpose(2, 0, 1, 3).reshape(128, BN)
            assert np.array_equal(blk, P[mt * 128:(mt + 1) * 128, nt * BN:(nt + 1) * BN])
    # a second call with the next epoch gives the same result (counters were reset)
    for x in case.out:
        x.fill_(float("nan"))
    tdx.check(case.run(opts(reduce_mode=2, epoch=8)))
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")


def test_rs_full_size_slotted_matches_chained():
    wl = wls.WORKLOADS["rs_w8"]
    inp = wls.make_inputs(wl, integer=False)
    bits = []
    for rm in (1, 2):
        case = RSCase(inp, opts=opts(reduce_mode=rm))
        tdx.check(case.run())
        status_ok(case)
        bits.append(case.result_bits())
        del case
        torch.cuda.empty_cache()
    assert np.array_equal(bits[0], bits[1])


@pytest.mark.parametrize("cluster", [3])
@pytest.mark.parametrize("rm", [1, 2])
def test_rs_pairs_parity_trace_and_identity(rm, cluster):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], W=4, M=512, K=512, N=512)
    inp = wls.make_inputs(wl, integer=False)
    grid = 8
    o = opts(num_sms=grid, cluster=cluster, block_n=256, reduce_mode=rm)
    plan = tdx.tdx_plan_info(tdx.OP_RS, 4, 512, 512, 512, tdx.TDX_BF16, o)
    assert plan["cluster"] == cluster
    items = plan["L"] * plan["T"]
    trace = torch.zeros(tdx.tdx_trace_size(grid, items, 0) // 4, dtype=torch.int32, device="cuda")
    case = RSCase(inp, opts=opts(num_sms=grid, cluster=cluster, block_n=256, reduce_mode=rm, trace=trace))
    tdx.check(case.run())
    status_ok(case)
    assert_within_tol(case.result(), case.oracle(), "bf16")
    paired = case.result_bits()
    tr = trace.cpu().numpy().astype(np.uint32)
    taken = trace_items(tr, grid, 0, cl=2)
    check_each_item_once(taken, plan["L"], plan["T"])
    check_rs_fold_order(taken, 4, plan["T"])
    single = RSCase(inp, opts=opts(cluster=1, block_n=256, reduce_mode=rm))
    tdx.check(single.run())
    status_ok(single)
    assert np.array_equal(single.result_bits(), paired)


def test_rs_many_n_tiles_trace():
    # 20 N-tiles of 128 per rank: whatever raster the kernel takes inside a rank, every (rank, tile)
    # is computed once and every tile's ranks come in the fold order 0..W-1
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], W=2, M=256, K=128, N=2560)
    inp = wls.make_inputs(wl, integer=True)
    grid = 6
    o = opts(num_sms=grid, block_n=128, reduce_mode=1, cluster=1)
    plan = tdx.tdx_plan_info(tdx.OP_RS, 2, 256, 128, 2560, tdx.TDX_BF16, o)
    assert plan["tiles_n"] == 20
    items = plan["L"] * plan["T"]
    trace = torch.zeros(tdx.tdx_trace_size(grid, items, 0) // 4, dtype=torch.int32, device="cuda")
    case = RSCase(inp, opts=opts(num_sms=grid, block_n=128, reduce_mode=1, cluster=1, trace=trace))
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    taken = trace_items(trace.cpu().numpy().astype(np.uint32), grid, 0)
    check_each_item_once(taken, plan["L"], plan["T"])
    check_rs_fold_order(taken, 2, plan["T"])


@pytest.mark.parametrize("variant", [dict(), dict(reduce_mode=1), dict(reduce_mode=2, block_n=256),
                                     dict(cluster=3, block_n=256, reduce_mode=1)])
@pytest.mark.parametrize("integer", [True, False])
def test_rs_e4m3(variant, integer):
    wl = wls.with_shape(wls.WORKLOADS["rs_fp8_w8"], W=4, M=512, K=1024, N=1024)
    inp = wls.make_inputs(wl, integer=integer)
    o = opts(scale_a=inp.scale_a, scale_b=inp.scale_b, **variant)
    case = RSCase(inp, opts=o)
    tdx.check(case.run())
    status_ok(case)
    if integer:
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    else:
        assert_within_tol(case.result(), case.oracle(), "e4m3")


@pytest.mark.parametrize("integer", [True, False])
def test_rs_e4m3_full_size_full_output_and_deterministic(integer):
    wl = wls.WORKLOADS["rs_fp8_w8"]
    inp = wls.make_inputs(wl, integer=integer)
    case = RSCase(inp, opts=opts(scale_a=inp.scale_a, scale_b=inp.scale_b))
    tdx.check(case.run())
    status_ok(case)
    first = case.result_bits()
    want = case.oracle()
    assert want.shape == first.shape == (wl.M, wl.N)
    if integer:
        assert_bit_exact(first, want, "bf16")
    else:
        assert_within_tol(R.decode_bf16(first), want, "e4m3")
    tdx.check(case.run(opts(scale_a=inp.scale_a, scale_b=inp.scale_b, perturb_seed=3)))
    assert np.array_equal(case.result_bits(), first)


# ------------------------------------------------------------------ bf16 partials


@pytest.mark.parametrize("shape", [
    dict(W=2, M=256, K=256, N=512),
    dict(W=3, M=384, K=200, N=136),
    dict(W=4, M=200, K=64, N=264),
    dict(W=8, M=1024, K=512, N=1024),
])
@pytest.mark.parametrize("integer", [True, False])
def test_rs_bf16_partials(shape, integer):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    for bn in (0, 256):
        case = RSCase(inp, opts=opts(bf16_partials=1, block_n=bn))
        plan = tdx.tdx_plan_info(tdx.OP_RS, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, case.opts)
        assert plan["partial_bytes"] == 2 and plan["reduce_mode"] == 2
        tdx.check(case.run())
        status_ok(case)
        want = case.oracle(partials="bf16")
        if integer:
            assert_bit_exact(case.result_bits(), want, "bf16")
        else:
            assert_within_tol(case.result(), want, "bf16")
            # the rounded partials stay close to the fp32-partial result too
            assert_within_tol(case.result(), case.oracle(), "bf16")


def test_rs_bf16_partial_slots_hold_rounded_partials():
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], W=4, M=512, K=1024, N=512)
    inp = wls.make_inputs(wl, integer=True)      # partials up to 16384: many need rounding in bf16
    o = opts(bf16_partials=1, block_n=128, epoch=4)
    plan = tdx.tdx_plan_info(tdx.OP_RS, 4, 512, 1024, 512, tdx.TDX_BF16, o)
    case = RSCase(inp, opts=o)
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(partials="bf16"), "bf16")
    T, BN = plan["T"], plan["BN"]
    S = case.ws[plan["off_S"]:plan["off_S"] + 2 * 4 * T * 128 * BN].view(torch.int16).cpu().numpy().view(np.uint16)
    for r in (0, 3):
        P = R.gemm_rs_rows([inp.a[r]], [inp.b[r]], np.arange(512), "bf16")
        want = R.round_bf16_rne(P)
        for (mt, nt) in [(0, 0), (3, 2)]:
            tile = mt * plan["tiles_n"] + nt
            blk = S[(r * T + tile) * 128 * BN:(r * T + tile + 1) * 128 * BN]
            # layout: ((cc*4 + j)*128 + i)*8 + t  ->  element (i, 32*cc + 8*j + t)
            blk = blk.reshape(BN // 32, 4, 128, 8).transpose(2, 0, 1, 3).reshape(128, BN)
            assert np.array_equal(blk, want[mt * 128:(mt + 1) * 128, nt * BN:(nt + 1) * BN])


def test_rs_bf16_partials_full_size_sampled_and_deterministic():
    wl = wls.WORKLOADS["rs_w8"]
    inp = wls.make_inputs(wl, integer=False)
    case = RSCase(inp, opts=opts(bf16_partials=1))
    tdx.check(case.run())
    status_ok(case)
    rows = sample_rows(wl.M, wl.M // wl.W)
    first = case.result_bits()
    assert_within_tol(R.decode_bf16(first[rows]), case.oracle(rows, partials="bf16"), "bf16")
    for o in case.out:
        o.fill_(float("nan"))
    tdx.check(case.run(opts(bf16_partials=1, perturb_seed=21)))
    status_ok(case)
    assert np.array_equal(case.result_bits(), first)


def test_rs_e4m3_bf16_partials():
    wl = wls.with_shape(wls.WORKLOADS["rs_fp8_w8"], W=4, M=512, K=1024, N=1024)
    inp = wls.make_inputs(wl, integer=True)
    case = RSCase(inp, opts=opts(scale_a=inp.scale_a, scale_b=inp.scale_b, bf16_partials=1))
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(partials="bf16"), "bf16")


@pytest.mark.parametrize("variant", [dict(reduce_mode=1), dict(reduce_mode=2)])
@pytest.mark.parametrize("shape", [dict(W=4, M=512, K=512, N=1024), dict(W=3, M=768, K=256, N=1344)])
def test_rs_wide_tiles(variant, shape):
    wl = wls.with_shape(wls.WORKLOADS["rs_w8"], **shape)
    for integer in (True, False):
        inp = wls.make_inputs(wl, integer=integer)
        bits = []
        for bn in (512, 256):
            case = RSCase(inp, opts=opts(cluster=3, block_n=bn, perturb_seed=5, **variant))
            tdx.check(case.run())
            status_ok(case)
            bits.append(case.result_bits())
            if integer:
                assert_bit_exact(bits[-1], case.oracle(), "bf16")
            else:
                assert_within_tol(case.result(), case.oracle(), "bf16")
        assert np.array_equal(bits[0], bits[1])


@pytest.mark.parametrize("integer", [True, False])
def test_rs_e4m3_wide_tiles(integer):
    wl = wls.with_shape(wls.WORKLOADS["rs_fp8_w8"], W=4, M=512, K=1024, N=1024)
    inp = wls.make_inputs(wl, integer=integer)
    case = RSCase(inp, opts=opts(scale_a=inp.scale_a, scale_b=inp.scale_b, cluster=3, block_n=512))
    tdx.check(case.run())
    status_ok(case)
    if integer:
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    else:
        assert_within_tol(case.result(), case.oracle(), "e4m3")
