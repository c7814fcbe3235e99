"""AllGather+GEMM on the GPU through the C ABI, element by element against the CPU oracle.

Integer inputs (U{-4..4}, scales 1) must match the oracle's single rounding of the exact sum bit
for bit; random inputs must satisfy max|gpu - oracle| <= 1e-2 * max|oracle| (bf16) or 4e-2 (e4m3),
the bound applied to the fp64 oracle before rounding.
"""
import numpy as np
import pytest
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import reference as R
import workloads as wls
from gpu_util import (AGCase, assert_bit_exact, dev_bits, dtype_code, assert_within_tol, check_ag_consumer_order,
                      check_each_item_once, host_bits, sample_rows, trace_items, trace_phases,
                      trace_releases)

pytestmark = pytest.mark.gpu

TMO = int(5e8)   # 0.5 s bound on every device wait in these tests


def opts(**kw):
    return tdx.make_opts(timeout_ns=TMO, **kw)


def status_ok(case):
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_OK, (tdx.tdx_status_string(st), detail)


def gathered(case, plan):
    g = case.ws[plan["off_G"]:plan["off_G"] + case.W * case.M_local * case.K * (1 if case.dt else 2)]
    return g


TINY = wls.WORKLOADS["ag_tiny"]


@pytest.mark.parametrize("variant", [
    {}, {"split_k": 1, "block_n": 256}, {"split_k": 1, "block_n": 128}, {"split_k": 1, "block_n": 64},
    {"self_rank": 1}, {"split_k": 2, "block_n": 256}, {"perturb_seed": 7}, {"split_k": 2, "reduce_mode": 1},
])
def test_ag_tiny_integer_bit_exact(variant):
    inp = wls.make_inputs(TINY, integer=True)
    o = opts(chunk_rows=32, out_dtype=tdx.TDX_FP32, **variant)
    case = AGCase(inp, out_dtype="fp32", opts=o)
    tdx.check(case.run(), "ag tiny")
    assert_bit_exact(case.C.cpu().numpy(), case.oracle(), "fp32")
    status_ok(case)
    plan = tdx.tdx_plan_info(tdx.OP_AG, 2, 64, 128, 256, tdx.TDX_BF16, o)
    g = gathered(case, plan)
    assert torch.equal(g, torch.cat(case.shards).view(torch.uint8).flatten())
    flags = case.ws[plan["off_chunk_flags"]:plan["off_chunk_flags"] + 4 * 2 * plan["n_chunks"]].view(torch.int32)
    assert np.array_equal(flags.cpu().numpy().astype(np.uint32), R.expected_flags(2 * plan["n_chunks"], 1))


def test_ag_tiny_random_within_tolerance():
    inp = wls.make_inputs(TINY, integer=False)
    case = AGCase(inp, out_dtype="fp32", opts=opts(chunk_rows=32, out_dtype=tdx.TDX_FP32))
    tdx.check(case.run())
    got = case.result()
    rel = assert_within_tol(got, case.oracle(), "bf16")
    assert rel < 1e-5   # fp32 output of an fp32-accumulated 128-term sum


@pytest.mark.parametrize("name", ["ag_w8", "ag_fp8_w8"])
@pytest.mark.parametrize("integer", [True, False])
def test_ag_full_size_full_output(name, integer):
    # the headline shapes, every element of C against the full fp64 oracle
    wl = wls.WORKLOADS[name]
    inp = wls.make_inputs(wl, integer=integer)
    o = opts(scale_a=inp.scale_a, scale_b=inp.scale_b[0]) if wl.dtype == "e4m3" else opts()
    case = AGCase(inp, opts=o)
    tdx.check(case.run(), name)
    status_ok(case)
    got_bits = case.result_bits()
    want = case.oracle()
    assert want.shape == got_bits.shape == (wl.W * wl.M, wl.N)
    if integer:
        assert_bit_exact(got_bits, want, "bf16")
    else:
        assert_within_tol(R.decode_bf16(got_bits), want, wl.dtype)
    plan = tdx.tdx_plan_info(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, case.dt, case.opts)
    assert torch.equal(gathered(case, plan), torch.cat(case.shards).view(torch.uint8).flatten())


@pytest.mark.parametrize("integer", [True, False])
def test_ag_small_m_full_output(integer):
    wl = wls.WORKLOADS["ag_small"]
    inp = wls.make_inputs(wl, integer=integer)
    case = AGCase(inp, opts=opts())
    tdx.check(case.run())
    status_ok(case)
    if integer:
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    else:
        assert_within_tol(case.result(), case.oracle(), "bf16")


@pytest.mark.parametrize("shape", [
    dict(W=3, M=96, K=320, N=200, chunk_rows=32),     # tiles span ranks, ragged K and N
    dict(W=1, M=200, K=136, N=264, chunk_rows=40),    # one rank, ragged M tile
    dict(W=5, M=64, K=1024, N=72, chunk_rows=16),
    dict(W=16, M=8, K=64, N=128, chunk_rows=8),       # maximum W
])
@pytest.mark.parametrize("integer", [True, False])
def test_ag_ragged_shapes(shape, integer):
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    for variant in [{}, {"split_k": 1}, {"split_k": 3, "block_n": 128, "reduce_mode": 1},
                    {"split_k": 4, "block_n": 256, "reduce_mode": 2}]:
        case = AGCase(inp, opts=opts(chunk_rows=shape["chunk_rows"], **variant))
        tdx.check(case.run(), str(variant))
        status_ok(case)
        if integer:
            assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
        else:
            assert_within_tol(case.result(), case.oracle(), "bf16")


def test_ag_fp8_ragged_and_scales():
    wl = wls.with_shape(wls.WORKLOADS["ag_fp8_w8"], W=3, M=128, K=384, N=384, chunk_rows=64)
    inp = wls.make_inputs(wl, integer=False)
    case = AGCase(inp, opts=opts(chunk_rows=64, scale_a=inp.scale_a, scale_b=inp.scale_b[0]))
    tdx.check(case.run())
    status_ok(case)
    assert_within_tol(case.result(), case.oracle(), "e4m3")


@pytest.mark.parametrize("self_rank", [0, 3, 7])
@pytest.mark.parametrize("grid", [1, 16])
def test_ag_trace_follows_the_oracle_orders(self_rank, grid):
    """Bookkeeping against what the method fixes: every (split, tile) is computed exactly once, the
    consumer takes the ranks' rows in the arrival order self, self+1, ... (in whatever raster inside
    a rank), and the producer releases every chunk exactly once; with one CTA (a single producer
    thread) the release sequence is exactly the oracle's release order."""
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=8, M=256, K=512, N=512, chunk_rows=128)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(self_rank=self_rank, num_sms=grid)
    plan = tdx.tdx_plan_info(tdx.OP_AG, 8, 256, 512, 512, tdx.TDX_BF16, o)
    items = plan["L"] * plan["T"]
    chunks = 8 * plan["n_chunks"]
    trace = torch.zeros(tdx.tdx_trace_size(grid, items, chunks) // 4, dtype=torch.int32, device="cuda")
    case = AGCase(inp, opts=opts(self_rank=self_rank, num_sms=grid, trace=trace))
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    tr = trace.cpu().numpy().astype(np.uint32)
    assert list(tr[:4]) == [grid, items, plan["L"], plan["T"]]
    taken = trace_items(tr, grid, chunks)
    check_each_item_once(taken, plan["L"], plan["T"])
    check_ag_consumer_order(taken, plan["L"], plan["tiles_n"], 8, 256, self_rank)
    rel = trace_releases(tr, grid, chunks)
    want = [r * plan["n_chunks"] + c for r, c in R.ag_chunk_release_order(8, 256, 128, self_rank)]
    assert sorted(rel) == list(range(chunks))
    if grid == 1:
        assert rel == want
    # phase stamps in order (entry, set-up, first item's loads issued, its MMAs issued, last MMA
    # completed, items done, epilogue done; two roles that see the same completion may stamp a
    # little apart, hence the 2 us allowance), all within the call
    ph = trace_phases(tr, grid)
    busy = tr[4 + 3:4 + 12 * grid:12] > 0
    assert busy.any()
    for a, b in zip(range(6), range(1, 7)):
        assert np.all(ph[busy, a] <= ph[busy, b] + 2000), (a, ph[busy][:4])
    assert np.all(ph[:, 6] < 10 ** 9)


def test_ag_modes_and_epochs():
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=4, M=256, K=512, N=768, chunk_rows=64)
    inp = wls.make_inputs(wl, integer=True)
    case = AGCase(inp, opts=opts(chunk_rows=64))
    want = R.round_out(case.oracle(), "bf16")
    # epoch mode: strictly increasing epochs, no clearing between calls
    for e in (5, 6, 9):
        case.C.fill_(float("nan"))
        tdx.check(case.run(opts(chunk_rows=64, epoch=e)))
        assert np.array_equal(case.result_bits(), want)
        plan = tdx.tdx_plan_info(tdx.OP_AG, 4, 256, 512, 768, tdx.TDX_BF16, case.opts)
        n = 4 * plan["n_chunks"]
        f = case.ws[plan["off_chunk_flags"]:plan["off_chunk_flags"] + 4 * n].view(torch.int32).cpu().numpy()
        assert np.array_equal(f.astype(np.uint32), R.expected_flags(n, e))
        status_ok(case)
    # GEMM_ONLY reads the already gathered buffer
    case.C.fill_(float("nan"))
    tdx.check(case.run(opts(chunk_rows=64, mode=tdx.TDX_GEMM_ONLY)))
    assert np.array_equal(case.result_bits(), want)
    # MOVE_ONLY gathers and leaves C alone
    plan = tdx.tdx_plan_info(tdx.OP_AG, 4, 256, 512, 768, tdx.TDX_BF16, case.opts)
    case.ws[plan["off_G"]:plan["off_G"] + 4 * 256 * 512 * 2].zero_()
    case.C.fill_(0.0)
    tdx.check(case.run(opts(chunk_rows=64, mode=tdx.TDX_MOVE_ONLY)))
    torch.cuda.synchronize()
    assert torch.equal(gathered(case, plan), torch.cat(case.shards).view(torch.uint8).flatten())
    assert int(torch.count_nonzero(case.C)) == 0
    status_ok(case)


def test_ag_device_epochs_eager_and_graph():
    # epochs kept in the workspace: no flag clearing between calls, and a captured call replays
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=4, M=256, K=512, N=768, chunk_rows=64)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(chunk_rows=64, epoch=tdx.TDX_EPOCH_DEVICE)
    case = AGCase(inp, opts=o)
    want = R.round_out(case.oracle(), "bf16")
    plan = tdx.tdx_plan_info(tdx.OP_AG, 4, 256, 512, 768, tdx.TDX_BF16, o)
    n = 4 * plan["n_chunks"]
    for call in range(1, 4):
        case.C.fill_(float("nan"))
        tdx.check(case.run())
        assert np.array_equal(case.result_bits(), want)
        status_ok(case)
        assert int(case.ws[64:68].view(torch.int32).item()) == call          # header word 16
        assert int(case.ws[68:72].view(torch.int32).item()) == 0             # start count, reset
        f = case.ws[plan["off_chunk_flags"]:plan["off_chunk_flags"] + 4 * n].view(torch.int32).cpu().numpy()
        assert np.array_equal(f.astype(np.uint32), R.expected_flags(n, call))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            tdx.check(tdx.tdx_ag_gemm(case.shards, case.B, case.C, case.ws, 4, 256, 512, 768, tdx.TDX_BF16, o,
                                      stream=s))
    torch.cuda.synchronize()
    for rep in range(3):
        case.C.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(case.result_bits(), want)
    status_ok(case)
    assert int(case.ws[64:68].view(torch.int32).item()) == 3 + 2 * 3


@pytest.mark.parametrize("shape", [dict(W=8, M=16, K=2048, N=512, chunk_rows=16),      # pull tiles, K splits
                                   dict(W=4, M=256, K=512, N=1024, chunk_rows=128)])  # 2-SM pairs
def test_ag_device_epochs_across_modes(shape):
    # every call advances the kept epoch by one whatever its mode (movement alone, GEMM alone on the
    # gathered buffer it left, fused), and the count of CTAs that read the epoch is back to zero
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], **shape)
    inp = wls.make_inputs(wl, integer=True)
    case = AGCase(inp, opts=opts(chunk_rows=wl.chunk_rows))
    want = R.round_out(case.oracle(), "bf16")
    modes = [tdx.TDX_MOVE_ONLY, tdx.TDX_GEMM_ONLY, tdx.TDX_FUSED, tdx.TDX_FUSED, tdx.TDX_MOVE_ONLY, tdx.TDX_FUSED]
    for call, mode in enumerate(modes, start=1):
        case.C.fill_(float("nan"))
        tdx.check(case.run(opts(chunk_rows=wl.chunk_rows, epoch=tdx.TDX_EPOCH_DEVICE, mode=mode)))
        torch.cuda.synchronize()
        status_ok(case)
        assert int(case.ws[64:68].view(torch.int32).item()) == call
        assert int(case.ws[68:72].view(torch.int32).item()) == 0
        if mode != tdx.TDX_MOVE_ONLY:
            assert np.array_equal(case.result_bits(), want), f"call {call}"


@pytest.mark.parametrize("shape2", [dict(M=64, N=128), dict(M=16, N=512)])
def test_ag_chained_calls_read_the_previous_output(shape2):
    # two calls queued back to back on one stream, the second gathering the first one's output rows
    # as its shards: the second kernel may start its set-up while the first still runs (programmatic
    # dependent launch) and must read the first's finished output (bit-exact on integers; every
    # value stays exact in bf16 and in the fp32 accumulation)
    wl1 = wls.with_shape(wls.WORKLOADS["ag_w8"], W=2, M=64, K=128, N=256, chunk_rows=64)
    inp1 = wls.make_inputs(wl1, integer=True)
    first = AGCase(inp1, opts=opts(chunk_rows=64))
    W2, M2, N2 = 128 // shape2["M"], shape2["M"], shape2["N"]
    wl2 = wls.with_shape(wls.WORKLOADS["ag_w8"], W=W2, M=M2, K=256, N=N2, chunk_rows=M2)
    b2 = wls.make_inputs(wl2, integer=True).b[0]
    B2 = dev_bits(b2)
    C2 = torch.full((128, N2), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws2 = torch.zeros(tdx.tdx_workspace_size(tdx.OP_AG, W2, M2, 256, N2, tdx.TDX_BF16, opts(chunk_rows=M2)),
                      dtype=torch.uint8, device="cuda")
    shards2 = [first.C[r * M2:(r + 1) * M2] for r in range(W2)]   # views into the first call's output
    for rep in range(3):
        first.C.fill_(float("nan"))
        C2.fill_(float("nan"))
        tdx.check(first.run(opts(chunk_rows=64, epoch=rep + 1)))
        tdx.check(tdx.tdx_ag_gemm(shards2, B2, C2, ws2, W2, M2, 256, N2, tdx.TDX_BF16,
                                  opts(chunk_rows=M2, epoch=rep + 1)))
        torch.cuda.synchronize()
        status_ok(first)
        c1 = R.round_out(first.oracle(), "bf16")
        assert np.array_equal(first.result_bits(), c1)
        want = R.round_out(R.ag_gemm([c1[r * M2:(r + 1) * M2] for r in range(W2)], b2, "bf16"), "bf16")
        assert np.array_equal(host_bits(C2), want), f"rep {rep}"


@pytest.mark.parametrize("self_rank", [0, 5])
@pytest.mark.parametrize("perturb", [0, 9])
def test_ag_first_wave_chunks_through_the_operand_ring(self_rank, perturb):
    # 16 CTAs: the first wave holds the self rank's 8 tiles and 8 tiles of the next rank, whose CTAs
    # copy that rank's chunks through their operand ring before loading operands into it (delays
    # injected into both copy phases with perturb); exact result, every chunk released once
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=8, M=256, K=512, N=1024, chunk_rows=64)
    inp = wls.make_inputs(wl, integer=True)
    o = opts(self_rank=self_rank, num_sms=16, chunk_rows=64, block_n=256, cluster=1)
    plan = tdx.tdx_plan_info(tdx.OP_AG, 8, 256, 512, 1024, tdx.TDX_BF16, o)
    assert plan["cluster"] == 1 and plan["BN"] == 256 and plan["L"] == 1 and plan["T"] == 64
    items, chunks = plan["T"], 8 * plan["n_chunks"]
    trace = torch.zeros(tdx.tdx_trace_size(16, items, chunks) // 4, dtype=torch.int32, device="cuda")
    case = AGCase(inp, opts=o)
    want = R.round_out(case.oracle(), "bf16")
    for call in range(2):
        trace.zero_()
        case.C.fill_(float("nan"))
        tdx.check(case.run(opts(self_rank=self_rank, num_sms=16, chunk_rows=64, block_n=256, cluster=1,
                                epoch=call + 1, perturb_seed=perturb + call if perturb else 0, trace=trace)))
        status_ok(case)
        assert np.array_equal(case.result_bits(), want)
        tr = trace.cpu().numpy().astype(np.uint32)
        assert sorted(trace_releases(tr, 16, chunks)) == list(range(chunks))
        check_each_item_once(trace_items(tr, 16, chunks), 1, plan["T"])
        n = chunks
        f = case.ws[plan["off_chunk_flags"]:plan["off_chunk_flags"] + 4 * n].view(torch.int32).cpu().numpy()
        assert np.array_equal(f.astype(np.uint32), R.expected_flags(n, call + 1))
        cnt = case.ws[plan["off_chunk_cnt"]:plan["off_chunk_cnt"] + 4 * n].view(torch.int32).cpu().numpy()
        assert not cnt.any()   # the completing copy reset every chunk's count


def test_ag_degenerate_sizes():
    # K == 0: C = 0 (empty sums); M_local == 0 and N == 0: nothing to do
    B = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    shards = [torch.zeros((64, 0), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    C = torch.full((128, 256), 3.0, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    # zero-size tensors may share address 0; pass aligned dummy pointers instead
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    tdx.check(tdx.tdx_ag_gemm([dummy, dummy], dummy, C, ws, 2, 64, 0, 256, tdx.TDX_BF16, opts()))
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(C)) == 0
    C2 = torch.full((4, 4), 3.0, dtype=torch.bfloat16, device="cuda")
    assert tdx.tdx_ag_gemm([dummy], dummy, C2, ws, 1, 0, 128, 256, tdx.TDX_BF16, opts()) == tdx.TDX_OK
    assert tdx.tdx_ag_gemm([dummy], dummy, C2, ws, 1, 4, 128, 0, tdx.TDX_BF16, opts()) == tdx.TDX_OK
    torch.cuda.synchronize()
    assert float(C2.float().sum()) == 48.0
    del B, shards


def test_ag_timeout_is_reported_and_workspace_recovers():
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=4, M=256, K=256, N=256, chunk_rows=128)
    inp = wls.make_inputs(wl, integer=True)
    case = AGCase(inp, opts=opts())
    # no producer releases the flags: every remote tile's wait must run out (2 ms) and report
    tdx.check(case.run(tdx.make_opts(mode=tdx.TDX_CONSUMER_ONLY, timeout_ns=2_000_000)))
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_ERR_TIMEOUT and detail[1] == 1
    # after re-initialising the workspace a normal call succeeds
    tdx.check(tdx.tdx_workspace_init(case.ws))
    tdx.check(case.run(opts()))
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")


def test_ag_stale_epoch_is_reported():
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=4, M=256, K=256, N=256, chunk_rows=128)
    inp = wls.make_inputs(wl, integer=True)
    case = AGCase(inp, opts=opts())
    tdx.check(case.run(opts(epoch=10)))
    status_ok(case)
    tdx.check(case.run(tdx.make_opts(epoch=5, timeout_ns=2_000_000)))
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_ERR_STALE_EPOCH
    assert detail[4] == 10 and detail[5] == 5


def test_ag_split_k_chained_and_slotted_identical():
    wl = wls.WORKLOADS["ag_small"]
    inp = wls.make_inputs(wl, integer=False)
    bits = []
    for rm in (1, 2):
        case = AGCase(inp, opts=opts(reduce_mode=rm, perturb_seed=5))
        tdx.check(case.run())
        status_ok(case)
        bits.append(case.result_bits())
    assert np.array_equal(bits[0], bits[1])


@pytest.mark.parametrize("self_rank", [0, 5])
def test_ag_pairs_parity_and_trace(self_rank):
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=8, M=256, K=1024, N=768, chunk_rows=128)
    inp = wls.make_inputs(wl, integer=True)
    grid = 16
    o = opts(self_rank=self_rank, num_sms=grid, cluster=3, block_n=256)
    plan = tdx.tdx_plan_info(tdx.OP_AG, 8, 256, 1024, 768, tdx.TDX_BF16, o)
    assert plan["cluster"] == 3 and plan["BN"] == 256
    items = plan["L"] * plan["T"]
    chunks = 8 * plan["n_chunks"]
    trace = torch.zeros(tdx.tdx_trace_size(grid, items, chunks) // 4, dtype=torch.int32, device="cuda")
    case = AGCase(inp, opts=opts(self_rank=self_rank, num_sms=grid, cluster=3, block_n=256, trace=trace))
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    tr = trace.cpu().numpy().astype(np.uint32)
    taken = trace_items(tr, grid, chunks, cl=2)
    check_each_item_once(taken, plan["L"], plan["T"])
    # the two CTAs of a pair take vertically adjacent tiles of the same N-tile
    for it in {k[0] for k in taken}:
        (c0, t0), (c1, t1) = taken[(it, 0)], taken[(it, 1)]
        assert c0 == c1 and t1 == t0 + plan["tiles_n"]
    check_ag_consumer_order(taken, plan["L"], plan["tiles_n"], 8, 256, self_rank)
    assert sorted(trace_releases(tr, grid, chunks)) == list(range(chunks))


@pytest.mark.parametrize("name", ["ag_w8", "ag_fp8_w8"])
def test_ag_pairs_and_singles_give_identical_bits(name):
    wl = wls.with_shape(wls.WORKLOADS[name], W=4, M=256, K=1024, N=512, chunk_rows=128)
    inp = wls.make_inputs(wl, integer=False)
    bits = []
    for cl in (1, 3):
        kw = dict(cluster=cl, block_n=256)
        if wl.dtype == "e4m3":
            kw.update(scale_a=inp.scale_a, scale_b=inp.scale_b[0])
        case = AGCase(inp, opts=opts(**kw))
        tdx.check(case.run())
        status_ok(case)
        bits.append(case.result_bits())
        assert_within_tol(case.result(), case.oracle(), wl.dtype)
    assert np.array_equal(bits[0], bits[1])


@pytest.mark.parametrize("cluster", [3])
def test_ag_pairs_timeout_recovers(cluster):
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], W=4, M=256, K=256, N=512, chunk_rows=128)
    inp = wls.make_inputs(wl, integer=True)
    case = AGCase(inp, opts=opts(cluster=cluster, block_n=256))
    tdx.check(case.run(tdx.make_opts(mode=tdx.TDX_CONSUMER_ONLY, timeout_ns=2_000_000, cluster=cluster,
                                     block_n=256)))
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_ERR_TIMEOUT and detail[1] == 1
    tdx.check(tdx.tdx_workspace_init(case.ws))
    tdx.check(case.run(opts(cluster=cluster, block_n=256)))
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")


def test_ag_small_shards_pull_and_flag_paths_agree():
    # shards smaller than a tile: tiles read A straight from the shards (pull), while the gathered
    # copy still completes G and releases every flag; a 96-row shard (not a divisor of 128) takes
    # the flag-waiting path. Both match the oracle bit for bit on integers.
    for shape, chunk in ((dict(W=8, M=16, K=2048, N=512), 16), (dict(W=4, M=96, K=512, N=512), 32)):
        wl = wls.with_shape(wls.WORKLOADS["ag_w8"], chunk_rows=chunk, **shape)
        inp = wls.make_inputs(wl, integer=True)
        o = opts(chunk_rows=chunk, epoch=4)
        plan = tdx.tdx_plan_info(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, tdx.TDX_BF16, o)
        assert plan["pull_a"] == (1 if wl.M == 16 else 0)
        case = AGCase(inp, opts=o)
        tdx.check(case.run())
        status_ok(case)
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
        assert torch.equal(gathered(case, plan), torch.cat(case.shards).view(torch.uint8).flatten())
        n = wl.W * plan["n_chunks"]
        f = case.ws[plan["off_chunk_flags"]:plan["off_chunk_flags"] + 4 * n].view(torch.int32).cpu().numpy()
        assert np.array_equal(f.astype(np.uint32), R.expected_flags(n, 4))


@pytest.mark.parametrize("layout", ["stacked", "scattered", "reversed"])
@pytest.mark.parametrize("shape", [
    dict(W=8, M=16, K=2048, N=512, dtype="bf16"),     # 8 shards per tile; B in one box per K slice
    dict(W=4, M=16, K=1024, N=200, dtype="bf16"),     # 4 of 8 shard rows exist; ragged N: 2D B boxes
    dict(W=16, M=8, K=512, N=256, dtype="bf16"),      # 16 shards per tile
    dict(W=2, M=32, K=704, N=384, dtype="e4m3"),      # e4m3, ragged K, 2 of 4 shard rows
    dict(W=8, M=16, K=200, N=320, dtype="bf16"),      # ragged K; the last tile's second column
                                                      # group lies past N (zero-filled)
])
def test_ag_pull_tiles_over_shard_layouts(shape, layout):
    # pull tiles read a tile's shards as one 3D box when the shards sit at one stride (stacked) and
    # shard by shard otherwise (uneven gaps, or descending addresses); both match the oracle bit for
    # bit, and so does the gathered copy
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], chunk_rows=shape["M"], **shape)
    inp = wls.make_inputs(wl, integer=True)
    kw = dict(scale_a=inp.scale_a, scale_b=inp.scale_b[0]) if wl.dtype == "e4m3" else {}
    o = opts(chunk_rows=wl.M, **kw)
    plan = tdx.tdx_plan_info(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, dtype_code(wl.dtype), o)
    assert plan["pull_a"] == 1
    case = AGCase(inp, opts=o, layout=layout)
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    assert torch.equal(gathered(case, plan), torch.cat([s.view(torch.uint8).flatten() for s in case.shards]))


@pytest.mark.parametrize("shape,extra", [
    (dict(W=3, M=256, K=320, N=384, dtype="bf16"), {}),                # B: one box per K slice
    (dict(W=3, M=256, K=320, N=392, dtype="bf16"), {}),                # ragged N: 2D B boxes
    (dict(W=4, M=256, K=512, N=640, dtype="bf16"), {"block_n": 256}),  # 4 groups; last tile half past N
    (dict(W=2, M=128, K=1024, N=1024, dtype="e4m3"), {}),              # e4m3: 128-column groups
])
def test_ag_single_cta_b_column_groups(shape, extra):
    # single-CTA tiles that wait on chunk flags load a K slice of B across the tile width as one 3D
    # box when N is whole 128-byte column groups (2D boxes otherwise); bit-exact on integers
    wl = wls.with_shape(wls.WORKLOADS["ag_w8"], chunk_rows=128, **shape)
    inp = wls.make_inputs(wl, integer=True)
    kw = dict(scale_a=inp.scale_a, scale_b=inp.scale_b[0]) if wl.dtype == "e4m3" else {}
    o = opts(chunk_rows=128, **kw, **extra)
    plan = tdx.tdx_plan_info(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, dtype_code(wl.dtype), o)
    assert plan["cluster"] == 1 and plan["pull_a"] == 0
    case = AGCase(inp, opts=o)
    tdx.check(case.run())
    status_ok(case)
    assert_bit_exact(case.result_bits(), case.oracle(), "bf16")


@pytest.mark.parametrize("integer", [True, False])
def test_ag_split_k_grid_fold(integer):
    # split-K items over several waves of a small grid, folded by every CTA after a grid barrier
    wl = wls.with_shape(wls.WORKLOADS["ag_small"], W=8, M=16, K=4096, N=512)
    inp = wls.make_inputs(wl, integer=integer)
    o = opts(chunk_rows=16, split_k=8, reduce_mode=3, num_sms=6)
    assert tdx.tdx_plan_info(tdx.OP_AG, 8, 16, 4096, 512, tdx.TDX_BF16, o)["coop_fold"] == 2
    case = AGCase(inp, opts=o)
    tdx.check(case.run())
    status_ok(case)
    if integer:
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    else:
        assert_within_tol(case.result(), case.oracle(), "bf16")
    first = case.result_bits()
    case.C.fill_(float("nan"))
    tdx.check(case.run(opts(chunk_rows=16, split_k=8, reduce_mode=3, num_sms=6, epoch=5, perturb_seed=2)))
    status_ok(case)
    assert np.array_equal(case.result_bits(), first)


@pytest.mark.parametrize("integer", [True, False])
def test_ag_split_k_cooperative_fold(integer):
    # one wave of split-K work items: every element of a tile folds 1/L of it after all L arrived
    wl = wls.with_shape(wls.WORKLOADS["ag_small"], W=8, M=16, K=4096, N=512)
    inp = wls.make_inputs(wl, integer=integer)
    o = tdx.make_opts(timeout_ns=int(5e8), chunk_rows=16, split_k=8)
    plan = tdx.tdx_plan_info(tdx.OP_AG, 8, 16, 4096, 512, tdx.TDX_BF16, o)
    assert plan["L"] == 8 and plan["reduce_mode"] == 2
    case = AGCase(inp, opts=o)
    tdx.check(case.run())
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_OK, detail
    assert tdx.tdx_plan_info(tdx.OP_AG, 8, 16, 4096, 512, tdx.TDX_BF16, o)["coop_fold"] == 1
    if integer:
        assert_bit_exact(case.result_bits(), case.oracle(), "bf16")
    else:
        assert_within_tol(case.result(), case.oracle(), "bf16")
    # counters are back to zero: a second call with the next epoch gives the same bits
    first = case.result_bits()
    case.C.fill_(float("nan"))
    tdx.check(case.run(tdx.make_opts(timeout_ns=int(5e8), chunk_rows=16, split_k=8, epoch=2, perturb_seed=5)))
    assert np.array_equal(case.result_bits(), first)


@pytest.mark.parametrize("name", ["ag_w8", "ag_fp8_w8"])
@pytest.mark.parametrize("shape", [dict(W=4, M=256, K=1024, N=1024), dict(W=2, M=384, K=512, N=1344)])
def test_ag_wide_tiles(name, shape):
    # 512-column tiles on 2-SM pairs (two MMAs per K step into one 512-column accumulator): exact on
    # integers, and the same bits as 256-column pairs on random inputs (ragged N included; one K
    # split for both, since the library would split K differently for the two tile counts)
    wl = wls.with_shape(wls.WORKLOADS[name], chunk_rows=128, **shape)
    for integer in (True, False):
        inp = wls.make_inputs(wl, integer=integer)
        kw = dict(scale_a=inp.scale_a, scale_b=inp.scale_b[0]) if wl.dtype == "e4m3" else {}
        bits = []
        for bn in (512, 256):
            o = opts(cluster=3, block_n=bn, split_k=1, **kw)
            assert tdx.tdx_plan_info(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, 1 if wl.dtype == "e4m3" else 0, o)["BN"] == bn
            case = AGCase(inp, opts=o)
            tdx.check(case.run())
            status_ok(case)
            bits.append(case.result_bits())
            if integer:
                assert_bit_exact(bits[-1], case.oracle(), "bf16")
            else:
                assert_within_tol(case.result(), case.oracle(), wl.dtype)
        assert np.array_equal(bits[0], bits[1])
