"""Grouped GEMM + AllToAll combine of a mixture-of-experts layer on the GPU through the C ABI,
against the CPU oracle: expert outputs (kept in the workspace) bit-exactly on integer inputs, the
gate-weighted per-token combine bit-exactly on integer inputs (gates powers of two) and within the
bf16 tolerance on random ones; modes and run-to-run bit identity under injected delays."""
import numpy as np
import pytest
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import moe as MO
from oracle import reference as R
import workloads as wls
from gpu_util import CombineCase, assert_bit_exact, assert_within_tol

pytestmark = pytest.mark.gpu

TMO = int(5e8)


def opts(**kw):
    return tdx.make_opts(timeout_ns=TMO, **kw)


def status_ok(case):
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_OK, (tdx.tdx_status_string(st), detail)


def oracle_out(inp):
    wl = inp.wl
    outs = MO.moe_gemm_combine(inp.a[0], inp.route, inp.b[0], inp.gates, wl.E, z_dtype="bf16")
    return np.stack(outs)


SHAPES = [
    dict(W=2, M=5, K=64, N=128, E=4, topk=2),
    dict(W=3, M=70, K=200, N=136, E=6, topk=3),        # ragged K and N
    dict(W=8, M=128, K=256, N=512, E=64, topk=8),
    dict(W=1, M=300, K=128, N=256, E=3, topk=1),
    dict(W=4, M=257, K=64, N=64, E=8, topk=2),
    dict(W=16, M=17, K=64, N=192, E=32, topk=4),
    dict(W=2, M=40, K=64, N=136, E=20, topk=12),       # two slot groups, the second partial
    dict(W=4, M=33, K=128, N=256, E=16, topk=16),      # the most slots a token may have: every expert
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("integer", [True, False])
def test_combine_small_shapes(shape, integer):
    wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    want = oracle_out(inp)
    Z = MO.moe_grouped_gemm(inp.a[0], inp.route, inp.b[0], wl.E)
    for bn, cl in ((0, 0), (64, 0), (256, 1), (256, 3)):
        case = CombineCase(inp, opts=opts(block_n=bn, cluster=cl))
        tdx.check(case.run(), f"combine {shape} bn={bn} cluster={cl}")
        status_ok(case)
        got = case.result_bits()
        if integer:
            assert_bit_exact(case.z_bits(), Z, "bf16")
            assert_bit_exact(got.reshape(-1, wl.N), want.reshape(-1, wl.N), "bf16")
        else:
            assert_within_tol(R.decode_bf16(case.z_bits()), Z, "bf16")
            assert_within_tol(R.decode_bf16(got.reshape(-1, wl.N)), want.reshape(-1, wl.N), "bf16")


def test_combine_modes_counters_and_determinism():
    wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], W=4, M=128, K=512, N=768, E=16, topk=4)
    inp = wls.make_inputs(wl, integer=False)
    case = CombineCase(inp, opts=opts())
    tdx.check(case.run(opts(epoch=1)))
    status_ok(case)
    first = case.result_bits()
    assert_within_tol(R.decode_bf16(first.reshape(-1, wl.N)), oracle_out(inp).reshape(-1, wl.N), "bf16")
    # every arrival counter is back to zero
    pl = case.plan()
    n = wl.W * wl.M * pl["tiles_n"]
    cnt = case.ws[pl["off_tokcnt"]:pl["off_tokcnt"] + 4 * n].view(torch.int32).cpu().numpy()
    assert not cnt.any()
    # GEMM alone then the combine alone, and fused runs with delays, give the same bits
    for o in case.out:
        o.fill_(float("nan"))
    tdx.check(case.run(opts(mode=tdx.TDX_GEMM_ONLY, epoch=2)))
    tdx.check(case.run(opts(mode=tdx.TDX_MOVE_ONLY, epoch=3)))
    status_ok(case)
    assert np.array_equal(case.result_bits(), first)
    for ep, seed in ((4, 7), (5, 99)):
        for o in case.out:
            o.fill_(float("nan"))
        tdx.check(case.run(opts(epoch=ep, perturb_seed=seed)))
        status_ok(case)
        assert np.array_equal(case.result_bits(), first)


def test_combine_invalid_expert_id_is_reported_not_run():
    wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], W=2, M=16, K=64, N=64, E=4, topk=2)
    inp = wls.make_inputs(wl, integer=True)
    inp.route[0] = inp.route[0].copy()
    inp.route[0][5, 0] = -3
    case = CombineCase(inp, opts=opts())
    tdx.check(case.run())
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_ERR_INVALID_ARG and detail[1] == 5
    assert all(bool(torch.isnan(o.float()).all()) for o in case.out)


def test_combine_full_size_sampled():
    wl = wls.WORKLOADS["moe_combine_w8"]
    inp = wls.make_inputs(wl, integer=False)
    case = CombineCase(inp, opts=opts())
    tdx.check(case.run())
    status_ok(case)
    got = case.result_bits()
    toks = [(s, t) for s in (0, 3, 7) for t in (0, 1, 777, wl.M - 1)]
    want = MO.moe_gemm_combine_rows(inp.a[0], inp.route, inp.b[0], inp.gates, wl.E, toks)
    sel = np.stack([got[s][t] for (s, t) in toks])
    assert_within_tol(R.decode_bf16(sel), want, "bf16")


@pytest.mark.parametrize("case_name", ["mostly_empty", "skewed"])
def test_combine_empty_and_skewed_experts(case_name):
    if case_name == "mostly_empty":
        wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], W=2, M=3, K=128, N=256, E=64, topk=2)
        inp = wls.make_inputs(wl, integer=True)
    else:
        wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], W=4, M=660, K=128, N=256, E=8, topk=2)
        inp = wls.make_inputs(wl, integer=True)
        for s in range(wl.W):
            r = np.empty_like(inp.route[s])
            r[:] = np.array([6, 1], dtype=np.int32)[None, :]
            inp.route[s] = r
    want = oracle_out(inp)
    for bn, cl in ((0, 0), (256, 3)):
        case = CombineCase(inp, opts=opts(block_n=bn, cluster=cl))
        tdx.check(case.run())
        status_ok(case)
        assert_bit_exact(case.result_bits().reshape(-1, wl.N), want.reshape(-1, wl.N), "bf16")


@pytest.mark.parametrize("topk", [5, 16])
def test_combine_alone_matches_fused(topk):
    """The combine alone (expert outputs already in place) walks (token, N-tile) units two at a
    time across the grid, the fused combine walks each tile's task list: both give the fused bits,
    also for an odd unit count per warp and for a token's slots in two groups of loads."""
    wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], W=3, M=37, K=64, N=328, E=18, topk=topk)
    inp = wls.make_inputs(wl, integer=False)
    for bn in (0, 64):
        case = CombineCase(inp, opts=opts(block_n=bn))
        tdx.check(case.run(opts(block_n=bn, epoch=1)))
        status_ok(case)
        fused = case.result_bits()
        assert_within_tol(R.decode_bf16(fused.reshape(-1, wl.N)), oracle_out(inp).reshape(-1, wl.N), "bf16")
        for o in case.out:
            o.fill_(float("nan"))
        tdx.check(case.run(opts(block_n=bn, mode=tdx.TDX_GEMM_ONLY, epoch=2)))
        tdx.check(case.run(opts(block_n=bn, mode=tdx.TDX_MOVE_ONLY, epoch=3)))
        status_ok(case)
        assert np.array_equal(case.result_bits(), fused), f"topk={topk} bn={bn}"


def test_combine_wide_tiles_match_256():
    # 512-column pair tiles for the combine's grouped GEMM: the same expert outputs and combined
    # tokens as 256 columns; exact on integers; ragged H (1344)
    wl = wls.with_shape(wls.WORKLOADS["moe_combine_w8"], W=4, M=300, K=512, N=1344, E=8, topk=3)
    for integer in (True, False):
        inp = wls.make_inputs(wl, integer=integer)
        bits = []
        for bn in (512, 256):
            case = CombineCase(inp, opts=opts(block_n=bn, cluster=3))
            assert case.plan()["BN"] == bn
            tdx.check(case.run())
            status_ok(case)
            bits.append(case.result_bits())
        want = np.stack(MO.moe_gemm_combine(inp.a[0], inp.route, inp.b[0], inp.gates, wl.E, z_dtype="bf16"))
        if integer:
            assert_bit_exact(bits[0], want, "bf16")
        assert np.array_equal(bits[0], bits[1])
