"""GEMM+AllReduce on the GPU through the C ABI against the CPU oracle: every rank's full output
equals the rounded sum, all W outputs are bit-identical, and the result matches the ReduceScatter
entry point's shards row for row (AllReduce = ReduceScatter + AllGather)."""
import numpy as np
import pytest
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import reference as R
import workloads as wls
from gpu_util import ARCase, RSCase, assert_bit_exact, assert_within_tol, host_bits, sample_rows

pytestmark = pytest.mark.gpu

TMO = int(5e8)


def opts(**kw):
    return tdx.make_opts(timeout_ns=TMO, **kw)


def status_ok(case):
    st, detail = tdx.tdx_read_device_status(case.ws)
    assert st == tdx.TDX_OK, (tdx.tdx_status_string(st), detail)


def all_ranks_identical(case):
    torch.cuda.synchronize()
    for o in case.out[1:]:
        assert torch.equal(o.view(torch.int16), case.out[0].view(torch.int16))


@pytest.mark.parametrize("shape", [
    dict(W=2, M=256, K=256, N=512),
    dict(W=3, M=200, K=200, N=136),     # M not a multiple of W, ragged K and N
    dict(W=4, M=130, K=64, N=264),      # two-row M tail
    dict(W=1, M=128, K=128, N=256),
    dict(W=16, M=136, K=64, N=64),
])
@pytest.mark.parametrize("integer", [True, False])
def test_ar_small_shapes(shape, integer):
    wl = wls.with_shape(wls.WORKLOADS["ar_w8"], **shape)
    inp = wls.make_inputs(wl, integer=integer)
    want = R.gemm_ar(inp.a, inp.b)
    for bn, rm in ((0, 0), (128, 1), (256, 2)):
        case = ARCase(inp, opts=opts(block_n=bn, reduce_mode=rm))
        tdx.check(case.run(), f"ar {shape} bn={bn} reduce_mode={rm}")
        status_ok(case)
        for r in range(wl.W):
            got = case.result_bits(r)
            if integer:
                assert_bit_exact(got, want[r], "bf16")
            else:
                assert_within_tol(R.decode_bf16(got), want[r], "bf16")
        all_ranks_identical(case)


def test_ar_matches_reducescatter_shards_bitwise():
    wl = wls.with_shape(wls.WORKLOADS["ar_w8"], W=4, M=512, K=512, N=768)
    inp = wls.make_inputs(wl, integer=False)
    for rm in (1, 2):
        ar = ARCase(inp, opts=opts(reduce_mode=rm, perturb_seed=5))
        tdx.check(ar.run())
        status_ok(ar)
        rs = RSCase(inp, opts=opts(reduce_mode=rm))
        tdx.check(rs.run())
        status_ok(rs)
        assert np.array_equal(ar.result_bits(3), rs.result_bits())
        all_ranks_identical(ar)


@pytest.mark.parametrize("variant", [dict(cluster=3, block_n=256, reduce_mode=1),
                                     dict(cluster=3, block_n=256, reduce_mode=2)])
def test_ar_pairs(variant):
    wl = wls.with_shape(wls.WORKLOADS["ar_w8"], W=4, M=512, K=512, N=512)
    inp = wls.make_inputs(wl, integer=True)
    case = ARCase(inp, opts=opts(**variant))
    tdx.check(case.run())
    status_ok(case)
    want = R.gemm_ar(inp.a, inp.b)[0]
    assert_bit_exact(case.result_bits(0), want, "bf16")
    all_ranks_identical(case)


@pytest.mark.parametrize("integer", [True, False])
def test_ar_e4m3(integer):
    wl = wls.with_shape(wls.WORKLOADS["rs_fp8_w8"], op="ar", W=4, M=384, K=1024, N=1024)
    inp = wls.make_inputs(wl, integer=integer)
    case = ARCase(inp, opts=opts(scale_a=inp.scale_a, scale_b=inp.scale_b))
    tdx.check(case.run())
    status_ok(case)
    want = case.oracle()
    if integer:
        assert_bit_exact(case.result_bits(1), want, "bf16")
    else:
        assert_within_tol(R.decode_bf16(case.result_bits(1)), want, "e4m3")
    all_ranks_identical(case)


def test_ar_full_size_sampled_and_deterministic():
    wl = wls.WORKLOADS["ar_w8"]
    inp = wls.make_inputs(wl, integer=False)
    case = ARCase(inp, opts=opts())
    tdx.check(case.run())
    status_ok(case)
    rows = sample_rows(wl.M, wl.M // wl.W)
    want = case.oracle(rows)
    for r in (0, wl.W - 1):
        assert_within_tol(R.decode_bf16(case.result_bits(r)[rows]), want, "bf16")
    all_ranks_identical(case)
    first = case.result_bits(0)
    for o in case.out:
        o.fill_(float("nan"))
    tdx.check(case.run(opts(perturb_seed=11)))
    status_ok(case)
    assert np.array_equal(case.result_bits(5), first)


def test_ar_degenerate_sizes():
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    outs = [torch.full((64, 128), 2.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    # K = 0: every rank's output is zero
    tdx.check(tdx.tdx_gemm_ar([dummy] * 3, [dummy] * 3, outs, ws, 3, 64, 0, 128, tdx.TDX_BF16, opts()))
    torch.cuda.synchronize()
    assert all(int(torch.count_nonzero(o)) == 0 for o in outs)
    # M = 0: nothing to do, outputs untouched
    for o in outs:
        o.fill_(2.0)
    tdx.check(tdx.tdx_gemm_ar([dummy] * 3, [dummy] * 3, outs, ws, 3, 0, 64, 128, tdx.TDX_BF16, opts()))
    torch.cuda.synchronize()
    assert all(bool((o == 2.0).all()) for o in outs)


def test_ar_modes_run():
    wl = wls.with_shape(wls.WORKLOADS["ar_w8"], W=4, M=512, K=256, N=512)
    inp = wls.make_inputs(wl, integer=True)
    case = ARCase(inp, opts=opts())
    for mode in (tdx.TDX_GEMM_ONLY, tdx.TDX_MOVE_ONLY, tdx.TDX_FUSED):
        tdx.check(case.run(opts(mode=mode)))
        status_ok(case)
    assert_bit_exact(case.result_bits(2), R.gemm_ar(inp.a, inp.b)[2], "bf16")
    assert host_bits(case.out[0]).shape == (512, 512)


@pytest.mark.parametrize("integer", [True, False])
def test_ar_bf16_partials(integer):
    wl = wls.with_shape(wls.WORKLOADS["ar_w8"], W=4, M=300, K=1024, N=512)
    inp = wls.make_inputs(wl, integer=integer)
    case = ARCase(inp, opts=opts(bf16_partials=1))
    tdx.check(case.run())
    status_ok(case)
    want = case.oracle(partials="bf16")
    if integer:
        assert_bit_exact(case.result_bits(2), want, "bf16")
    else:
        assert_within_tol(R.decode_bf16(case.result_bits(2)), want, "bf16")
    all_ranks_identical(case)
