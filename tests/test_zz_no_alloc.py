"""The allocation-free AllGather+GEMM entry point (tdx_ag_gemm_noalloc).

Some callers cannot allocate device memory: code running inside a host framework that owns every
device allocation and gives the caller no allocator (an inference-runtime plugin with a fixed
memory budget), or a latency-critical loop that cannot accept the device-wide synchronisation of
cudaMalloc. For them the library offers one entry point that takes no workspace and allocates
nothing: it runs on a scratch array the library declares statically in device memory
(TDX_NOALLOC_SCRATCH_BYTES per device).

This file is collected last on purpose, so that a run that stops at the first failure has already
run every other test. It must pass both alone in a fresh process and after the other tests: the
scratch array keeps the previous call's contents, and every call must clear what has to start at
zero. Each case below checks the output of two calls in a row against the output of the existing
tdx_ag_gemm entry point (with its own caller-owned workspace) on the same inputs: bit for bit on
integer inputs (where both must equal the oracle's single rounding of the exact sum), otherwise
within the tolerance the parity tests use.
"""
import numpy as np
import pytest
import torch

import comm_overlapped_gemm_gb300 as tdx
from oracle import reference as R
import workloads as wls
from gpu_util import AGCase, TOL

pytestmark = pytest.mark.gpu


def _close(got_bits: np.ndarray, ref_bits: np.ndarray, out_dtype: str, dtype: str):
    if out_dtype == "fp32":
        got = np.asarray(got_bits, dtype=np.float64)
        ref = np.asarray(ref_bits, dtype=np.float64)
    else:
        got, ref = R.decode_bf16(got_bits), R.decode_bf16(ref_bits)
    assert np.all(np.isfinite(got))
    scale = float(np.max(np.abs(ref)))
    assert float(np.max(np.abs(got - ref))) <= TOL[dtype] * scale


@pytest.mark.parametrize("name,integer", [("ag_small", False), ("ag_small", True), ("ag_tiny", False),
                                          ("ag_tiny", True), ("ag_fp8_small", False)])
def test_noalloc_matches_existing_entry_point_twice(name, integer):
    if name == "ag_fp8_small":
        wl = wls.with_shape(wls.WORKLOADS["ag_fp8_w8"], W=4, M=64, K=1024, N=512, chunk_rows=64)
    else:
        wl = wls.WORKLOADS[name]
    inp = wls.make_inputs(wl, integer=integer)
    out_dtype = "fp32" if wl.out_dtype == "fp32" else "bf16"
    kw = dict(chunk_rows=wl.chunk_rows, timeout_ns=500_000_000)
    if out_dtype == "fp32":
        kw["out_dtype"] = tdx.TDX_FP32
    if wl.dtype == "e4m3":
        kw.update(scale_a=inp.scale_a, scale_b=inp.scale_b[0])
    opts = tdx.make_opts(**kw)
    need = tdx.tdx_workspace_size(tdx.OP_AG, wl.W, wl.M, wl.K, wl.N, 0 if wl.dtype == "bf16" else 1, opts)
    assert need <= tdx.TDX_NOALLOC_SCRATCH_BYTES

    # existing entry point, caller-owned workspace
    ref_case = AGCase(inp, out_dtype=out_dtype, opts=opts)
    tdx.check(ref_case.run(), "tdx_ag_gemm")
    st, detail = tdx.tdx_read_device_status(ref_case.ws)
    assert st == tdx.TDX_OK, detail
    ref = ref_case.result_bits() if out_dtype == "bf16" else ref_case.C.cpu().numpy()

    status = torch.zeros(8, dtype=torch.int32, device="cuda")
    for call in range(2):
        C = torch.full_like(ref_case.C, float("nan"))
        rc = tdx.tdx_ag_gemm_noalloc(ref_case.shards, ref_case.B, C, wl.W, wl.M, wl.K, wl.N, ref_case.dt,
                                     opts, device_status=status)
        assert rc == tdx.TDX_OK, tdx.tdx_status_string(rc)
        torch.cuda.synchronize()
        assert int(status[0]) == tdx.TDX_OK, status.tolist()
        got = C.view(torch.int16).cpu().numpy().view(np.uint16) if out_dtype == "bf16" else C.cpu().numpy()
        if integer:
            assert np.array_equal(got, ref)
            assert np.array_equal(got, R.round_out(ref_case.oracle(), out_dtype))
        else:
            _close(got, ref, out_dtype, wl.dtype)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    # W=8 x 1024 x 8192 bf16 needs a 128 MiB gathered buffer: rejected before any launch
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    rc = tdx.tdx_ag_gemm_noalloc([dummy] * 8, dummy, dummy, 8, 1024, 8192, 3584, tdx.TDX_BF16, None)
    assert rc == tdx.TDX_ERR_WORKSPACE
