"""C-ABI boundary checks that need no GPU: the library loads, exports every function declared in
include/tdx.h, and its host-side validation returns the documented status codes without touching a
device (every pointer below is a fake address that is never dereferenced on the host)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _load_build_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "tdx_build", os.path.join(ROOT, "comm_overlapped_gemm_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _lib_or_skip():
    build = _load_build_module()
    if not os.path.exists(build.LIB):
        build.build()
    import comm_overlapped_gemm_gb300 as tdx
    return tdx


@pytest.fixture(scope="module")
def tdx():
    return _lib_or_skip()


def declared_functions():
    with open(os.path.join(ROOT, "include", "tdx.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:tdx_status|size_t|uint32_t|const char\*)\s+(tdx_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["tdx_ag_gemm", "tdx_gemm_rs", "tdx_workspace_size", "tdx_read_device_status", "tdx_status_string"]:
        assert n in names


def test_header_is_plain_c(tmp_path):
    """include/tdx.h compiles as C99 on its own (no C++, CUDA or torch types in the ABI), and a C
    program that calls every entry point links against the library."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_tdx.c"
    calls = "\n".join(f"  (void)&{n};" for n in declared_functions())
    src.write_text('#include "tdx.h"\nint main(void) {\n' + calls + "\n  return 0;\n}\n")
    inc = os.path.join(ROOT, "include")
    res = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", inc, "-c", str(src),
                          "-o", str(tmp_path / "use_tdx.o")], capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    lib = _load_build_module().LIB
    if os.path.exists(lib):
        res = subprocess.run([cc, str(tmp_path / "use_tdx.o"), lib, "-o", str(tmp_path / "use_tdx")],
                             capture_output=True, text=True)
        assert res.returncode == 0, res.stderr


def test_library_exports_every_declared_symbol(tdx):
    lib = ctypes.CDLL(tdx.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(tdx.EXPORTED)


def test_status_strings_and_version(tdx):
    for s in range(8):
        assert tdx.tdx_status_string(s).startswith("TDX_")
    assert "unknown" in tdx.tdx_status_string(99)
    assert tdx.tdx_version() >> 16 == 1


def test_opts_default(tdx):
    o = tdx.tdx_opts_default()
    assert o.self_rank == 0 and o.mode == tdx.TDX_FUSED and o.timeout_ns == 2_000_000_000
    assert o.epoch == 0 and o.out_dtype == tdx.TDX_BF16
    assert ctypes.sizeof(tdx.tdx_opts) == 96 and o.reduce_mode == 0 and o.cluster == 0


def test_workspace_sizes(tdx):
    # AG W=8: gathered buffer 8192 x 8192 bf16 = 128 MiB plus a small control region
    ws = tdx.tdx_workspace_size(tdx.OP_AG, 8, 1024, 8192, 3584, tdx.TDX_BF16)
    assert 128 << 20 < ws < (128 << 20) + (1 << 20)
    # RS W=8: fp32 running sum of one 8192 x 8192 output = 256 MiB plus 7 x 2048 chain flags
    ws = tdx.tdx_workspace_size(tdx.OP_RS, 8, 8192, 3584, 8192, tdx.TDX_BF16)
    assert 256 << 20 < ws < (256 << 20) + (1 << 20)
    # fp8 AG: 16384 x 8192 e4m3 gathered buffer = 128 MiB
    ws = tdx.tdx_workspace_size(tdx.OP_AG, 8, 2048, 8192, 8192, tdx.TDX_FP8_E4M3)
    assert 128 << 20 < ws < (128 << 20) + (1 << 20)


def test_allreduce_workspace_any_m(tdx):
    # GEMM+AllReduce keeps every row on every rank, so M need not be a multiple of W
    ws = tdx.tdx_workspace_size(tdx.OP_AR, 3, 200, 136, 264, tdx.TDX_BF16)
    assert ws > 0
    info = tdx.tdx_plan_info(tdx.OP_AR, 3, 200, 136, 264, tdx.TDX_BF16)
    assert info["tiles_m"] == 2 and info["L"] == 3


@pytest.mark.parametrize("args,code", [
    ((0, 0, 64, 128, 256, 0), 1),      # W = 0
    ((0, 17, 64, 128, 256, 0), 1),     # W > 16
    ((0, 2, -1, 128, 256, 0), 1),      # negative size
    ((1, 3, 128, 128, 256, 0), 1),     # RS: M not a multiple of W
    ((3, 2, 64, 128, 256, 0), 1),      # bad op
    ((0, 2, 64, 128, 256, 7), 1),      # bad dtype
])
def test_workspace_size_rejects(tdx, args, code):
    with pytest.raises(tdx.TdxError) as e:
        tdx.tdx_workspace_size(*args)
    assert e.value.status == code


def test_chunk_rows_must_divide_shard(tdx):
    o = tdx.make_opts(chunk_rows=48)
    with pytest.raises(tdx.TdxError) as e:
        tdx.tdx_workspace_size(tdx.OP_AG, 2, 64, 128, 256, tdx.TDX_BF16, o)
    assert e.value.status == tdx.TDX_ERR_INVALID_ARG


FAKE = 0x7F0000000000   # 256-byte aligned fake device address, never dereferenced on the host


def _ag(tdx, shards=None, B=FAKE, C=FAKE, ws=FAKE, wsb=1 << 30, W=2, M_local=64, K=128, N=256,
        dtype=0, opts=None):
    shards = [FAKE] * W if shards is None else shards
    return tdx.tdx_ag_gemm(shards, B, C, ws, W, M_local, K, N, dtype, opts, stream=0, workspace_bytes=wsb)


def test_ag_validation_codes(tdx):
    assert _ag(tdx, B=0) == tdx.TDX_ERR_INVALID_ARG
    assert _ag(tdx, shards=[FAKE, 0]) == tdx.TDX_ERR_INVALID_ARG
    assert _ag(tdx, W=0, shards=[FAKE]) == tdx.TDX_ERR_INVALID_ARG
    assert _ag(tdx, shards=[FAKE + 8, FAKE]) == tdx.TDX_ERR_ALIGNMENT
    assert _ag(tdx, C=FAKE + 4) == tdx.TDX_ERR_ALIGNMENT
    assert _ag(tdx, K=100) == tdx.TDX_ERR_ALIGNMENT           # 200-byte rows
    assert _ag(tdx, N=100) == tdx.TDX_ERR_ALIGNMENT
    assert _ag(tdx, ws=0) == tdx.TDX_ERR_WORKSPACE
    assert _ag(tdx, ws=FAKE + 16) == tdx.TDX_ERR_WORKSPACE
    assert _ag(tdx, wsb=1024) == tdx.TDX_ERR_WORKSPACE
    assert _ag(tdx, opts=tdx.make_opts(self_rank=2)) == tdx.TDX_ERR_INVALID_ARG
    assert _ag(tdx, opts=tdx.make_opts(out_dtype=1)) == tdx.TDX_ERR_INVALID_ARG
    assert _ag(tdx, opts=tdx.make_opts(mode=9)) == tdx.TDX_ERR_INVALID_ARG
    assert _ag(tdx, opts=tdx.make_opts(block_n=96)) == tdx.TDX_ERR_UNSUPPORTED
    assert _ag(tdx, opts=tdx.make_opts(cluster=4)) == tdx.TDX_ERR_INVALID_ARG
    assert _ag(tdx, opts=tdx.make_opts(cluster=3, block_n=128)) == tdx.TDX_ERR_UNSUPPORTED
    # 512-wide tiles need 2-SM pairs
    assert _ag(tdx, opts=tdx.make_opts(cluster=1, block_n=512)) == tdx.TDX_ERR_UNSUPPORTED
    # pairs sharing B through multicast loads are not offered
    assert _ag(tdx, M_local=256, opts=tdx.make_opts(cluster=2, block_n=256)) == tdx.TDX_ERR_UNSUPPORTED
    assert _ag(tdx, dtype=1, opts=tdx.make_opts(block_n=64)) == tdx.TDX_ERR_UNSUPPORTED
    # empty problems launch nothing and succeed
    assert _ag(tdx, M_local=0) == tdx.TDX_OK
    assert _ag(tdx, N=0) == tdx.TDX_OK


def test_rs_validation_codes(tdx):
    def rs(A=None, B=None, O=None, W=2, M=128, K=128, N=256, dtype=0, opts=None, wsb=1 << 30, ws=FAKE):
        A = [FAKE] * W if A is None else A
        B = [FAKE] * W if B is None else B
        O = [FAKE] * W if O is None else O
        return tdx.tdx_gemm_rs(A, B, O, ws, W, M, K, N, dtype, opts, stream=0, workspace_bytes=wsb)
    assert rs(A=[FAKE, 0]) == tdx.TDX_ERR_INVALID_ARG
    assert rs(O=[0, FAKE]) == tdx.TDX_ERR_INVALID_ARG
    assert rs(M=129) == tdx.TDX_ERR_INVALID_ARG
    assert rs(dtype=1, M=256, opts=tdx.make_opts(cluster=2, block_n=256)) == tdx.TDX_ERR_UNSUPPORTED
    assert rs(M=256, opts=tdx.make_opts(cluster=2, block_n=256)) == tdx.TDX_ERR_UNSUPPORTED
    assert rs(dtype=1, K=120) == tdx.TDX_ERR_ALIGNMENT      # 120-byte e4m3 rows
    assert rs(opts=tdx.make_opts(out_dtype=2)) == tdx.TDX_ERR_UNSUPPORTED
    assert rs(B=[FAKE, FAKE + 2]) == tdx.TDX_ERR_ALIGNMENT
    assert rs(wsb=100) == tdx.TDX_ERR_WORKSPACE
    assert rs(M=0) == tdx.TDX_OK


def test_ar_validation_codes(tdx):
    def ar(A=None, B=None, O=None, W=2, M=128, K=128, N=256, dtype=0, opts=None, wsb=1 << 30, ws=FAKE):
        A = [FAKE] * W if A is None else A
        B = [FAKE] * W if B is None else B
        O = [FAKE] * W if O is None else O
        return tdx.tdx_gemm_ar(A, B, O, ws, W, M, K, N, dtype, opts, stream=0, workspace_bytes=wsb)
    assert ar(A=[FAKE, 0]) == tdx.TDX_ERR_INVALID_ARG
    assert ar(O=[FAKE, 0]) == tdx.TDX_ERR_INVALID_ARG
    assert ar(O=[FAKE, FAKE + 4]) == tdx.TDX_ERR_ALIGNMENT
    assert ar(opts=tdx.make_opts(out_dtype=2)) == tdx.TDX_ERR_UNSUPPORTED
    assert ar(wsb=100) == tdx.TDX_ERR_WORKSPACE
    assert ar(W=17, A=[FAKE] * 17, B=[FAKE] * 17, O=[FAKE] * 17) == tdx.TDX_ERR_INVALID_ARG
    assert ar(M=0) == tdx.TDX_OK
    assert ar(opts=tdx.make_opts(bf16_partials=1, reduce_mode=1)) == tdx.TDX_ERR_UNSUPPORTED
    assert ar(opts=tdx.make_opts(bf16_partials=2)) == tdx.TDX_ERR_INVALID_ARG


def test_bf16_partials_plan(tdx):
    # the partial slots shrink to half, and the slotted reduction is chosen even for many tiles
    full = tdx.tdx_plan_info(tdx.OP_RS, 8, 8192, 3584, 8192, tdx.TDX_BF16)
    half = tdx.tdx_plan_info(tdx.OP_RS, 8, 8192, 3584, 8192, tdx.TDX_BF16, tdx.make_opts(bf16_partials=1))
    assert full["reduce_mode"] == 1 and full["partial_bytes"] == 4
    assert half["reduce_mode"] == 2 and half["partial_bytes"] == 2
    assert half["total"] - half["off_S"] == 8 * half["T"] * 128 * half["BN"] * 2
    with pytest.raises(tdx.TdxError):
        tdx.tdx_workspace_size(tdx.OP_AG, 2, 64, 128, 256, tdx.TDX_BF16, tdx.make_opts(bf16_partials=1))


PLANS = [
    # (name, op, W, M_local or M, K, N, chunk_rows, expected plan words)
    ("AG W=8", "OP_AG", 8, 1024, 8192, 3584, 0,
     dict(BN=512, L=1, cluster=3, tiles_m=64, tiles_n=7, n_chunks=8, chunk_rows=128, pull_a=0)),
    ("RS W=8", "OP_RS", 8, 8192, 3584, 8192, 0,
     dict(BN=256, L=8, cluster=3, reduce_mode=1, group_n=16, tiles_m=64, tiles_n=32, coop_fold=0)),
    ("small-M AG", "OP_AG", 8, 16, 8192, 1024, 16,
     dict(BN=128, L=19, cluster=1, reduce_mode=2, pull_a=1, coop_fold=1, T=8, n_chunks=1)),
    ("small-M RS", "OP_RS", 8, 128, 1024, 8192, 0,
     dict(BN=256, L=8, cluster=1, reduce_mode=2, coop_fold=2, T=32)),
    ("RS, 8 M-tiles", "OP_RS", 8, 1024, 1024, 8192, 0,
     dict(BN=128, L=8, cluster=1, reduce_mode=1, T=512)),
    ("AG, N=64, 2-row shards", "OP_AG", 8, 2, 8192, 64, 0,
     dict(BN=64, L=19, cluster=1, reduce_mode=2, pull_a=0)),
    ("tiny AG", "OP_AG", 2, 64, 128, 256, 32,
     dict(BN=128, L=2, cluster=1, reduce_mode=2, pull_a=1, n_chunks=2)),
]


@pytest.mark.parametrize("case", PLANS, ids=[c[0] for c in PLANS])
def test_planner_choices_for_the_workloads(tdx, case):
    """Tile width, K splits, CTA cooperation and reduction chosen for the measured workloads and a
    few neighbours (a 152-SM device): 512-wide 2-SM pair tiles for the large AllGather, 2-SM pairs
    of 256-wide tiles with a chained running sum for the large RS,
    128-wide tiles over 19 K splits (one wave on 152 SMs) that read the shards in place and fold
    cooperatively for the small-M AllGather, 256-wide tiles with a grid-wide fold for the small-M
    ReduceScatter (two waves of work but only 32 tiles)."""
    _, op, W, M, K, N, cr, want = case
    p = tdx.tdx_plan_info(getattr(tdx, op), W, M, K, N, tdx.TDX_BF16, tdx.make_opts(chunk_rows=cr, num_sms=152))
    got = {k: p[k] for k in want}
    assert got == want
    assert p["T"] == p["tiles_m"] * p["tiles_n"]


def test_grid_fold_plan_and_limits(tdx):
    o3 = tdx.make_opts(reduce_mode=3, num_sms=152)
    p = tdx.tdx_plan_info(tdx.OP_RS, 4, 512, 256, 512, tdx.TDX_BF16, o3)
    assert p["reduce_mode"] == 2 and p["coop_fold"] == 2
    # a large problem that would take CTA pairs runs on single CTAs under reduce_mode 3
    assert tdx.tdx_plan_info(tdx.OP_RS, 8, 8192, 3584, 8192, tdx.TDX_BF16, o3)["cluster"] == 1
    for bad in (dict(reduce_mode=3, cluster=3, block_n=256), dict(reduce_mode=3, bf16_partials=1)):
        with pytest.raises(tdx.TdxError):
            tdx.tdx_plan_info(tdx.OP_RS, 4, 512, 256, 512, tdx.TDX_BF16, tdx.make_opts(**bad))
    with pytest.raises(tdx.TdxError):
        tdx.tdx_plan_info(tdx.OP_RS, 4, 512, 256, 512, tdx.TDX_BF16, tdx.make_opts(reduce_mode=4))


def test_trace_size(tdx):
    # header, 4 statistics words per CTA, the producer's release count and sequence, items per CTA
    assert tdx.tdx_trace_size(4, 10) == 4 * (4 + 48 + 1 + 4 * 3)
    assert tdx.tdx_trace_size(4, 10, 64) == 4 * (4 + 48 + 1 + 64 + 4 * 3)
    assert tdx.tdx_trace_size(0, 10) == 0
    assert tdx.tdx_trace_size(4, 10, -1) == 0


def test_copy_engine_producer_is_not_offered(tdx):
    rc = tdx.tdx_ag_gemm([FAKE] * 2, FAKE, FAKE, FAKE, 2, 64, 128, 256, tdx.TDX_BF16,
                         tdx.make_opts(producer=tdx.TDX_PRODUCER_COPY_ENGINE), stream=0, workspace_bytes=1 << 30)
    assert rc == tdx.TDX_ERR_UNSUPPORTED


def test_noalloc_rejects_copy_engine_producer_before_any_device_work(tdx):
    o = tdx.make_opts(producer=tdx.TDX_PRODUCER_COPY_ENGINE)
    rc = tdx.tdx_ag_gemm_noalloc([FAKE] * 2, FAKE, FAKE, 2, 64, 128, 256, tdx.TDX_BF16, o, stream=0)
    assert rc == tdx.TDX_ERR_UNSUPPORTED


def test_noalloc_rejects_oversized_problem_before_any_device_work(tdx):
    rc = tdx.tdx_ag_gemm_noalloc([FAKE] * 8, FAKE, FAKE, 8, 1024, 8192, 3584, tdx.TDX_BF16, None, stream=0)
    assert rc == tdx.TDX_ERR_WORKSPACE


@pytest.mark.parametrize("bad", ["B", "shard", "C", "K", "self_rank", "out_dtype", "null_shard", "status"])
def test_noalloc_checks_every_argument_before_any_device_work(tdx, bad):
    # No GPU here: a call that reached the scratch set-up or a launch would fail with
    # TDX_ERR_CUDA, so the specific code proves the argument was rejected before anything was
    # enqueued on the shared scratch array.
    shards, B, C, K, o, status = [FAKE] * 2, FAKE, FAKE, 128, None, None
    want = tdx.TDX_ERR_ALIGNMENT
    if bad == "B":
        B = FAKE + 8
    elif bad == "shard":
        shards = [FAKE, FAKE + 4]
    elif bad == "C":
        C = FAKE + 2
    elif bad == "K":
        K = 100                                    # 200-byte rows
    elif bad == "self_rank":
        o, want = tdx.make_opts(self_rank=5), tdx.TDX_ERR_INVALID_ARG
    elif bad == "out_dtype":
        o, want = tdx.make_opts(out_dtype=tdx.TDX_FP8_E4M3), tdx.TDX_ERR_INVALID_ARG
    elif bad == "null_shard":
        shards, want = [FAKE, 0], tdx.TDX_ERR_INVALID_ARG
    elif bad == "status":
        status = FAKE + 4
    rc = tdx.tdx_ag_gemm_noalloc(shards, B, C, 2, 64, K, 256, tdx.TDX_BF16, o, device_status=status, stream=0)
    assert rc == want, tdx.tdx_status_string(rc)


def test_moe_validation_codes(tdx):
    def ws_size(W=2, T=8, H=64, F=64, E=4, k=2, dtype=0, opts=None):
        try:
            tdx.tdx_moe_workspace_size(W, T, H, F, E, k, dtype, opts)
            return tdx.TDX_OK
        except tdx.TdxError as e:
            return e.status

    assert ws_size() == tdx.TDX_OK
    assert ws_size(E=513) == tdx.TDX_ERR_UNSUPPORTED
    assert ws_size(k=5) == tdx.TDX_ERR_INVALID_ARG          # topk > E
    assert ws_size(k=0) == tdx.TDX_ERR_INVALID_ARG
    assert ws_size(W=17) == tdx.TDX_ERR_INVALID_ARG
    assert ws_size(dtype=1) == tdx.TDX_OK                       # e4m3 dispatch
    assert ws_size(dtype=1, opts=tdx.make_opts(block_n=64)) == tdx.TDX_ERR_UNSUPPORTED
    assert ws_size(dtype=2) == tdx.TDX_ERR_INVALID_ARG
    assert ws_size(opts=tdx.make_opts(cluster=3)) == tdx.TDX_ERR_UNSUPPORTED
    assert ws_size(opts=tdx.make_opts(block_n=96)) == tdx.TDX_ERR_UNSUPPORTED

    def moe(X=None, R=None, B=FAKE, Y=FAKE, dest=FAKE, offs=0, W=2, T=8, H=64, F=64, E=4, k=2, opts=None,
            wsb=1 << 30, ws=FAKE):
        X = [FAKE] * W if X is None else X
        R = [FAKE] * W if R is None else R
        return tdx.tdx_moe_dispatch_gemm(X, R, B, Y, dest, offs, ws, W, T, H, F, E, k, tdx.TDX_BF16, opts,
                                         stream=0, workspace_bytes=wsb)

    assert moe(X=[FAKE, 0]) == tdx.TDX_ERR_INVALID_ARG
    assert moe(R=[0, FAKE]) == tdx.TDX_ERR_INVALID_ARG
    assert moe(dest=0) == tdx.TDX_ERR_INVALID_ARG
    assert moe(X=[FAKE, FAKE + 8]) == tdx.TDX_ERR_ALIGNMENT
    assert moe(dest=FAKE + 2) == tdx.TDX_ERR_ALIGNMENT
    assert moe(H=60) == tdx.TDX_ERR_ALIGNMENT                # 120-byte rows
    assert tdx.tdx_moe_dispatch_gemm([FAKE] * 2, [FAKE] * 2, FAKE, FAKE, FAKE, 0, FAKE, 2, 8, 72, 64, 4, 2,
                                     tdx.TDX_FP8_E4M3, None, stream=0, workspace_bytes=1 << 30) == tdx.TDX_ERR_ALIGNMENT
    assert moe(wsb=100) == tdx.TDX_ERR_WORKSPACE
    assert moe(opts=tdx.make_opts(mode=tdx.TDX_CONSUMER_ONLY)) == tdx.TDX_ERR_UNSUPPORTED
    assert moe(opts=tdx.make_opts(producer=tdx.TDX_PRODUCER_COPY_ENGINE)) == tdx.TDX_ERR_UNSUPPORTED


def test_moe_plan(tdx):
    # 262144 dispatched rows of 7168: 2048 chunks; 2-SM pairs (4096 rows per expert on average), so
    # the tile table holds a partial and a padding tile per expert: 2048 + 2 * 64; receive buffer 3.5 GiB
    p = tdx.tdx_moe_plan_info(8, 4096, 7168, 2048, 64, 8, tdx.TDX_BF16)
    assert p["total_rows"] == 262144 and p["n_chunks"] == 2048 and p["max_tiles"] == 2048 + 128
    assert p["cluster"] == 3
    # 128 tokens per rank: 128 rows per expert on average; bf16 on pairs of 256-wide tiles (a partial
    # and a padding tile per expert), e4m3 on single CTAs
    q = tdx.tdx_moe_plan_info(8, 128, 7168, 2048, 64, 8, tdx.TDX_BF16)
    assert q["cluster"] == 3 and q["BN"] == 256 and q["max_tiles"] == 64 + 2 * 64
    q8 = tdx.tdx_moe_plan_info(8, 128, 7168, 2048, 64, 8, tdx.TDX_FP8_E4M3)
    assert q8["cluster"] == 1 and q8["BN"] == 256 and q8["max_tiles"] == 64 + 64
    assert tdx.tdx_moe_plan_info(8, 128, 7168, 2048, 64, 8, tdx.TDX_BF16, tdx.make_opts(cluster=1))["cluster"] == 1
    assert tdx.tdx_moe_plan_info(8, 128, 7168, 2048, 64, 8, tdx.TDX_FP8_E4M3, tdx.make_opts(cluster=3))["cluster"] == 3
    with pytest.raises(tdx.TdxError):
        tdx.tdx_moe_plan_info(8, 128, 7168, 2048, 64, 8, tdx.TDX_BF16, tdx.make_opts(cluster=3, block_n=128))
    # 512-column pair tiles for the dispatch's grouped GEMM (library choice on pairs)
    assert p["BN"] == 512 and p["tiles_n"] == 4 and p["num_kb"] == 112
    assert tdx.tdx_moe_plan_info(8, 4096, 7168, 2048, 64, 8, tdx.TDX_BF16, tdx.make_opts(block_n=256))["BN"] == 256
    with pytest.raises(tdx.TdxError):
        tdx.tdx_moe_plan_info(8, 4096, 7168, 2048, 64, 8, tdx.TDX_BF16, tdx.make_opts(block_n=512, cluster=1))
    # the combine keeps 256-column tiles unless asked for 512 (pairs)
    assert tdx.tdx_moe_combine_plan_info(8, 4096, 2048, 7168, 64, 8, tdx.TDX_BF16)["BN"] == 256
    assert tdx.tdx_moe_combine_plan_info(8, 4096, 2048, 7168, 64, 8, tdx.TDX_BF16, tdx.make_opts(block_n=512))["BN"] == 512
    assert p["total"] - p["off_R"] == 262144 * 7168 * 2


def test_moe_combine_validation_codes(tdx):
    def ws_size(W=2, T=8, F=64, H=64, E=4, k=2, dtype=0):
        try:
            tdx.tdx_moe_combine_workspace_size(W, T, F, H, E, k, dtype)
            return tdx.TDX_OK
        except tdx.TdxError as e:
            return e.status

    assert ws_size() == tdx.TDX_OK
    assert ws_size(E=32, k=17) == tdx.TDX_ERR_UNSUPPORTED      # more than 16 slots per token
    assert ws_size(k=5) == tdx.TDX_ERR_INVALID_ARG
    assert ws_size(dtype=1) == tdx.TDX_ERR_UNSUPPORTED

    def comb(Hd=FAKE, R=None, B=FAKE, G=None, O=None, W=2, T=8, F=64, H=64, E=4, k=2, opts=None, wsb=1 << 30):
        R = [FAKE] * W if R is None else R
        G = [FAKE] * W if G is None else G
        O = [FAKE] * W if O is None else O
        return tdx.tdx_moe_gemm_combine(Hd, R, B, G, O, FAKE, W, T, F, H, E, k, tdx.TDX_BF16, opts, stream=0,
                                        workspace_bytes=wsb)

    assert comb(Hd=0) == tdx.TDX_ERR_INVALID_ARG
    assert comb(G=[FAKE, 0]) == tdx.TDX_ERR_INVALID_ARG
    assert comb(O=[0, FAKE]) == tdx.TDX_ERR_INVALID_ARG
    assert comb(O=[FAKE, FAKE + 8]) == tdx.TDX_ERR_ALIGNMENT
    assert comb(G=[FAKE + 2, FAKE]) == tdx.TDX_ERR_ALIGNMENT
    assert comb(F=60) == tdx.TDX_ERR_ALIGNMENT
    assert comb(wsb=64) == tdx.TDX_ERR_WORKSPACE
    assert comb(opts=tdx.make_opts(mode=tdx.TDX_CONSUMER_ONLY)) == tdx.TDX_ERR_UNSUPPORTED
    # the plan keeps per-(token, N-tile) counters and the slot table
    p = tdx.tdx_moe_combine_plan_info(8, 4096, 2048, 7168, 64, 8, tdx.TDX_BF16)
    assert p["tiles_n"] == 28 and p["off_tokcnt"] > 0 and p["off_dest"] > p["off_src"]
    assert p["total"] - p["off_R"] == 262144 * 7168 * 2
