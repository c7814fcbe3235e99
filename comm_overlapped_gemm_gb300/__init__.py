"""Python binding of libtdx (tile-pipelined collective+GEMM kernels on sm_103a: AllGather+GEMM,
GEMM+ReduceScatter, GEMM+AllReduce, mixture-of-experts AllToAll dispatch + grouped GEMM and grouped
GEMM + combine).

Argument marshalling only: every function below converts its arguments (torch tensors or raw
device pointers) into the plain pointers and sizes of the C ABI in ``include/tdx.h`` and calls the
function of the same name in ``_lib/libtdx.so``. All computation happens in the library's CUDA
kernels; there is no other implementation behind these names, and importing this package fails
loudly when the library has not been built (``python comm_overlapped_gemm_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libtdx.so")

TDX_OK, TDX_ERR_INVALID_ARG, TDX_ERR_UNSUPPORTED, TDX_ERR_ALIGNMENT = 0, 1, 2, 3
TDX_ERR_WORKSPACE, TDX_ERR_CUDA, TDX_ERR_TIMEOUT, TDX_ERR_STALE_EPOCH = 4, 5, 6, 7
TDX_BF16, TDX_FP8_E4M3, TDX_FP32 = 0, 1, 2
TDX_FUSED, TDX_GEMM_ONLY, TDX_MOVE_ONLY, TDX_CONSUMER_ONLY = 0, 1, 2, 3
TDX_PRODUCER_SM, TDX_PRODUCER_COPY_ENGINE = 0, 1
OP_AG, OP_RS, OP_AR = 0, 1, 2
TDX_EPOCH_DEVICE = 0xFFFFFFFF

EXPORTED = ["tdx_opts_default", "tdx_workspace_size", "tdx_workspace_init", "tdx_ag_gemm", "tdx_gemm_rs",
            "tdx_read_device_status", "tdx_trace_size", "tdx_status_string", "tdx_version", "tdx_plan_info",
            "tdx_ag_gemm_noalloc", "tdx_gemm_ar", "tdx_moe_workspace_size", "tdx_moe_plan_info",
            "tdx_moe_dispatch_gemm", "tdx_moe_combine_workspace_size", "tdx_moe_combine_plan_info",
            "tdx_moe_gemm_combine"]


class tdx_opts(ctypes.Structure):
    _fields_ = [
        ("self_rank", ctypes.c_int),
        ("chunk_rows", ctypes.c_int),
        ("out_dtype", ctypes.c_int),
        ("scale_a", ctypes.POINTER(ctypes.c_float)),
        ("scale_b", ctypes.POINTER(ctypes.c_float)),
        ("mode", ctypes.c_int),
        ("producer", ctypes.c_int),
        ("epoch", ctypes.c_uint32),
        ("timeout_ns", ctypes.c_uint64),
        ("perturb_seed", ctypes.c_uint32),
        ("trace", ctypes.c_void_p),
        ("num_sms", ctypes.c_int),
        ("split_k", ctypes.c_int),
        ("block_n", ctypes.c_int),
        ("reduce_mode", ctypes.c_int),
        ("cluster", ctypes.c_int),
        ("bf16_partials", ctypes.c_int),
    ]


class TdxError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {tdx_status_string(status)}" if what else tdx_status_string(status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libtdx.so is not built ({LIB_PATH}); run python comm_overlapped_gemm_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, U32, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_size_t
    PP = ctypes.POINTER(ctypes.c_void_p)
    OP = ctypes.POINTER(tdx_opts)
    sig = {
        "tdx_opts_default": (I, [OP]),
        "tdx_workspace_size": (I, [I, I, I, I, I, I, OP, ctypes.POINTER(SZ)]),
        "tdx_workspace_init": (I, [P, SZ, P]),
        "tdx_ag_gemm": (I, [PP, P, P, P, SZ, I, I, I, I, I, OP, P]),
        "tdx_gemm_rs": (I, [PP, PP, PP, P, SZ, I, I, I, I, I, OP, P]),
        "tdx_gemm_ar": (I, [PP, PP, PP, P, SZ, I, I, I, I, I, OP, P]),
        "tdx_read_device_status": (I, [P, P, ctypes.POINTER(I), ctypes.POINTER(U32)]),
        "tdx_trace_size": (SZ, [I, I, I]),
        "tdx_status_string": (ctypes.c_char_p, [I]),
        "tdx_version": (U32, []),
        "tdx_plan_info": (I, [I, I, I, I, I, I, OP, ctypes.POINTER(ctypes.c_int64)]),
        "tdx_ag_gemm_noalloc": (I, [PP, P, P, I, I, I, I, I, OP, P, P]),
        "tdx_moe_workspace_size": (I, [I, I, I, I, I, I, I, OP, ctypes.POINTER(SZ)]),
        "tdx_moe_plan_info": (I, [I, I, I, I, I, I, I, OP, ctypes.POINTER(ctypes.c_int64)]),
        "tdx_moe_dispatch_gemm": (I, [PP, PP, P, P, P, P, P, SZ, I, I, I, I, I, I, I, OP, P]),
        "tdx_moe_combine_workspace_size": (I, [I, I, I, I, I, I, I, OP, ctypes.POINTER(SZ)]),
        "tdx_moe_combine_plan_info": (I, [I, I, I, I, I, I, I, OP, ctypes.POINTER(ctypes.c_int64)]),
        "tdx_moe_gemm_combine": (I, [P, PP, P, PP, PP, P, SZ, I, I, I, I, I, I, I, OP, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


# ---------------------------------------------------------------------------------- marshalling
def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _nbytes(x) -> int:
    return int(x.numel() * x.element_size())


def _ptr_array(xs):
    arr = (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])
    return arr


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) if torch.cuda.is_available() else 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def make_opts(**kw) -> tdx_opts:
    """A tdx_opts filled with the library defaults, then the given fields. ``scale_a`` (list of W
    floats) and ``scale_b`` (a float for AllGather, a list of W floats for ReduceScatter) are
    converted to host arrays kept alive by the struct."""
    o = tdx_opts()
    _lib.tdx_opts_default(ctypes.byref(o))
    keep = []
    for k, v in kw.items():
        if k == "scale_a" and v is not None:
            arr = (ctypes.c_float * len(v))(*[float(s) for s in v])
            keep.append(arr)
            o.scale_a = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
        elif k == "scale_b" and v is not None:
            vals = [float(s) for s in v] if isinstance(v, (list, tuple)) else [float(v)]
            arr = (ctypes.c_float * len(vals))(*vals)
            keep.append(arr)
            o.scale_b = ctypes.cast(arr, ctypes.POINTER(ctypes.c_float))
        elif k == "trace":
            o.trace = _ptr(v)
        elif v is not None:
            setattr(o, k, v)
    o._keep = keep
    return o


def _opts_ref(opts):
    return ctypes.byref(opts) if opts is not None else None


# ---------------------------------------------------------------------------------- C ABI names
def tdx_opts_default() -> tdx_opts:
    return make_opts()


def tdx_status_string(status: int) -> str:
    return _lib.tdx_status_string(int(status)).decode()


def tdx_version() -> int:
    return int(_lib.tdx_version())


def tdx_trace_size(grid: int, items: int, chunks: int = 0) -> int:
    return int(_lib.tdx_trace_size(grid, items, chunks))


def tdx_workspace_size(op: int, W: int, M_local_or_M: int, K: int, N: int, dtype: int, opts=None) -> int:
    out = ctypes.c_size_t(0)
    st = _lib.tdx_workspace_size(op, W, M_local_or_M, K, N, dtype, _opts_ref(opts), ctypes.byref(out))
    if st != TDX_OK:
        raise TdxError(st, "tdx_workspace_size")
    return int(out.value)


def tdx_workspace_init(workspace, nbytes: int | None = None, stream=None) -> int:
    n = _nbytes(workspace) if nbytes is None else nbytes
    return int(_lib.tdx_workspace_init(_ptr(workspace), n, _stream(stream)))


PLAN_KEYS = ["BN", "L", "tiles_m", "tiles_n", "T", "num_kb", "chunk_rows", "n_chunks", "off_chunk_flags",
             "off_chunk_cnt", "off_chain_flags", "off_G", "off_S", "total", "reduce_mode", "off_tile_cnt",
             "cluster", "group_n", "rank_block", "pull_a", "partial_bytes", "coop_fold"]


def tdx_plan_info(op: int, W: int, M_local_or_M: int, K: int, N: int, dtype: int, opts=None) -> dict:
    info = (ctypes.c_int64 * len(PLAN_KEYS))()
    st = _lib.tdx_plan_info(op, W, M_local_or_M, K, N, dtype, _opts_ref(opts), info)
    if st != TDX_OK:
        raise TdxError(st, "tdx_plan_info")
    return {k: int(info[i]) for i, k in enumerate(PLAN_KEYS)}


def tdx_ag_gemm(shards, B, C, workspace, W: int, M_local: int, K: int, N: int, dtype: int, opts=None,
                stream=None, workspace_bytes: int | None = None) -> int:
    wsb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return int(_lib.tdx_ag_gemm(_ptr_array(shards), _ptr(B), _ptr(C), _ptr(workspace), wsb, W, M_local, K, N,
                                dtype, _opts_ref(opts), _stream(stream)))


TDX_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024


def tdx_ag_gemm_noalloc(shards, B, C, W: int, M_local: int, K: int, N: int, dtype: int, opts=None,
                        device_status=None, stream=None) -> int:
    """AllGather+GEMM on the library's built-in scratch array (no workspace argument, nothing
    allocated by the call); see include/tdx.h for its limit and sharing rules."""
    return int(_lib.tdx_ag_gemm_noalloc(_ptr_array(shards), _ptr(B), _ptr(C), W, M_local, K, N, dtype,
                                        _opts_ref(opts), _ptr(device_status), _stream(stream)))


def tdx_gemm_rs(A_parts, B_parts, out_shards, workspace, W: int, M: int, K: int, N: int, dtype: int,
                opts=None, stream=None, workspace_bytes: int | None = None) -> int:
    wsb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return int(_lib.tdx_gemm_rs(_ptr_array(A_parts), _ptr_array(B_parts), _ptr_array(out_shards), _ptr(workspace),
                                wsb, W, M, K, N, dtype, _opts_ref(opts), _stream(stream)))


def tdx_gemm_ar(A_parts, B_parts, out_full, workspace, W: int, M: int, K: int, N: int, dtype: int,
                opts=None, stream=None, workspace_bytes: int | None = None) -> int:
    wsb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return int(_lib.tdx_gemm_ar(_ptr_array(A_parts), _ptr_array(B_parts), _ptr_array(out_full), _ptr(workspace),
                                wsb, W, M, K, N, dtype, _opts_ref(opts), _stream(stream)))


def tdx_read_device_status(workspace, stream=None):
    """Returns (status, detail[8])."""
    st = ctypes.c_int(0)
    detail = (ctypes.c_uint32 * 8)()
    rc = _lib.tdx_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(st), detail)
    if rc != TDX_OK:
        raise TdxError(rc, "tdx_read_device_status")
    return int(st.value), list(detail)


def check(status: int, what: str = "tdx") -> None:
    """Raise TdxError unless status is TDX_OK."""
    if status != TDX_OK:
        raise TdxError(status, what)


# ------------------------------------------------------------------ mixture-of-experts dispatch
MOE_PLAN_KEYS = ["BN", "tiles_n", "max_tiles", "n_chunks", "total_rows", "off_chunk_flags", "off_ntiles",
                 "off_offsets", "off_src", "off_tiles", "off_R", "total", "num_kb", "off_tokcnt", "off_dest",
                 "cluster"]


def tdx_moe_workspace_size(W: int, T: int, H: int, F: int, E: int, topk: int, dtype: int, opts=None) -> int:
    out = ctypes.c_size_t(0)
    st = _lib.tdx_moe_workspace_size(W, T, H, F, E, topk, dtype, _opts_ref(opts), ctypes.byref(out))
    if st != TDX_OK:
        raise TdxError(st, "tdx_moe_workspace_size")
    return int(out.value)


def tdx_moe_plan_info(W: int, T: int, H: int, F: int, E: int, topk: int, dtype: int, opts=None) -> dict:
    info = (ctypes.c_int64 * len(MOE_PLAN_KEYS))()
    st = _lib.tdx_moe_plan_info(W, T, H, F, E, topk, dtype, _opts_ref(opts), info)
    if st != TDX_OK:
        raise TdxError(st, "tdx_moe_plan_info")
    return {k: int(info[i]) for i, k in enumerate(MOE_PLAN_KEYS)}


def tdx_moe_dispatch_gemm(X, topk_idx, B_experts, Y, dest, expert_offsets, workspace, W: int, T: int, H: int,
                          F: int, E: int, topk: int, dtype: int, opts=None, stream=None,
                          workspace_bytes: int | None = None) -> int:
    wsb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return int(_lib.tdx_moe_dispatch_gemm(_ptr_array(X), _ptr_array(topk_idx), _ptr(B_experts), _ptr(Y), _ptr(dest),
                                          _ptr(expert_offsets), _ptr(workspace), wsb, W, T, H, F, E, topk, dtype,
                                          _opts_ref(opts), _stream(stream)))


def tdx_moe_combine_workspace_size(W: int, T: int, F: int, H: int, E: int, topk: int, dtype: int, opts=None) -> int:
    out = ctypes.c_size_t(0)
    st = _lib.tdx_moe_combine_workspace_size(W, T, F, H, E, topk, dtype, _opts_ref(opts), ctypes.byref(out))
    if st != TDX_OK:
        raise TdxError(st, "tdx_moe_combine_workspace_size")
    return int(out.value)


def tdx_moe_combine_plan_info(W: int, T: int, F: int, H: int, E: int, topk: int, dtype: int, opts=None) -> dict:
    info = (ctypes.c_int64 * len(MOE_PLAN_KEYS))()
    st = _lib.tdx_moe_combine_plan_info(W, T, F, H, E, topk, dtype, _opts_ref(opts), info)
    if st != TDX_OK:
        raise TdxError(st, "tdx_moe_combine_plan_info")
    return {k: int(info[i]) for i, k in enumerate(MOE_PLAN_KEYS)}


def tdx_moe_gemm_combine(Hd, topk_idx, B_experts, gates, out, workspace, W: int, T: int, F: int, H: int, E: int,
                         topk: int, dtype: int, opts=None, stream=None, workspace_bytes: int | None = None) -> int:
    wsb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    return int(_lib.tdx_moe_gemm_combine(_ptr(Hd), _ptr_array(topk_idx), _ptr(B_experts), _ptr_array(gates),
                                         _ptr_array(out), _ptr(workspace), wsb, W, T, F, H, E, topk, dtype,
                                         _opts_ref(opts), _stream(stream)))
