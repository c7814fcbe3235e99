"""CPU oracle for tile-pipelined AllGather+GEMM, GEMM+ReduceScatter / AllReduce and the
AllToAll-overlapped grouped GEMM of a mixture-of-experts layer (``moe.py``).

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` use it. It shares no code with the CUDA library (no kernels, headers,
helpers, tables or constants); both sides take their inputs from ``workloads.py``, which holds
none of the method's arithmetic.

The oracle computes what the overlapped kernels must produce, written as the plain definition in
fp64 (see ``reference.py`` and ``moe.py``). Every function there is pinned by
``tests/test_oracle.py`` / ``tests/test_oracle_moe.py`` against
brute force in exact rational arithmetic, closed forms, the identity-matrix special cases, a
hand-worked fixture and library routines (torch's bf16 and e4m3 casts).
"""
from .reference import (  # noqa: F401
    decode_bf16, decode_e4m3, round_bf16_rne, round_fp32_rne,
    ag_gemm, ag_gemm_rows, gemm_rs, gemm_rs_rows, gemm_ar, round_out,
    ag_chunk_release_order, ag_arrival_rank_order, ag_consumer_order_ok, rs_fold_order, expected_flags,
)
