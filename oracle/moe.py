"""Plain fp64 definition of the AllToAll-overlapped grouped GEMM of a mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never imports this file.

What the pages fix (Triton-distributed / DITRON article, cronfeed.work): the section "DITRON adds
three levels of tiling" names AllToAll among the collectives that are broken into chunks and
paired with computation tiles, and says that device-level tiles are dynamically sized because the
number of tokens routed to each expert of a mixture-of-experts model is known only at run time.
The Triton-distributed repository page lists MoE kernels among its examples and quotes an AllToAll
of 128 tokens per rank. As with AllGather+GEMM, overlap changes when work happens, not what is
computed, so the result is the plain definition below.

Where the pages are silent this file takes the plainest reading:

* W ranks; rank s holds ``T`` tokens ``X_s`` (T x H) and their routing ``topk_s`` (T x k expert
  ids in [0, E), distinct within a token). Experts are split into W equal contiguous groups: rank
  rho owns experts ``rho*E/W .. (rho+1)*E/W - 1``.
* Dispatch (the AllToAll): every (s, t, j) sends row ``X_s[t]`` to the owner of expert
  ``e = topk_s[t, j]``. The receive side lays the rows out grouped by expert, experts ascending
  (so each rank's experts are one contiguous block, and the blocks follow in rank order); inside
  one expert, rows come in ascending source rank s, then ascending token t. ``dest[s][t, j]`` is
  the row that (s, t, j) lands in.
* Grouped GEMM: expert e multiplies its rows by its own weight ``B_e`` (H x F); the output keeps
  the dispatched row order: ``Y[dest[s][t, j]] = X_s[t] @ B_{topk_s[t, j]}``, rounded once.
* Combine (the reverse AllToAll with the gate-weighted sum): given per-row expert outputs ``Z``
  in the dispatched order and gates ``g_s`` (T x k),
  ``out_s[t] = sum_{j=0}^{k-1} g_s[t, j] * Z[dest[s][t, j]]`` (ascending j), rounded once.
* e4m3 inputs carry per-tensor scales as in the AllGather: one scale per source rank's X_s and
  one per expert weight, multiplied into the product before rounding.
"""
from __future__ import annotations

import numpy as np

from .reference import decode, decode_bf16, round_bf16_rne


def moe_layout(topk, E: int):
    """Routing layout of the dispatch. ``topk`` is a list of W int arrays (T x k).

    Returns ``(counts, offsets, dest, src)``: ``counts[s, e]`` tokens of rank s routed to expert e;
    ``offsets[e]`` first dispatched row of expert e (``offsets[E]`` = total rows = W*T*k);
    ``dest[s]`` (T x k) the dispatched row of every (s, t, j); ``src[row] = (s, t)``.
    Expert by expert, the rows are taken rank by rank; inside a rank, ``np.nonzero`` lists the
    (t, j) hits of the expert in row-major order, i.e. token ascending."""
    W = len(topk)
    for s in range(W):
        bad = (topk[s] < 0) | (topk[s] >= E)
        if bad.any():
            raise ValueError(f"expert id {int(topk[s][bad][0])} out of range")
    counts = np.array([[int((topk[s] == e).sum()) for e in range(E)] for s in range(W)], dtype=np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts.sum(axis=0))
    dest = [np.zeros(topk[s].shape, dtype=np.int64) for s in range(W)]
    src = [None] * int(offsets[E])
    for e in range(E):
        row = int(offsets[e])
        for s in range(W):
            tt, jj = np.nonzero(topk[s] == e)
            dest[s][tt, jj] = np.arange(row, row + len(tt))
            for i, t in enumerate(tt):
                src[row + i] = (s, int(t))
            row += len(tt)
    return counts, offsets, dest, src


def row_expert(offsets: np.ndarray, row: int) -> int:
    """The expert whose block of dispatched rows contains ``row``."""
    return int(np.searchsorted(offsets, row, side="right") - 1)


def moe_dispatch_gemm(x, topk, b_experts, E: int, dtype: str = "bf16", scale_x=None, scale_b=None):
    """AllToAll dispatch + grouped GEMM, unrounded fp64: ``Y`` (W*T*k x F) in the dispatched row
    order, plus the layout of :func:`moe_layout`. ``b_experts`` is E x H x F (bf16 bits or e4m3
    codes); ``scale_x[s]``, ``scale_b[e]`` are e4m3 dequantisation scales (None = 1)."""
    counts, offsets, dest, src = moe_layout(topk, E)
    F = b_experts.shape[2]
    Y = np.zeros((int(offsets[E]), F), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 == r1:
            continue
        rows = np.stack([decode(x[s][t], dtype) for (s, t) in src[r0:r1]])
        sx = np.array([1.0 if scale_x is None else float(scale_x[s]) for (s, _) in src[r0:r1]])
        sb = 1.0 if scale_b is None else float(scale_b[e])
        Y[r0:r1] = (rows @ decode(b_experts[e], dtype)) * (sx[:, None] * sb)
    return Y, (counts, offsets, dest, src)


def moe_dispatch_gemm_rows(x, topk, b_experts, E: int, rows, dtype: str = "bf16", scale_x=None, scale_b=None):
    """Rows ``rows`` (dispatched row indices) of :func:`moe_dispatch_gemm` only."""
    _, offsets, _, src = moe_layout(topk, E)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(rows), b_experts.shape[2]), dtype=np.float64)
    experts = np.array([row_expert(offsets, int(r)) for r in rows], dtype=np.int64)
    for e in np.unique(experts):
        sel = np.nonzero(experts == e)[0]
        b = decode(b_experts[e], dtype)                   # decoded once per expert
        sb = 1.0 if scale_b is None else float(scale_b[e])
        for i in sel:
            s, t = src[int(rows[i])]
            sx = 1.0 if scale_x is None else float(scale_x[s])
            out[i] = (decode(x[s][t][None, :], dtype) @ b)[0] * (sx * sb)
    return out


def moe_combine(Z: np.ndarray, dest, gates):
    """Combine: ``out_s[t] = sum_j gates_s[t, j] * Z[dest_s[t, j]]`` in fp64, ascending j (unrounded).
    ``Z`` holds fp64 values in the dispatched row order; ``gates`` a list of W fp32 arrays (T x k)."""
    outs = []
    for s in range(len(dest)):
        T, k = dest[s].shape
        o = np.zeros((T, Z.shape[1]), dtype=np.float64)
        for t in range(T):
            for j in range(k):
                o[t] += float(gates[s][t, j]) * Z[int(dest[s][t, j])]
        outs.append(o)
    return outs


def moe_grouped_gemm(h, topk, b_experts, E: int, dtype: str = "bf16", rows=None):
    """Grouped GEMM over rows already in the dispatched order, unrounded fp64: row r of expert e
    (``offsets[e] <= r < offsets[e+1]`` for the layout of ``topk``) gives ``h[r] @ B_e``. All rows,
    or only ``rows`` when given."""
    _, offsets, _, _ = moe_layout(topk, E)
    H = b_experts.shape[2]
    if rows is not None:
        rows = np.asarray(rows, dtype=np.int64)
        out = np.zeros((len(rows), H), dtype=np.float64)
        for e in np.unique([row_expert(offsets, int(r)) for r in rows]):
            sel = [i for i, r in enumerate(rows) if row_expert(offsets, int(r)) == e]
            out[sel] = decode(h[rows[sel]], dtype) @ decode(b_experts[e], dtype)
        return out
    Z = np.zeros((h.shape[0], H), dtype=np.float64)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r0 < r1:
            Z[r0:r1] = decode(h[r0:r1], dtype) @ decode(b_experts[e], dtype)
    return Z


def moe_gemm_combine_rows(h, topk, b_experts, gates, E: int, tokens, dtype: str = "bf16", z_dtype: str = "bf16"):
    """Combined outputs of the (rank, token) pairs in ``tokens`` only: ``out_s[t]`` of
    :func:`moe_gemm_combine` for each pair, as an array (len(tokens) x H)."""
    _, _, dest, _ = moe_layout(topk, E)
    rows = sorted({int(dest[s][t, j]) for (s, t) in tokens for j in range(dest[s].shape[1])})
    Zr = moe_grouped_gemm(h, topk, b_experts, E, dtype, rows=rows)
    if z_dtype == "bf16":
        Zr = decode_bf16(round_bf16_rne(Zr))
    at = {r: i for i, r in enumerate(rows)}
    out = np.zeros((len(tokens), b_experts.shape[2]), dtype=np.float64)
    for i, (s, t) in enumerate(tokens):
        for j in range(dest[s].shape[1]):
            out[i] += float(gates[s][t, j]) * Zr[at[int(dest[s][t, j])]]
    return out


def moe_gemm_combine(h, topk, b_experts, gates, E: int, dtype: str = "bf16", z_dtype: str = "fp32"):
    """Grouped GEMM + AllToAll combine, unrounded fp64. ``h`` is the dispatched activations
    (W*T*k x F, bf16 bits, the rows in the dispatch layout of ``topk``), ``b_experts`` E x F x H.
    Row r of expert e gives ``Z[r] = h[r] @ B_e``; with ``z_dtype="bf16"`` each Z row is rounded to
    bf16 first (the type a rank would send back), else it enters the sum exactly. Returns the W
    combined outputs (T x H) of :func:`moe_combine`."""
    _, _, dest, _ = moe_layout(topk, E)
    Z = moe_grouped_gemm(h, topk, b_experts, E, dtype)
    if z_dtype == "bf16":
        Z = decode_bf16(round_bf16_rne(Z))
    elif z_dtype != "fp32":
        raise ValueError(z_dtype)
    return moe_combine(Z, dest, gates)
