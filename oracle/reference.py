"""Plain fp64 definition of what the overlapped AllGather+GEMM and GEMM+ReduceScatter compute.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never imports this file.

What the pages fix (Triton-distributed / DITRON article, cronfeed.work, section "The first move
was to expose the overlap"): an AllGather moves row shards into place and a GEMM consumes the
gathered matrix; the overlapped kernel splits the gather into chunks and computes on arrived
chunks while others still move. The same section names the mirror operation,
GEMM-plus-ReduceScatter; the section "DITRON adds three levels of tiling" lists AllGather and
ReduceScatter among the collectives that are broken into chunks and paired with compute tiles.
Overlap changes *when* work happens, never *what* is computed, so the result the kernels must
reach is the plain definition:

* AllGather+GEMM: ``G = concat_r shards[r]`` (rank order 0..W-1, rows stacked) and
  ``C = s_r * (G @ B)`` where the per-row factor ``s_r = scale_a[r] * scale_b`` is 1 for bf16
  and the product of the per-tensor dequantisation scales for e4m3. Rounded once to the output
  type.
* GEMM+ReduceScatter: ``S = sum_{r=0}^{W-1} A_r @ B_r`` (ascending r) and output shard j is rows
  ``[j*M/W, (j+1)*M/W)`` of S, rounded once to bf16.
* GEMM+AllReduce (AllReduce is listed among the chunked collectives in "DITRON adds three levels of
  tiling"): every rank receives the whole of the same S, rounded once to bf16; M is any size.
* Both with ``partials="bf16"``: every rank's partial ``P_r = s_r * A_r @ B_r`` is first rounded to
  bf16 (the type a rank would put on the wire), then the rounded partials are summed exactly and
  the sum rounded once more to bf16. The pages do not say in which type partials travel; fp32 is
  the default reading and bf16 the variant real ReduceScatters send.

Where the pages are silent this file takes the plainest reading: inputs are decoded exactly to
fp64, products and sums are fp64 (a library fp64 matmul serves as the GEMM step; on the integer
inputs of the bit-exact checks every partial sum is an integer below 2**53, so the summation order
cannot matter there), and the single final rounding is round-to-nearest-even.

Bookkeeping (flags, schedules) is defined at the end of the file; it follows the rank-swizzled
arrival order of the same section ("begin computing on one chunk while another is still moving").
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------------------------
# Number formats
# ----------------------------------------------------------------------------------------------


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp64 values. A bf16 number is the upper half of an IEEE binary32
    (1 sign, 8 exponent, 7 fraction bits), so widening the pattern by 16 zero bits is exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _e4m3_table() -> np.ndarray:
    """fp64 value of every e4m3 (OCP FP8 "E4M3FN") code: 1 sign bit, 4 exponent bits with bias 7,
    3 fraction bits; exponent field 0 encodes subnormals m/8 * 2**-6; the all-ones pattern
    S.1111.111 is NaN; there is no infinity, so S.1111.110 = 448 is the largest finite value."""
    t = np.empty(256, dtype=np.float64)
    for c in range(256):
        sign = -1.0 if (c >> 7) & 1 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            t[c] = np.nan
        elif e == 0:
            t[c] = sign * (m / 8.0) * 2.0 ** -6
        else:
            t[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


_E4M3 = _e4m3_table()


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes (uint8) -> exact fp64 values through the format definition above."""
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def decode(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return decode_bf16(x)
    if dtype == "e4m3":
        return decode_e4m3(x)
    if dtype == "fp32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(dtype)


def round_bf16_rne(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 with ONE round-to-nearest-even step; returns the uint16 bit patterns.

    bf16 keeps 8 significant bits. For |x| in [2**(E-1), 2**E) the spacing of bf16 numbers is
    2**(E-8); below the smallest normal (2**-126) the spacing stays 2**-133 (subnormals). The value
    is divided by the spacing (exact: a power of two), rounded half-to-even, and scaled back. A
    result of magnitude 2**128 or more is an overflow and becomes infinity. NaN stays NaN."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, E = np.frexp(xf)                      # xf = f * 2**E, 0.5 <= |f| < 1
    q_exp = np.maximum(E.astype(np.int64) - 8, -133)
    quantum = np.ldexp(1.0, q_exp)
    r = np.rint(xf / quantum) * quantum      # np.rint rounds half to even
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, r), r)
    out[finite] = r[finite]
    out[~finite] = x[~finite]
    bits = out.astype(np.float32).view(np.uint32)   # exact: every bf16 value is a binary32 value
    return (bits >> np.uint32(16)).astype(np.uint16)


def round_fp32_rne(x: np.ndarray) -> np.ndarray:
    """fp64 -> binary32, round to nearest even (numpy's cast, a library routine)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def round_out(x: np.ndarray, out_dtype: str) -> np.ndarray:
    """The single final rounding to the output type: bf16 bit patterns or fp32 values."""
    if out_dtype == "bf16":
        return round_bf16_rne(x)
    if out_dtype == "fp32":
        return round_fp32_rne(x)
    raise ValueError(out_dtype)


# ----------------------------------------------------------------------------------------------
# AllGather + GEMM
# ----------------------------------------------------------------------------------------------


def _row_scales(W: int, M_local: int, scale_a, scale_b) -> np.ndarray:
    sa = np.ones(W) if scale_a is None else np.asarray(scale_a, dtype=np.float64)
    sb = 1.0 if scale_b is None else float(scale_b)
    return np.repeat(sa * sb, M_local)


def ag_gemm(shards, b, dtype: str = "bf16", scale_a=None, scale_b=None) -> np.ndarray:
    """AllGather+GEMM, unrounded fp64: ``C = diag(s) @ concat_r(shards[r]) @ B``.

    ``shards`` is a list of W arrays (M_local x K) of bf16 bits / e4m3 codes, ``b`` is K x N.
    ``scale_a[r]`` and ``scale_b`` are the per-tensor dequantisation scales (None = 1)."""
    W = len(shards)
    M_local = shards[0].shape[0]
    G = np.concatenate([decode(s, dtype) for s in shards], axis=0)   # the gathered buffer
    C = G @ decode(b, dtype)
    return C * _row_scales(W, M_local, scale_a, scale_b)[:, None]


def ag_gemm_rows(shards, b, rows, dtype: str = "bf16", scale_a=None, scale_b=None) -> np.ndarray:
    """Rows ``rows`` of :func:`ag_gemm` only (row i of G is row i % M_local of shard
    i // M_local), for sampled checks of large outputs."""
    W = len(shards)
    M_local = shards[0].shape[0]
    rows = np.asarray(rows, dtype=np.int64)
    G_rows = np.stack([decode(shards[i // M_local][i % M_local], dtype) for i in rows])
    C = G_rows @ decode(b, dtype)
    return C * _row_scales(W, M_local, scale_a, scale_b)[rows][:, None]


# ----------------------------------------------------------------------------------------------
# GEMM + ReduceScatter
# ----------------------------------------------------------------------------------------------


def _partial(P: np.ndarray, partials: str) -> np.ndarray:
    """A rank's partial as it enters the sum: exact (``"fp32"``: the kernels keep it in fp32, and
    the fp64 value is the exact one it approximates) or rounded once to bf16 (``"bf16"``)."""
    if partials == "fp32":
        return P
    if partials == "bf16":
        return decode_bf16(round_bf16_rne(P))
    raise ValueError(partials)


def gemm_rs(a_parts, b_parts, dtype: str = "bf16", scale_a=None, scale_b=None, partials: str = "fp32"):
    """GEMM+ReduceScatter, unrounded fp64: ``S = sum_r s_r * A_r @ B_r`` (ascending r), returned
    as the list of W row shards ``S[j*M/W:(j+1)*M/W]``. ``s_r = scale_a[r]*scale_b[r]`` (None = 1).
    ``partials="bf16"`` rounds every term of the sum to bf16 first."""
    W = len(a_parts)
    M = a_parts[0].shape[0]
    if M % W:
        raise ValueError("M must be a multiple of W")
    S = None
    for r in range(W):
        s = 1.0
        if scale_a is not None:
            s *= float(scale_a[r])
        if scale_b is not None:
            s *= float(scale_b[r])
        P = _partial((decode(a_parts[r], dtype) @ decode(b_parts[r], dtype)) * s, partials)
        S = P if S is None else S + P
    h = M // W
    return [S[j * h:(j + 1) * h] for j in range(W)]


def gemm_ar(a_parts, b_parts, dtype: str = "bf16", scale_a=None, scale_b=None, partials: str = "fp32"):
    """GEMM+AllReduce, unrounded fp64: the full ``S = sum_r s_r * A_r @ B_r`` (ascending r), one
    entry per rank (every rank holds the same S). ``s_r`` and ``partials`` as in :func:`gemm_rs`;
    M need not be a multiple of W."""
    W = len(a_parts)
    S = None
    for r in range(W):
        s = (1.0 if scale_a is None else float(scale_a[r])) * (1.0 if scale_b is None else float(scale_b[r]))
        P = _partial((decode(a_parts[r], dtype) @ decode(b_parts[r], dtype)) * s, partials)
        S = P if S is None else S + P
    return [S.copy() for _ in range(W)]


def gemm_rs_rows(a_parts, b_parts, rows, dtype: str = "bf16", scale_a=None, scale_b=None, partials: str = "fp32"):
    """Rows ``rows`` (indices into the M rows of S) of the reduced sum, before scattering."""
    rows = np.asarray(rows, dtype=np.int64)
    S = None
    for r in range(len(a_parts)):
        s = 1.0
        if scale_a is not None:
            s *= float(scale_a[r])
        if scale_b is not None:
            s *= float(scale_b[r])
        P = _partial((decode(a_parts[r][rows], dtype) @ decode(b_parts[r], dtype)) * s, partials)
        S = P if S is None else S + P
    return S


# ----------------------------------------------------------------------------------------------
# Bookkeeping: flags, arrival order and reduction order
#
# What the method fixes about order (Triton-distributed article, section "The first move was to
# expose the overlap": compute on one chunk while another is still moving; section "DITRON adds
# three levels of tiling": collectives broken into chunks paired with compute tiles, synchronised by
# signals) is stated here at the level of ranks and chunks only. How a kernel cuts the output into
# tiles, and in which raster it walks the tiles that one rank owns, is its own choice and is not
# part of the definition: the checks below take the consumed work as row ranges of the output.
# ----------------------------------------------------------------------------------------------


def ag_chunk_release_order(W: int, M_local: int, chunk: int, self_rank: int = 0):
    """Order in which the AllGather producer moves chunks into the gathered buffer: the peers
    in ring order self+1, self+2, ..., self+W-1 (mod W), chunks ascending within a rank, and the
    self shard last (the consumer reads its own shard in place, so nothing waits on that copy).
    Returns (rank, chunk index) pairs."""
    n_chunks = M_local // chunk
    ranks = [(self_rank + i) % W for i in range(1, W)] + [self_rank]
    return [(r, c) for r in ranks for c in range(n_chunks)]


def ag_arrival_rank_order(W: int, self_rank: int = 0):
    """Order in which the AllGather's consumer takes the ranks' rows: its own shard first (local,
    no wait), then the peers in the order their chunks arrive, self+1, self+2, ... (mod W)."""
    return [(self_rank + i) % W for i in range(W)]


def ag_consumer_order_ok(row_starts, W: int, M_local: int, self_rank: int = 0) -> bool:
    """True if a sequence of consumed output row blocks (the first row of each block, in the order
    the consumer took them) visits the ranks in :func:`ag_arrival_rank_order`: the rank that owns a
    block's first row never moves back to an earlier position of that order."""
    pos = {r: i for i, r in enumerate(ag_arrival_rank_order(W, self_rank))}
    seq = [pos[int(r0) // M_local] for r0 in row_starts]
    return all(b >= a for a, b in zip(seq, seq[1:]))


def rs_fold_order(W: int):
    """Order in which the ranks' partial products enter the ReduceScatter's sum of one output tile:
    ranks 0, 1, ..., W-1, a left fold ((P_0 + P_1) + P_2) + ..., the same for every tile and
    independent of timing and of which rank is local."""
    return list(range(W))


def expected_flags(n: int, epoch: int) -> np.ndarray:
    """After a completed call with epoch ``epoch`` every flag it released holds ``epoch``."""
    return np.full(n, epoch, dtype=np.uint32)
