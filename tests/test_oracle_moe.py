"""Pins of the mixture-of-experts oracle (AllToAll dispatch + grouped GEMM, grouped GEMM + combine)
against hand-worked fixtures, exact rational brute force, layout invariants, identity experts and
the reduction to the AllGather+GEMM oracle; planted mistakes must fail them."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import workloads
from oracle import moe as MO
from oracle import reference as R
from test_oracle import bf16_bits_to_fraction, rand_bf16_bits

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def golden():
    with open(os.path.join(HERE, "golden", "moe_hand_examples.json")) as f:
        return json.load(f)


def _bf16(a):
    return workloads.to_bf16_bits(np.asarray(a, dtype=np.float32))


def _route(a):
    return np.asarray(a, dtype=np.int32)


def check_golden_dispatch(dispatch, golden):
    ex = golden["dispatch"]
    x = [_bf16(v) for v in ex["x"]]
    topk = [_route(v) for v in ex["topk"]]
    b = np.stack([_bf16(v) for v in ex["b"]])
    Y, (counts, offsets, dest, _) = dispatch(x, topk, b, ex["E"])
    assert np.array_equal(counts, ex["counts"])
    assert np.array_equal(offsets, ex["offsets"])
    for s in range(len(x)):
        assert np.array_equal(dest[s], ex["dest"][s])
    assert np.array_equal(Y, np.asarray(ex["y"], dtype=np.float64))


def test_golden_dispatch(golden):
    check_golden_dispatch(MO.moe_dispatch_gemm, golden)


def test_golden_dispatch_and_combine(golden):
    ex = golden["dispatch_combine"]
    x = [_bf16(v) for v in ex["x"]]
    topk = [_route(v) for v in ex["topk"]]
    b = np.stack([_bf16(v) for v in ex["b"]])
    Y, (_, _, dest, _) = MO.moe_dispatch_gemm(x, topk, b, ex["E"])
    assert np.array_equal(Y, np.asarray(ex["y"], dtype=np.float64))
    assert np.array_equal(dest[0], ex["dest"][0])
    gates = [np.asarray(g, dtype=np.float32) for g in ex["gates"]]
    out = MO.moe_combine(Y, dest, gates)
    assert np.array_equal(out[0], np.asarray(ex["out"][0], dtype=np.float64))
    # the same through the grouped GEMM + combine: h = dispatched x, B_e = the expert weights
    h = _bf16(np.array([[1], [2], [1], [2]]))     # dispatched rows: expert 0 gets x0, x1; expert 1 x0, x1
    out2 = MO.moe_gemm_combine(h, topk, b, gates, ex["E"])
    assert np.array_equal(out2[0], np.asarray(ex["out"][0], dtype=np.float64))


def random_routing(rng, W, T, E, k):
    return [np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32) for _ in range(W)]


def check_layout_invariants(layout, topk, E):
    counts, offsets, dest, src = layout
    W = len(topk)
    T, k = topk[0].shape
    total = W * T * k
    assert offsets[0] == 0 and offsets[E] == total
    assert counts.sum() == total
    for e in range(E):
        assert offsets[e + 1] - offsets[e] == counts[:, e].sum()
    seen = np.zeros(total, dtype=bool)
    for s in range(W):
        for t in range(T):
            for j in range(k):
                r = int(dest[s][t, j])
                assert not seen[r]
                seen[r] = True
                e = int(topk[s][t, j])
                assert offsets[e] <= r < offsets[e + 1]          # lands in its expert's block
                assert src[r] == (s, t)
    assert seen.all()
    for e in range(E):                                           # (source, token) ascending
        block = src[int(offsets[e]):int(offsets[e + 1])]
        assert block == sorted(block)


@pytest.mark.parametrize("W,T,E,k", [(1, 5, 3, 2), (2, 4, 4, 2), (3, 6, 6, 3), (4, 3, 8, 1)])
def test_layout_invariants(W, T, E, k):
    rng = np.random.default_rng(10 * W + T)
    topk = random_routing(rng, W, T, E, k)
    check_layout_invariants(MO.moe_layout(topk, E), topk, E)


def test_layout_rejects_bad_expert_ids():
    with pytest.raises(ValueError):
        MO.moe_layout([np.array([[0, 5]], dtype=np.int32)], 4)


def check_dispatch_brute(dispatch, W, T, E, k, H, F, integer, seed):
    rng = np.random.default_rng(seed)
    x = [rand_bf16_bits(rng, (T, H), integer) for _ in range(W)]
    b = np.stack([rand_bf16_bits(rng, (H, F), integer) for _ in range(E)])
    topk = random_routing(rng, W, T, E, k)
    Y, (_, _, dest, _) = dispatch(x, topk, b, E)
    assert Y.shape == (W * T * k, F)
    for s in range(W):
        for t in range(T):
            xq = [bf16_bits_to_fraction(int(v)) for v in x[s][t]]
            for j in range(k):
                e = int(topk[s][t, j])
                bq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in b[e]]
                r = int(dest[s][t, j])
                for n in range(F):
                    exact = sum((xq[h] * bq[h][n] for h in range(H)), Fraction(0))
                    if integer:
                        assert Y[r, n] == exact
                    else:
                        mag = sum(abs(xq[h] * bq[h][n]) for h in range(H))
                        assert abs(Fraction(Y[r, n]) - exact) <= mag * Fraction(H, 2 ** 52)


@pytest.mark.parametrize("W,T,E,k", [(1, 3, 2, 1), (2, 3, 4, 2), (3, 2, 3, 3)])
@pytest.mark.parametrize("integer", [True, False])
def test_dispatch_brute_force(W, T, E, k, integer):
    check_dispatch_brute(MO.moe_dispatch_gemm, W, T, E, k, H=5, F=3, integer=integer, seed=W * 31 + k)


def test_identity_experts_give_dispatched_tokens():
    rng = np.random.default_rng(3)
    W, T, E, k, H = 3, 5, 6, 2, 8
    x = [rand_bf16_bits(rng, (T, H), False) for _ in range(W)]
    eye = np.stack([_bf16(np.eye(H)) for _ in range(E)])
    topk = random_routing(rng, W, T, E, k)
    Y, (_, _, dest, _) = MO.moe_dispatch_gemm(x, topk, eye, E)
    for s in range(W):
        for t in range(T):
            for j in range(k):
                assert np.array_equal(Y[dest[s][t, j]], R.decode_bf16(x[s][t]))


def test_single_expert_top1_is_allgather_gemm():
    # every token of every rank to expert 0: the dispatch is the AllGather, the grouped GEMM one GEMM
    wl = workloads.with_shape(workloads.WORKLOADS["ag_w8"], W=3, M=4, K=16, N=8)
    inp = workloads.make_inputs(wl)
    topk = [np.zeros((4, 1), dtype=np.int32) for _ in range(3)]
    Y, _ = MO.moe_dispatch_gemm(inp.a, topk, inp.b[0][None], 1)
    assert np.array_equal(Y, R.ag_gemm(inp.a, inp.b[0]))


def test_sampled_rows_match_full():
    wl = workloads.with_shape(workloads.WORKLOADS["moe_w8"], W=2, M=6, K=16, N=8, E=4, topk=2)
    inp = workloads.make_inputs(wl)
    Y, _ = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E)
    rows = np.array([0, 5, 11, 23])
    assert np.array_equal(MO.moe_dispatch_gemm_rows(inp.a, inp.route, inp.b[0], wl.E, rows), Y[rows])


def test_e4m3_scales_per_source_and_expert():
    wl = workloads.with_shape(workloads.WORKLOADS["moe_w8"], W=2, M=4, K=16, N=8, E=4, topk=2, dtype="e4m3")
    inp = workloads.make_inputs(wl)
    Y, (_, offsets, _, src) = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E, "e4m3", inp.scale_a, inp.scale_b)
    Y1, _ = MO.moe_dispatch_gemm(inp.a, inp.route, inp.b[0], wl.E, "e4m3")
    for r in range(Y.shape[0]):
        s, _ = src[r]
        e = MO.row_expert(offsets, r)
        assert np.allclose(Y[r], Y1[r] * inp.scale_a[s] * inp.scale_b[e], rtol=1e-15, atol=0)


def test_combine_with_identity_experts_sums_gates():
    rng = np.random.default_rng(9)
    W, T, E, k, H = 2, 4, 4, 3, 6
    topk = random_routing(rng, W, T, E, k)
    wl = workloads.with_shape(workloads.WORKLOADS["moe_combine_w8"], W=W, M=T, K=H, N=H, E=E, topk=k)
    _, gates = workloads.make_routing(wl, integer=True)
    x = [rand_bf16_bits(rng, (T, H), True) for _ in range(W)]
    eye = np.stack([_bf16(np.eye(H)) for _ in range(E)])
    Y, (_, _, dest, _) = MO.moe_dispatch_gemm(x, topk, eye, E)
    h = workloads.to_bf16_bits(Y.astype(np.float32))          # exact: the dispatched bf16 tokens
    out = MO.moe_gemm_combine(h, topk, eye, gates, E)
    for s in range(W):
        want = R.decode_bf16(x[s]) * gates[s].astype(np.float64).sum(axis=1, keepdims=True)
        assert np.array_equal(out[s], want)


def check_combine_brute(combine):
    """``combine(h, topk, b, gates, E, z_dtype)`` against exact rational arithmetic on a tiny case,
    with the expert outputs entering exactly (fp32 reading) or rounded once to bf16 first."""
    rng = np.random.default_rng(12)
    W, T, E, k, F, H = 2, 3, 3, 2, 4, 3
    topk = random_routing(rng, W, T, E, k)
    h = rand_bf16_bits(rng, (W * T * k, F), False)
    b = np.stack([rand_bf16_bits(rng, (F, H), False) for _ in range(E)])
    gates = [rng.uniform(0, 1, size=(T, k)).astype(np.float32) for _ in range(W)]
    _, offsets, dest, _ = MO.moe_layout(topk, E)
    outs = {z: combine(h, topk, b, gates, E, z) for z in ("fp32", "bf16")}
    for s in range(W):
        for t in range(T):
            for n in range(H):
                exact = Fraction(0)
                exact_rz = Fraction(0)
                for j in range(k):
                    r = int(dest[s][t, j])
                    e = MO.row_expert(offsets, r)
                    z = sum((bf16_bits_to_fraction(int(h[r, f])) * bf16_bits_to_fraction(int(b[e, f, n]))
                             for f in range(F)), Fraction(0))
                    g = Fraction(float(gates[s][t, j]))
                    exact += g * z
                    zr = Fraction(float(R.decode_bf16(R.round_bf16_rne(np.array([float(z)])))[0]))
                    exact_rz += g * zr
                assert abs(Fraction(outs["fp32"][s][t, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 60)
                assert abs(Fraction(outs["bf16"][s][t, n]) - exact_rz) <= abs(exact_rz) * Fraction(1, 2 ** 48) + Fraction(1, 2 ** 60)


def test_combine_brute_force_and_z_rounding():
    check_combine_brute(lambda h, topk, b, gates, E, z: MO.moe_gemm_combine(h, topk, b, gates, E, z_dtype=z))


# ------------------------------------------------------------------ planted mistakes

def _mut_token_major(x, topk, b, E, dtype="bf16", scale_x=None, scale_b=None):
    # rows of an expert ordered token-major across sources instead of source-major
    Y, lay = MO.moe_dispatch_gemm(x, topk, b, E, dtype)
    counts, offsets, dest, src = lay
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        order = sorted(range(r0, r1), key=lambda r: (src[r][1], src[r][0]))
        Y[r0:r1] = Y[order]
    return Y, lay


def _mut_wrong_expert(x, topk, b, E, dtype="bf16", scale_x=None, scale_b=None):
    return MO.moe_dispatch_gemm(x, topk, b[::-1].copy(), E, dtype)


def _mut_dropped_slot(x, topk, b, E, dtype="bf16", scale_x=None, scale_b=None):
    Y, lay = MO.moe_dispatch_gemm(x, topk, b, E, dtype)
    Y[-1] = 0.0
    return Y, lay


@pytest.mark.parametrize("mut", [_mut_token_major, _mut_wrong_expert, _mut_dropped_slot])
def test_planted_dispatch_mistakes_are_caught(mut, golden):
    caught = 0
    try:
        check_golden_dispatch(mut, golden)
    except AssertionError:
        caught += 1
    try:
        check_dispatch_brute(mut, 2, 3, 4, 2, 3, 2, True, 5)
    except AssertionError:
        caught += 1
    assert caught > 0


def _cmut_rotated_gates(h, topk, b, gates, E, z):
    # slot j weighted by the gate of slot j+1
    return MO.moe_gemm_combine(h, topk, b, [np.roll(g, -1, axis=1) for g in gates], E, z_dtype=z)


def _cmut_unrounded_z(h, topk, b, gates, E, z):
    # expert outputs never rounded to bf16
    return MO.moe_gemm_combine(h, topk, b, gates, E, z_dtype="fp32")


def _cmut_wrong_experts(h, topk, b, gates, E, z):
    return MO.moe_gemm_combine(h, topk, b[::-1].copy(), gates, E, z_dtype=z)


def _cmut_first_slot_row(h, topk, b, gates, E, z):
    # every slot reads the expert output of slot 0
    _, _, dest, _ = MO.moe_layout(topk, E)
    Z = MO.moe_grouped_gemm(h, topk, b, E)
    if z == "bf16":
        Z = R.decode_bf16(R.round_bf16_rne(Z))
    bad = [np.repeat(d[:, :1], d.shape[1], axis=1) for d in dest]
    return MO.moe_combine(Z, bad, gates)


@pytest.mark.parametrize("mut", [_cmut_rotated_gates, _cmut_unrounded_z, _cmut_wrong_experts, _cmut_first_slot_row])
def test_planted_combine_mistakes_are_caught(mut):
    with pytest.raises(AssertionError):
        check_combine_brute(mut)


def test_grouped_gemm_rows_and_combine_rows_match_full():
    rng = np.random.default_rng(21)
    W, T, E, k, F, H = 2, 5, 4, 2, 6, 5
    topk = random_routing(rng, W, T, E, k)
    h = rand_bf16_bits(rng, (W * T * k, F), False)
    b = np.stack([rand_bf16_bits(rng, (F, H), False) for _ in range(E)])
    gates = [rng.uniform(0, 1, size=(T, k)).astype(np.float32) for _ in range(W)]
    Z = MO.moe_grouped_gemm(h, topk, b, E)
    rows = [0, 3, 7, 19]
    assert np.array_equal(MO.moe_grouped_gemm(h, topk, b, E, rows=rows), Z[rows])
    _, offsets, _, _ = MO.moe_layout(topk, E)
    for r in rows:                                   # brute force: h[r] @ B_e in exact rationals
        e = MO.row_expert(offsets, r)
        for n in range(H):
            exact = sum((bf16_bits_to_fraction(int(h[r, f])) * bf16_bits_to_fraction(int(b[e, f, n]))
                         for f in range(F)), Fraction(0))
            assert abs(Fraction(Z[r, n]) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 70)
    full = MO.moe_gemm_combine(h, topk, b, gates, E, z_dtype="bf16")
    toks = [(0, 0), (1, 4), (0, 3)]
    got = MO.moe_gemm_combine_rows(h, topk, b, gates, E, toks)
    for i, (s, t) in enumerate(toks):
        assert np.array_equal(got[i], full[s][t])
