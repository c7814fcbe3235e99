"""Pins for the CPU oracle (CPU only; no GPU, no CUDA library).

Each pin checks the oracle against something other than itself: brute force in exact rational
arithmetic on tiny inputs, hand-worked fixtures (tests/golden/hand_examples.json), closed forms,
the identity-matrix special cases, invariants (rank permutation, linearity) and library routines
(torch's bf16 and float8_e4m3fn casts). The mutation tests at the end plant plausible mistakes in
copies of the oracle's functions and check that some pin fails for each.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import reference as R
import workloads

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ brute force (exact rationals)

def bf16_bits_to_fraction(b: int) -> Fraction:
    """bf16 bit pattern -> exact rational, from the bit fields (independent of the oracle)."""
    s = -1 if (b >> 15) & 1 else 1
    e = (b >> 7) & 0xFF
    m = b & 0x7F
    assert e != 0xFF, "no inf/nan in these tests"
    if e == 0:
        return s * Fraction(m, 128) * Fraction(2) ** -126
    return s * (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)


def brute_gemm(A, B):
    M, K = len(A), len(A[0])
    N = len(B[0])
    return [[sum((A[i][k] * B[k][n] for k in range(K)), Fraction(0)) for n in range(N)]
            for i in range(M)]


def rand_bf16_bits(rng, shape, integer):
    if integer:
        x = rng.integers(-4, 5, size=shape).astype(np.float32)
    else:
        x = rng.standard_normal(size=shape).astype(np.float32)
    return workloads.to_bf16_bits(x)


def check_ag_brute(ag_gemm, W, M_local, K, N, integer, seed):
    rng = np.random.default_rng(seed)
    shards = [rand_bf16_bits(rng, (M_local, K), integer) for _ in range(W)]
    b = rand_bf16_bits(rng, (K, N), integer)
    Gq = [[bf16_bits_to_fraction(int(v)) for v in row] for s in shards for row in s]
    Bq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in b]
    exact = brute_gemm(Gq, Bq)
    got = ag_gemm(shards, b, "bf16")
    assert got.shape == (W * M_local, N)
    for i in range(W * M_local):
        for n in range(N):
            if integer:
                assert got[i, n] == exact[i][n]
            else:
                bound = sum(abs(Gq[i][k] * Bq[k][n]) for k in range(K)) * Fraction(K, 2 ** 52)
                assert abs(Fraction(got[i, n]) - exact[i][n]) <= bound


def check_rs_brute(gemm_rs, W, M, K, N, integer, seed):
    rng = np.random.default_rng(seed)
    A = [rand_bf16_bits(rng, (M, K), integer) for _ in range(W)]
    B = [rand_bf16_bits(rng, (K, N), integer) for _ in range(W)]
    exact = [[Fraction(0)] * N for _ in range(M)]
    mag = [[Fraction(0)] * N for _ in range(M)]
    for r in range(W):
        Aq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in A[r]]
        Bq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in B[r]]
        P = brute_gemm(Aq, Bq)
        for i in range(M):
            for n in range(N):
                exact[i][n] += P[i][n]
                mag[i][n] += sum(abs(Aq[i][k] * Bq[k][n]) for k in range(K))
    shards = gemm_rs(A, B, "bf16")
    assert len(shards) == W
    h = M // W
    for j in range(W):
        assert shards[j].shape == (h, N)
        for i in range(h):
            for n in range(N):
                e = exact[j * h + i][n]
                if integer:
                    assert shards[j][i, n] == e
                else:
                    assert abs(Fraction(shards[j][i, n]) - e) <= mag[j * h + i][n] * Fraction(W * K + W, 2 ** 52)


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("M_local", [1, 2, 5])
@pytest.mark.parametrize("integer", [True, False])
def test_ag_brute_force(W, M_local, integer):
    check_ag_brute(R.ag_gemm, W, M_local, K=7 + W, N=3 + 2 * M_local, integer=integer,
                   seed=1000 * W + 10 * M_local + integer)


@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("integer", [True, False])
def test_rs_brute_force(W, integer):
    check_rs_brute(R.gemm_rs, W, M=2 * W, K=5 + W, N=6, integer=integer, seed=77 + W + integer)


def check_ar_brute(gemm_ar, W, M, K, N, integer, seed):
    """Every rank's output of GEMM+AllReduce is the exact sum of the W products (any M)."""
    rng = np.random.default_rng(seed)
    A = [rand_bf16_bits(rng, (M, K), integer) for _ in range(W)]
    B = [rand_bf16_bits(rng, (K, N), integer) for _ in range(W)]
    exact = [[Fraction(0)] * N for _ in range(M)]
    mag = [[Fraction(0)] * N for _ in range(M)]
    for r in range(W):
        Aq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in A[r]]
        Bq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in B[r]]
        P = brute_gemm(Aq, Bq)
        for i in range(M):
            for n in range(N):
                exact[i][n] += P[i][n]
                mag[i][n] += sum(abs(Aq[i][k] * Bq[k][n]) for k in range(K))
    outs = gemm_ar(A, B, "bf16")
    assert len(outs) == W
    for o in outs:
        assert o.shape == (M, N)
        for i in range(M):
            for n in range(N):
                if integer:
                    assert o[i, n] == exact[i][n]
                else:
                    assert abs(Fraction(o[i, n]) - exact[i][n]) <= mag[i][n] * Fraction(W * K + W, 2 ** 52)


@pytest.mark.parametrize("W,M", [(1, 3), (2, 3), (3, 5), (4, 2)])
@pytest.mark.parametrize("integer", [True, False])
def test_ar_brute_force(W, M, integer):
    # M = 3, 5, 2 against W = 2, 3, 4: row counts that do not divide among the ranks
    check_ar_brute(R.gemm_ar, W, M, K=4 + W, N=5, integer=integer, seed=91 + 7 * W + integer)


def test_ar_is_reducescatter_then_allgather():
    # AllReduce = ReduceScatter followed by AllGather of the shards (where M divides by W)
    wl = workloads.with_shape(workloads.WORKLOADS["rs_w8"], W=4, M=64, K=48, N=40)
    inp = workloads.make_inputs(wl)
    outs = R.gemm_ar(inp.a, inp.b)
    gathered = np.concatenate(R.gemm_rs(inp.a, inp.b))
    for o in outs:
        assert np.array_equal(o, gathered)
    rows = np.array([0, 17, 63])
    assert np.array_equal(R.gemm_rs_rows(inp.a, inp.b, rows), outs[2][rows])


def _mut_ar_one_rank_missing(a, b, dtype="bf16", scale_a=None, scale_b=None):
    outs = R.gemm_ar(a, b, dtype)
    outs[-1] = R.gemm_ar(a[:-1], b[:-1], dtype)[0] if len(a) > 1 else outs[-1] * 0
    return outs


def _mut_ar_shard_only(a, b, dtype="bf16", scale_a=None, scale_b=None):
    S = R.gemm_ar(a, b, dtype)[0]
    outs = [S.copy() for _ in a]
    outs[0][1:] = 0          # rank 0 keeps only its own first row, as if the AllGather were skipped
    return outs


@pytest.mark.parametrize("mut", [_mut_ar_one_rank_missing, _mut_ar_shard_only])
def test_planted_ar_mistakes_are_caught(mut):
    with pytest.raises(AssertionError):
        check_ar_brute(mut, 3, 4, 3, 3, True, 5)


# ------------------------------------------------------------------ hand-worked fixtures

def _bf16(a):
    return workloads.to_bf16_bits(np.asarray(a, dtype=np.float32))


def check_golden_ag(ag_gemm, golden):
    for ex in golden["ag_gemm"]:
        shards = [_bf16(s) for s in ex["shards"]]
        got = ag_gemm(shards, _bf16(ex["B"]), "bf16")
        assert np.array_equal(got, np.asarray(ex["C"], dtype=np.float64))
    ex = golden["ag_gemm_e4m3"]
    shards = [np.asarray(s, dtype=np.uint8) for s in ex["shards"]]
    got = ag_gemm(shards, np.asarray(ex["B"], dtype=np.uint8), "e4m3", ex["scale_a"], ex["scale_b"])
    assert np.array_equal(got, np.asarray(ex["C"], dtype=np.float64))


def check_golden_rs(gemm_rs, golden):
    for ex in golden["gemm_rs"]:
        A = [_bf16(a) for a in ex["A"]]
        B = [_bf16(b) for b in ex["B"]]
        got = gemm_rs(A, B, "bf16")
        for j, want in enumerate(ex["out"]):
            assert np.array_equal(got[j], np.asarray(want, dtype=np.float64))


def test_golden_rs_bf16_partials(golden):
    ex = golden["gemm_rs_bf16_partials"]
    A = [_bf16(a) for a in ex["A"]]
    B = [_bf16(b) for b in ex["B"]]
    for mode, key in (("fp32", "out_fp32_partials"), ("bf16", "out_bf16_partials")):
        got = R.gemm_rs(A, B, "bf16", partials=mode)
        for j, want in enumerate(ex[key]):
            assert np.array_equal(R.decode_bf16(R.round_out(got[j], "bf16")), np.asarray(want, dtype=np.float64))
    ar = R.gemm_ar(A, B, "bf16", partials="bf16")
    assert R.decode_bf16(R.round_out(ar[1], "bf16"))[0, 0] == 256


def fraction_to_bf16(x: Fraction) -> Fraction:
    """Round an exact rational to the nearest bf16 value, ties to an even significand (8 significant
    bits), by exact rational arithmetic: an independent restatement for the pins."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = 0
    while a >= 2:
        a /= 2
        e += 1
    while a < 1:
        a *= 2
        e -= 1
    e = max(e, -126)                       # subnormals share the smallest exponent's spacing
    ulp = Fraction(2) ** (e - 7)
    q = abs(x) / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * ulp


def test_fraction_bf16_rounding_agrees_with_torch():
    rng = np.random.default_rng(8)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 6, 2000),
                        np.arange(250, 270, dtype=np.float64)]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    for xi, wi in zip(x, want):
        assert fraction_to_bf16(Fraction(float(xi))) == Fraction(float(wi))


def check_rs_bf16_partials_brute(gemm_rs, W, seed):
    rng = np.random.default_rng(seed)
    M, K, N = W, 3, 4
    A = [rand_bf16_bits(rng, (M, K), False) for _ in range(W)]
    B = [rand_bf16_bits(rng, (K, N), False) for _ in range(W)]
    exact = [[Fraction(0)] * N for _ in range(M)]
    for r in range(W):
        Aq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in A[r]]
        Bq = [[bf16_bits_to_fraction(int(v)) for v in row] for row in B[r]]
        P = brute_gemm(Aq, Bq)
        for i in range(M):
            for n in range(N):
                exact[i][n] += fraction_to_bf16(P[i][n])
    shards = gemm_rs(A, B, "bf16", partials="bf16")
    for j in range(W):
        for n in range(N):
            # the sum of W bf16 values is exact in fp64 here (few terms, close exponents)
            assert Fraction(shards[j][0, n]) == exact[j][n]
    # the final rounding of the exact sum, also by the independent rule
    out = R.decode_bf16(R.round_out(np.concatenate(shards), "bf16"))
    for i in range(M):
        for n in range(N):
            assert Fraction(out[i, n]) == fraction_to_bf16(exact[i][n])


@pytest.mark.parametrize("W", [2, 3])
def test_rs_bf16_partials_brute_force(W):
    check_rs_bf16_partials_brute(R.gemm_rs, W, 500 + W)
    check_rs_bf16_partials_brute(
        lambda a, b, dt, partials: [R.gemm_ar(a, b, dt, partials=partials)[W - 1][j:j + 1] for j in range(W)],
        W, 600 + W)


def test_bf16_partials_equal_fp32_when_partials_are_representable():
    wl = workloads.with_shape(workloads.WORKLOADS["rs_w8"], W=4, M=8, K=2, N=8)
    inp = workloads.make_inputs(wl, integer=True)     # |P_r| <= 32: every integer partial fits bf16
    a = np.concatenate(R.gemm_rs(inp.a, inp.b, partials="fp32"))
    b = np.concatenate(R.gemm_rs(inp.a, inp.b, partials="bf16"))
    assert np.array_equal(a, b)
    rows = np.array([1, 6])
    assert np.array_equal(R.gemm_rs_rows(inp.a, inp.b, rows, partials="bf16"), b[rows])


def _mut_round_running_sum(a, b, dtype="bf16", partials="fp32"):
    # a ring's rounding: the running sum is rounded at every hand-over instead of each partial
    S = None
    for r in range(len(a)):
        P = R.decode(a[r], dtype) @ R.decode(b[r], dtype)
        S = P if S is None else S + P
        S = R.decode_bf16(R.round_bf16_rne(S))
    h = S.shape[0] // len(a)
    return [S[j * h:(j + 1) * h] for j in range(len(a))]


def _mut_truncated_partials(a, b, dtype="bf16", partials="fp32"):
    S = None
    for r in range(len(a)):
        P = (R.decode(a[r], dtype) @ R.decode(b[r], dtype)).astype(np.float32)
        P = (P.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
        S = P if S is None else S + P
    h = S.shape[0] // len(a)
    return [S[j * h:(j + 1) * h] for j in range(len(a))]


def _mut_fp32_partials(a, b, dtype="bf16", partials="fp32"):
    return R.gemm_rs(a, b, dtype)


@pytest.mark.parametrize("mut", [_mut_round_running_sum, _mut_truncated_partials, _mut_fp32_partials])
def test_planted_partial_rounding_mistakes_are_caught(mut):
    with pytest.raises(AssertionError):
        for seed in range(5):
            check_rs_bf16_partials_brute(mut, 3, 700 + seed)


def test_golden_ag(golden):
    check_golden_ag(R.ag_gemm, golden)


def test_golden_rs(golden):
    check_golden_rs(R.gemm_rs, golden)


def test_golden_e4m3_codes(golden):
    ex = golden["e4m3_codes"]
    for code, val in ex.items():
        if code.startswith("_") or code == "nan":
            continue
        got = R.decode_e4m3(np.array([int(code)], dtype=np.uint8))[0]
        assert got == val and np.signbit(got) == np.signbit(val)
    for code in ex["nan"]:
        assert np.isnan(R.decode_e4m3(np.array([code], dtype=np.uint8))[0])


def test_golden_bf16_rne(golden):
    for expr, bits in golden["bf16_rne"]["cases"]:
        x = float(eval(expr))   # the fixture's own arithmetic on exact powers of two
        assert int(R.round_bf16_rne(np.array([x]))[0]) == bits, expr


# ------------------------------------------------------------------ number formats vs library

def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = R.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = R.decode_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_bf16_rne_matches_torch_on_fp32_inputs():
    # For inputs that are already binary32 values there is no double rounding, so torch's
    # fp32 -> bf16 cast (round to nearest even) is an independent reference.
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),   # subnormal range
        (rng.standard_normal(20000) * 1e38).astype(np.float32),    # near overflow
        np.array([0.0, -0.0, np.inf, -np.inf], dtype=np.float32),
    ])
    # force exact ties: low 16 bits = 0x8000
    ties = (rng.integers(0, 1 << 31, 20000, dtype=np.uint32) & np.uint32(0x7F7F0000)) | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32)])
    ours = R.round_bf16_rne(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rne_single_rounding_from_fp64():
    # A value just above a bf16 tie that rounds to the tie in binary32: one rounding (fp64 ->
    # bf16) must go up; rounding through fp32 first would go to even (down).
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert int(R.round_bf16_rne(np.array([x]))[0]) == 0x3F81
    assert np.float32(x) == np.float32(1.0 + 2.0 ** -8)


def test_round_out_fp32():
    x = np.array([1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 0.1])
    assert np.array_equal(R.round_out(x, "fp32"), np.array([1.0, 1.0 + 2.0 ** -22, np.float32(0.1)], dtype=np.float32))


# ------------------------------------------------------------------ special cases / invariants

def test_identity_B_gives_gathered_shards():
    rng = np.random.default_rng(11)
    W, M_local, K = 4, 3, 16
    shards = [rand_bf16_bits(rng, (M_local, K), False) for _ in range(W)]
    eye = _bf16(np.eye(K))
    C = R.ag_gemm(shards, eye, "bf16")
    want = np.concatenate([R.decode_bf16(s) for s in shards])
    assert np.array_equal(C, want)
    assert np.array_equal(R.decode_bf16(R.round_out(C, "bf16")), want)   # bf16 values round to themselves


def test_identity_B_gives_summed_slices():
    rng = np.random.default_rng(12)
    W, M, K = 4, 8, 8
    A = [rand_bf16_bits(rng, (M, K), False) for _ in range(W)]
    eye = [_bf16(np.eye(K)) for _ in range(W)]
    out = R.gemm_rs(A, eye, "bf16")
    for j in range(W):
        for i in range(M // W):
            for k in range(K):
                want = sum((bf16_bits_to_fraction(int(A[r][j * (M // W) + i, k])) for r in range(W)),
                           Fraction(0))
                assert Fraction(out[j][i, k]) == want


def test_ones_closed_form():
    W, M_local, K, N = 3, 4, 37, 5
    ones = _bf16(np.ones((M_local, K)))
    C = R.ag_gemm([ones] * W, _bf16(np.ones((K, N))), "bf16")
    assert np.array_equal(C, np.full((W * M_local, N), float(K)))
    out = R.gemm_rs([_bf16(np.ones((8, K)))] * 2, [_bf16(np.ones((K, N)))] * 2, "bf16")
    assert all(np.array_equal(o, np.full((4, N), 2.0 * K)) for o in out)


def test_rank_permutation_equivariance():
    rng = np.random.default_rng(13)
    W, M_local, K, N = 4, 2, 9, 5
    shards = [rand_bf16_bits(rng, (M_local, K), True) for _ in range(W)]
    b = rand_bf16_bits(rng, (K, N), True)
    C = R.ag_gemm(shards, b, "bf16")
    perm = [2, 0, 3, 1]
    Cp = R.ag_gemm([shards[p] for p in perm], b, "bf16")
    for i, p in enumerate(perm):
        assert np.array_equal(Cp[i * M_local:(i + 1) * M_local], C[p * M_local:(p + 1) * M_local])
    # GEMM-RS output does not depend on the rank order (exact on integers)
    A = [rand_bf16_bits(rng, (8, K), True) for _ in range(W)]
    B = [rand_bf16_bits(rng, (K, N), True) for _ in range(W)]
    o1 = R.gemm_rs(A, B, "bf16")
    o2 = R.gemm_rs([A[p] for p in perm], [B[p] for p in perm], "bf16")
    assert all(np.array_equal(x, y) for x, y in zip(o1, o2))


def test_linearity_exact():
    rng = np.random.default_rng(14)
    shards = [rand_bf16_bits(rng, (3, 8), False) for _ in range(2)]
    b = rand_bf16_bits(rng, (8, 4), False)
    twice = [workloads.to_bf16_bits(2 * R.decode_bf16(s).astype(np.float32)) for s in shards]
    assert np.array_equal(R.ag_gemm(twice, b, "bf16"), 2 * R.ag_gemm(shards, b, "bf16"))


def test_scales_apply_per_rank():
    codes = [np.full((2, 4), 0x38, dtype=np.uint8), np.full((2, 4), 0x40, dtype=np.uint8)]
    b = np.full((4, 3), 0x38, dtype=np.uint8)
    C = R.ag_gemm(codes, b, "e4m3", [2.0, 0.5], 0.25)
    assert np.array_equal(C[:2], np.full((2, 3), 2.0 * 0.25 * 4))
    assert np.array_equal(C[2:], np.full((2, 3), 0.5 * 0.25 * 8))


def test_sampled_rows_match_full():
    wl = workloads.with_shape(workloads.WORKLOADS["ag_w8"], W=3, M=8, K=32, N=16)
    inp = workloads.make_inputs(wl)
    full = R.ag_gemm(inp.a, inp.b[0], "bf16")
    rows = [0, 5, 8, 23]
    assert np.array_equal(R.ag_gemm_rows(inp.a, inp.b[0], rows, "bf16"), full[rows])
    wl = workloads.with_shape(workloads.WORKLOADS["rs_w8"], W=4, M=8, K=16, N=8)
    inp = workloads.make_inputs(wl)
    shards = R.gemm_rs(inp.a, inp.b, "bf16")
    S = np.concatenate(shards)
    rows = [1, 2, 7]
    assert np.allclose(R.gemm_rs_rows(inp.a, inp.b, rows, "bf16"), S[rows], rtol=1e-15, atol=0)


def test_integer_mode_is_exact_at_config_magnitudes():
    # Integer inputs in [-4, 4]: |sum| <= 16*K*W < 2**24, so every value is an exact integer
    # and the bf16/fp32 rounding of it is deterministic.
    wl = workloads.with_shape(workloads.WORKLOADS["rs_w8"], M=16, K=3584, N=8)
    inp = workloads.make_inputs(wl, integer=True)
    out = np.concatenate(R.gemm_rs(inp.a, inp.b, "bf16"))
    assert np.array_equal(out, np.round(out))
    assert np.abs(out).max() < 2 ** 24


# ------------------------------------------------------------------ bookkeeping definitions

def _check_release_order(order, W, M_local, chunk, self_rank):
    """What the pages fix about the producer's order, as invariants: every chunk exactly once,
    ranks in ring order from self+1 with the local shard last, chunks ascending within a rank."""
    n = M_local // chunk
    assert sorted(order) == [(r, c) for r in range(W) for c in range(n)]
    ranks = [order[i * n][0] for i in range(W)]
    assert ranks[-1] == self_rank
    assert all((b - a) % W == 1 for a, b in zip(ranks, ranks[1:]))
    for i in range(W):
        assert [c for _, c in order[i * n:(i + 1) * n]] == list(range(n))
        assert len({r for r, _ in order[i * n:(i + 1) * n]}) == 1


@pytest.mark.parametrize("W,M_local,chunk,self_rank", [(8, 1024, 128, 3), (8, 16, 16, 0), (2, 64, 32, 1),
                                                       (5, 96, 32, 4), (1, 128, 64, 0)])
def test_chunk_release_order_invariants(W, M_local, chunk, self_rank):
    _check_release_order(R.ag_chunk_release_order(W, M_local, chunk, self_rank), W, M_local, chunk, self_rank)


def test_arrival_order_matches_release_order():
    # the consumer takes the ranks in the order their rows become available: its own shard first
    # (read in place), then the peers in the producer's release order
    for W in (1, 2, 5, 8, 16):
        for s in range(W):
            arr = R.ag_arrival_rank_order(W, s)
            assert sorted(arr) == list(range(W)) and arr[0] == s
            rel = R.ag_chunk_release_order(W, 4 * W, 4, s)
            peers = [r for i, (r, c) in enumerate(rel) if c == 0 and r != s]
            assert arr[1:] == peers


def test_consumer_order_check():
    W, M_local = 4, 256
    # any raster inside a rank is accepted: rows of rank 2 (self) in any order, then 3, 0, 1
    ok = [600, 512, 700, 768, 1000, 0, 100, 300]
    assert R.ag_consumer_order_ok(ok, W, M_local, self_rank=2)
    # going back to an earlier rank, or starting with a peer, is rejected
    assert not R.ag_consumer_order_ok([512, 768, 600], W, M_local, self_rank=2)
    assert not R.ag_consumer_order_ok([0, 512], W, M_local, self_rank=2)
    # a block whose first row is in rank 0 counts as rank 0's (the tiny config: one 128-row tile
    # covers both 64-row shards)
    assert R.ag_consumer_order_ok([0], 2, 64, self_rank=1)
    assert R.ag_consumer_order_ok([], 8, 1024, self_rank=5)


def test_fold_order_and_flags():
    for W in (1, 2, 8, 16):
        f = R.rs_fold_order(W)
        assert f == sorted(f) and f[0] == 0 and len(set(f)) == W == len(f)
    # the fold order decides the fp32 bits: the left fold of these partials in rank order differs
    # from the reverse order, so a fixed order is what makes the result identical run to run
    p = np.array([2.0 ** 24, 1.0, 1.0, -(2.0 ** 24)], dtype=np.float32)
    fwd = np.float32(0)
    for r in R.rs_fold_order(4):
        fwd = np.float32(fwd + p[r])
    rev = np.float32(0)
    for r in reversed(R.rs_fold_order(4)):
        rev = np.float32(rev + p[r])
    assert fwd != rev
    assert np.array_equal(R.expected_flags(3, 7), np.array([7, 7, 7], dtype=np.uint32))


def test_planted_order_mistakes_are_caught():
    W, M_local, chunk, s = 8, 256, 128, 3
    good = R.ag_chunk_release_order(W, M_local, chunk, s)
    self_first = [(s, c) for c in range(2)] + [x for x in good if x[0] != s]
    reversed_ring = sorted(good, key=lambda rc: ((s - rc[0]) % W == 0, (s - rc[0]) % W, rc[1]))
    chunks_descending = [(r, 1 - c) for r, c in good]
    for bad in (self_first, reversed_ring, chunks_descending):
        with pytest.raises(AssertionError):
            _check_release_order(bad, W, M_local, chunk, s)


# ------------------------------------------------------------------ planted mistakes

def _mut_transposed_b(shards, b, dtype="bf16", scale_a=None, scale_b=None):
    G = np.concatenate([R.decode(s, dtype) for s in shards])
    Bd = R.decode(b, dtype)
    return G @ Bd.T if Bd.shape[0] == Bd.shape[1] else G @ Bd[:, ::-1]


def _mut_reversed_concat(shards, b, dtype="bf16", scale_a=None, scale_b=None):
    return R.ag_gemm(list(reversed(shards)), b, dtype, scale_a, scale_b)


def _mut_dropped_term(shards, b, dtype="bf16", scale_a=None, scale_b=None):
    G = np.concatenate([R.decode(s, dtype) for s in shards])
    return G[:, 1:] @ R.decode(b, dtype)[1:] if G.shape[1] > 1 else 0 * G @ R.decode(b, dtype)


def _mut_rs_dropped_rank(a, b, dtype="bf16", scale_a=None, scale_b=None):
    return R.gemm_rs(a[1:] + [a[0] * 0], b, dtype) if len(a) > 1 else R.gemm_rs(a, b, dtype)


def _mut_rs_wrong_slice(a, b, dtype="bf16", scale_a=None, scale_b=None):
    return list(reversed(R.gemm_rs(a, b, dtype)))


def _mut_rs_sign(a, b, dtype="bf16", scale_a=None, scale_b=None):
    out = R.gemm_rs(a[:1], b[:1], dtype)
    rest = R.gemm_rs(a[1:], b[1:], dtype) if len(a) > 1 else None
    if rest is None:
        return out
    # partial of rank >= 1 subtracted instead of added (shard count follows the full W)
    full = np.concatenate(R.gemm_rs(a, b, dtype))
    p0 = R.decode(a[0], dtype) @ R.decode(b[0], dtype)
    wrong = 2 * p0 - full
    h = wrong.shape[0] // len(a)
    return [wrong[j * h:(j + 1) * h] for j in range(len(a))]


@pytest.mark.parametrize("mut", [_mut_transposed_b, _mut_reversed_concat, _mut_dropped_term])
def test_planted_ag_mistakes_are_caught(mut, golden):
    caught = 0
    try:
        check_golden_ag(mut, golden)
    except AssertionError:
        caught += 1
    try:
        check_ag_brute(mut, 2, 2, 4, 4, True, 3)
    except (AssertionError, ValueError):
        caught += 1
    assert caught > 0


@pytest.mark.parametrize("mut", [_mut_rs_dropped_rank, _mut_rs_wrong_slice, _mut_rs_sign])
def test_planted_rs_mistakes_are_caught(mut, golden):
    caught = 0
    try:
        check_golden_rs(mut, golden)
    except AssertionError:
        caught += 1
    try:
        check_rs_brute(mut, 3, 6, 4, 3, True, 4)
    except AssertionError:
        caught += 1
    assert caught > 0


def test_planted_format_mistakes_are_caught():
    # wrong exponent bias in e4m3, and truncation instead of rounding in bf16
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    bad = R.decode_e4m3(codes) * 2.0
    ok = ~np.isnan(ref)
    assert not np.array_equal(bad[ok], ref[ok])
    x = np.array([1.0 + 3 * 2.0 ** -8])
    trunc = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert int(trunc[0]) != int(R.round_bf16_rne(x)[0])


def test_oracle_package_exports():
    for name in ["ag_gemm", "gemm_rs", "gemm_ar", "round_out", "ag_chunk_release_order", "ag_arrival_rank_order",
                 "ag_consumer_order_ok", "rs_fold_order"]:
        assert hasattr(oracle, name)
