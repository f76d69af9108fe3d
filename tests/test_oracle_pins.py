"""Pins for the oracle: each check ties it to something other than itself.

Brute force on tiny integer inputs, algebraic identities, closed forms and
library special cases (torch's float8_e4m3fn and bfloat16 casts). The cases are
chosen so that a plausible slip (a transposed operand, a dropped beta term, a
wrong exponent bias, rounding ties the wrong way) fails at least one of them.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle


def brute_int(A, B, b_layout, C, alpha, beta):
    """Independent int64 triple loop on integer inputs."""
    M, K = len(A), len(A[0])
    N = len(B[0]) if b_layout == "kn" else len(B)
    out = [[0] * N for _ in range(M)]
    for i in range(M):
        for n in range(N):
            s = 0
            for k in range(K):
                s += A[i][k] * (B[k][n] if b_layout == "kn" else B[n][k])
            out[i][n] = alpha * s + (beta * C[i][n] if beta else 0)
    return np.array(out, dtype=np.int64)


# ---------------------------------------------------------------- GEMM core

@pytest.mark.parametrize("b_layout", ["kn", "nk"])
def test_gemm_brute_force_tiny(b_layout):
    rng = np.random.default_rng(7)
    for M, N, K in itertools.product([1, 2, 3, 5, 8], [1, 4, 7], [1, 2, 6, 8]):
        A = rng.integers(-4, 5, size=(M, K))
        B = rng.integers(-4, 5, size=(K, N) if b_layout == "kn" else (N, K))
        C = rng.integers(-4, 5, size=(M, N))
        for alpha, beta in [(1, 0), (2, 3), (-1, 1), (0, 2)]:
            want = brute_int(A.tolist(), B.tolist(), b_layout, C.tolist(), alpha, beta)
            got = oracle.gemm(A, B, b_layout, C, alpha, beta)
            assert np.array_equal(got, want.astype(np.float64)), (M, N, K, alpha, beta)


def test_gemm_hand_case_4x4():
    """A 4x4 case small enough to check by hand (the CUDA-tile page's advice,
    §6: compare a 4x4 result element by element): A = I + J (ones on the
    diagonal plus all-ones), B = diag(1..4), so (AB)[i][n] = (n+1) * (1 + [i==n])."""
    A = np.eye(4) + np.ones((4, 4))
    B = np.diag([1.0, 2.0, 3.0, 4.0])
    got = oracle.gemm(A, B, "kn")
    for i in range(4):
        for n in range(4):
            assert got[i, n] == (n + 1) * (2 if i == n else 1)


def test_gemm_identity_and_transpose():
    rng = np.random.default_rng(11)
    A = rng.standard_normal((37, 29))
    B = rng.standard_normal((29, 23))
    # A . I = A exactly
    assert np.array_equal(oracle.gemm(A, np.eye(29), "kn"), A)
    assert np.array_equal(oracle.gemm(A, np.eye(29), "nk"), A)
    # (A B)^T = B^T A^T, the second evaluated through the NxK layout
    X = oracle.gemm(A, B, "kn")
    Y = oracle.gemm(np.ascontiguousarray(B.T), A, "nk")
    assert np.array_equal(Y, X.T)
    # the two layouts agree on the same mathematical operand
    Z = oracle.gemm(A, np.ascontiguousarray(B.T), "nk")
    assert np.array_equal(Z, X)
    # and a library product agrees to rounding
    assert np.allclose(X, A @ B, rtol=1e-12, atol=1e-12)


def test_gemm_alpha_beta_cases():
    rng = np.random.default_rng(12)
    A = rng.standard_normal((16, 40))
    B = rng.standard_normal((40, 24))
    C = rng.standard_normal((16, 24))
    AB = oracle.gemm(A, B, "kn")
    # alpha = 0: beta * C only
    assert np.array_equal(oracle.gemm(A, B, "kn", C, 0.0, 0.5), 0.5 * C)
    # beta = 0: C is not read, so NaN in C cannot leak
    Cnan = np.full_like(C, np.nan)
    assert np.array_equal(oracle.gemm(A, B, "kn", Cnan, 1.0, 0.0), AB)
    # alpha = 2 scales exactly (power of two)
    assert np.array_equal(oracle.gemm(A, B, "kn", None, 2.0, 0.0), 2.0 * AB)
    # beta term is added once, with the right operand
    got = oracle.gemm(A, B, "kn", C, 1.5, -2.0)
    assert np.allclose(got, 1.5 * AB - 2.0 * C, rtol=1e-14, atol=1e-13)


def test_gemm_row_subset_matches_full():
    rng = np.random.default_rng(13)
    A = rng.standard_normal((50, 33))
    B = rng.standard_normal((21, 33))
    full = oracle.gemm(A, B, "nk")
    part = oracle.gemm(A, B, "nk", rows=(17, 41))
    assert np.array_equal(part, full[17:41])


# ---------------------------------------------------------------- E4M3

def torch_e4m3_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_every_code_matches_torch():
    ours = oracle.decode_e4m3(np.arange(256, dtype=np.uint8))
    ref = torch_e4m3_decode_all()
    nan_o, nan_r = np.isnan(ours), np.isnan(ref)
    assert np.array_equal(nan_o, nan_r)
    assert list(np.nonzero(nan_o)[0]) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan_o], ref[~nan_r])


def test_e4m3_special_values():
    d = lambda c: oracle.decode_e4m3(np.array([c], np.uint8))[0]
    assert d(0x7E) == 448.0
    assert d(0xFE) == -448.0
    assert d(0x08) == 2.0 ** -6          # smallest normal
    assert d(0x01) == 2.0 ** -9          # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9      # largest subnormal
    assert d(0x38) == 1.0                # exponent field 7 = bias
    assert d(0x00) == 0.0 and math.copysign(1, d(0x80)) == -1.0


def test_e4m3_round_trip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.decode_e4m3(codes)
    assert np.array_equal(oracle.encode_e4m3(vals), codes)


def test_e4m3_midpoints_round_to_even():
    finite = oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448
    mids = (finite[:-1] + finite[1:]) / 2
    got = oracle.encode_e4m3(mids)
    lo = np.arange(0x7E, dtype=np.uint8)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    # negative side mirrors
    assert np.array_equal(oracle.encode_e4m3(-mids), want | 0x80)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 0.05, 1, 30, 200)])
    x = x[np.abs(x) <= 448].astype(np.float32).astype(np.float64)
    ours = oracle.encode_e4m3(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.decode_e4m3(ours), oracle.decode_e4m3(ref))


def test_e4m3_saturates():
    assert oracle.decode_e4m3(oracle.encode_e4m3(np.array([449.0, 1e9, -500.0]))).tolist() == [448.0, 448.0, -448.0]
    assert oracle.encode_e4m3(np.array([np.nan]))[0] == 0x7F


# ---------------------------------------------------------------- BF16

def test_bf16_round_matches_torch():
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.standard_normal(50000) * s for s in (1e-30, 1e-3, 1, 1e5, 1e30)])
    x = np.concatenate([x, [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 2 ** -130 * 1.5, 3.0e38, -0.0]])
    x32 = x.astype(np.float32)           # float32 inputs: torch rounds once, from binary32
    ours = oracle.round_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)
    bits = oracle.encode_bf16(x32.astype(np.float64))
    assert np.array_equal(bits, torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_bf16_ties_to_even_and_decode():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties to even -> 1
    assert oracle.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    # 1 + 3*2^-8 lies halfway between 1+2^-7 and 1+2^-6: even mantissa is 1+2^-6
    assert oracle.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6
    assert oracle.decode_bf16(np.array([0x3F80, 0xC000, 0x0001], np.uint16)).tolist() == [1.0, -2.0, 2.0 ** -133]


# ---------------------------------------------------------------- activations

def test_silu_and_gelu_closed_forms():
    assert oracle.silu(0.0) == 0.0 and oracle.gelu(0.0) == 0.0
    for x in [0.1, 0.7, 1.3, 2.5, 7.0, 30.0]:
        # sigmoid(x) + sigmoid(-x) = 1  =>  silu(x) - silu(-x) = x
        assert abs(oracle.silu(x) - oracle.silu(-x) - x) < 1e-15 * max(1, x)
        # Phi(x) + Phi(-x) = 1  =>  gelu(x) - gelu(-x) = x
        assert abs(oracle.gelu(x) - oracle.gelu(-x) - x) < 1e-15 * max(1, x)
    # silu(ln 3) = ln3 * 3/4 (sigmoid(ln 3) = 3/4); gelu at large x tends to x
    assert abs(oracle.silu(math.log(3)) - 0.75 * math.log(3)) < 1e-15
    assert oracle.gelu(40.0) == 40.0 and oracle.silu(-800.0) == 0.0


def test_gelu_is_the_erf_form():
    # gelu(x) = x * Phi(x) with the exact normal CDF: standard-normal table values
    # Phi(1) = 0.841344746068543, Phi(2) = 0.977249868051821, Phi(-0.5) =
    # 0.308537538725987. The tanh approximation misses these by 2e-5 to 2e-4.
    assert abs(oracle.gelu(1.0) - 0.841344746068543) < 1e-14
    assert abs(oracle.gelu(2.0) - 2 * 0.977249868051821) < 1e-14
    assert abs(oracle.gelu(-0.5) - (-0.5) * 0.308537538725987) < 1e-14


def test_epilogue_bias_then_activation():
    X = np.array([[-1.0, 0.0, 2.0]])
    bias = np.array([0.5, -0.25, 1.0], np.float32)
    assert oracle.epilogue(X, bias, "none").tolist() == [[-0.5, -0.25, 3.0]]
    assert oracle.epilogue(X, bias, "relu").tolist() == [[0.0, 0.0, 3.0]]
    y = oracle.epilogue(X, bias, "silu")[0]
    assert abs(y[2] - 3.0 / (1 + math.exp(-3.0))) < 1e-15


# ---------------------------------------------------------------- FP8 path

def test_fp8_unit_scales_reduce_to_plain_gemm():
    rng = np.random.default_rng(8)
    Aq = rng.integers(0, 256, size=(9, 64), dtype=np.uint8)
    Bq = rng.integers(0, 256, size=(13, 64), dtype=np.uint8)
    Aq[(Aq & 0x7F) == 0x7F] = 0x10     # no NaN codes
    Bq[(Bq & 0x7F) == 0x7F] = 0x22
    one_a, one_b = np.ones(9, np.float32), np.ones(13, np.float32)
    got = oracle.fp8_gemm_ref(Aq, Bq, "nk", one_a, one_b)
    plain = oracle.gemm(oracle.decode_e4m3(Aq), oracle.decode_e4m3(Bq), "nk")
    assert np.array_equal(got, plain)


def test_fp8_scales_are_per_row_and_per_column():
    """Distinct scales per row of A and per output channel of B: a transposed scale
    vector (the stride pitfall of the FP8 page, §5.2) changes the answer."""
    rng = np.random.default_rng(9)
    Aq = np.full((4, 32), 0x38, np.uint8)          # all 1.0
    Bq = np.full((6, 32), 0x38, np.uint8)
    sa = np.array([1, 2, 4, 8], np.float32)
    sb = np.array([1, 3, 5, 7, 9, 11], np.float32)
    got = oracle.fp8_gemm_ref(Aq, Bq, "nk", sa, sb)
    assert np.array_equal(got, 32.0 * np.outer(sa, sb))
    # the K x N layout with a per-column scale gives the same
    got_kn = oracle.fp8_gemm_ref(Aq, np.ascontiguousarray(Bq.T), "kn", sa, sb)
    assert np.array_equal(got_kn, got)
    # row sampling
    part = oracle.fp8_gemm_ref(Aq, Bq, "nk", sa, sb, rows=(1, 3))
    assert np.array_equal(part, got[1:3])


def test_requant_rows_invariants():
    rng = np.random.default_rng(10)
    Z = rng.standard_normal((64, 300)) * np.exp(rng.uniform(-5, 5, size=(64, 1)))
    Z[3] = 0.0
    q, s = oracle.requant_rows(Z)
    dq = oracle.decode_e4m3(q)
    assert s[3] == 1.0 and not q[3].any()
    for r in range(64):
        if r == 3:
            continue
        amax_pos = np.argmax(np.abs(Z[r]))
        assert q[r, amax_pos] in (0x7E, 0xFE)
        assert s[r] == np.abs(Z[r]).max() / 448
    assert np.all(np.abs(dq) <= 448)
    # every code is the nearest E4M3 value to z/s: within half a spacing
    x = Z / s[:, None]
    grid = oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    idx = np.searchsorted(grid, np.abs(x)).clip(1, 126)
    spacing = grid[idx] - grid[idx - 1]
    assert np.all(np.abs(np.abs(dq) - np.abs(x)) <= spacing / 2 + 1e-12)


# ---------------------------------------------------------------- FP8 per-K-group scales

def _int_codes(rng, shape):
    """E4M3 codes of small integers in [-8, 8] (exact values, exact sums)."""
    vals = rng.integers(-8, 9, size=shape).astype(np.float64)
    return oracle.encode_e4m3(vals), vals


@pytest.mark.parametrize("b_layout", ["nk", "kn"])
def test_fp8_grouped_brute_force_ragged_k(b_layout):
    """Tiny case, written out index by index: K = 7 in groups of 3 (the last group
    is partial), power-of-two scales, so every product and sum is exact."""
    rng = np.random.default_rng(21)
    M, N, K, g = 3, 4, 7, 3
    G = 3
    Aq, Av = _int_codes(rng, (M, K))
    Bq, Bv = _int_codes(rng, (N, K))
    sa = (2.0 ** rng.integers(-3, 4, size=(G, M))).astype(np.float32)
    sb = (2.0 ** rng.integers(-3, 4, size=(G, N))).astype(np.float32)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            for k in range(K):
                want[m, n] += Av[m, k] * sa[k // g, m] * Bv[n, k] * sb[k // g, n]
    B_in = Bq if b_layout == "nk" else np.ascontiguousarray(Bq.T)
    got = oracle.fp8_gemm_ref(Aq, B_in, b_layout, sa, sb, k_group=g)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("b_layout", ["nk", "kn"])
def test_fp8_grouped_is_sum_of_per_group_gemms(b_layout):
    """Per-group scaling = the sum over K groups of per-row x per-channel scaled
    GEMMs on that group's K slice (each already pinned above)."""
    rng = np.random.default_rng(22)
    M, N, K, g = 10, 12, 40, 16
    G = 3
    Aq, _ = _int_codes(rng, (M, K))
    Bq, _ = _int_codes(rng, (N, K))
    sa = (2.0 ** rng.integers(-4, 5, size=(G, M))).astype(np.float32)
    sb = (2.0 ** rng.integers(-4, 5, size=(G, N))).astype(np.float32)
    want = np.zeros((M, N))
    for j in range(G):
        ks = slice(j * g, min(K, (j + 1) * g))
        want += oracle.fp8_gemm_ref(np.ascontiguousarray(Aq[:, ks]), np.ascontiguousarray(Bq[:, ks]), "nk",
                                    sa[j], sb[j])
    B_in = Bq if b_layout == "nk" else np.ascontiguousarray(Bq.T)
    got = oracle.fp8_gemm_ref(Aq, B_in, b_layout, sa, sb, k_group=g)
    assert np.array_equal(got, want)
    # rows of the result are the GEMM on those rows of A (and of a_scale's columns)
    part = oracle.fp8_gemm_ref(Aq, B_in, b_layout, sa, sb, k_group=g, rows=np.array([7, 2]))
    assert np.array_equal(part, got[[7, 2]])


def test_fp8_grouped_constant_scales_reduce_to_per_row():
    """Scales equal across K groups give the per-row x per-channel result exactly;
    a group size >= K is one group."""
    rng = np.random.default_rng(23)
    Aq, _ = _int_codes(rng, (5, 64))
    Bq, _ = _int_codes(rng, (7, 64))
    sa = rng.uniform(0.5, 2, size=5).astype(np.float32)
    sb = rng.uniform(0.5, 2, size=7).astype(np.float32)
    plain = oracle.fp8_gemm_ref(Aq, Bq, "nk", sa, sb)
    grouped = oracle.fp8_gemm_ref(Aq, Bq, "nk", np.tile(sa, (4, 1)), np.tile(sb, (4, 1)), k_group=16)
    assert np.allclose(grouped, plain, rtol=1e-14, atol=0)
    one = oracle.fp8_gemm_ref(Aq, Bq, "nk", sa[None, :], sb[None, :], k_group=64)
    assert np.array_equal(one, plain)
    with pytest.raises(ValueError):   # a scale table of the wrong orientation
        oracle.fp8_gemm_ref(Aq, Bq, "nk", np.tile(sa, (4, 1)).T.copy(), np.tile(sb, (4, 1)), k_group=16)


def test_fp8_grouped_scale_layout_is_group_major():
    """All-ones codes, scale (j, i) = distinct powers: entry (m, n) is
    sum_j |group j| * sa[j, m] * sb[j, n], which a [L, G] table would not give."""
    M, N, K, g = 2, 3, 10, 4
    Aq = np.full((M, K), 0x38, np.uint8)   # 1.0
    Bq = np.full((N, K), 0x38, np.uint8)
    sa = np.array([[1, 2], [4, 8], [16, 32]], np.float32)          # [G=3, M=2]
    sb = np.array([[1, 3, 5], [7, 9, 11], [13, 15, 17]], np.float32)   # [G=3, N=3]
    sizes = np.array([4, 4, 2], np.float64)
    want = np.einsum("j,jm,jn->mn", sizes, sa.astype(np.float64), sb.astype(np.float64))
    assert np.array_equal(oracle.fp8_gemm_ref(Aq, Bq, "nk", sa, sb, k_group=g), want)
    assert want[0, 0] == 4 * 1 * 1 + 4 * 4 * 7 + 2 * 16 * 13


@pytest.mark.parametrize("b_layout", ["nk", "kn"])
def test_fp8_block_scaled_brute_force(b_layout):
    """Block-scaled weights written out index by index: N = 260 output channels
    in blocks of 128 (the last block 4 wide), K = 10 in groups of 4, one weight
    scale per (K group, channel block); power-of-two scales keep it exact."""
    rng = np.random.default_rng(24)
    M, N, K, g, blk = 3, 260, 10, 4, 128
    G, NB = 3, 3
    Aq, Av = _int_codes(rng, (M, K))
    Bq, Bv = _int_codes(rng, (N, K))
    sa = (2.0 ** rng.integers(-3, 4, size=(G, M))).astype(np.float32)
    sb = (2.0 ** rng.integers(-3, 4, size=(G, NB))).astype(np.float32)
    want = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            for k in range(K):
                want[m, n] += Av[m, k] * sa[k // g, m] * Bv[n, k] * sb[k // g, n // blk]
    B_in = Bq if b_layout == "nk" else np.ascontiguousarray(Bq.T)
    got = oracle.fp8_gemm_ref(Aq, B_in, b_layout, sa, sb, k_group=g, b_block=blk)
    assert np.array_equal(got, want)
    with pytest.raises(ValueError):   # a per-channel table is not a block table
        oracle.fp8_gemm_ref(Aq, B_in, b_layout, sa, np.ones((G, N), np.float32), k_group=g, b_block=blk)
    with pytest.raises(ValueError):   # blocks are a per-group form
        oracle.fp8_gemm_ref(Aq, B_in, b_layout, sa[0], sb[0], b_block=blk)
