"""Pins for the oracle, on the CPU: each checks it against something other than
itself (library routines, exact integer brute force, closed forms, a worked
example), so that a dropped term, a wrong sign or index or a transposed
operand anywhere in it fails at least one test.
"""
import numpy as np
import pytest

import oracle
from dense_gemm_fp16_gb300 import workloads as wl


# ----------------------------------------------------------------------------
# binary16 conversions against numpy's own float16 <-> float64 casts
# ----------------------------------------------------------------------------

def test_half_decode_all_bit_patterns_match_numpy():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.half_to_f64(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros decode with their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_half_encode_round_nearest_even_matches_numpy():
    rng = np.random.default_rng(7)
    halves = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).view(np.float16)
    finite = halves[np.isfinite(halves)].astype(np.float64)
    # every finite half, the midpoints between neighbours (ties), and nudges around them
    srt = np.unique(finite)
    mids = (srt[:-1] + srt[1:]) / 2
    nudged = np.concatenate([mids * (1 + 2.0 ** -40), mids * (1 - 2.0 ** -40)])
    special = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, -1e9,
                        2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26, 2.0 ** -14,
                        np.inf, -np.inf])
    rand = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-5, 20000),
                           rng.uniform(-7e4, 7e4, 20000)])
    x = np.concatenate([finite, mids, nudged, special, rand])
    got = oracle.f64_to_half_rn(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)
    assert oracle.f64_to_half_rn(np.array([np.nan]))[0] & 0x7C00 == 0x7C00


# ----------------------------------------------------------------------------
# fp16 NT:  C = A·Bᵀ,  A [M,K], B [N,K]
# ----------------------------------------------------------------------------

def _rand_half(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def test_f16_nt_identity_is_exact():
    A = _rand_half((7, 13), 1)
    B = np.eye(13, dtype=np.float16)           # B [N=K, K] = I
    C, S = oracle.gemm_f16_nt(A, B)
    assert C.shape == (7, 13)
    assert np.array_equal(C, A.astype(np.float64))
    assert np.array_equal(S, np.abs(A.astype(np.float64)))


def test_f16_nt_permutation_permutes_columns():
    A = _rand_half((9, 11), 2)
    perm = np.random.default_rng(3).permutation(11)
    B = np.eye(11, dtype=np.float16)[perm]     # row j of B is e_{perm[j]}
    C, _ = oracle.gemm_f16_nt(A, B)
    assert np.array_equal(C, A.astype(np.float64)[:, perm])


def test_f16_nt_small_integers_exact_against_brute_force():
    rng = np.random.default_rng(4)
    M, N, K = 5, 6, 9
    Ai = rng.integers(-3, 4, (M, K))
    Bi = rng.integers(-3, 4, (N, K))
    C, S = oracle.gemm_f16_nt(Ai.astype(np.float16), Bi.astype(np.float16))
    for i in range(M):
        for j in range(N):
            exact = sum(int(Ai[i, k]) * int(Bi[j, k]) for k in range(K))
            mag = sum(abs(int(Ai[i, k]) * int(Bi[j, k])) for k in range(K))
            assert C[i, j] == exact
            assert S[i, j] == mag


def test_f16_nt_hand_example_2x3x4():
    # A = [[1,2,3,4],[5,6,7,8]], B (rows are the right operand's columns):
    #   B = [[1,0,0,0],[0,1,0,0],[1,1,1,1]]
    # row 0: (1, 2, 1+2+3+4 = 10);  row 1: (5, 6, 5+6+7+8 = 26)
    A = np.array([[1, 2, 3, 4], [5, 6, 7, 8]], dtype=np.float16)
    B = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [1, 1, 1, 1]], dtype=np.float16)
    C, S = oracle.gemm_f16_nt(A, B)
    assert C.tolist() == [[1, 2, 10], [5, 6, 26]]
    assert S.tolist() == [[1, 2, 10], [5, 6, 26]]


@pytest.mark.parametrize("M,N,K", [(37, 23, 51), (1, 64, 200), (65, 1, 3), (16, 16, 1)])
def test_f16_nt_matches_numpy_matmul(M, N, K):
    A = _rand_half((M, K), 10 + M)
    B = _rand_half((N, K), 20 + N)
    C, S = oracle.gemm_f16_nt(A, B)
    a, b = A.astype(np.float64), B.astype(np.float64)
    Cn = a @ b.T
    Sn = np.abs(a) @ np.abs(b).T
    assert np.all(np.abs(C - Cn) <= 1e-12 * Sn + 1e-300)
    assert np.allclose(S, Sn, rtol=1e-12, atol=0)


def test_f16_nt_rejects_inner_dimension_mismatch():
    with pytest.raises(ValueError):
        oracle.gemm_f16_nt(np.zeros((2, 3), np.float16), np.zeros((2, 4), np.float16))


def test_f16_nt_empty_and_k0():
    C, S = oracle.gemm_f16_nt(np.zeros((0, 5), np.float16), np.zeros((3, 5), np.float16))
    assert C.shape == (0, 3)
    C, S = oracle.gemm_f16_nt(np.zeros((4, 0), np.float16), np.zeros((3, 0), np.float16))
    assert C.shape == (4, 3) and not C.any() and not S.any()


def test_f16_nt_sampled_equals_full():
    A = _rand_half((40, 70), 5)
    B = _rand_half((33, 70), 6)
    C, S = oracle.gemm_f16_nt(A, B)
    rows, cols = wl.sample_positions(40, 33, 100, seed=9, tail_rows=[38, 39])
    Cs, Ss = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    assert np.array_equal(Cs, C[rows, cols])
    assert np.array_equal(Ss, S[rows, cols])


def test_half_of_acc_is_the_pages_stored_value():
    # the page stores half(acc): rounding the f64 result must agree with numpy's cast
    A = _rand_half((8, 300), 11)
    B = _rand_half((8, 300), 12)
    C, _ = oracle.gemm_f16_nt(A, B)
    assert np.array_equal(oracle.f64_to_half_rn(C), C.astype(np.float16).view(np.uint16))


# ----------------------------------------------------------------------------
# fp32 SGEMM:  C = alpha·A·B + beta·C0,  row-major A [M,K], B [K,N]
# ----------------------------------------------------------------------------

def test_sgemm_hand_example_alpha_beta():
    # A·B = [[1,2,10],[5,6,26]]; alpha = 2, beta = 0.5, C0 = 2 everywhere:
    # 2*[[1,2,10],[5,6,26]] + 1 = [[3,5,21],[11,13,53]]
    A = np.array([[1, 2, 3, 4], [5, 6, 7, 8]], dtype=np.float32)
    B = np.array([[1, 0, 1], [0, 1, 1], [0, 0, 1], [0, 0, 1]], dtype=np.float32)
    C0 = np.full((2, 3), 2.0, dtype=np.float32)
    C, S = oracle.sgemm(A, B, alpha=2.0, beta=0.5, C0=C0)
    assert C.tolist() == [[3, 5, 21], [11, 13, 53]]
    assert S.tolist() == [[2, 4, 20], [10, 12, 52]]


def test_sgemm_small_integers_exact_against_brute_force():
    rng = np.random.default_rng(13)
    M, N, K = 4, 7, 6
    Ai = rng.integers(-4, 5, (M, K))
    Bi = rng.integers(-4, 5, (K, N))
    Ci = rng.integers(-4, 5, (M, N))
    C, _ = oracle.sgemm(Ai.astype(np.float32), Bi.astype(np.float32), alpha=3.0, beta=-2.0,
                        C0=Ci.astype(np.float32))
    for i in range(M):
        for j in range(N):
            exact = 3 * sum(int(Ai[i, k]) * int(Bi[k, j]) for k in range(K)) - 2 * int(Ci[i, j])
            assert C[i, j] == exact


@pytest.mark.parametrize("M,N,K,alpha,beta", [(31, 17, 45, 1.5, -0.25), (1, 40, 7, 1.0, 0.0),
                                              (50, 3, 64, -2.0, 1.0)])
def test_sgemm_matches_numpy_matmul(M, N, K, alpha, beta):
    rng = np.random.default_rng(M * 100 + N)
    A = rng.uniform(-1, 1, (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (M, N)).astype(np.float32)
    C, S = oracle.sgemm(A, B, alpha=alpha, beta=beta, C0=C0)
    a, b, c0 = A.astype(np.float64), B.astype(np.float64), C0.astype(np.float64)
    Cn = alpha * (a @ b) + beta * c0
    Sn = abs(alpha) * (np.abs(a) @ np.abs(b))
    assert np.all(np.abs(C - Cn) <= 1e-12 * (Sn + np.abs(beta * c0)) + 1e-300)
    assert np.allclose(S, Sn, rtol=1e-12, atol=0)


def test_sgemm_beta_zero_does_not_read_c0():
    A = np.ones((3, 4), np.float32)
    B = np.ones((4, 5), np.float32)
    C0 = np.full((3, 5), np.nan, np.float32)
    C, _ = oracle.sgemm(A, B, alpha=1.0, beta=0.0, C0=C0)
    assert np.all(C == 4.0)


def test_sgemm_k0_is_beta_c0():
    C0 = np.arange(6, dtype=np.float32).reshape(2, 3)
    C, S = oracle.sgemm(np.zeros((2, 0), np.float32), np.zeros((0, 3), np.float32),
                        alpha=1.0, beta=0.5, C0=C0)
    assert np.array_equal(C, 0.5 * C0.astype(np.float64))
    assert not S.any()


def test_sgemm_sampled_equals_full():
    rng = np.random.default_rng(21)
    A = rng.uniform(-1, 1, (30, 20)).astype(np.float32)
    B = rng.uniform(-1, 1, (20, 25)).astype(np.float32)
    C0 = rng.uniform(-1, 1, (30, 25)).astype(np.float32)
    C, S = oracle.sgemm(A, B, 1.0, 0.5, C0)
    rows, cols = wl.sample_positions(30, 25, 60, seed=1)
    Cs, Ss = oracle.sgemm_sampled(A, B, rows, cols, 1.0, 0.5, C0)
    assert np.array_equal(Cs, C[rows, cols])
    assert np.array_equal(Ss, S[rows, cols])


def test_oracle_reports_threads():
    assert oracle.num_threads() >= 1


# ----------------------------------------------------------------------------
# fused epilogue: act(alpha·A·Bᵀ + bias[n] + beta·R[m,n])
# ----------------------------------------------------------------------------

def test_activations_against_library_and_identities():
    from scipy.special import erf, expit

    xs = np.linspace(-12, 12, 481)
    silu = np.array([oracle.activation(x, "silu") for x in xs])
    assert np.allclose(silu, xs * expit(xs), rtol=1e-13, atol=1e-15)
    gelu = np.array([oracle.activation(x, "gelu_tanh") for x in xs])
    exact_gelu = 0.5 * xs * (1 + erf(xs / np.sqrt(2)))
    assert np.max(np.abs(gelu - exact_gelu)) < 1e-3      # the tanh form's approximation error
    relu = np.array([oracle.activation(x, "relu") for x in xs])
    assert np.array_equal(relu, np.maximum(xs, 0))
    # x·σ(x) and the tanh GELU are both of the form x·(1+g(x))/2 with g odd:
    # act(x) − act(−x) = x
    for act in ("silu", "gelu_tanh", "relu"):
        for x in (0.3, 1.7, -4.2, 9.0):
            assert abs(oracle.activation(x, act) - oracle.activation(-x, act) - x) < 1e-12
    assert oracle.activation(0.0, "silu") == 0.0 and oracle.activation(0.0, "gelu_tanh") == 0.0


def test_epilogue_exact_through_identity():
    # B = I: alpha·A + bias + beta·R exactly for small integers; ReLU clips.
    rng = np.random.default_rng(31)
    M, K = 6, 10
    A = rng.integers(-4, 5, (M, K)).astype(np.float16)
    bias = rng.integers(-3, 4, K).astype(np.float16)
    R = rng.integers(-5, 6, (M, K)).astype(np.float16)
    B = np.eye(K, dtype=np.float16)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=2.0, bias=bias, beta=-1.5, R=R)
    exact = 2.0 * A.astype(np.float64) + bias.astype(np.float64) - 1.5 * R.astype(np.float64)
    assert np.array_equal(Y, exact)
    assert np.array_equal(S, 2 * np.abs(A.astype(np.float64)) + np.abs(bias.astype(np.float64))
                          + 1.5 * np.abs(R.astype(np.float64)))
    Yr, _ = oracle.gemm_f16_nt_epilogue(A, B, alpha=2.0, bias=bias, beta=-1.5, R=R, act="relu")
    assert np.array_equal(Yr, np.maximum(exact, 0))


@pytest.mark.parametrize("act", ["none", "relu", "silu", "gelu_tanh"])
def test_epilogue_matches_numpy(act):
    from scipy.special import expit

    rng = np.random.default_rng(41)
    M, N, K = 13, 29, 37
    A = rng.standard_normal((M, K)).astype(np.float16)
    B = rng.standard_normal((N, K)).astype(np.float16)
    bias = rng.standard_normal(N).astype(np.float16)
    R = rng.standard_normal((M, N)).astype(np.float16)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=0.5, bias=bias, beta=2.0, R=R, act=act)
    v = 0.5 * (A.astype(np.float64) @ B.astype(np.float64).T) + bias.astype(np.float64) \
        + 2.0 * R.astype(np.float64)
    f = {"none": lambda x: x, "relu": lambda x: np.maximum(x, 0), "silu": lambda x: x * expit(x),
         "gelu_tanh": lambda x: 0.5 * x * (1 + np.tanh(np.sqrt(2 / np.pi) * (x + 0.044715 * x ** 3)))}
    assert np.allclose(Y, f[act](v), rtol=1e-12, atol=1e-12)
    # without bias or residual the epilogue reduces to the plain product
    Y0, S0 = oracle.gemm_f16_nt_epilogue(A, B)
    C, Sc = oracle.gemm_f16_nt(A, B)
    assert np.array_equal(Y0, C) and np.array_equal(S0, Sc)


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_epilogue_sampled_agrees_with_full(act):
    rng = np.random.default_rng(43)
    M, N, K = 11, 17, 24
    A = rng.standard_normal((M, K)).astype(np.float16)
    B = rng.standard_normal((N, K)).astype(np.float16)
    bias = rng.standard_normal(N).astype(np.float16)
    R = rng.standard_normal((M, N)).astype(np.float16)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=-0.75, bias=bias, beta=0.5, R=R, act=act)
    rows = np.array([0, 10, 3, 7, 10])
    cols = np.array([0, 16, 5, 0, 2])
    Ys, Ss = oracle.gemm_f16_nt_epilogue_sampled(A, B, rows, cols, alpha=-0.75, bias=bias,
                                                 beta=0.5, R=R, act=act)
    assert np.array_equal(Ys, Y[rows, cols]) and np.array_equal(Ss, S[rows, cols])
    with pytest.raises(RuntimeError):
        oracle.gemm_f16_nt_epilogue_sampled(A, B, [M], [0], act=act)
