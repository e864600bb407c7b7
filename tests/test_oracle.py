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


def _library_activation(xs, act):
    """PyTorch's own float64 activations, an implementation independent of the oracle's C."""
    import torch

    x = torch.tensor(xs, dtype=torch.float64)
    f = {"silu": torch.nn.functional.silu,
         "gelu_tanh": lambda t: torch.nn.functional.gelu(t, approximate="tanh")}[act]
    return f(x).numpy()


# Pointwise agreement with the library: the two differ only in the rounding
# order of a handful of float64 operations, while a wrong digit in a constant
# (0.0447 for 0.044715 moves GELU by up to 4.7e-4) or a wrong sign is many
# orders of magnitude above this bound.
ACT_PIN_REL = 1e-13
ACT_PIN_ABS = 1e-15
ACT_PIN_XS = np.linspace(-8, 8, 1601)


def _activation_pin_error(fn, act):
    ref = _library_activation(ACT_PIN_XS, act)
    got = np.array([fn(x) for x in ACT_PIN_XS])
    return np.max(np.abs(got - ref) / (ACT_PIN_REL * np.abs(ref) + ACT_PIN_ABS))


@pytest.mark.parametrize("act", ["silu", "gelu_tanh"])
def test_activation_pinned_to_library_values(act):
    # tanh-GELU 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) and SiLU v σ(v)
    # point by point against torch.nn.functional (gelu(approximate="tanh"),
    # silu) in float64, e.g. GELU_tanh(1) = 0.8411919906082768.
    assert _activation_pin_error(lambda x: oracle.activation(x, act), act) <= 1.0
    assert oracle.activation(1.0, "gelu_tanh") == pytest.approx(0.8411919906082768, rel=1e-15)


@pytest.mark.parametrize("old,new", [
    ("0.044715 * v * v * v", "0.0447 * v * v * v"),          # a dropped digit
    ("sqrt(2.0 / M_PI)", "sqrt(2.0 / 3.1416)"),              # a rounded pi
    ("0.5 * v * (1.0 + tanh", "0.5 * v * (1.0 - tanh"),      # a wrong sign
])
def test_activation_pin_rejects_a_planted_mistake(tmp_path, old, new):
    # The GELU pin above must fail for a plausible typo: build a scratch copy
    # of the oracle with the mistake planted and evaluate it through the pin.
    import ctypes
    import subprocess

    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation anchor {old!r} not found once"
    path = tmp_path / "gemm_oracle_mutant.c"
    path.write_text(src.replace(old, new))
    lib_path = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", *oracle.GCC_FLAGS, "-o", str(lib_path), str(path), "-lm"])
    lib = ctypes.CDLL(str(lib_path))
    lib.oracle_activation.restype = ctypes.c_double
    lib.oracle_activation.argtypes = [ctypes.c_double, ctypes.c_int]
    code = oracle.ACTIVATIONS["gelu_tanh"]
    assert _activation_pin_error(lambda x: lib.oracle_activation(x, code), "gelu_tanh") > 1e3


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


# ---------------------------------------------------------------------------
# Block-scaled FP8 (MXFP8)
# ---------------------------------------------------------------------------

def test_e4m3_and_ue8m0_decode_every_code_like_torch():
    import torch

    codes = np.arange(256, dtype=np.uint8)
    for ours, dt in ((oracle.e4m3_to_f64(codes), torch.float8_e4m3fn),
                     (oracle.ue8m0_to_f64(codes), getattr(torch, "float8_e8m0fnu", None))):
        if dt is None:
            continue
        ref = torch.from_numpy(codes).view(dt).double().numpy()
        assert np.array_equal(np.isnan(ours), np.isnan(ref))
        assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    # the closed forms: largest finite E4M3 is 448, smallest subnormal 2^-9,
    # UE8M0 127 is 1 and every code e is 2^(e-127)
    e = oracle.e4m3_to_f64(np.array([0x7E, 0x01, 0x38, 0xB8, 0x7F], dtype=np.uint8))
    assert e[0] == 448.0 and e[1] == 2.0 ** -9 and e[2] == 1.0 and e[3] == -1.0 and np.isnan(e[4])
    u = oracle.ue8m0_to_f64(np.arange(255, dtype=np.uint8))
    assert np.array_equal(u, 2.0 ** (np.arange(255) - 127.0))


def _mx_decode_ref(codes, scales):
    # independent decode for the pins: PyTorch's float8 cast, scale repeated
    import torch

    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()
    return v * np.repeat(2.0 ** (scales.astype(np.float64) - 127.0), 32, axis=1)


def test_mxfp8_small_integers_exact_against_brute_force():
    # E4M3 represents the integers -8..8 exactly; scales 127 (x1), 128 (x2)
    # and 126 (x1/2) keep every product and sum exact.
    rng = np.random.default_rng(51)
    M, N, K = 5, 7, 64
    import torch

    ai = rng.integers(-8, 9, (M, K))
    bi = rng.integers(-8, 9, (N, K))
    A = torch.from_numpy(ai.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    B = torch.from_numpy(bi.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    SA = rng.integers(126, 129, (M, K // 32)).astype(np.uint8)
    SB = rng.integers(126, 129, (N, K // 32)).astype(np.uint8)
    C, S = oracle.gemm_mxfp8_nt(A, SA, B, SB)
    from fractions import Fraction

    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(int(ai[i, k]) * int(bi[j, k])) *
                        Fraction(2) ** (int(SA[i, k // 32]) + int(SB[j, k // 32]) - 254)
                        for k in range(K))
            assert C[i, j] == float(exact)
            assert S[i, j] == float(sum(abs(Fraction(int(ai[i, k]) * int(bi[j, k]))) *
                                        Fraction(2) ** (int(SA[i, k // 32]) + int(SB[j, k // 32]) - 254)
                                        for k in range(K)))


def test_mxfp8_each_scale_covers_its_own_32_elements():
    # Ones everywhere; only block b of row 0 of A gets scale 2^3: the result
    # grows by exactly 7 * 32 (one block of ones now worth 8 instead of 1).
    M, N, K = 2, 3, 128
    one = 0x38
    A = np.full((M, K), one, np.uint8)
    B = np.full((N, K), one, np.uint8)
    SA = np.full((M, K // 32), 127, np.uint8)
    SB = np.full((N, K // 32), 127, np.uint8)
    base, _ = oracle.gemm_mxfp8_nt(A, SA, B, SB)
    assert np.all(base == K)
    for b in range(K // 32):
        SA2 = SA.copy()
        SA2[0, b] = 130
        C, _ = oracle.gemm_mxfp8_nt(A, SA2, B, SB)
        assert np.all(C[0] == K + 7 * 32) and np.all(C[1] == K)
        SB2 = SB.copy()
        SB2[2, b] = 125
        C, _ = oracle.gemm_mxfp8_nt(A, SA, B, SB2)
        assert np.all(C[:, 2] == K - 0.75 * 32) and np.all(C[:, :2] == K)


def test_mxfp8_matches_numpy_and_sampled():
    from dense_gemm_fp16_gb300 import workloads as wl

    M, N, K = 37, 29, 160
    A, SA = wl.draw_mxfp8(M, K, seed=61)
    B, SB = wl.draw_mxfp8(N, K, seed=62)
    A, SA, B, SB = A.numpy(), SA.numpy(), B.numpy(), SB.numpy()
    C, S = oracle.gemm_mxfp8_nt(A, SA, B, SB)
    a, b = _mx_decode_ref(A, SA), _mx_decode_ref(B, SB)
    assert np.allclose(C, a @ b.T, rtol=0, atol=1e-12 * S.max())
    assert np.allclose(S, np.abs(a) @ np.abs(b).T, rtol=1e-13)
    rows = np.array([0, 36, 5, 17])
    cols = np.array([0, 28, 3, 11])
    Cs, Ss = oracle.gemm_mxfp8_nt_sampled(A, SA, B, SB, rows, cols)
    assert np.array_equal(Cs, C[rows, cols]) and np.array_equal(Ss, S[rows, cols])
    with pytest.raises(ValueError):
        oracle.gemm_mxfp8_nt(A[:, :40], SA[:, :1], B[:, :40], SB[:, :1])


# ---------------------------------------------------------------------------
# Block-scaled FP4 (NVFP4)
# ---------------------------------------------------------------------------

def _e2m1_via_e4m3(nib):
    # widen each E2M1 field into an E4M3 code (exponent bias 1 -> 7, the
    # mantissa bit to the top of three, the subnormal 0.5 = 2^-1) and let
    # PyTorch's float8_e4m3fn cast decode it
    import torch

    s, e, m = (nib >> 3) & 1, (nib >> 1) & 3, nib & 1
    if e == 0:
        code = (s << 7) | ((6 << 3) if m else 0)
    else:
        code = (s << 7) | ((e + 6) << 3) | (m << 2)
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).float())


def _nv_decode_ref(packed, scales):
    import torch

    lo, hi = packed & 0xF, packed >> 4
    nib = np.stack([lo, hi], axis=-1).reshape(packed.shape[0], -1)
    lut = np.array([_e2m1_via_e4m3(c) for c in range(16)])
    sv = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).double().numpy()
    return lut[nib] * np.repeat(sv, 16, axis=1)


def test_e2m1_decode_every_code():
    ours = oracle.e2m1_to_f64(np.arange(16, dtype=np.uint8))
    ref = np.array([_e2m1_via_e4m3(c) for c in range(16)])
    assert np.array_equal(ours, ref)
    assert ours.max() == 6.0 and ours[1] == 0.5 and np.all(np.diff(ours[:8]) > 0)


def test_nvfp4_nibble_order_and_block_scales():
    # B's single row holds distinct values; A selects one element k at a time:
    # C = value at k, so the packing order (element 2i in the low nibble) and
    # the 16-element scale blocks are both checked position by position.
    K = 64
    bcodes = np.array([(k % 7) + 1 for k in range(K)], dtype=np.uint8)  # 0.5 .. 4
    B = (bcodes[0::2] | (bcodes[1::2] << 4)).astype(np.uint8)[None, :]
    SB = np.array([[0x38, 0x40, 0x30, 0x48]], dtype=np.uint8)  # 1, 2, 0.5, 4
    for k in range(K):
        a = np.zeros(K, dtype=np.uint8)
        a[k] = 0x2  # 1.0
        A = (a[0::2] | (a[1::2] << 4)).astype(np.uint8)[None, :]
        SA = np.full((1, K // 16), 0x38, np.uint8)
        C, _ = oracle.gemm_nvfp4_nt(A, SA, B, SB, alpha=1.0)
        want = _e2m1_via_e4m3(int(bcodes[k])) * [1.0, 2.0, 0.5, 4.0][k // 16]
        assert C[0, 0] == want, k


def test_nvfp4_small_values_exact_against_brute_force():
    from fractions import Fraction
    from dense_gemm_fp16_gb300 import workloads as wl

    M, N, K = 4, 5, 64
    A, SA = wl.draw_nvfp4(M, K, seed=71)
    B, SB = wl.draw_nvfp4(N, K, seed=72)
    A, SA, B, SB = A.numpy(), SA.numpy(), B.numpy(), SB.numpy()
    C, S = oracle.gemm_nvfp4_nt(A, SA, B, SB, alpha=0.375)
    a, b = _nv_decode_ref(A, SA), _nv_decode_ref(B, SB)
    for i in range(M):
        for j in range(N):
            exact = Fraction(0.375) * sum(Fraction(a[i, k]) * Fraction(b[j, k]) for k in range(K))
            assert C[i, j] == float(exact)
            assert S[i, j] == float(Fraction(0.375) * sum(abs(Fraction(a[i, k]) * Fraction(b[j, k]))
                                                          for k in range(K)))


def test_nvfp4_matches_numpy_and_sampled():
    from dense_gemm_fp16_gb300 import workloads as wl

    M, N, K = 33, 27, 192
    A, SA = wl.draw_nvfp4(M, K, seed=73)
    B, SB = wl.draw_nvfp4(N, K, seed=74)
    A, SA, B, SB = A.numpy(), SA.numpy(), B.numpy(), SB.numpy()
    C, S = oracle.gemm_nvfp4_nt(A, SA, B, SB, alpha=-2.0)
    a, b = _nv_decode_ref(A, SA), _nv_decode_ref(B, SB)
    assert np.allclose(C, -2.0 * (a @ b.T), rtol=0, atol=1e-12 * S.max())
    assert np.allclose(S, 2.0 * (np.abs(a) @ np.abs(b).T), rtol=1e-13)
    rows = np.array([0, 32, 7, 19])
    cols = np.array([0, 26, 3, 13])
    Cs, Ss = oracle.gemm_nvfp4_nt_sampled(A, SA, B, SB, rows, cols, alpha=-2.0)
    assert np.array_equal(Cs, C[rows, cols]) and np.array_equal(Ss, S[rows, cols])
    with pytest.raises(ValueError):
        oracle.gemm_nvfp4_nt(A[:, :5], SA[:, :1], B[:, :5], SB[:, :1])
