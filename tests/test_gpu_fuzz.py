"""Seeded random shapes through the library's own selection, every output
compared with the float64 oracle (element by element).

Shapes are drawn so that each selector rule is reached: one row (matrix-
vector), 2..64 rows (skinny), few tiles over a long K (the skinny kernel's
cluster split), the tile kernels, rows off the 128-byte grid (K % 64 != 0:
two CTA pairs sharing B), ragged M, N and K everywhere.  The SGEMM draws
cover its tiles and split counts.  A sentinel guard around C catches stray
writes.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_f16, check_f16_epilogue, check_sgemm

pytestmark = pytest.mark.gpu

SENTINEL = 0x7E5A
GUARD = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _f16_shapes(seed, count):
    rng = np.random.default_rng(seed)
    shapes = []
    for i in range(count):
        kind = i % 6
        N = int(rng.integers(1, 1800))
        K = 8 * int(rng.integers(1, 500 if kind != 4 else 2000))
        if kind == 0:
            M = 1
        elif kind == 1:
            M = int(rng.integers(2, 65))
        elif kind == 2:
            M = int(rng.integers(65, 400))
        elif kind == 3:
            M = int(rng.integers(129, 1700))
        else:
            # enough 256 x 256 tiles for the pair kernel, and for K % 64 != 0
            # the two pairs sharing B
            M = int(rng.integers(1800, 2600))
            N = int(rng.integers(1800, 2600))
            K = 8 * int(rng.integers(32, 260))
        shapes.append((M, N, K))
    return shapes


F16_SHAPES = _f16_shapes(2024, 36)


def _guarded_half(M, N):
    buf = torch.empty(M * N + 2 * GUARD, dtype=torch.int16, device="cuda")
    buf.fill_(SENTINEL)
    return buf


def _check_guard(buf, M, N):
    host = buf.cpu().numpy().view(np.uint16)
    assert np.all(host[:GUARD] == SENTINEL) and np.all(host[GUARD + M * N:] == SENTINEL), \
        "kernel wrote outside C"
    return host[GUARD:GUARD + M * N].view(np.float16).reshape(M, N)


@pytest.mark.parametrize("M,N,K", F16_SHAPES)
def test_f16_random_shapes_through_the_selector(M, N, K):
    A = wl.draw_f16((M, K), seed=M * 7 + K, dist="normal")
    B = wl.draw_f16((N, K), seed=N * 11 + K, dist="normal")
    buf = _guarded_half(M, N)
    C = buf[GUARD:GUARD + M * N].view(torch.float16)
    stream = torch.cuda.current_stream().cuda_stream
    dA, dB = A.cuda(), B.cuda()   # kept alive until the asynchronous call has run
    g.gemm_f16_nt(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), stream)
    g.gemm_check_device_status(stream)
    Cref, S = oracle.gemm_f16_nt(A, B)
    variant = g.gemm_f16_select(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)[0]
    check_f16(_check_guard(buf, M, N), Cref, S, what=f"{M}x{N}x{K} variant {variant}")


@pytest.mark.parametrize("M,N,K", F16_SHAPES[::3])
@pytest.mark.parametrize("act", ["relu", "silu", "gelu_tanh"])
def test_f16_fused_random_shapes(M, N, K, act):
    A = wl.draw_f16((M, K), seed=M + 3 * K, dist="normal")
    B = wl.draw_f16((N, K), seed=N + 5 * K, dist="normal")
    bias = wl.draw_f16((N,), seed=N + 1, dist="normal")
    R = wl.draw_f16((M, N), seed=M + N, dist="normal")
    alpha, beta = 0.5, -0.75
    C = g.f16_nt_fused(A.cuda(), B.cuda(), alpha=alpha, bias=bias.cuda(), beta=beta,
                       residual=R.cuda(), activation=act)
    g.gemm_check_device_status(torch.cuda.current_stream().cuda_stream)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=alpha, bias=bias, beta=beta, R=R, act=act)
    check_f16_epilogue(C.cpu().numpy(), Y, S, what=f"fused {act} {M}x{N}x{K}")


def _sgemm_shapes(seed, count):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(count):
        M = int(rng.integers(1, 1200))
        N = int(rng.integers(1, 1200))
        K = int(rng.integers(1, 3000 if i % 3 else 12000))
        alpha = float(rng.choice([1.0, -0.5, 2.0]))
        beta = float(rng.choice([0.0, 0.5, -1.0]))
        out.append((M, N, K, alpha, beta))
    return out


@pytest.mark.parametrize("M,N,K,alpha,beta", _sgemm_shapes(77, 24))
def test_sgemm_random_shapes_through_the_planner(M, N, K, alpha, beta):
    A = wl.draw_f32((M, K), seed=M + K)
    B = wl.draw_f32((K, N), seed=N + 2 * K)
    C0 = wl.draw_f32((M, N), seed=M + N)
    dC = torch.empty(M * N + 2 * GUARD, dtype=torch.float32, device="cuda")
    dC.fill_(float("nan"))
    dC[GUARD:GUARD + M * N] = C0.cuda().reshape(-1)
    stream = torch.cuda.current_stream().cuda_stream
    dA, dB = A.cuda(), B.cuda()   # kept alive until the asynchronous call has run
    g.sgemm(M, N, K, alpha, dA.data_ptr(), dB.data_ptr(), beta, dC[GUARD:].data_ptr(), stream)
    torch.cuda.synchronize()
    host = dC.cpu().numpy()
    assert np.all(np.isnan(host[:GUARD])) and np.all(np.isnan(host[GUARD + M * N:])), \
        "kernel wrote outside C"
    Cref, S = oracle.sgemm(A, B, alpha, beta, C0)
    plan = g.gemm_sgemm_select(M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)
    check_sgemm(host[GUARD:GUARD + M * N].reshape(M, N), Cref, S,
                what=f"{M}x{N}x{K} alpha={alpha} beta={beta} plan {plan}")
