"""GPU parity at sizes whose element counts pass 2^31: every row or element
offset must be computed in 64 bits.

* fp16 C of 49152 x 49152 (2.4e9 halves, 4.8 GB) through every tile variant;
* fp16 B of 262400 x 8192 (2.15e9 halves, 4.3 GB) through the matrix-vector
  kernel (M = 1) and the skinny kernel (M = 16);
* fp32 C of 46400 x 46400 (2.15e9 floats, 8.6 GB) through the SGEMM.

The big operand is built on the device by repeating a seeded block, so the
float64 oracle, given the block, computes any sampled output; samples are
gathered on the device (the last rows and columns, where the offsets pass
2^31, are always among them) and a guard region past C is checked.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_f16, check_sgemm

pytestmark = pytest.mark.gpu

GUARD = 256
SENTINEL = 0x7E5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _positions(M, N, seed):
    rows, cols = wl.sample_positions(M, N, 65536, seed=seed, tail_rows=[M - 2])
    return rows, cols


def _gather(C, rows, cols):
    r = torch.as_tensor(rows, device=C.device)
    c = torch.as_tensor(cols, device=C.device)
    return C[r, c].cpu().numpy()


def _guarded(count, dtype, fill):
    """A device buffer of count + GUARD elements; the guard holds a sentinel."""
    buf = torch.empty(count + GUARD, dtype=dtype, device="cuda")
    buf.fill_(fill)
    if dtype == torch.float16:
        buf[count:].view(torch.int16).fill_(SENTINEL)
    return buf


def _guard_intact(buf, count):
    tail = buf[count:]
    if buf.dtype == torch.float16:
        return bool((tail.view(torch.int16) == SENTINEL).all())
    return bool(torch.isnan(tail).all())


@pytest.mark.parametrize("variant", [g.GEMM_F16_AUTO, g.GEMM_F16_256x256_PAIR, g.GEMM_F16_256x256_QUAD,
                                     g.GEMM_F16_128x128, g.GEMM_F16_128x256])
def test_f16_output_past_2_31_elements(variant):
    M, N, K = 49152, 49152, 64
    assert M * N > 2 ** 31
    A = wl.draw_f16((M, K), seed=111, dist="normal")
    B = wl.draw_f16((N, K), seed=112, dist="normal")
    dA, dB = A.cuda(), B.cuda()
    buf = _guarded(M * N, torch.float16, float("nan"))
    C = buf[:M * N].view(M, N)
    stream = torch.cuda.current_stream().cuda_stream
    g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), stream, variant)
    g.gemm_check_device_status(stream)
    assert _guard_intact(buf, M * N), "kernel wrote past C"
    rows, cols = _positions(M, N, seed=113)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(_gather(C, rows, cols), Cref, S, what=f"49152^2 x 64 variant {variant}")
    del buf, C


def _repeated_b(reps, block_rows, K, seed):
    """B of reps x block_rows rows on the device: a seeded block repeated."""
    block = wl.draw_f16((block_rows, K), seed=seed, dist="uniform")
    return block, block.cuda().repeat(reps, 1)


@pytest.mark.parametrize("M", [1, 16])
def test_f16_b_operand_past_2_31_elements(M):
    # 262400 = 64 x 4100 rows of 8192: 2.15e9 elements of B.  M = 1 takes the
    # matrix-vector kernel, M = 16 the skinny one.
    block_rows, reps, K = 4100, 64, 8192
    N = block_rows * reps
    assert N * K > 2 ** 31
    block, dB = _repeated_b(reps, block_rows, K, seed=114)
    A = wl.draw_f16((M, K), seed=115, dist="uniform")
    dA = A.cuda()
    buf = _guarded(M * N, torch.float16, float("nan"))
    C = buf[:M * N].view(M, N)
    stream = torch.cuda.current_stream().cuda_stream
    g.gemm_f16_nt(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), stream)
    g.gemm_check_device_status(stream)
    assert _guard_intact(buf, M * N), "kernel wrote past C"
    del dB
    rows, cols = wl.sample_positions(M, N, 16384, seed=116)
    # output (m, n) reads row n % block_rows of the block
    Cref, S = oracle.gemm_f16_nt_sampled(A, block, rows, cols % block_rows)
    check_f16(_gather(C, rows, cols), Cref, S, what=f"M={M} N={N} K={K}")


def test_sgemm_output_past_2_31_elements():
    M, N, K = 46400, 46400, 16
    assert M * N > 2 ** 31
    A = wl.draw_f32((M, K), seed=117)
    B = wl.draw_f32((K, N), seed=118)
    dA, dB = A.cuda(), B.cuda()
    buf = _guarded(M * N, torch.float32, float("nan"))
    C = buf[:M * N].view(M, N)
    stream = torch.cuda.current_stream().cuda_stream
    g.sgemm(M, N, K, 1.0, dA.data_ptr(), dB.data_ptr(), 0.0, C.data_ptr(), stream)
    torch.cuda.synchronize()
    assert _guard_intact(buf, M * N), "kernel wrote past C"
    rows, cols = _positions(M, N, seed=119)
    Cref, S = oracle.sgemm_sampled(A, B, rows, cols)
    check_sgemm(_gather(C, rows, cols), Cref, S, what="46400^2 x 16")
