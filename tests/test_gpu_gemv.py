"""GPU parity of the matrix-vector path of gemm_f16_nt (M <= 4 rows of A;
chosen by the selector for M = 1, forced through gemm_f16_nt_ex, against the float64
oracle: ragged N and K, several rows per warp, and the decode-sized shape the
benchmark times (sampled)."""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_f16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _run(A, B, variant=g.GEMM_F16_AUTO):
    M, K = A.shape
    N = B.shape[0]
    dA, dB = A.cuda(), B.cuda()
    buf = torch.full((M * N + 128,), 0x7E5A, dtype=torch.int16, device="cuda").view(torch.float16)
    C = buf[64:64 + M * N].view(M, N)
    g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                     torch.cuda.current_stream().cuda_stream, variant, 0)
    g.gemm_check_device_status(0)
    host = buf.cpu()
    guard = torch.cat([host[:64], host[64 + M * N:]]).view(torch.int16).numpy()
    assert np.all(guard == 0x7E5A), "wrote outside C"
    return host[64:64 + M * N].view(M, N).numpy()


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("N,K", [(1, 8), (77, 72), (5376, 2048), (3000, 1032), (1000, 12008), (9, 4096)])
def test_small_m_full_compare(M, N, K):
    # M = 1 takes the matrix-vector kernel, larger M the tensor cores; both
    # agree with the oracle, and the matrix-vector kernel can be forced up to
    # M = 4.  (9 rows of B: more warps than rows, odd row blocks.)
    A = wl.draw_f16((M, K), seed=M + 100, dist="normal")
    B = wl.draw_f16((N, K), seed=N + 200, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert (g.gemm_f16_select(M, N, K, sm)[0] == g.GEMM_F16_GEMV) == (M == 1)
    check_f16(_run(A, B), Cref, S, what=f"M={M} {N}x{K}")
    if M <= 4:
        check_f16(_run(A, B, g.GEMM_F16_GEMV), Cref, S, what=f"gemv forced {M}x{N}x{K}")


def test_gemv_bench_shape_sampled():
    # The decode-sized product the benchmark times: B is 256 MB, larger than L2.
    w = wl.WORKLOADS["f16_gemv_1x16384x8192"]
    A, B, _ = wl.make_inputs(w)
    dA, dB = A.cuda(), B.cuda()
    C = g.f16_nt(dA, dB)
    g.gemm_check_device_status(0)
    rows, cols = wl.sample_positions(w.M, w.N, 4096, seed=5)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(C.cpu().numpy()[rows, cols], Cref, S, what="gemv bench shape")


def test_gemv_variant_rejects_too_many_rows():
    A = torch.zeros((5, 64), dtype=torch.float16, device="cuda")
    C = torch.zeros((5, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt_ex(5, 64, 64, A.data_ptr(), A.data_ptr(), C.data_ptr(), 0, g.GEMM_F16_GEMV)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED
