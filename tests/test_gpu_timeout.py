"""Failure detection without a GPU fault: a TMA load is left out on purpose
so that the fp16 kernel's bounded waits run out (a stage nothing fills).  The
kernel must report GEMM_ERR_DEVICE_TIMEOUT through the host status query,
release its resources and leave the CUDA context usable."""
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


# The first two shapes run the 1-CTA 128 x 128 kernel, the third the CTA-pair
# kernel (enough 256 x 256 tiles for every SM pair), the last two the skinny
# kernel: one CTA per tile, and clusters of 8 CTAs splitting K (every CTA of
# the cluster gives up, and they still meet at the cluster barriers).
@pytest.mark.parametrize("M,N,K,skip", [(256, 512, 256, 0), (600, 700, 392, 3),
                                        (2560, 2560, 256, 1), (8, 77, 72, 1),
                                        (8, 1000, 4096, 1)])
def test_missing_load_times_out_and_context_survives(M, N, K, skip):
    A = wl.draw_f16((M, K), seed=1)
    B = wl.draw_f16((N, K), seed=2)
    dA, dB = A.cuda(), B.cuda()
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_debug_f16_nt_skip_load(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                                       stream, skip, 20_000_000)   # 20 ms per wait
    assert rc == g.GEMM_OK
    with pytest.raises(g.GemmError) as e:
        g.gemm_check_device_status(stream)
    assert e.value.status == g.GEMM_ERR_DEVICE_TIMEOUT
    # the status word was cleared and the context still works
    assert g.gemm_check_device_status(stream) == g.GEMM_OK
    C2 = g.f16_nt(dA, dB)
    g.gemm_check_device_status(stream)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C2.cpu().numpy(), Cref, S, what="after timeout")
