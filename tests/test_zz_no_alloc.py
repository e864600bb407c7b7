"""The allocation-free fp16 entry point, gemm_f16_nt_stream_k_noalloc.

Some callers cannot let a library call cudaMalloc: a server that reserved its
whole device-memory budget in its own pool up front, a latency-critical path
where an allocation could synchronise the device, a framework whose allocator
must account for every byte.  For them this entry point runs the CTA-pair
kernel with its stream-K split but keeps the partial tiles and flags in a
static array inside the library instead of a workspace it allocates.

Through the C ABI, it must give gemm_f16_nt's result within the fp16
tolerance (|difference| <= 4e-3 * sum_k |A*B| + 1e-6 per element), on two
calls in a row: the second call finds the first call's partials and flags
still in the shared array and must not be misled by them.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import F16_ABS, F16_REL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def test_noalloc_entry_point_matches_gemm_f16_nt_on_two_calls():
    # 2304 x 2304 gives 9 x 9 = 81 tiles of 256 x 256 for the 76 CTA pairs of a
    # GB300: the 5 tiles left after the full round have 5 x 16 = 80 k-blocks,
    # split over all pairs, so partials pass through the static array.
    M, N, K = 2304, 2304, 1024
    A = wl.draw_f16((M, K), seed=81, dist="normal")
    B = wl.draw_f16((N, K), seed=82, dist="normal")
    _, S = oracle.gemm_f16_nt(A, B)
    bound = F16_REL * S + F16_ABS

    stream = torch.cuda.current_stream().cuda_stream
    dA, dB = A.cuda(), B.cuda()
    C_ref = torch.empty((M, N), dtype=torch.float16, device="cuda")
    g.gemm_f16_nt(M, N, K, dA.data_ptr(), dB.data_ptr(), C_ref.data_ptr(), stream)
    g.gemm_check_device_status(stream)
    ref = C_ref.cpu().numpy().astype(np.float64)

    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        assert g.gemm_f16_nt_stream_k_noalloc(M, N, K, dA.data_ptr(), dB.data_ptr(),
                                              C.data_ptr(), stream) == g.GEMM_OK
        g.gemm_check_device_status(stream)
        got = C.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(got)), f"call {call}: unwritten or non-finite outputs"
        err = np.abs(got - ref)
        assert np.all(err <= bound), \
            f"call {call}: {(err > bound).sum()} outputs differ from gemm_f16_nt beyond tolerance"
