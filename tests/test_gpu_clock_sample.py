"""The measurement hook gemm_debug_sm_clocks: two samples around a stretch of
GEMM work give each SM seen in both a mean clock within the GPU's range, and
every SM id it reports exists."""
import pytest
import torch

import bench
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def test_clock_samples_around_work_give_each_sm_a_plausible_clock():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    stream = torch.cuda.current_stream()
    probe = bench.SmClockProbe(g, sms, stream)
    M = N = 2048
    K = 1024
    A = wl.draw_f16((M, K), seed=1).cuda()
    B = wl.draw_f16((N, K), seed=2).cuda()
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    probe.sample(0)
    for _ in range(200):
        g.gemm_f16_nt(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), stream.cuda_stream)
    probe.sample(1)
    g.gemm_check_device_status(stream.cuda_stream)
    host = probe.buf.cpu().tolist()
    for sample in host:
        ids = sample[0::3]
        assert all(0 <= i < sms for i in ids)
        assert all(ns > 0 for ns in sample[2::3])
    mhz, seen = probe.mhz()
    assert seen >= sms // 2, f"only {seen} of {sms} SMs seen in both samples"
    assert 300.0 < mhz < 2600.0, f"mean SM clock {mhz} MHz"
