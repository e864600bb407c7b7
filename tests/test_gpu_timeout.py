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
# kernel (enough 256 x 256 tiles for every SM pair), the next two the skinny
# kernel: one CTA per tile, and clusters of 8 CTAs splitting K (every CTA of
# the cluster gives up, and they still meet at the cluster barriers); the
# sixth two CTA pairs sharing B (K = 1016: rows off the 128-byte grid), whose
# stages also wait for the other pair's multicast; the last the skinny kernel
# with 4 clusters per tile, whose parts still meet in the workspace after the
# timeout, and whose tagged counters must not mislead the next call; and two
# CTA pairs splitting one tile's K (1024 x 2048 x 8192), where pair 0 gives
# up while pair 1 finishes and publishes its share, and both still meet at
# the cluster's closing barrier.
@pytest.mark.parametrize("M,N,K,skip", [(256, 512, 256, 0), (600, 700, 392, 3),
                                        (2560, 2560, 256, 1), (8, 77, 72, 1),
                                        (8, 1000, 4096, 1), (2048, 2048, 1016, 1),
                                        (8, 512, 32768, 1), (1024, 2048, 8192, 1)])
def test_missing_load_times_out_and_context_survives(M, N, K, skip):
    if (M, N, K) == (1024, 2048, 8192):
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert g.gemm_f16_select(M, N, K, sms)[0] == g.GEMM_F16_256x256_KSPLIT
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


# The block-scaled kernels use the same bounded waits, status word and
# abort/drain teardown: each CTA (the even CTA of each pair) leaves out one
# k-block of its first tile, in both formats and every tile variant.
BLOCKSCALED_VARIANTS = [g.GEMM_MXFP8_128x128, g.GEMM_MXFP8_256x128_PAIR, g.GEMM_MXFP8_128x256,
                        g.GEMM_MXFP8_256x256_PAIR]


@pytest.mark.parametrize("variant", BLOCKSCALED_VARIANTS)
@pytest.mark.parametrize("fmt", [0, 1], ids=["mxfp8", "nvfp4"])
def test_blockscaled_missing_load_times_out_and_context_survives(fmt, variant):
    M, N, K = 640, 768, 512      # 4 (MXFP8) or 2 (NVFP4) k-blocks; several tiles per variant
    if fmt == 0:
        A, SA = wl.draw_mxfp8(M, K, seed=71)
        B, SB = wl.draw_mxfp8(N, K, seed=72)
        pack, run, ref = g.mxfp8_pack_scales, g.mxfp8_nt, oracle.gemm_mxfp8_nt
    else:
        A, SA = wl.draw_nvfp4(M, K, seed=73)
        B, SB = wl.draw_nvfp4(N, K, seed=74)
        pack, run, ref = g.nvfp4_pack_scales, g.nvfp4_nt, oracle.gemm_nvfp4_nt
    dA, dB = A.cuda(), B.cuda()
    pa, pb = pack(SA.cuda()), pack(SB.cuda())
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_debug_blockscaled_skip_load(fmt, M, N, K, dA.data_ptr(), pa.data_ptr(), dB.data_ptr(),
                                            pb.data_ptr(), C.data_ptr(), stream, variant, 1,
                                            20_000_000)
    assert rc == g.GEMM_OK
    with pytest.raises(g.GemmError) as e:
        g.gemm_check_device_status(stream)
    assert e.value.status == g.GEMM_ERR_DEVICE_TIMEOUT
    assert g.gemm_check_device_status(stream) == g.GEMM_OK
    C2 = run(dA, pa, dB, pb, packed=True, variant=variant)
    g.gemm_check_device_status(stream)
    Cref, S = ref(A, SA, B, SB)
    check_f16(C2.cpu().numpy(), Cref, S, what=f"fmt {fmt} variant {variant} after timeout")


def test_stream_k_partial_wait_times_out_and_context_survives():
    # 81 pair tiles for 76 pairs: the last 5 tiles' k-blocks are shared over
    # all pairs, whose partials are written but never flagged; every such
    # tile's first pair gives up waiting for them (status role 4).
    M, N, K = 2304, 2304, 1024
    A = wl.draw_f16((M, K), seed=75, dist="normal")
    B = wl.draw_f16((N, K), seed=76, dist="normal")
    dA, dB = A.cuda(), B.cuda()
    C = torch.zeros((M, N), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = g.gemm_debug_f16_nt_stream_k_skip_publish(M, N, K, dA.data_ptr(), dB.data_ptr(),
                                                   C.data_ptr(), stream, 20_000_000)
    assert rc == g.GEMM_OK
    pairs, whole, shared, kind = g.gemm_debug_last_pair_launch()
    assert shared > 0, "the launch did not split any tile"
    with pytest.raises(g.GemmError) as e:
        g.gemm_check_device_status(stream)
    assert e.value.status == g.GEMM_ERR_DEVICE_TIMEOUT
    assert g.gemm_check_device_status(stream) == g.GEMM_OK
    # the same split with the partials flagged: correct on the same context
    C2 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C2.data_ptr(), stream,
                     g.GEMM_F16_256x256_PAIR, 0, g.GEMM_F16_FLAG_STREAM_K)
    g.gemm_check_device_status(stream)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C2.cpu().numpy(), Cref, S, what="stream-K after timeout")
