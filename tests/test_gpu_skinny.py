"""GPU parity of the skinny variant of gemm_f16_nt (a few rows of A, computed
as B·Aᵀ on the tensor cores with the K range split over a cluster of CTAs)
against the float64 oracle: every MMA width (16, 32, 64, 128 rows of A), ragged
M, N and K, 1, 2, 4 and 8 shares, the fused epilogue on both paths, an
unaligned C, graph capture, and run-to-run equality of the split sums."""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_f16, check_f16_epilogue

pytestmark = pytest.mark.gpu

SENTINEL = 0x7E5A  # a NaN payload nothing in the product writes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _guarded(M, N, pad=64):
    buf = torch.full((M * N + 2 * pad,), SENTINEL, dtype=torch.int16, device="cuda").view(torch.float16)
    return buf, buf[pad:pad + M * N].view(M, N)


def _unguard(buf, M, N, pad=64):
    host = buf.cpu()
    guard = torch.cat([host[:pad], host[pad + M * N:]]).view(torch.int16).numpy()
    assert np.all(guard == SENTINEL), "kernel wrote outside C"
    return host[pad:pad + M * N].view(M, N).numpy()


def _run(A, B, variant=g.GEMM_F16_SKINNY, pad=64):
    M, K = A.shape
    N = B.shape[0]
    dA, dB = A.cuda(), B.cuda()
    buf, C = _guarded(M, N, pad)
    stream = torch.cuda.current_stream().cuda_stream
    g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), stream, variant, 0)
    g.gemm_check_device_status(stream)
    return _unguard(buf, M, N, pad)


# (N, K) and the plan on 152 SMs (shares): one partial group over two
# k-blocks (1), a partial k-block (2), ragged groups and k-blocks (4), a long
# K (8), N % 4 != 0 (8: the split sum's scalar stores), exactly one wave of
# groups (1).  Shorter groups (the multi-wave plan) have a test of their own.
SHAPES = [(77, 72), (3000, 1032), (4000, 2056), (1000, 12008), (1001, 4104), (19456, 1024)]


@pytest.mark.parametrize("M", [1, 5, 16, 17, 32, 33, 64, 65, 128])
@pytest.mark.parametrize("N,K", SHAPES)
def test_skinny_full_compare(M, N, K):
    A = wl.draw_f16((M, K), seed=M + 300, dist="normal")
    B = wl.draw_f16((N, K), seed=N + K, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(_run(A, B), Cref, S, what=f"skinny {M}x{N}x{K}")


def test_skinny_bench_shape_sampled():
    # The 16-row product the benchmark times, as the selector runs it: B is
    # 256 MB, larger than L2; sampled outputs against the oracle.
    w = wl.WORKLOADS["f16_skinny_16x16384x8192"]
    A, B, _ = wl.make_inputs(w)
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert g.gemm_f16_select(w.M, w.N, w.K, sm)[0] == g.GEMM_F16_SKINNY
    dA, dB = A.cuda(), B.cuda()
    C = g.f16_nt(dA, dB)
    g.gemm_check_device_status(0)
    rows, cols = wl.sample_positions(w.M, w.N, 4096, seed=9)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(C.cpu().numpy()[rows, cols], Cref, S, what="skinny bench shape")


def test_skinny_two_even_waves():
    # 128-row groups would need just over one wave: groups of 72 rows (not a
    # power of two) fill two waves instead.
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 3, sm * 128 + 500, 256
    A = wl.draw_f16((M, K), seed=81, dist="normal")
    B = wl.draw_f16((N, K), seed=82, dist="normal")
    assert g.gemm_debug_skinny_plan(M, N, K, sm)[1] < 128
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(_run(A, B), Cref, S, what=f"skinny two waves {M}x{N}x{K}")


@pytest.mark.parametrize("M", [100, 128])
def test_skinny_128_rows_split_by_the_selector(M):
    # 65 to 128 rows with a long K: the selector's skinny kernel, K split
    # over clusters of 4 (the MMA's N = 128 instance).
    N, K = 3000, 4104
    A = wl.draw_f16((M, K), seed=91, dist="normal")
    B = wl.draw_f16((N, K), seed=92, dist="normal")
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert g.gemm_f16_select(M, N, K, sm)[0] == g.GEMM_F16_SKINNY
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(_run(A, B, variant=g.GEMM_F16_AUTO), Cref, S, what=f"skinny selected {M}x{N}x{K}")


def test_skinny_unaligned_output():
    # C two bytes off an 8-byte boundary: the split sum stores half by half.
    M, N, K = 20, 1000, 4096
    A = wl.draw_f16((M, K), seed=61, dist="normal")
    B = wl.draw_f16((N, K), seed=62, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(_run(A, B, pad=65), Cref, S, what="skinny unaligned C")


def test_skinny_is_selected_for_few_rows():
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    for M in (2, 5, 64, 100, 128):
        assert g.gemm_f16_select(M, 8192, 8192, sm)[0] == g.GEMM_F16_SKINNY
    M, N, K = 7, 2000, 3000
    A = wl.draw_f16((M, K), seed=71, dist="normal")
    B = wl.draw_f16((N, K), seed=72, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(_run(A, B, variant=g.GEMM_F16_AUTO), Cref, S, what="skinny by the selector")


def test_skinny_split_sum_is_deterministic():
    # The shares are added in split order: equal runs give equal bits.
    M, N, K = 24, 1000, 12008
    A = wl.draw_f16((M, K), seed=41, dist="normal")
    B = wl.draw_f16((N, K), seed=42, dist="normal")
    first = _run(A, B)
    for _ in range(3):
        assert np.array_equal(_run(A, B).view(np.uint16), first.view(np.uint16))


@pytest.mark.parametrize("act", ["none", "relu", "gelu_tanh"])
@pytest.mark.parametrize("M,N,K", [(9, 300, 136), (40, 1000, 12008), (300, 1000, 4104)])
def test_skinny_fused_epilogue(M, N, K, act):
    # (the first shape runs unsplit, the second with 8 shares summed over the
    # cluster, the third as three 128-row tiles of A with 4 shares each: the
    # residual rows offset by each tile's first row)
    A = wl.draw_f16((M, K), seed=M, dist="normal")
    B = wl.draw_f16((N, K), seed=N, dist="normal")
    bias = wl.draw_f16((N,), seed=7, dist="normal")
    R = wl.draw_f16((M, N), seed=8, dist="normal")
    dA, dB, dbias, dR = A.cuda(), B.cuda(), bias.cuda(), R.cuda()
    buf, C = _guarded(M, N)
    stream = torch.cuda.current_stream().cuda_stream
    g.gemm_f16_nt_fused(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 0.5, -1.25,
                        dbias.data_ptr(), dR.data_ptr(), g.ACTIVATIONS[act], stream, g.GEMM_F16_SKINNY)
    g.gemm_check_device_status(stream)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=0.5, bias=bias, beta=-1.25, R=R, act=act)
    check_f16_epilogue(_unguard(buf, M, N), Y, S, what=f"skinny fused {M}x{N}x{K} {act}")


def test_skinny_under_graph_capture():
    # The split (8 shares per tile here) needs no workspace, so a captured
    # call runs as a plain one; the replayed graph gives the oracle's result.
    M, N, K = 12, 640, 4096
    A = wl.draw_f16((M, K), seed=51, dist="normal")
    B = wl.draw_f16((N, K), seed=52, dist="normal")
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty((M, N), dtype=torch.float16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), side.cuda_stream,
                         g.GEMM_F16_SKINNY)
    C.zero_()
    graph.replay()
    torch.cuda.synchronize()
    g.gemm_check_device_status(0)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C.cpu().numpy(), Cref, S, what="skinny captured")


@pytest.mark.parametrize("M,N,K", [(300, 1000, 4104), (300, 77, 72), (129, 2000, 2056)])
def test_skinny_several_row_tiles_of_a(M, N, K):
    # More than 128 rows of A: 128-row tiles of A on the grid's third
    # dimension (the last one partial), with and without the K split.
    A = wl.draw_f16((M, K), seed=M + 7, dist="normal")
    B = wl.draw_f16((N, K), seed=N + 7, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(_run(A, B), Cref, S, what=f"skinny {M}x{N}x{K}")


# A few tiles over a very long K: each tile's K range goes to several 8-CTA
# clusters (parts), whose fp32 sums meet in a workspace; the last cluster of
# a tile adds them in part order.  (M, N, K) -> parts on 152 SMs: 4 tiles x 4,
# one tile x 8, 4 tiles of 8 rows x 4.
PARTS_SHAPES = [(256, 256, 65536), (128, 128, 65536), (8, 512, 32768)]


@pytest.mark.parametrize("M,N,K", PARTS_SHAPES)
def test_skinny_several_clusters_per_tile(M, N, K):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert g.gemm_debug_skinny_parts(M, N, K, sms) > 1
    A = wl.draw_f16((M, K), seed=M + 71, dist="normal")
    B = wl.draw_f16((N, K), seed=N + 72, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    first = _run(A, B)
    check_f16(first, Cref, S, what=f"skinny parts {M}x{N}x{K}")
    for rep in range(3):   # the parts add in a fixed order: the same bits every time
        assert np.array_equal(_run(A, B).view(np.uint16), first.view(np.uint16)), f"rep {rep}"


def test_skinny_several_clusters_per_tile_fused_and_captured():
    M, N, K = 256, 256, 65536
    A = wl.draw_f16((M, K), seed=81, dist="normal")
    B = wl.draw_f16((N, K), seed=82, dist="normal")
    bias = wl.draw_f16((N,), seed=83, dist="normal")
    R = wl.draw_f16((M, N), seed=84, dist="normal")
    dA, dB, dbias, dR = A.cuda(), B.cuda(), bias.cuda(), R.cuda()
    buf, C = _guarded(M, N)
    stream = torch.cuda.current_stream().cuda_stream
    g.gemm_f16_nt_fused(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), 0.5, 1.0,
                        dbias.data_ptr(), dR.data_ptr(), g.ACTIVATIONS["silu"], stream, g.GEMM_F16_SKINNY)
    g.gemm_check_device_status(stream)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=0.5, bias=bias, beta=1.0, R=R, act="silu")
    check_f16_epilogue(_unguard(buf, M, N), Y, S, what="skinny parts fused")
    # under stream capture the tile keeps one cluster (no workspace use)
    Cg = torch.empty((M, N), dtype=torch.float16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), Cg.data_ptr(), side.cuda_stream,
                         g.GEMM_F16_SKINNY)
    graph.replay()
    torch.cuda.synchronize()
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(Cg.cpu().numpy(), Cref, S, what="skinny parts captured")


def test_skinny_several_clusters_per_tile_on_two_streams_at_once():
    # Each stream has its own workspace and counters: two streams whose
    # multi-cluster products overlap on the GPU must not mix their parts.
    M, N, K = 256, 256, 65536
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert g.gemm_debug_skinny_parts(M, N, K, sms) > 1
    ins = [(wl.draw_f16((M, K), seed=91 + j, dist="normal"), wl.draw_f16((N, K), seed=93 + j, dist="normal"))
           for j in range(2)]
    devs = [(A.cuda(), B.cuda()) for A, B in ins]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.empty((M, N), dtype=torch.float16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(4):
        for j in range(2):
            dA, dB = devs[j]
            g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), outs[j].data_ptr(), streams[j].cuda_stream,
                             g.GEMM_F16_SKINNY)
    for s in streams:
        s.synchronize()
    g.gemm_check_device_status(0)
    for j in range(2):
        Cref, S = oracle.gemm_f16_nt(*ins[j])
        check_f16(outs[j].cpu().numpy(), Cref, S, what=f"skinny parts, stream {j}")
