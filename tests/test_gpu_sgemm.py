"""GPU parity of sgemm (C = alpha·A·B + beta·C, fp32 FFMA) against the
float64 oracle, called through the C ABI: the three SGEMM workloads, ragged
shapes on both tile variants and both load paths, and the BLAS conventions
(beta == 0 never reads C; K == 0 gives beta·C)."""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_sgemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _run(A, B, C0, alpha, beta, variant=g.GEMM_SGEMM_AUTO, pad=64, splits=0):
    M, K = A.shape
    N = B.shape[1]
    dA, dB = A.cuda(), B.cuda()
    buf = torch.full((M * N + 2 * pad,), -7.25, dtype=torch.float32, device="cuda")
    C = buf[pad:pad + M * N].view(M, N)
    if C0 is not None:
        C.copy_(C0.cuda())
    g.sgemm_ex(M, N, K, alpha, dA.data_ptr(), dB.data_ptr(), beta, C.data_ptr(),
               torch.cuda.current_stream().cuda_stream, variant, splits)
    torch.cuda.synchronize()
    host = buf.cpu().numpy()
    assert np.all(host[:pad] == -7.25) and np.all(host[pad + M * N:] == -7.25), "wrote outside C"
    return host[pad:pad + M * N].reshape(M, N)


@pytest.mark.parametrize("name", ["sgemm_256", "sgemm_1024"])
def test_sgemm_workloads_full_compare(name):
    w = wl.WORKLOADS[name]
    A, B, C0 = wl.make_inputs(w)
    C = _run(A, B, torch.zeros(w.M, w.N), w.alpha, w.beta)
    Cref, S = oracle.sgemm(A, B, w.alpha, w.beta, C0)
    check_sgemm(C, Cref, S, what=name)


def test_sgemm_4096_alpha_beta_sampled():
    w = wl.WORKLOADS["sgemm_4096"]
    A, B, C0 = wl.make_inputs(w)
    C = _run(A, B, C0, w.alpha, w.beta, pad=4)
    rows, cols = wl.sample_positions(w.M, w.N, 65536, seed=77)
    Cref, S = oracle.sgemm_sampled(A, B, rows, cols, w.alpha, w.beta, C0)
    check_sgemm(C[rows, cols], Cref, S, what="sgemm_4096")


@pytest.mark.parametrize("variant", [g.GEMM_SGEMM_128x128, g.GEMM_SGEMM_64x64, g.GEMM_SGEMM_128x64])
@pytest.mark.parametrize("M,N,K,alpha,beta", [
    (100, 70, 33, 1.0, 0.0),       # ragged everything, scalar loads (K, N odd-ish)
    (257, 129, 17, -1.5, 0.25),    # one past the tile edges
    (1, 1, 1, 2.0, 0.0),
    (300, 260, 64, 1.0, -1.0),     # vector loads, ragged M/N
    (128, 128, 8, 0.5, 2.0),       # exactly one tile and one k-slice
    (513, 384, 200, 1.0, 0.5),
])
def test_sgemm_ragged(M, N, K, alpha, beta, variant):
    A = wl.draw_f32((M, K), seed=M)
    B = wl.draw_f32((K, N), seed=N + 1)
    C0 = wl.draw_f32((M, N), seed=K + 2)
    C = _run(A, B, C0, alpha, beta, variant)
    Cref, S = oracle.sgemm(A, B, alpha, beta, C0)
    check_sgemm(C, Cref, S, what=f"{M}x{N}x{K} v{variant}")


def test_sgemm_misaligned_pointers_use_scalar_path():
    M, N, K = 96, 80, 48
    A = wl.draw_f32((M, K), seed=1)
    B = wl.draw_f32((K, N), seed=2)
    C = _run(A, B, None, 1.0, 0.0, pad=1)      # C offset by 4 bytes
    Cref, S = oracle.sgemm(A, B)
    check_sgemm(C, Cref, S, what="misaligned C")


def test_sgemm_small_integers_exact():
    M, N, K = 200, 150, 96
    A = wl.draw_int((M, K), 3, -4, 4)
    B = wl.draw_int((K, N), 4, -4, 4)
    C0 = wl.draw_int((M, N), 5, -4, 4)
    C = _run(A, B, C0, 2.0, -3.0)
    Cref, _ = oracle.sgemm(A, B, 2.0, -3.0, C0)
    assert np.array_equal(C.astype(np.float64), Cref)


def test_sgemm_beta_zero_ignores_nan_c():
    M, N, K = 130, 140, 40
    A = wl.draw_f32((M, K), seed=11)
    B = wl.draw_f32((K, N), seed=12)
    C = _run(A, B, torch.full((M, N), float("nan")), 1.0, 0.0)
    Cref, S = oracle.sgemm(A, B)
    check_sgemm(C, Cref, S, what="beta=0 NaN C")


def test_sgemm_k0_is_beta_c():
    M, N = 65, 33
    C0 = wl.draw_f32((M, N), seed=13)
    dummy = torch.zeros(4, device="cuda")
    C = C0.cuda()
    g.sgemm(M, N, 0, 1.0, dummy.data_ptr(), dummy.data_ptr(), 0.5, C.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert np.array_equal(C.cpu().numpy(), (0.5 * C0).numpy())
    g.sgemm(M, N, 0, 1.0, dummy.data_ptr(), dummy.data_ptr(), 0.0, C.data_ptr(),
            torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert (C == 0).all()


def test_sgemm_tensor_wrapper():
    A = wl.draw_f32((64, 32), seed=20).cuda()
    B = wl.draw_f32((32, 48), seed=21).cuda()
    C = torch.zeros(64, 48, device="cuda")
    g.sgemm_(A, B, C)
    Cref, S = oracle.sgemm(A.cpu(), B.cpu())
    check_sgemm(C.cpu().numpy(), Cref, S, what="wrapper")


V1, V2, V3 = g.GEMM_SGEMM_128x128, g.GEMM_SGEMM_64x64, g.GEMM_SGEMM_128x64


@pytest.mark.parametrize("M,N,K,alpha,beta,variant,splits", [
    (1024, 1024, 1024, 1.0, 0.5, V1, 4),    # the 1024-cube size with a beta term: 64 tiles
    (1024, 1024, 1024, 1.0, 0.5, 0, 0),     # the library's own plan for it
    (300, 200, 1000, -2.0, 0.25, V1, 8),    # 6 ragged tiles, a partial last share
    (130, 260, 4099, 0.5, 0.0, V1, 0),      # K not a multiple of 4: the element-wise loads
    (128, 128, 65536, 1.0, 1.0, V1, 8),     # one tile, 8 shares of 8192
    (200, 150, 3000, 1.0, 0.5, V2, 6),      # the 64 x 64 tile, ragged
    (64, 1024, 4096, 1.5, 0.0, V2, 7),      # skinny M
    (96, 80, 150, 1.0, 1.0, V1, 8),         # short K: 8 requested, 3 shares of >= 64
    (256, 256, 4096, 1.0, 0.0, 0, 0),
    (1024, 1024, 1024, 1.0, 0.5, V3, 1),    # the 128 x 64 tile over the whole K
    (300, 200, 1000, -2.0, 0.25, V3, 4),    # ... split, ragged
    (130, 70, 4099, 0.5, 0.0, V3, 3),       # ... element-wise loads, a partial tile column
])
def test_sgemm_split_k(M, N, K, alpha, beta, variant, splits):
    # Each tile's K is shared over several CTAs; the last to finish adds the
    # partials in split order and applies beta * C.  Three calls on one
    # stream: the per-tile counters reset.
    A = wl.draw_f32((M, K), seed=M + 11)
    B = wl.draw_f32((K, N), seed=N + 12)
    C0 = wl.draw_f32((M, N), seed=13)
    Cref, S = oracle.sgemm(A, B, alpha, beta, C0)
    for rep in range(3):
        C = _run(A, B, C0, alpha, beta, variant, splits=splits)
        check_sgemm(C, Cref, S, what=f"split-K {M}x{N}x{K} v{variant} s{splits} rep {rep}")


def test_sgemm_split_k_matches_unsplit_within_rounding():
    # The same product with 1..8 shares: every result within the bound of the
    # oracle, and 1 share gives the plain kernel's bits.
    M, N, K = 256, 192, 2048
    A = wl.draw_f32((M, K), seed=41)
    B = wl.draw_f32((K, N), seed=42)
    Cref, S = oracle.sgemm(A, B, 1.0, 0.0, None)
    for v in (V1, V2, V3):
        plain = _run(A, B, None, 1.0, 0.0, v, splits=1)
        for sp in range(1, 9):
            C = _run(A, B, None, 1.0, 0.0, v, splits=sp)
            check_sgemm(C, Cref, S, what=f"v{v} splits {sp}")
            if sp == 1:
                assert np.array_equal(C, plain)


def test_sgemm_split_k_beta_zero_ignores_nan_c_and_is_deterministic():
    M, N, K = 256, 384, 2048
    A = wl.draw_f32((M, K), seed=21)
    B = wl.draw_f32((K, N), seed=22)
    dA, dB = A.cuda(), B.cuda()
    outs = []
    for _ in range(2):
        C = torch.full((M, N), float("nan"), device="cuda")
        g.sgemm(M, N, K, 1.0, dA.data_ptr(), dB.data_ptr(), 0.0, C.data_ptr(), 0)
        torch.cuda.synchronize()
        outs.append(C.cpu().numpy())
    Cref, S = oracle.sgemm(A, B, 1.0, 0.0, None)
    check_sgemm(outs[0], Cref, S, what="split-K beta 0")
    assert np.array_equal(outs[0], outs[1]), "split-K partials must add in a fixed order"


def test_sgemm_split_k_under_graph_capture():
    # Inside a capture the workspace cannot be allocated; a stream that has
    # one already splits, a fresh stream runs unsplit.  Either way: correct.
    M, N, K = 512, 512, 2048
    A = wl.draw_f32((M, K), seed=31)
    B = wl.draw_f32((K, N), seed=32)
    dA, dB = A.cuda(), B.cuda()
    Cref, S = oracle.sgemm(A, B, 1.0, 0.0, None)
    s = torch.cuda.Stream()
    C = torch.zeros((M, N), device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        g.sgemm(M, N, K, 1.0, dA.data_ptr(), dB.data_ptr(), 0.0, C.data_ptr(), s.cuda_stream)
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    check_sgemm(C.cpu().numpy(), Cref, S, what="captured")


def test_sgemm_split_k_on_two_streams_at_once():
    # Split-K slots and tile counters are per stream: two streams whose split
    # products overlap on the GPU must not mix their partials.
    M, N, K = 512, 512, 8192
    ins = [(wl.draw_f32((M, K), seed=41 + j), wl.draw_f32((K, N), seed=43 + j)) for j in range(2)]
    devs = [(A.cuda(), B.cuda()) for A, B in ins]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [torch.zeros((M, N), device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(4):
        for j in range(2):
            dA, dB = devs[j]
            g.sgemm_ex(M, N, K, 1.0, dA.data_ptr(), dB.data_ptr(), 0.0, outs[j].data_ptr(), streams[j].cuda_stream,
                       g.GEMM_SGEMM_128x64, 8)
    for s in streams:
        s.synchronize()
    for j in range(2):
        Cref, S = oracle.sgemm(*ins[j], 1.0, 0.0, None)
        check_sgemm(outs[j].cpu().numpy(), Cref, S, what=f"split-K, stream {j}")
