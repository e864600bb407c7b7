"""GPU parity of gemm_mxfp8_nt (block-scaled FP8: E4M3 elements, one UE8M0
scale per 32 elements of K, fp32 accumulation, half out) against the float64
oracle ("异步拷贝与 Hopper/Blackwell 新特性", section "Blackwell 概览 sm_100"),
through the C ABI.

The cases are staged so that each isolates one part of the path: unit scales
with small integers (bit-exact: the FP8 operands and the MMA), scales that
vary by row only (which TMEM lane and column hold each row's scale), scales
that vary along K (which scale each 32-element slice of K takes), then random
data over several tiles with ragged M, N and K, and the packing of plain
scales into the kernel's chunk layout.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_f16

pytestmark = pytest.mark.gpu

SENTINEL = 0x7E5A


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _e4m3(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)


VARIANTS = [g.GEMM_MXFP8_128x128, g.GEMM_MXFP8_256x128_PAIR, g.GEMM_MXFP8_128x256,
            g.GEMM_MXFP8_256x256_PAIR]


def _run(A, SA, B, SB, pad=64, variant=g.GEMM_MXFP8_AUTO, grid=0):
    M, K = A.shape
    N = B.shape[0]
    buf = torch.empty((M * N + 2 * pad,), dtype=torch.int16, device="cuda")
    buf.fill_(SENTINEL)
    buf = buf.view(torch.float16)
    C = buf[pad:pad + M * N].view(M, N)
    g.mxfp8_nt(A.cuda(), SA.cuda(), B.cuda(), SB.cuda(), C, variant=variant, grid=grid)
    g.gemm_check_device_status(torch.cuda.current_stream().cuda_stream)
    host = buf.cpu()
    guard = torch.cat([host[:pad], host[pad + M * N:]]).view(torch.int16).numpy().view(np.uint16)
    assert np.all(guard == SENTINEL), "kernel wrote outside C"
    return host[pad:pad + M * N].view(M, N).numpy()


def _pack_ref(S, rows, K):
    # the chunk layout of gemm.h, written out with plain index loops
    kbt = (K + 127) // 128
    rt = (rows + 127) // 128
    out = np.full(rt * kbt * 512, 127, dtype=np.uint8)
    for r in range(rows):
        for j in range(K // 32):
            t, b = r // 128, j // 4
            rr, jj = r % 128, j % 4
            out[(t * kbt + b) * 512 + 16 * (rr % 32) + 4 * (rr // 32) + jj] = S[r, j]
    return out


@pytest.mark.parametrize("rows,K", [(1, 32), (128, 128), (300, 160), (129, 544)])
def test_pack_scales_layout(rows, K):
    S = torch.randint(0, 255, (rows, K // 32), dtype=torch.uint8)
    packed = g.mxfp8_pack_scales(S.cuda()).cpu().numpy()
    assert packed.size == g.gemm_mxfp8_scale_bytes(rows, K)
    assert np.array_equal(packed, _pack_ref(S.numpy(), rows, K))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (256, 384, 256), (130, 136, 96)])
def test_unit_scales_small_integers_bit_exact(M, N, K, variant):
    rng = np.random.default_rng(M + N + K)
    ai = rng.integers(-2, 3, (M, K))
    bi = rng.integers(-2, 3, (N, K))
    A, B = _e4m3(ai), _e4m3(bi)
    SA = torch.full((M, K // 32), 127, dtype=torch.uint8)
    SB = torch.full((N, K // 32), 127, dtype=torch.uint8)
    C = _run(A, SA, B, SB, variant=variant)
    assert np.array_equal(C.astype(np.float64), (ai @ bi.T).astype(np.float64))


@pytest.mark.parametrize("variant", VARIANTS)
def test_row_scales_place_each_rows_scale(variant):
    # Scales constant along K but different for every row of A and of B:
    # integers times powers of two, still exact.
    M, N, K = 256, 256, 256
    rng = np.random.default_rng(7)
    ai = rng.integers(-2, 3, (M, K))
    bi = rng.integers(-2, 3, (N, K))
    ea = rng.integers(-3, 4, M)
    eb = rng.integers(-3, 4, N)
    SA = torch.from_numpy(np.repeat((127 + ea)[:, None], K // 32, axis=1).astype(np.uint8))
    SB = torch.from_numpy(np.repeat((127 + eb)[:, None], K // 32, axis=1).astype(np.uint8))
    C = _run(_e4m3(ai), SA, _e4m3(bi), SB, variant=variant)
    ref = (ai @ bi.T).astype(np.float64) * np.ldexp(1.0, ea)[:, None] * np.ldexp(1.0, eb)[None, :]
    Cref, S = oracle.gemm_mxfp8_nt(_e4m3(ai), SA, _e4m3(bi), SB)
    assert np.array_equal(Cref, ref)
    check_f16(C, Cref, S, what="row scales")


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_scales_pick_their_32_elements(variant):
    # Ones everywhere; scales vary along K only: each 32-element block
    # contributes 32 * 2^(ea_b + eb_b) exactly, and the sum is rounded to half
    # once (a scale taken from the wrong block would move it by far more).
    M, N, K = 128, 128, 512
    rng = np.random.default_rng(11)
    ea = rng.integers(-3, 4, K // 32)
    eb = rng.integers(-3, 4, K // 32)
    A = _e4m3(np.ones((M, K)))
    B = _e4m3(np.ones((N, K)))
    SA = torch.from_numpy(np.tile((127 + ea).astype(np.uint8), (M, 1)))
    SB = torch.from_numpy(np.tile((127 + eb).astype(np.uint8), (N, 1)))
    C = _run(A, SA, B, SB, variant=variant)
    exact = float(np.sum(32 * np.ldexp(1.0, ea + eb)))
    want = float(np.float16(exact))  # round to nearest even
    assert np.all(C.astype(np.float64) == want), (C[0, :4], exact)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", [
    (128, 128, 128),
    (256, 512, 1024),     # several tiles, 8 k-blocks
    (300, 520, 160),      # ragged M, N; a partial last k-block (160 = 128 + 32)
    (1000, 24, 2080),     # thin N, long K
    (7, 1000, 96),        # thin M, K below one k-block
])
def test_random_full_compare(M, N, K, variant):
    A, SA = wl.draw_mxfp8(M, K, seed=M + 3)
    B, SB = wl.draw_mxfp8(N, K, seed=N + 4)
    C = _run(A, SA, B, SB, variant=variant)
    Cref, S = oracle.gemm_mxfp8_nt(A, SA, B, SB)
    check_f16(C, Cref, S, what=f"mxfp8 {M}x{N}x{K} v{variant}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_scalar_store_path_and_k0(variant):
    # N % 8 != 0 takes the element-wise epilogue; K = 0 writes zeros.
    M, N, K = 200, 250, 256
    A, SA = wl.draw_mxfp8(M, K, seed=21)
    B, SB = wl.draw_mxfp8(N, K, seed=22)
    C = _run(A, SA, B, SB, variant=variant)
    Cref, S = oracle.gemm_mxfp8_nt(A, SA, B, SB)
    check_f16(C, Cref, S, what="scalar stores")
    Cz = torch.full((33, 17), 3.0, dtype=torch.float16, device="cuda")
    g.gemm_mxfp8_nt(33, 17, 0, 0, 0, 0, 0, Cz.data_ptr(), 0)
    torch.cuda.synchronize()
    assert (Cz == 0).all()


@pytest.mark.parametrize("variant,grid", [(g.GEMM_MXFP8_AUTO, 0), (g.GEMM_MXFP8_128x128, 0),
                                          (g.GEMM_MXFP8_256x128_PAIR, 6)])
def test_persistent_many_tiles_per_cta(variant, grid):
    # every CTA (pair) walks several tiles: accumulator buffers and stages cycle
    M, N, K = 768, 640, 512
    A, SA = wl.draw_mxfp8(M, K, seed=41)
    B, SB = wl.draw_mxfp8(N, K, seed=42)
    C = _run(A, SA, B, SB, variant=variant, grid=grid if grid else 3)
    Cref, S = oracle.gemm_mxfp8_nt(A, SA, B, SB)
    check_f16(C, Cref, S, what=f"persistent v{variant}")


def test_full_size_sampled():
    M, N, K = 5376, 5376, 2048
    A, SA = wl.draw_mxfp8(M, K, seed=31)
    B, SB = wl.draw_mxfp8(N, K, seed=32)
    C = g.mxfp8_nt(A.cuda(), SA.cuda(), B.cuda(), SB.cuda())
    g.gemm_check_device_status(0)
    Ch = C.cpu().numpy()
    rows, cols = wl.sample_positions(M, N, 16384, seed=2028)
    Cref, S = oracle.gemm_mxfp8_nt_sampled(A, SA, B, SB, rows, cols)
    check_f16(Ch[rows, cols], Cref, S, what="mxfp8 full size")
