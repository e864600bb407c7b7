"""GPU parity of gemm_nvfp4_nt (block-scaled FP4: E2M1 elements packed two
per byte, one E4M3 scale per 16 elements of K, a tensor-level scale alpha,
fp32 accumulation, half out) against the float64 oracle ("异步拷贝与
Hopper/Blackwell 新特性", section "Blackwell 概览 sm_100"), through the C ABI.

Staged like the MXFP8 tests: unit scales with small values (bit-exact: the
packed FP4 operands and the MMA), scales varying by row only (where each
row's scale sits), scales varying along K (which scale each 16-element slice
and each of the four MMAs of a k-block take), alpha, then random data with
ragged shapes and the packing of plain scales.
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
VARIANTS = [g.GEMM_MXFP8_128x128, g.GEMM_MXFP8_256x128_PAIR, g.GEMM_MXFP8_128x256,
            g.GEMM_MXFP8_256x256_PAIR]
E2M1 = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}
ONE, TWO, HALF = 0x38, 0x40, 0x30  # E4M3 scale codes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _pack(vals):
    # values in ±{0, .5, 1, 1.5, 2, 3, 4, 6} -> E2M1 pairs, element 2i low
    v = np.asarray(vals, dtype=np.float64)
    codes = np.vectorize(lambda x: E2M1[abs(x)] | (8 if x < 0 else 0))(v).astype(np.uint8)
    return torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))


def _run(A, SA, B, SB, alpha=1.0, pad=64, variant=g.GEMM_MXFP8_AUTO):
    M, N = A.shape[0], B.shape[0]
    buf = torch.empty((M * N + 2 * pad,), dtype=torch.int16, device="cuda")
    buf.fill_(SENTINEL)
    buf = buf.view(torch.float16)
    C = buf[pad:pad + M * N].view(M, N)
    g.nvfp4_nt(A.cuda(), SA.cuda(), B.cuda(), SB.cuda(), alpha, C, variant=variant)
    g.gemm_check_device_status(torch.cuda.current_stream().cuda_stream)
    host = buf.cpu()
    guard = torch.cat([host[:pad], host[pad + M * N:]]).view(torch.int16).numpy().view(np.uint16)
    assert np.all(guard == SENTINEL), "kernel wrote outside C"
    return host[pad:pad + M * N].view(M, N).numpy()


def _pack_ref(S, rows, K):
    cpr = 4 * ((K + 255) // 256)
    out = np.full(((rows + 127) // 128) * cpr * 512, 0x38, dtype=np.uint8)
    for r in range(rows):
        for j in range(K // 16):
            t, c = r // 128, j // 4
            rr, jj = r % 128, j % 4
            out[(t * cpr + c) * 512 + 16 * (rr % 32) + 4 * (rr // 32) + jj] = S[r, j]
    return out


@pytest.mark.parametrize("rows,K", [(1, 32), (128, 256), (300, 320), (129, 544)])
def test_pack_scales_layout(rows, K):
    S = torch.randint(0, 127, (rows, K // 16), dtype=torch.uint8)
    packed = g.nvfp4_pack_scales(S.cuda()).cpu().numpy()
    assert packed.size == g.gemm_nvfp4_scale_bytes(rows, K)
    assert np.array_equal(packed, _pack_ref(S.numpy(), rows, K))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 384, 512), (130, 136, 96)])
def test_unit_scales_small_values_bit_exact(M, N, K, variant):
    rng = np.random.default_rng(M + N + K)
    av = rng.choice([-1.0, -0.5, 0.0, 0.5, 1.0], (M, K))
    bv = rng.choice([-1.0, -0.5, 0.0, 0.5, 1.0], (N, K))
    SA = torch.full((M, K // 16), ONE, dtype=torch.uint8)
    SB = torch.full((N, K // 16), ONE, dtype=torch.uint8)
    C = _run(_pack(av), SA, _pack(bv), SB, variant=variant)
    assert np.array_equal(C.astype(np.float64), av @ bv.T)


@pytest.mark.parametrize("variant", VARIANTS)
def test_row_scales_place_each_rows_scale(variant):
    M, N, K = 256, 256, 256
    rng = np.random.default_rng(5)
    av = rng.choice([-1.0, 0.0, 0.5, 1.0], (M, K))
    bv = rng.choice([-1.0, 0.0, 0.5, 1.0], (N, K))
    ca = rng.choice([HALF, ONE, TWO], M)
    cb = rng.choice([HALF, ONE, TWO], N)
    SA = torch.from_numpy(np.repeat(ca[:, None], K // 16, axis=1).astype(np.uint8))
    SB = torch.from_numpy(np.repeat(cb[:, None], K // 16, axis=1).astype(np.uint8))
    C = _run(_pack(av), SA, _pack(bv), SB, variant=variant)
    Cref, S = oracle.gemm_nvfp4_nt(_pack(av), SA, _pack(bv), SB)
    sv = {HALF: 0.5, ONE: 1.0, TWO: 2.0}
    want = (av @ bv.T) * np.vectorize(sv.get)(ca)[:, None] * np.vectorize(sv.get)(cb)[None, :]
    assert np.array_equal(Cref, want)
    check_f16(C, Cref, S, what="row scales")


@pytest.mark.parametrize("variant", VARIANTS)
def test_block_scales_pick_their_16_elements(variant):
    # Ones everywhere; the scales vary along K only (every 16-element block
    # and so every MMA of a k-block differs): C = sum_b 16 * sa_b * sb_b.
    M, N, K = 128, 256, 512
    rng = np.random.default_rng(9)
    ca = rng.choice([HALF, ONE, TWO], K // 16)
    cb = rng.choice([HALF, ONE, TWO], K // 16)
    SA = torch.from_numpy(np.tile(ca.astype(np.uint8), (M, 1)))
    SB = torch.from_numpy(np.tile(cb.astype(np.uint8), (N, 1)))
    C = _run(_pack(np.ones((M, K))), SA, _pack(np.ones((N, K))), SB, variant=variant)
    sv = {HALF: 0.5, ONE: 1.0, TWO: 2.0}
    exact = float(sum(16 * sv[a] * sv[b] for a, b in zip(ca, cb)))
    assert np.all(C.astype(np.float64) == float(np.float16(exact))), (C[0, :4], exact)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K,alpha", [
    (128, 128, 256, 1.0),
    (256, 512, 1024, 0.25),   # several tiles and k-blocks, alpha
    (300, 520, 160, -1.5),    # ragged M, N; a partial last k-block
    (1000, 24, 2080, 1.0),    # thin N, long K
    (7, 1000, 96, 2.0),       # thin M, K below one k-block
])
def test_random_full_compare(M, N, K, alpha, variant):
    A, SA = wl.draw_nvfp4(M, K, seed=M + 5)
    B, SB = wl.draw_nvfp4(N, K, seed=N + 6)
    C = _run(A, SA, B, SB, alpha=alpha, variant=variant)
    Cref, S = oracle.gemm_nvfp4_nt(A, SA, B, SB, alpha=alpha)
    check_f16(C, Cref, S, what=f"nvfp4 {M}x{N}x{K} v{variant}")


def test_scalar_store_path_and_k0():
    M, N, K = 200, 250, 256
    A, SA = wl.draw_nvfp4(M, K, seed=23)
    B, SB = wl.draw_nvfp4(N, K, seed=24)
    C = _run(A, SA, B, SB, alpha=0.5)
    Cref, S = oracle.gemm_nvfp4_nt(A, SA, B, SB, alpha=0.5)
    check_f16(C, Cref, S, what="scalar stores")
    Cz = torch.full((33, 17), 3.0, dtype=torch.float16, device="cuda")
    g.gemm_nvfp4_nt(33, 17, 0, 0, 0, 0, 0, 1.0, Cz.data_ptr(), 0)
    torch.cuda.synchronize()
    assert (Cz == 0).all()


def test_full_size_sampled():
    M, N, K = 5376, 5376, 2048
    A, SA = wl.draw_nvfp4(M, K, seed=51)
    B, SB = wl.draw_nvfp4(N, K, seed=52)
    C = g.nvfp4_nt(A.cuda(), SA.cuda(), B.cuda(), SB.cuda(), 0.125)
    g.gemm_check_device_status(0)
    Ch = C.cpu().numpy()
    rows, cols = wl.sample_positions(M, N, 16384, seed=2029)
    Cref, S = oracle.gemm_nvfp4_nt_sampled(A, SA, B, SB, rows, cols, alpha=0.125)
    check_f16(Ch[rows, cols], Cref, S, what="nvfp4 full size")
