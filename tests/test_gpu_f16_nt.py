"""GPU parity of gemm_f16_nt (C = A·Bᵀ, fp16 in, fp32 accumulate, fp16 out)
against the float64 oracle, called through the C ABI.

Small shapes are compared element by element (several tiles, ragged M/N/K
tails, every compiled tile variant, persistent loops forced through many
tiles per CTA); the two full-size workloads are compared on a seeded sample
of 65,536 outputs plus the last row, last column and the partial M tile.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_f16

pytestmark = pytest.mark.gpu

SENTINEL = 0x7E5A  # a NaN payload nothing in the product writes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _run(A, B, variant=g.GEMM_F16_AUTO, grid=0, pad=64, flags=0, raster=0):
    """Run on the GPU with a sentinel guard of `pad` halves around C."""
    M, K = A.shape
    N = B.shape[0]
    dA, dB = A.cuda(), B.cuda()
    buf = torch.full((M * N + 2 * pad,), 0, dtype=torch.int16, device="cuda")
    buf.fill_(SENTINEL - (1 << 16) if SENTINEL >= (1 << 15) else SENTINEL)
    buf = buf.view(torch.float16)
    C = buf[pad:pad + M * N].view(M, N)
    g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                     torch.cuda.current_stream().cuda_stream, variant, grid, flags, raster)
    g.gemm_check_device_status(torch.cuda.current_stream().cuda_stream)
    host = buf.cpu()
    guard = torch.cat([host[:pad], host[pad + M * N:]]).view(torch.int16).numpy().view(np.uint16)
    assert np.all(guard == SENTINEL), "kernel wrote outside C"
    return host[pad:pad + M * N].view(M, N).numpy()


SHAPES = [
    (128, 256, 64),      # exactly one wide tile, one k-block
    (256, 512, 128),     # 2 x 2 wide tiles
    (300, 520, 136),     # ragged M, N and a partial k-block (136 = 2*64 + 8)
    (129, 257, 72),      # one row / column past the tile edge
    (1, 1, 8),           # smallest legal problem
    (7, 1000, 2048),     # thin M, long K
    (1000, 24, 520),     # thin N
    (640, 768, 1024),    # several tiles per CTA under the selector's grid
]


VARIANTS = [g.GEMM_F16_128x256, g.GEMM_F16_128x128, g.GEMM_F16_256x256_PAIR]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_f16_nt_full_compare(M, N, K, variant):
    A = wl.draw_f16((M, K), seed=M + 1)
    B = wl.draw_f16((N, K), seed=N + 2)
    C = _run(A, B, variant)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C, Cref, S, what=f"{M}x{N}x{K} v{variant}")


@pytest.mark.parametrize("variant,grid", [(g.GEMM_F16_128x256, 1), (g.GEMM_F16_128x256, 3),
                                          (g.GEMM_F16_128x128, 1), (g.GEMM_F16_128x128, 5),
                                          (g.GEMM_F16_256x256_PAIR, 2),
                                          (g.GEMM_F16_256x256_PAIR, 6)])
def test_f16_nt_persistent_many_tiles_per_cta(variant, grid):
    # 5 x 3 (wide), 5 x 6 (narrow) or 3 x 3 (pair) tiles on 1..5 CTAs or 1..3
    # CTA pairs: every stage and accumulator barrier goes through several phases.
    M, N, K = 600, 700, 392
    A = wl.draw_f16((M, K), seed=31, dist="normal")
    B = wl.draw_f16((N, K), seed=32, dist="normal")
    C = _run(A, B, variant, grid)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C, Cref, S, what=f"grid={grid} v{variant}")


# Two CTA pairs sharing B (a 4-CTA cluster, B multicast to both pairs): each
# tile is computed with the very MMAs of the pair kernel, so the two variants
# must agree bit for bit, and both with the oracle.  Shapes: rows of A and B
# off the 128-byte grid (K % 64 != 0), a cluster whose second pair falls
# wholly past the last row (M = 600: its tile rows 768.. are empty), aligned
# K, several tiles per cluster (grid of 2 or 3 clusters), a ragged N.
@pytest.mark.parametrize("M,N,K,grid", [(600, 520, 136, 0), (1024, 768, 1000, 0),
                                        (300, 300, 64, 0), (1536, 1280, 520, 8),
                                        (1100, 700, 392, 12), (2048, 2048, 1016, 0)])
def test_f16_nt_two_pairs_sharing_b_match_the_pair_kernel(M, N, K, grid):
    A = wl.draw_f16((M, K), seed=M + 5, dist="normal")
    B = wl.draw_f16((N, K), seed=N + 6, dist="normal")
    C = _run(A, B, g.GEMM_F16_256x256_QUAD, grid)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C, Cref, S, what=f"quad {M}x{N}x{K} grid {grid}")
    Cpair = _run(A, B, g.GEMM_F16_256x256_PAIR)
    assert np.array_equal(C.view(np.uint16), Cpair.view(np.uint16)), \
        "two pairs sharing B differ from the pair kernel"


def test_f16_nt_two_pairs_sharing_b_scalar_store_paths():
    # N % 8 != 0 and a C offset by one element take the per-element epilogue
    # (no TMA store) in both pairs of the cluster.
    for (M, N, K), pad in [((700, 250, 136), 64), ((530, 264, 200), 1)]:
        A = wl.draw_f16((M, K), seed=M + 7, dist="normal")
        B = wl.draw_f16((N, K), seed=N + 8, dist="normal")
        C = _run(A, B, g.GEMM_F16_256x256_QUAD, pad=pad)
        Cref, S = oracle.gemm_f16_nt(A, B)
        check_f16(C, Cref, S, what=f"quad scalar {M}x{N}x{K} pad={pad}")


def test_f16_nt_two_pairs_sharing_b_repeatable():
    # the same launch many times on one stream: every run bit-identical (a
    # stage refilled before both pairs have read it would show as a change)
    M, N, K = 2048, 2048, 2040
    A = wl.draw_f16((M, K), seed=61, dist="normal")
    B = wl.draw_f16((N, K), seed=62, dist="normal")
    dA, dB = A.cuda(), B.cuda()
    stream = torch.cuda.current_stream().cuda_stream
    outs = []
    for _ in range(20):
        C = torch.empty((M, N), dtype=torch.float16, device="cuda")
        g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), stream,
                         g.GEMM_F16_256x256_QUAD)
        outs.append(C)
    g.gemm_check_device_status(stream)
    first = outs[0].cpu().numpy()
    for i, C in enumerate(outs[1:]):
        assert np.array_equal(C.cpu().numpy().view(np.uint16), first.view(np.uint16)), f"run {i + 1}"
    rows, cols = wl.sample_positions(M, N, 65536, seed=63)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(first[rows, cols], Cref, S, what="quad repeated")


# Two CTA pairs of a 4-CTA cluster splitting one tile's K range: the second
# pair's fp32 sum reaches the first through distributed shared memory.
# Shapes: one tile, ragged M, N and K (a partial last k-block), the fewest
# k-blocks the split takes (2 and 3), tiles past the clusters that fit at
# once (80 tiles: clusters start later), a long K, and K = 64 (a single
# k-block: the pair variant runs instead).
@pytest.mark.parametrize("M,N,K", [(256, 256, 128), (300, 700, 520), (200, 600, 136), (512, 384, 4104),
                                   (2560, 2048, 256), (1024, 1024, 8192), (256, 512, 64)])
def test_f16_nt_k_split_cluster(M, N, K):
    A = wl.draw_f16((M, K), seed=M + 21, dist="normal")
    B = wl.draw_f16((N, K), seed=N + 22, dist="normal")
    C = _run(A, B, g.GEMM_F16_256x256_KSPLIT)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C, Cref, S, what=f"k-split {M}x{N}x{K}")


def test_f16_nt_k_split_cluster_repeatable_and_exact():
    # small integers: every partial sum is an exact integer, so the result
    # must equal the exact product bit for bit; and repeated runs agree
    M, N, K = 768, 1024, 2048
    rng = np.random.default_rng(5)
    A = torch.from_numpy(rng.integers(-1, 2, (M, K)).astype(np.float16))
    B = torch.from_numpy(rng.integers(-1, 2, (N, K)).astype(np.float16))
    exact = (A.double() @ B.double().t()).numpy()
    first = _run(A, B, g.GEMM_F16_256x256_KSPLIT)
    assert np.array_equal(first.astype(np.float64), exact)
    for _ in range(3):
        assert np.array_equal(_run(A, B, g.GEMM_F16_256x256_KSPLIT).view(np.uint16), first.view(np.uint16))


def test_f16_nt_k_split_cluster_sampled_large():
    M, N, K = 1024, 2048, 8192
    A = wl.draw_f16((M, K), seed=31, dist="normal")
    B = wl.draw_f16((N, K), seed=32, dist="normal")
    C = _run(A, B, g.GEMM_F16_256x256_KSPLIT)
    rows, cols = wl.sample_positions(M, N, 65536, seed=33)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(C[rows, cols], Cref, S, what="k-split sampled")


def test_f16_nt_small_integers_bit_exact():
    # entries in {-1, 0, 1}, K = 1024: every partial sum is an integer below
    # 2^11, exact in fp32 and in half, so the output must match bit for bit.
    M, N, K = 384, 640, 1024
    A = wl.draw_int((M, K), 41, -1, 1, torch.float16)
    B = wl.draw_int((N, K), 42, -1, 1, torch.float16)
    C = _run(A, B)
    Cref, _ = oracle.gemm_f16_nt(A, B)
    assert np.array_equal(C.astype(np.float64), Cref)


def test_f16_nt_identity_and_permutation():
    M, K = 256, 256
    A = wl.draw_f16((M, K), seed=5)
    perm = torch.randperm(K, generator=torch.Generator().manual_seed(6))
    B = torch.eye(K, dtype=torch.float16)[perm]
    C = _run(A, B)
    assert np.array_equal(C, A.numpy()[:, perm.numpy()])


def test_f16_nt_scalar_store_paths():
    # N % 8 != 0 forces the per-element epilogue; a C offset by one element
    # (2-byte aligned) does too.
    for (M, N, K), pad in [((200, 250, 64), 64), ((130, 136, 128), 1)]:
        A = wl.draw_f16((M, K), seed=7)
        B = wl.draw_f16((N, K), seed=8)
        C = _run(A, B, pad=pad)
        Cref, S = oracle.gemm_f16_nt(A, B)
        check_f16(C, Cref, S, what=f"scalar {M}x{N}x{K} pad={pad}")


def test_f16_nt_k0_writes_zeros():
    A = torch.zeros((0,), dtype=torch.float16).reshape(33, 0)
    B = torch.zeros((0,), dtype=torch.float16).reshape(17, 0)
    dA = torch.zeros(8, dtype=torch.float16, device="cuda")
    C = torch.full((33, 17), 3.0, dtype=torch.float16, device="cuda")
    g.gemm_f16_nt(33, 17, 0, dA.data_ptr(), dA.data_ptr(), C.data_ptr(),
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert A.shape[1] == 0 and B.shape[1] == 0
    assert (C == 0).all()


def test_f16_nt_unsupported_k_leaves_c_untouched():
    A = torch.zeros((16, 12), dtype=torch.float16, device="cuda")
    C = torch.full((16, 16), 5.0, dtype=torch.float16, device="cuda")
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt(16, 16, 12, A.data_ptr(), A.data_ptr(), C.data_ptr(), 0)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (C == 5.0).all()


def test_f16_nt_on_a_side_stream_and_tensor_wrapper():
    A = wl.draw_f16((512, 256), seed=9)
    B = wl.draw_f16((384, 256), seed=10)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dA, dB = A.cuda(), B.cuda()
        C = g.f16_nt(dA, dB)
    s.synchronize()
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C.cpu().numpy(), Cref, S, what="side stream")


@pytest.mark.parametrize("variant", VARIANTS)
def test_f16_nt_long_k_many_tiles(variant):
    # K = 4096 (64 k-blocks) over a grid that cycles each CTA through tiles.
    M, N, K = 1024, 1280, 4096
    A = wl.draw_f16((M, K), seed=51, dist="normal")
    B = wl.draw_f16((N, K), seed=52, dist="normal")
    C = _run(A, B, variant, grid=8)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C, Cref, S, what=f"long K v{variant}")


@pytest.mark.parametrize("name", ["f16_nt_5376x5376x2048", "f16_nt_5000x5376x2040"])
def test_f16_nt_full_size_stream_k_sampled(name):
    # The same workloads with the last round of tiles split along K.
    w = wl.WORKLOADS[name]
    A, B, _ = wl.make_inputs(w)
    dA, dB = A.cuda(), B.cuda()
    C = g.f16_nt(dA, dB, variant=g.GEMM_F16_256x256_PAIR, flags=g.GEMM_F16_FLAG_STREAM_K)
    g.gemm_check_device_status(0)
    Ch = C.cpu().numpy()
    rows, cols = wl.sample_positions(w.M, w.N, 65536, seed=2025)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(Ch[rows, cols], Cref, S, what=name + " stream-K")


@pytest.mark.parametrize("name", ["f16_nt_5376x5376x2048", "f16_nt_5000x5376x2040"])
def test_f16_nt_full_size_sampled(name):
    # The launch configuration the benchmark times (selector default).
    w = wl.WORKLOADS[name]
    A, B, _ = wl.make_inputs(w)
    dA, dB = A.cuda(), B.cuda()
    C = torch.empty((w.M, w.N), dtype=torch.float16, device="cuda")
    g.gemm_f16_nt(w.M, w.N, w.K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                  torch.cuda.current_stream().cuda_stream)
    g.gemm_check_device_status(torch.cuda.current_stream().cuda_stream)
    Ch = C.cpu().numpy()
    assert np.all(np.isfinite(Ch.astype(np.float32)))
    tail = list(range((w.M // 128) * 128, w.M))[:8] if w.M % 128 else []
    rows, cols = wl.sample_positions(w.M, w.N, 65536, seed=2024, tail_rows=tail)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(Ch[rows, cols], Cref, S, what=name)


@pytest.mark.parametrize("M,N,K,grid", [
    (1024, 1024, 512, 6),     # 16 pair tiles on 3 pairs: the 16th tile split over all three
    (1024, 1024, 512, 10),    # 5 pairs, one leftover tile
    (1024, 1024, 512, 14),    # 7 pairs, two leftover tiles: each split over ~4 pairs
    (1000, 1100, 1000, 10),   # ragged M, N, K with split tiles
    (2304, 2304, 256, 152),   # 81 tiles on 76 pairs: the selector's grid
])
def test_f16_nt_pair_stream_k(M, N, K, grid):
    # The leftover round of pair tiles is split along K across the pairs;
    # owners add the fp32 partials of the following shares before rounding.
    A = wl.draw_f16((M, K), seed=61, dist="normal")
    B = wl.draw_f16((N, K), seed=62, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    for rep in range(3):   # sequence numbers advance between calls on one stream
        C = _run(A, B, g.GEMM_F16_256x256_PAIR, grid, flags=g.GEMM_F16_FLAG_STREAM_K)
        check_f16(C, Cref, S, what=f"stream-K {M}x{N}x{K} grid {grid} rep {rep}")


def test_f16_nt_pair_stream_k_two_streams():
    M, N, K = 1024, 1024, 512
    A = wl.draw_f16((M, K), seed=71)
    B = wl.draw_f16((N, K), seed=72)
    Cref, S = oracle.gemm_f16_nt(A, B)
    dA, dB = A.cuda(), B.cuda()
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        with torch.cuda.stream(s):
            C = torch.empty((M, N), dtype=torch.float16, device="cuda")
            g.gemm_f16_nt_ex(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), s.cuda_stream,
                             g.GEMM_F16_256x256_PAIR, 10, g.GEMM_F16_FLAG_STREAM_K)
            outs.append(C)
    for s in streams:
        s.synchronize()
    g.gemm_check_device_status(0)
    for C in outs:
        check_f16(C.cpu().numpy(), Cref, S, what="two streams")


@pytest.mark.parametrize("M,N,K,grid", [
    (256, 256, 8192, 8),      # one tile split four ways (4 pairs, 32 k-blocks each)
    (200, 300, 8200, 16),     # two ragged tiles split eight ways, a partial last k-block
    (512, 256, 16384, 152),   # two tiles over the full grid: eight ways each
])
def test_f16_nt_split_k_underfilled(M, N, K, grid):
    # Few pair tiles over a long K: every tile's k-blocks are shared out over
    # several pairs by default (no flag); the owner adds the partials.
    A = wl.draw_f16((M, K), seed=81, dist="normal")
    B = wl.draw_f16((N, K), seed=82, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    for rep in range(2):
        C = _run(A, B, g.GEMM_F16_256x256_PAIR, grid)
        check_f16(C, Cref, S, what=f"split-K {M}x{N}x{K} grid {grid} rep {rep}")


@pytest.mark.parametrize("M,N,K", [(512, 512, 32768), (256, 256, 65536), (256, 4096, 8192)])
def test_f16_nt_split_k_selector_shapes_sampled(M, N, K):
    # Few tiles over a long K, through the selector: the skinny kernel with
    # 128-row tiles of A and the K range split over clusters (the pair
    # kernel's split stays reachable through gemm_f16_nt_ex, tested above).
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert g.gemm_f16_select(M, N, K, sm)[0] == g.GEMM_F16_SKINNY
    A = wl.draw_f16((M, K), seed=83)
    B = wl.draw_f16((N, K), seed=84)
    dA, dB = A.cuda(), B.cuda()
    C = g.f16_nt(dA, dB)
    g.gemm_check_device_status(0)
    Ch = C.cpu().numpy()
    rows, cols = wl.sample_positions(M, N, 8192, seed=2027)
    Cref, S = oracle.gemm_f16_nt_sampled(A, B, rows, cols)
    check_f16(Ch[rows, cols], Cref, S, what=f"split-K default {M}x{N}x{K}")



@pytest.mark.parametrize("variant,grid,flags", [
    (g.GEMM_F16_256x256_PAIR, 0, 0),
    (g.GEMM_F16_256x256_PAIR, 6, g.GEMM_F16_FLAG_STREAM_K),  # 3 pairs: stream-K over the last round
    (g.GEMM_F16_128x128, 7, 0),
    (g.GEMM_F16_128x256, 0, 0),
])
@pytest.mark.parametrize("raster", [1, 2, 3, 8])
def test_f16_nt_banded_tile_order(variant, grid, flags, raster):
    # The persistent CTAs walk the tiles in bands of `raster` tile rows (the
    # last band shorter); every tile is computed once, whatever the band.
    M, N, K = 1160, 1100, 192
    A = wl.draw_f16((M, K), seed=71, dist="normal")
    B = wl.draw_f16((N, K), seed=72, dist="normal")
    Cref, S = oracle.gemm_f16_nt(A, B)
    C = _run(A, B, variant, grid, flags=flags, raster=raster)
    check_f16(C, Cref, S, what=f"raster {raster} v{variant} grid {grid} flags {flags}")
