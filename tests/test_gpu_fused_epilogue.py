"""GPU parity of gemm_f16_nt_fused: C = act(alpha·A·Bᵀ + bias + beta·R),
rounded to half once, against the float64 oracle ("第 6 章 · Shared Memory &
Tile", section "6.5.4 Epilogue 融合"), through the C ABI.

Every fp16 kernel variant carries the epilogue: the 1-CTA tiles, the CTA pair
(also with stream-K partials), the M <= 4 matrix-vector kernel and the K = 0
fill.  Covered: all four activations, bias and residual present or absent,
the residual aliasing C, the scalar paths (N % 8 != 0, a bias that is not
16-byte aligned, C offset by one element), beta = 0 never reading R, and the
full-size 5376 × 5376 × 2048 product on a sample of outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import workloads as wl
from parity import check_f16_epilogue

pytestmark = pytest.mark.gpu

SENTINEL = 0x7E5A  # a NaN payload nothing in the product writes
ACTS = ["none", "relu", "silu", "gelu_tanh"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    g.load_library()
    torch.cuda.init()


def _inputs(M, N, K, seed, with_bias=True, with_res=True):
    A = wl.draw_f16((M, K), seed=seed, dist="normal")
    B = wl.draw_f16((N, K), seed=seed + 1, dist="normal")
    bias = wl.draw_f16((N,), seed=seed + 2, dist="normal") if with_bias else None
    R = wl.draw_f16((M, N), seed=seed + 3, dist="normal") if with_res else None
    return A, B, bias, R


def _run(A, B, bias, R, alpha, beta, act, variant=g.GEMM_F16_AUTO, grid=0, flags=0, pad=64,
         bias_offset=0):
    """The fused product on the GPU with a sentinel guard of `pad` halves
    around C; `bias_offset` shifts bias by that many halves off its
    allocation's alignment."""
    M, K = A.shape
    N = B.shape[0]
    dA, dB = A.cuda(), B.cuda()
    dbias = None
    if bias is not None:
        store = torch.empty(N + bias_offset, dtype=torch.float16, device="cuda")
        store[bias_offset:] = bias.cuda()
        dbias = store[bias_offset:]
    dR = R.cuda() if R is not None else None
    buf = torch.empty((M * N + 2 * pad,), dtype=torch.int16, device="cuda")
    buf.fill_(SENTINEL)
    buf = buf.view(torch.float16)
    C = buf[pad:pad + M * N].view(M, N)
    stream = torch.cuda.current_stream().cuda_stream
    g.gemm_f16_nt_fused(M, N, K, dA.data_ptr(), dB.data_ptr(), C.data_ptr(), alpha, beta,
                        dbias.data_ptr() if dbias is not None else 0,
                        dR.data_ptr() if dR is not None else 0, g.ACTIVATIONS[act], stream,
                        variant, grid, flags)
    g.gemm_check_device_status(stream)
    host = buf.cpu()
    guard = torch.cat([host[:pad], host[pad + M * N:]]).view(torch.int16).numpy().view(np.uint16)
    assert np.all(guard == SENTINEL), "kernel wrote outside C"
    return host[pad:pad + M * N].view(M, N).numpy()


VARIANTS = [g.GEMM_F16_128x256, g.GEMM_F16_128x128, g.GEMM_F16_256x256_PAIR]
SHAPES = [
    (256, 512, 128),   # whole tiles
    (300, 520, 136),   # ragged M, N and a partial k-block
    (129, 257, 72),    # one row / column past the tile edge (N % 8 != 0: scalar stores)
]


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_fused_full_compare(M, N, K, variant, act):
    A, B, bias, R = _inputs(M, N, K, seed=M + N)
    C = _run(A, B, bias, R, 0.5, -1.25, act, variant)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=0.5, bias=bias, beta=-1.25, R=R, act=act)
    check_f16_epilogue(C, Y, S, what=f"{M}x{N}x{K} v{variant} {act}")


@pytest.mark.parametrize("with_bias,with_res", [(True, False), (False, True), (False, False)])
def test_fused_optional_terms(with_bias, with_res):
    M, N, K = 384, 640, 256
    A, B, bias, R = _inputs(M, N, K, seed=11, with_bias=with_bias, with_res=with_res)
    C = _run(A, B, bias, R, 2.0, 0.75, "silu")
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=2.0, bias=bias, beta=0.75, R=R, act="silu")
    check_f16_epilogue(C, Y, S, what=f"bias={with_bias} res={with_res}")


def test_fused_identity_epilogue_equals_plain_product():
    # alpha = 1 and nothing else: the plain product, value for value.
    M, N, K = 300, 520, 136
    A, B, _, _ = _inputs(M, N, K, seed=21, with_bias=False, with_res=False)
    dA, dB = A.cuda(), B.cuda()
    plain = g.f16_nt(dA, dB)
    fused = g.f16_nt_fused(dA, dB)
    torch.cuda.synchronize()
    assert torch.equal(plain, fused)


@pytest.mark.parametrize("variant", [g.GEMM_F16_AUTO, g.GEMM_F16_256x256_PAIR])
def test_fused_in_place_residual(variant):
    # C = gelu(A·Bᵀ + bias + C): the residual is the output buffer itself
    # (the pair kernel fetches it by TMA into the staging it stores from).
    M, N, K = 520, 776, 200
    A, B, bias, R = _inputs(M, N, K, seed=31)
    dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
    C = R.cuda()
    g.f16_nt_fused(dA, dB, C, alpha=1.0, bias=dbias, beta=1.0, residual=C, activation="gelu_tanh",
                   variant=variant)
    torch.cuda.synchronize()
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=1.0, bias=bias, beta=1.0, R=R, act="gelu_tanh")
    check_f16_epilogue(C.cpu().numpy(), Y, S, what="in place")


def test_fused_scalar_paths():
    # A bias one half off 16-byte alignment and a C one half off alignment
    # take the element-wise loads and stores.
    M, N, K = 200, 256, 64
    A, B, bias, R = _inputs(M, N, K, seed=41)
    C = _run(A, B, bias, R, -1.0, 0.5, "relu", bias_offset=1, pad=1)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=-1.0, bias=bias, beta=0.5, R=R, act="relu")
    check_f16_epilogue(C, Y, S, what="scalar paths")


def test_fused_beta_zero_never_reads_the_residual():
    # beta = 0 with a residual full of NaN: R must not be read at all.
    M, N, K = 256, 512, 128
    A, B, bias, _ = _inputs(M, N, K, seed=51, with_res=False)
    dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
    Rnan = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    C = g.f16_nt_fused(dA, dB, alpha=1.0, bias=dbias, beta=0.0, residual=Rnan, activation="relu")
    torch.cuda.synchronize()
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=1.0, bias=bias, act="relu")
    check_f16_epilogue(C.cpu().numpy(), Y, S, what="beta 0")


@pytest.mark.parametrize("M,N,K,grid", [(1024, 1024, 512, 6), (1000, 1100, 1000, 10)])
def test_fused_with_stream_k(M, N, K, grid):
    # Owners add the fp32 partials of the split tiles before the epilogue.
    A, B, bias, R = _inputs(M, N, K, seed=61)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=0.25, bias=bias, beta=1.5, R=R, act="gelu_tanh")
    for rep in range(2):
        C = _run(A, B, bias, R, 0.25, 1.5, "gelu_tanh", g.GEMM_F16_256x256_PAIR, grid,
                 g.GEMM_F16_FLAG_STREAM_K)
        check_f16_epilogue(C, Y, S, what=f"stream-K grid {grid} rep {rep}")


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_fused_with_split_k(act):
    # One tile split four ways (4 pairs): the owner adds the partials, then
    # applies the epilogue with the residual from its TMA ring.
    M, N, K = 256, 256, 8192
    A, B, bias, R = _inputs(M, N, K, seed=65)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=0.5, bias=bias, beta=-1.0, R=R, act=act)
    C = _run(A, B, bias, R, 0.5, -1.0, act, g.GEMM_F16_256x256_PAIR, 8)
    check_f16_epilogue(C, Y, S, what=f"split-K {act}")


@pytest.mark.parametrize("act", ACTS)
@pytest.mark.parametrize("M,N,K", [(1, 1000, 4096), (2, 777, 520)])
def test_fused_gemv(M, N, K, act):
    A, B, bias, R = _inputs(M, N, K, seed=71 + M)
    C = _run(A, B, bias, R, 1.5, -0.5, act, g.GEMM_F16_GEMV)
    Y, S = oracle.gemm_f16_nt_epilogue(A, B, alpha=1.5, bias=bias, beta=-0.5, R=R, act=act)
    check_f16_epilogue(C, Y, S, what=f"gemv {M}x{N}x{K} {act}")


def test_fused_k0_is_the_epilogue_of_zero():
    M, N = 33, 17
    bias = wl.draw_f16((N,), seed=81, dist="normal")
    R = wl.draw_f16((M, N), seed=82, dist="normal")
    dbias, dR = bias.cuda(), R.cuda()
    dA = torch.zeros(8, dtype=torch.float16, device="cuda")
    C = torch.full((M, N), 3.0, dtype=torch.float16, device="cuda")
    g.gemm_f16_nt_fused(M, N, 0, dA.data_ptr(), dA.data_ptr(), C.data_ptr(), 1.0, 2.0,
                        dbias.data_ptr(), dR.data_ptr(), g.GEMM_ACT_SILU,
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    A0 = torch.zeros((M, 0), dtype=torch.float16)
    B0 = torch.zeros((N, 0), dtype=torch.float16)
    Y, S = oracle.gemm_f16_nt_epilogue(A0, B0, alpha=1.0, bias=bias, beta=2.0, R=R, act="silu")
    check_f16_epilogue(C.cpu().numpy(), Y, S, what="K = 0")


@pytest.mark.parametrize("act", ["relu", "gelu_tanh"])
def test_fused_full_size_sampled(act):
    # The 5376 × 5376 × 2048 workload under the selector's kernel.
    w = wl.WORKLOADS["f16_nt_5376x5376x2048"]
    A, B, _ = wl.make_inputs(w)
    bias = wl.draw_f16((w.N,), seed=91)
    R = wl.draw_f16((w.M, w.N), seed=92)
    dA, dB, dbias, dR = A.cuda(), B.cuda(), bias.cuda(), R.cuda()
    C = g.f16_nt_fused(dA, dB, alpha=0.125, bias=dbias, beta=1.0, residual=dR, activation=act)
    g.gemm_check_device_status(0)
    Ch = C.cpu().numpy()
    rows, cols = wl.sample_positions(w.M, w.N, 32768, seed=2026)
    Y, S = oracle.gemm_f16_nt_epilogue_sampled(A, B, rows, cols, alpha=0.125, bias=bias, beta=1.0,
                                               R=R, act=act)
    check_f16_epilogue(Ch[rows, cols], Y, S, what=f"full size {act}")
