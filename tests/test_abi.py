"""CPU-only checks of the C ABI: the library loads, exports every function
the headers declare, validates arguments on the host before touching a
device, and selects tiles by shape."""
import glob
import os
import re

import pytest

import dense_gemm_fp16_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_fp16_gb300 import build

    build.build()
    return g.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h, encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_headers_declare_the_boundary():
    names = _declared_functions()
    for n in ["gemm_f16_nt", "sgemm", "gemm_last_error", "gemm_check_device_status",
              "gemm_f16_select", "gemm_sgemm_select", "gemm_f16_nt_ex", "sgemm_ex",
              "gemm_debug_f16_nt_skip_load", "gemm_debug_skinny_plan",
              "gemm_f16_nt_fused", "gemm_f16_nt_stream_k_noalloc",
              "gemm_mxfp8_nt", "gemm_mxfp8_scale_bytes", "gemm_mxfp8_pack_scales",
              "gemm_nvfp4_nt", "gemm_nvfp4_nt_ex", "gemm_nvfp4_scale_bytes", "gemm_nvfp4_pack_scales",
              "gemm_debug_last_pair_launch", "gemm_debug_sm_clocks"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"libgemm.so does not export {name}"


def test_negative_sizes_are_rejected_on_the_host(lib):
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt(-1, 4, 8, 16, 16, 16)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    assert "negative" in g.gemm_last_error()
    with pytest.raises(g.GemmError) as e:
        g.sgemm(4, -4, 4, 1.0, 16, 16, 0.0, 16)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG


def test_pair_launch_record_is_empty_before_any_launch(lib):
    # host-side state of the test hook: nothing launched in this process yet
    assert g.gemm_debug_last_pair_launch() is None


def test_clock_sample_rejects_bad_arguments_on_the_host(lib):
    # checked before any CUDA call: nothing is enqueued
    for out, ctas in [(0, 4), (4096, 0), (4096, 65536), (4100, 4)]:
        with pytest.raises(g.GemmError) as e:
            g.gemm_debug_sm_clocks(out, ctas, 0)
        assert e.value.status == g.GEMM_ERR_INVALID_ARG
    assert "gemm_debug_sm_clocks" in g.gemm_last_error()


def test_empty_problems_are_no_ops(lib):
    assert g.gemm_f16_nt(0, 10, 64, 0, 0, 0) == g.GEMM_OK
    assert g.gemm_f16_nt(10, 0, 64, 0, 0, 0) == g.GEMM_OK
    assert g.sgemm(0, 5, 5, 1.0, 0, 0, 0.0, 0) == g.GEMM_OK


def test_null_and_misaligned_pointers(lib):
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt(4, 4, 8, 0, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt(4, 4, 8, 0x1002, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_MISALIGNED
    with pytest.raises(g.GemmError) as e:
        g.sgemm(4, 4, 4, 1.0, 0x1000, 0x1000, 0.0, 0)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG


def test_k_not_multiple_of_8_is_unsupported_for_f16(lib):
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt(16, 16, 12, 0x1000, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED
    assert "K=12" in str(e.value)


def test_bad_config_is_rejected(lib):
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt_ex(16, 16, 16, 0x1000, 0x1000, 0x1000, variant=99)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt_ex(16, 16, 16, 0x1000, 0x1000, 0x1000, flags=4)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.sgemm_ex(16, 16, 16, 1.0, 0x1000, 0x1000, 0.0, 0x1000, variant=7)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG


def test_fused_epilogue_arguments_are_checked_on_the_host(lib):
    for act in (-1, 4, 99):
        with pytest.raises(g.GemmError) as e:
            g.gemm_f16_nt_fused(16, 16, 16, 0x1000, 0x1000, 0x1000, activation=act)
        assert e.value.status == g.GEMM_ERR_INVALID_ARG
        assert "activation" in str(e.value)
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt_fused(-2, 16, 16, 0x1000, 0x1000, 0x1000, activation=g.GEMM_ACT_RELU)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt_fused(16, 16, 16, 0x1008, 0x1000, 0x1000, activation=g.GEMM_ACT_SILU)
    assert e.value.status == g.GEMM_ERR_MISALIGNED
    assert g.gemm_f16_nt_fused(0, 16, 16, 0, 0, 0, activation=g.GEMM_ACT_GELU_TANH) == g.GEMM_OK
    assert g.ACTIVATIONS == {"none": 0, "relu": 1, "silu": 2, "gelu_tanh": 3}


def test_mxfp8_arguments_are_checked_on_the_host(lib):
    assert g.gemm_mxfp8_scale_bytes(0, 64) == 0 and g.gemm_mxfp8_scale_bytes(64, 0) == 0
    assert g.gemm_mxfp8_scale_bytes(1, 32) == 512
    assert g.gemm_mxfp8_scale_bytes(129, 160) == 2 * 2 * 512
    assert g.gemm_mxfp8_scale_bytes(5376, 2048) == 42 * 16 * 512
    with pytest.raises(g.GemmError) as e:
        g.gemm_mxfp8_nt(16, 16, 48, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED and "K=48" in str(e.value)
    with pytest.raises(g.GemmError) as e:
        g.gemm_mxfp8_nt(16, 16, 64, 0x1000, 0x1004, 0x1000, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_MISALIGNED
    with pytest.raises(g.GemmError) as e:
        g.gemm_mxfp8_nt(16, 16, 64, 0, 0x1000, 0x1000, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    with pytest.raises(g.GemmError) as e:
        g.gemm_mxfp8_nt(-1, 16, 64, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_mxfp8_nt(0, 16, 64, 0, 0, 0, 0, 0) == g.GEMM_OK
    with pytest.raises(g.GemmError) as e:
        g.gemm_mxfp8_pack_scales(16, 40, 0x1000, 0x1000)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED


def test_nvfp4_arguments_are_checked_on_the_host(lib):
    assert g.gemm_nvfp4_scale_bytes(0, 64) == 0
    assert g.gemm_nvfp4_scale_bytes(1, 32) == 4 * 512
    assert g.gemm_nvfp4_scale_bytes(129, 320) == 2 * 4 * 2 * 512
    with pytest.raises(g.GemmError) as e:
        g.gemm_nvfp4_nt(16, 16, 48, 0x1000, 0x1000, 0x1000, 0x1000, 1.0, 0x1000)
    assert e.value.status == g.GEMM_ERR_UNSUPPORTED and "K=48" in str(e.value)
    with pytest.raises(g.GemmError) as e:
        g.gemm_nvfp4_nt(16, 16, 64, 0x1008, 0x1000, 0x1000, 0x1000, 1.0, 0x1000)
    assert e.value.status == g.GEMM_ERR_MISALIGNED
    with pytest.raises(g.GemmError) as e:
        g.gemm_nvfp4_nt_ex(16, 16, 64, 0x1000, 0x1000, 0x1000, 0x1000, 1.0, 0x1000,
                           variant=g.GEMM_MXFP8_NUM_VARIANTS)
    assert e.value.status == g.GEMM_ERR_INVALID_ARG
    assert g.gemm_nvfp4_nt(16, 0, 64, 0, 0, 0, 0, 1.0, 0) == g.GEMM_OK


def test_f16_selector(lib):
    # the two fp16 workloads: CTA-pair 256 x 256 tiles, one CTA per SM
    assert g.gemm_f16_select(5376, 5376, 2048, 152)[:2] == (g.GEMM_F16_256x256_PAIR, 152)
    # rows of 4080 bytes (K = 2040), off the 128-byte grid: two pairs sharing B
    # few pair tiles over a long K: two pairs per cluster split each tile's K
    assert g.gemm_f16_select(1024, 2048, 8192, 152)[:2] == (g.GEMM_F16_256x256_KSPLIT, 128)
    assert g.gemm_f16_select(512, 4096, 14336, 152)[0] == g.GEMM_F16_256x256_KSPLIT
    assert g.gemm_f16_select(1024, 2048, 2048, 152)[0] != g.GEMM_F16_256x256_KSPLIT   # halves too short
    assert g.gemm_f16_select(768, 4096, 8192, 152)[0] != g.GEMM_F16_256x256_KSPLIT    # 48 tiles > 36 clusters
    assert g.gemm_f16_select(1024, 1024, 8192, 152)[0] == g.GEMM_F16_SKINNY           # 16 tiles: the skinny split
    assert g.gemm_f16_select(5000, 5376, 2040, 152)[:2] == (g.GEMM_F16_256x256_QUAD, 152)
    assert g.gemm_f16_select(5376, 5376, 2040, 152)[0] == g.GEMM_F16_256x256_QUAD
    assert g.gemm_f16_select(8192, 8192, 8184, 152)[0] == g.GEMM_F16_256x256_QUAD
    assert g.gemm_f16_select(2048, 2048, 1016, 152)[:2] == (g.GEMM_F16_256x256_QUAD, 128)
    assert g.gemm_f16_select(5376, 5376, 2048, 152)[0] == g.GEMM_F16_256x256_PAIR   # whole lines
    assert g.gemm_f16_select(5376, 5376, 2048, 151)[:2] == (g.GEMM_F16_256x256_PAIR, 150)
    assert g.gemm_f16_select(8192, 8192, 8192, 152)[:2] == (g.GEMM_F16_256x256_PAIR, 152)
    # one row of A: the HBM-bound matrix-vector kernel, planned per SM
    assert g.gemm_f16_select(1, 5376, 2048, 152)[:2] == (g.GEMM_F16_GEMV, 152)
    assert g.gemm_f16_select(1, 4096, 65536, 152)[0] == g.GEMM_F16_GEMV
    # two to 64 rows: the skinny tensor-core kernel, one CTA per SM as the
    # target of its K split
    assert g.gemm_f16_select(2, 16384, 8192, 152)[:2] == (g.GEMM_F16_SKINNY, 152)
    assert g.gemm_f16_select(4, 16384, 8192, 148)[:2] == (g.GEMM_F16_SKINNY, 148)
    assert g.gemm_f16_select(5, 4096, 65536, 152)[0] == g.GEMM_F16_SKINNY
    assert g.gemm_f16_select(64, 8192, 8192, 152)[0] == g.GEMM_F16_SKINNY
    assert g.gemm_f16_select(64, 65536, 4096, 152)[0] == g.GEMM_F16_SKINNY
    # any M whose 128 x 128 tiles leave SMs idle: the skinny kernel when it
    # splits K in two shares of 16+ k-blocks, or in four or more
    assert g.gemm_f16_select(65, 8192, 8192, 152)[0] == g.GEMM_F16_SKINNY       # 2 x 64
    assert g.gemm_f16_select(128, 4096, 4096, 152)[0] == g.GEMM_F16_SKINNY      # 4 x 16
    assert g.gemm_f16_select(160, 2048, 8192, 152)[0] == g.GEMM_F16_SKINNY      # 4 x 32
    assert g.gemm_f16_select(512, 512, 32768, 152)[0] == g.GEMM_F16_SKINNY      # 8 x 64
    assert g.gemm_f16_select(256, 256, 65536, 152)[0] == g.GEMM_F16_SKINNY      # 8 x 128
    assert g.gemm_f16_select(1024, 1024, 4096, 152)[0] == g.GEMM_F16_SKINNY     # 2 x 32
    assert g.gemm_f16_select(128, 8192, 1024, 152)[0] == g.GEMM_F16_128x128     # 2 x 8 only
    assert g.gemm_f16_select(1024, 1024, 1024, 152)[:2] == (g.GEMM_F16_128x128, 64)
    # up to 128 rows without such a split: the 128 x 128 tile (a pair tile
    # would be half empty), grid = tile count up to one per SM
    assert g.gemm_f16_select(96, 16384, 8192, 152)[:2] == (g.GEMM_F16_128x128, 128)
    assert g.gemm_f16_select(128, 28672, 8192, 152)[:2] == (g.GEMM_F16_128x128, 152)
    assert g.gemm_f16_select(100, 100, 64, 152)[:2] == (g.GEMM_F16_128x128, 1)
    assert g.gemm_f16_select(128, 8192, 64, 148)[:2] == (g.GEMM_F16_128x128, 64)
    # more rows: the tile whose waves cost least (a 128 x 256 or pair wave
    # about 1.15 / 1.1 of a 128 x 128 wave, 1.5 / 1.5 for K <= 512)
    assert g.gemm_f16_select(192, 8192, 8192, 152)[:2] == (g.GEMM_F16_128x128, 128)   # 1 wave
    assert g.gemm_f16_select(384, 8192, 8192, 152)[0] == g.GEMM_F16_256x256_PAIR      # 2 vs 1.1
    assert g.gemm_f16_select(160, 16384, 8192, 152)[0] == g.GEMM_F16_256x256_PAIR
    assert g.gemm_f16_select(129, 28672, 8192, 152)[0] == g.GEMM_F16_256x256_PAIR
    assert g.gemm_f16_select(2048, 2048, 512, 152)[:2] == (g.GEMM_F16_128x256, 128)  # short K
    assert g.gemm_f16_select(4096, 2048, 512, 148)[:2] == (g.GEMM_F16_128x256, 148)
    with pytest.raises(g.GemmError):
        g.gemm_f16_select(1, 1, 1, 0)


def test_f16_selector_rule_over_a_shape_grid(lib):
    # The documented order of rules, checked against the skinny plan the
    # library exposes and the wave counts restated here.
    cdiv = lambda a, b: -(-a // b)
    for sm in (148, 152):
        for M in (1, 2, 64, 65, 128, 129, 200, 512, 1000, 4096):
            for N in (64, 1000, 4096, 16384):
                for K in (64, 512, 520, 4096, 32768):
                    v, grid, _ = g.gemm_f16_select(M, N, K, sm)
                    s, _, _, kb = g.gemm_debug_skinny_plan(M, N, K, sm)
                    split = s >= 4 or (s == 2 and kb >= 16)
                    if M == 1:
                        assert v == g.GEMM_F16_GEMV
                    elif M <= 64 or split:
                        assert v == g.GEMM_F16_SKINNY and grid == sm
                    elif M <= 128:
                        assert v == g.GEMM_F16_128x128
                    else:
                        short = cdiv(K, 64) <= 8
                        w = {g.GEMM_F16_128x128: cdiv(cdiv(M, 128) * cdiv(N, 128), sm),
                             g.GEMM_F16_128x256: (1.5 if short else 1.15) * cdiv(cdiv(M, 128) * cdiv(N, 256), sm),
                             g.GEMM_F16_256x256_PAIR: (1.5 if short else 1.1) * cdiv(cdiv(M, 256) * cdiv(N, 256), sm // 2)}
                        quad = K % 64 != 0 and M > 256
                        tpair = cdiv(M, 256) * cdiv(N, 256)
                        ks = (M >= 256 and K % 64 == 0 and cdiv(K, 64) >= 128 and
                              2 * tpair > sm // 4 - 2 and tpair <= sm // 4 - 2)
                        assert (v == g.GEMM_F16_256x256_KSPLIT) == ks, (M, N, K, sm, v)
                        if ks:
                            assert grid == 4 * tpair
                            continue
                        if v == g.GEMM_F16_256x256_QUAD:
                            # the pair's waves were cheapest and the rows are
                            # off the 128-byte grid
                            assert quad
                            v = g.GEMM_F16_256x256_PAIR
                        else:
                            assert not (v == g.GEMM_F16_256x256_PAIR and quad)
                        assert v in w and w[v] == min(w.values()), (M, N, K, sm, v, w)
                        assert 1 <= grid <= sm


def test_skinny_plan(lib):
    # Worked cases on 152 SMs: (shares, rows per group, groups, k-blocks a share).
    assert g.gemm_debug_skinny_plan(1, 8192, 8192, 152) == (2, 128, 64, 64)
    assert g.gemm_debug_skinny_plan(1, 16384, 8192, 152) == (1, 112, 147, 128)  # no room to split: rows spread
    assert g.gemm_debug_skinny_plan(1, 4096, 4096, 152) == (4, 128, 32, 16)
    assert g.gemm_debug_skinny_plan(1, 1000, 12008, 152) == (8, 128, 8, 12)     # 188 k-blocks, 2 parts
    assert g.gemm_debug_skinny_parts(1, 1000, 12008, 152) == 2
    assert g.gemm_debug_skinny_plan(1, 4000, 2056, 152) == (4, 128, 32, 9)      # 33 k-blocks: ragged
    assert g.gemm_debug_skinny_plan(1, 19456, 1024, 152) == (1, 128, 152, 16)   # exactly one wave
    assert g.gemm_debug_skinny_plan(1, 28672, 8192, 152) == (1, 96, 299, 128)   # two even waves
    assert g.gemm_debug_skinny_plan(1, 77, 72, 152) == (1, 128, 1, 2)           # too shallow to split
    assert g.gemm_debug_skinny_plan(1, 77, 0, 152) == (1, 128, 1, 1)            # K = 0
    # more than 128 rows of A: 128-row tiles of A count towards the SMs too
    assert g.gemm_debug_skinny_plan(160, 2048, 8192, 152) == (4, 128, 16, 32)   # 2 x 16 tiles
    assert g.gemm_debug_skinny_plan(512, 512, 32768, 152) == (8, 128, 4, 64)    # 4 x 4 tiles
    assert g.gemm_debug_skinny_plan(2048, 2048, 8192, 152) == (1, 128, 16, 128)  # 256 tiles
    assert g.gemm_debug_skinny_plan(300, 20000, 64, 152)[1] == 128             # no wave evening
    # a few tiles over a very long K: several 8-CTA clusters per tile
    assert g.gemm_debug_skinny_plan(256, 256, 65536, 152) == (8, 128, 2, 32)    # 4 tiles x 4 parts
    assert g.gemm_debug_skinny_parts(256, 256, 65536, 152) == 4
    assert g.gemm_debug_skinny_parts(128, 128, 65536, 152) == 8                 # 1 tile, at most 8
    assert g.gemm_debug_skinny_parts(512, 512, 32768, 152) == 1                 # 16 tiles: no room
    assert g.gemm_debug_skinny_parts(1, 4096, 4096, 152) == 1                   # 4 shares: no parts
    with pytest.raises(ValueError):
        g.gemm_debug_skinny_plan(1, 0, 64, 152)


def test_skinny_plan_properties(lib):
    # Against the rule itself, over a grid of shapes: the shares a power of
    # two up to 8, each at least 8 k-blocks, their CTAs within the slots, and
    # the next power of two breaking one of these; groups of 128 rows unless
    # 128-row groups need several waves (then the multiple of 8 that fills
    # that many waves) or fill more than half but not all of the slots (then
    # the multiple of 8 that fills them); groups and k-blocks covering N and K.
    for N in (1, 127, 128, 129, 1000, 4096, 8192, 16384, 19456, 19457, 28672):
        for K in (0, 8, 64, 512, 520, 4096, 12008, 65536):
            for ctas in (1, 19, 152, 304):
                s, rows, groups, kb = g.gemm_debug_skinny_plan(1, N, K, ctas)
                parts = g.gemm_debug_skinny_parts(1, N, K, ctas)
                tiles, nkb = -(-N // 128), -(-K // 64)
                assert s in (1, 2, 4, 8)
                if s > 1:
                    assert tiles * s <= ctas and nkb // s >= 8
                assert 2 * s > 8 or tiles * 2 * s > ctas or nkb // (2 * s) < 8
                if s > 1 or tiles == ctas or 2 * tiles <= ctas:
                    assert rows == 128
                elif tiles < ctas:
                    # fewer groups than slots, more than half: rows spread over the slots
                    assert rows % 8 == 0 and rows <= 128 and rows * ctas >= N
                    assert rows - 8 < -(-N // ctas)
                else:
                    waves = -(-tiles // ctas)
                    assert rows % 8 == 0 and rows <= 128 and rows * waves * ctas >= N
                    assert rows - 8 < -(-N // (waves * ctas))
                assert groups == -(-N // rows) and (groups - 1) * rows < N
                # parts: only with 8-CTA clusters, all resident, shares of 8+
                # k-blocks, at most 8, and one more would break one of these
                assert 1 <= parts <= 8 and (parts == 1 or s == 8)
                if parts > 1:
                    assert tiles * 8 * parts <= ctas and nkb // (8 * parts) >= 8
                if s == 8:
                    assert parts == 8 or tiles * 8 * (parts + 1) > ctas or nkb // (8 * (parts + 1)) < 8
                assert kb == max(1, -(-nkb // (s * parts))) and kb * s * parts >= nkb


def test_f16_selector_raster(lib):
    plain = 1 << 30
    # operands that fit in L2 keep the plain column order of tiles
    assert g.gemm_f16_select(5376, 5376, 2048, 152)[2] == plain
    assert g.gemm_f16_select(5000, 5376, 2040, 152)[2] == plain
    # beyond it, bands of tile rows (8 pair tiles = 2048 rows)
    assert g.gemm_f16_select(8192, 8192, 8192, 152)[2] == 8
    assert g.gemm_f16_select(16384, 16384, 2048, 152)[2] == 8
    assert g.gemm_f16_select(1, 16384, 8192, 152)[2] == plain  # GEMV has no tiles
    assert g.gemm_f16_select(8, 16384, 8192, 152)[2] == plain  # nor has the skinny kernel a band order
    with pytest.raises(g.GemmError):
        g.gemm_f16_nt_ex(16, 16, 16, 0x1000, 0x1000, 0x1000, raster=-1)


def _tile_mn(tile, m_tiles, n_tiles, raster):
    # the kernels' band order, restated: bands of `raster` tile rows, column by column
    gsz = min(raster, m_tiles)
    band, r = divmod(tile, gsz * n_tiles)
    first = band * gsz
    h = min(gsz, m_tiles - first)
    return first + r % h, r // h


@pytest.mark.parametrize("m_tiles,n_tiles,raster", [(21, 21, 8), (32, 32, 8), (5, 7, 3), (7, 3, 1 << 30),
                                                    (9, 4, 4), (1, 5, 8)])
def test_band_order_visits_every_tile_once(m_tiles, n_tiles, raster):
    seen = {_tile_mn(t, m_tiles, n_tiles, raster) for t in range(m_tiles * n_tiles)}
    assert seen == {(m, n) for m in range(m_tiles) for n in range(n_tiles)}
    if raster >= m_tiles:
        assert [_tile_mn(t, m_tiles, n_tiles, raster) for t in range(m_tiles * n_tiles)] == \
            [(t % m_tiles, t // m_tiles) for t in range(m_tiles * n_tiles)]


def test_sgemm_selector(lib):
    sel = g.gemm_sgemm_select
    # many tiles: the 128 x 128 tile, unsplit
    assert sel(4096, 4096, 4096, 152) == (g.GEMM_SGEMM_128x128, 1)
    assert sel(3000, 3000, 3000, 152) == (g.GEMM_SGEMM_128x128, 1)
    # shapes where the GB300 sweep of every (tile, splits) pair had a clear winner
    assert sel(2048, 2048, 2048, 152) == (g.GEMM_SGEMM_128x128, 4)   # 256 tiles: 4 splits even the waves
    assert sel(256, 256, 4096, 152) == (g.GEMM_SGEMM_64x64, 8)
    assert sel(1536, 1536, 1536, 152)[1] == 1                       # 144 tiles: one wave already
    # the 128 x 64 tile where its splits fill the SMs better (measured 2-12 % faster)
    assert sel(512, 512, 8192, 152) == (g.GEMM_SGEMM_128x64, 8)
    assert sel(768, 768, 768, 152) == (g.GEMM_SGEMM_128x64, 4)
    assert sel(1024, 1024, 1024, 152) == (g.GEMM_SGEMM_128x64, 8)
    assert sel(8192, 64, 1024, 152) == (g.GEMM_SGEMM_128x64, 7)
    # no K: nothing to split
    assert sel(4096, 4096, 0, 152)[1] == 1
    assert sel(16, 16, 16, 152)[1] == 1


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (100, 100, 64), (1024, 1024, 256), (64, 4096, 4096),
                                   (8192, 64, 1024), (128, 128, 65536), (777, 333, 5000)])
@pytest.mark.parametrize("sms", [1, 148, 152])
def test_sgemm_selector_plans_are_valid(lib, M, N, K, sms):
    variant, splits = g.gemm_sgemm_select(M, N, K, sms)
    assert variant in (g.GEMM_SGEMM_128x128, g.GEMM_SGEMM_64x64, g.GEMM_SGEMM_128x64)
    assert 1 <= splits <= 8
    # each share of K is at least 64 deep, and splits only come with few tiles
    assert splits == 1 or splits <= -(-K // 64)
    bm = 64 if variant == g.GEMM_SGEMM_64x64 else 128
    bn = 128 if variant == g.GEMM_SGEMM_128x128 else 64
    assert splits == 1 or -(-M // bm) * -(-N // bn) <= 2 * sms


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "dense_gemm_fp16_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if not path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            continue
        text = open(path, encoding="utf-8").read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), path
        assert "gemm_oracle" not in text and "liboracle" not in text, path
