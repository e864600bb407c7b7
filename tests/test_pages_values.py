"""Pins from numbers the pages print: the 2·M·N·K throughput arithmetic, the
ceil-div launch grid and tile counts, read from tests/golden/pages_values.txt
(each value there carries its page and section)."""
import math
import os

import numpy as np

from dense_gemm_fp16_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_values.txt")


def _values():
    out = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = (s.strip() for s in line.split("="))
                out[k] = float(v)
    return out


def test_flop_count_reproduces_printed_throughputs():
    v = _values()
    w = wl.WORKLOADS[wl.HEADLINE]
    assert (w.M, w.N, w.K) == (v["f16_nt_M"], v["f16_nt_N"], v["f16_nt_K"])
    tflops = lambda ms: w.flop / (ms * 1e-3) / 1e12
    assert round(tflops(1.0), 2) == v["tflops_at_1ms"]
    assert round(tflops(0.5), 2) == v["tflops_at_0p5ms"]
    assert round(tflops(v["naive_ms"]), 3) == v["naive_tflops"]


def test_ceil_div_grid_and_tile_counts():
    v = _values()
    w = wl.WORKLOADS[wl.HEADLINE]
    assert math.ceil(w.N / v["naive_block_x"]) == v["naive_grid_x"]
    assert math.ceil(w.M / v["naive_block_y"]) == v["naive_grid_y"]
    t = math.ceil(w.M / 128)
    assert t == v["tiles_128_per_dim"]
    # 42*42 CTAs x 8 warps x (K/32) steps
    assert t * t * 8 * (w.K // 32) == v["per_warp_k32_steps"]


def test_stage_bytes():
    v = _values()
    assert (128 * 8 + 8 * 128) * 4 == v["sgemm_stage_bytes"]


def test_workloads_are_seeded_and_shaped():
    for w in wl.WORKLOADS.values():
        if (w.M + w.N) * w.K > 6_000_000:
            continue
        A1, B1, C1 = wl.make_inputs(w)
        A2, B2, C2 = wl.make_inputs(w)
        assert A1.shape == (w.M, w.K)
        assert B1.shape == ((w.N, w.K) if w.form == "f16_nt" else (w.K, w.N))
        assert (A1 == A2).all() and (B1 == B2).all()
        assert A1.abs().max() <= 1.0


def test_sample_positions_cover_edges_without_duplicates():
    rows, cols = wl.sample_positions(50, 40, 300, seed=3, tail_rows=[45])
    pairs = set(zip(rows.tolist(), cols.tolist()))
    assert len(pairs) == len(rows)
    for c in range(40):
        assert (49, c) in pairs and (45, c) in pairs
    for r in range(50):
        assert (r, 39) in pairs
    assert (0, 0) in pairs
    assert np.all((rows >= 0) & (rows < 50) & (cols >= 0) & (cols < 40))
