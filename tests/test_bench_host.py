"""CPU checks of bench.py's host logic: the clock-sample summary, the
roofline traffic lookup, and the multi-rank (replica) plumbing over gloo with
world_size 2 — barrier and the max over ranks the timing takes."""
import os
import socket
import subprocess
import sys
import textwrap

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_clock_summary_filters_gpu_and_collects_reasons():
    rows = [
        "00000009:01:00.0, 1900, 2070, 900.1, 0x4, Not Active, Not Active, Not Active, Active",
        "00000009:01:00.0, 1800, 2070, 950.0, 0x4, Not Active, Not Active, Not Active, Active",
        "00000009:01:00.0, 345, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "00000019:01:00.0, 2070, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    s = bench.summarize_clock_samples(rows, "00000009:01:00.0")
    assert s["samples"] == 3
    assert s["sm_mhz"] == 1850.0          # idle sample (345 MHz) excluded from the load median
    assert s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]   # the other GPU's hw_slowdown is not ours


def test_clock_summary_single_gpu_without_bus_match():
    rows = ["00000001:02:00.0, 1500, 2070, 1.0, 0x0, Not Active, Active, Not Active, Not Active"]
    s = bench.summarize_clock_samples(rows, None)
    assert s["samples"] == 1 and s["reasons"] == ["hw_thermal_slowdown"]
    assert bench.summarize_clock_samples([], None)["reasons"] == ["no samples"]


def test_sm_clock_from_two_device_samples():
    # (SM id, cycles, ns) triples: SM 3 ran 2e6 cycles in 1e6 ns = 2000 MHz,
    # SM 5 1.5e6 in 1e6 = 1500 MHz (its second record in a sample is ignored),
    # SM 9 appears only once and does not count.
    before = [3, 1000, 10_000, 5, 0, 10_000, 5, 777, 10_500, 9, 0, 0]
    after = [5, 1_500_000, 1_010_000, 3, 2_001_000, 1_010_000]
    mhz, sms = bench.sm_clock_mhz(before, after)
    assert sms == 2 and abs(mhz - 1750.0) < 1e-9
    assert bench.sm_clock_mhz([1, 5, 5], [2, 9, 9]) == (None, 0)
    assert bench.sm_clock_mhz([1, 5, 5], [1, 9, 5]) == (None, 0)     # no time elapsed


def test_traffic_is_null_unless_the_kernel_hash_matches(tmp_path, monkeypatch):
    f = tmp_path / "t.txt"
    f.write_text("kernel_source_sha256_16: deadbeef\ndram_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", "t.txt")
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "deadbeef")
    assert bench.profiled_traffic() == 123.0
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "other")
    assert bench.profiled_traffic() is None


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_replica_timing_max_over_two_gloo_ranks():
    script = textwrap.dedent(f"""
        import os, sys
        sys.path.insert(0, {ROOT!r})
        import bench
        rank, local, world = bench.dist_setup(2)
        assert world == 2
        bench.barrier(world)
        t = bench.max_over_ranks(1.5 + rank, world)
        print(f"rank{{rank}} {{t}}")
        import torch.distributed as dist
        dist.destroy_process_group()
    """)
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", script], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    assert "rank0 2.5" in outs[0][0] and "rank1 2.5" in outs[1][0]


def test_reference_arm_nonzero_rank_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
