"""The C ABI from C: a C99 program (tests/c/abi_check.c) compiled against
include/gemm.h and include/gemm_testing.h with warnings as errors and linked
to libgemm.so.

* CPU: the headers compile as C, every host-only call links and runs, and its
  answers match the same calls made through the Python binding.
* GPU: the same program runs gemm_f16_nt and sgemm on cudaMalloc'd buffers;
  its outputs are checked against the oracle within the path's tolerances.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import dense_gemm_fp16_gb300 as g
from dense_gemm_fp16_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_check.c")
INCLUDE = os.path.join(ROOT, "include")
C_FLAGS = ["-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O1"]


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    return None


def _compile(out, gpu=False):
    lib = gbuild.build()
    libdir = os.path.dirname(lib)
    cmd = ["gcc", *C_FLAGS, "-I", INCLUDE, SRC, "-o", str(out), "-L", libdir, "-l:libgemm.so",
           f"-Wl,-rpath,{libdir}"]
    if gpu:
        cuda = _cuda_home()
        libs = [d for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib")
                if os.path.exists(os.path.join(cuda, d, "libcudart.so"))]
        assert libs, "libcudart.so not found under the CUDA toolkit"
        cudart = os.path.join(cuda, libs[0])
        cmd += ["-DABI_CHECK_GPU", "-isystem", os.path.join(cuda, "include"), "-L", cudart, "-lcudart",
                f"-Wl,-rpath,{cudart}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, f"C build failed:\n{' '.join(cmd)}\n{res.stdout}{res.stderr}"


def test_each_header_compiles_alone_as_c99(tmp_path):
    for header in ("gemm.h", "gemm_testing.h"):
        tu = tmp_path / f"only_{header}.c"
        tu.write_text(f'#include "{header}"\nint main(void) {{ return 0; }}\n')
        res = subprocess.run(["gcc", *C_FLAGS, "-fsyntax-only", "-I", INCLUDE, str(tu)],
                             capture_output=True, text=True)
        assert res.returncode == 0, f"{header} is not valid C99:\n{res.stderr}"


def test_c_program_host_calls_match_the_binding(tmp_path):
    exe = tmp_path / "abi_check"
    _compile(exe)
    res = subprocess.run([str(exe), "host"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, f"abi_check host failed:\n{res.stdout}\n{res.stderr}"
    kv = dict(line.split("=", 1) for line in res.stdout.splitlines() if "=" in line)
    ints = lambda s: tuple(int(x) for x in s.split(","))
    assert ints(kv["f16_select_5376x5376x2048"]) == g.gemm_f16_select(5376, 5376, 2048, 152)
    assert ints(kv["f16_select_1x16384x8192"]) == g.gemm_f16_select(1, 16384, 8192, 152)
    assert ints(kv["sgemm_select_4096"]) == g.gemm_sgemm_select(4096, 4096, 4096, 152)
    assert ints(kv["sgemm_select_256"]) == g.gemm_sgemm_select(256, 256, 256, 152)
    assert ints(kv["skinny_plan_16x16384x8192"]) == g.gemm_debug_skinny_plan(16, 16384, 8192, 152)
    assert int(kv["mxfp8_scale_bytes_5376x2048"]) == g.gemm_mxfp8_scale_bytes(5376, 2048)
    assert int(kv["nvfp4_scale_bytes_5376x2048"]) == g.gemm_nvfp4_scale_bytes(5376, 2048)
    status, msg = kv["f16_negative_m"].split(":", 1)
    assert int(status) == g.GEMM_ERR_INVALID_ARG and "negative" in msg
    status, msg = kv["sgemm_negative_n"].split(":", 1)
    assert int(status) == g.GEMM_ERR_INVALID_ARG and msg


@pytest.mark.gpu
def test_c_program_runs_both_products_on_the_gpu(tmp_path):
    import oracle
    from dense_gemm_fp16_gb300 import workloads as wl
    from parity import check_f16, check_sgemm

    if _cuda_home() is None or shutil.which("gcc") is None:
        pytest.fail("the CUDA toolkit headers and gcc are needed to build the C caller")
    exe = tmp_path / "abi_check_gpu"
    _compile(exe, gpu=True)
    # ragged in every dimension, several tiles of each kernel
    M, N, K = 300, 520, 264
    Ms, Ns, Ks, alpha, beta = 257, 131, 200, 1.5, -0.5
    A = wl.draw_f16((M, K), seed=101, dist="normal")
    B = wl.draw_f16((N, K), seed=102, dist="normal")
    As = wl.draw_f32((Ms, Ks), seed=103)
    Bs = wl.draw_f32((Ks, Ns), seed=104)
    C0 = wl.draw_f32((Ms, Ns), seed=105)
    (tmp_path / "params.txt").write_text(f"{M} {N} {K} {Ms} {Ns} {Ks} {alpha!r} {beta!r}\n")
    for name, t in (("A", A), ("B", B), ("As", As), ("Bs", Bs), ("C0", C0)):
        (tmp_path / f"{name}.bin").write_bytes(t.numpy().tobytes())
    res = subprocess.run([str(exe), "gpu", str(tmp_path)], capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, f"abi_check gpu failed:\n{res.stdout}\n{res.stderr}"
    C = np.frombuffer((tmp_path / "C.bin").read_bytes(), dtype=np.float16).reshape(M, N)
    Cs = np.frombuffer((tmp_path / "Cs.bin").read_bytes(), dtype=np.float32).reshape(Ms, Ns)
    Cref, S = oracle.gemm_f16_nt(A, B)
    check_f16(C, Cref, S, what="gemm_f16_nt from C")
    Csref, Ss = oracle.sgemm(As, Bs, alpha, beta, C0)
    check_sgemm(Cs, Csref, Ss, what="sgemm from C")
