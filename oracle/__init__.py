"""The parity oracle: plain float64 CPU definitions of the two products.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` are the only callers allowed.  The
product path (``dense_gemm_fp16_gb300`` and its CUDA library) never imports
this package, and this package never imports the product path.

The arithmetic lives in ``gemm_oracle.c`` (nested loops, one float64
accumulator per output, ascending k, OpenMP over output rows).  This module
only marshals numpy arrays into it.  See that file's header for the pages
each function follows:

* ``gemm_f16_nt``: "从零开始的 AI Infra: 算子基础与GPU架构", section
  "0. Naive Implementation" (C = A·Bᵀ, A [M,K], B [N,K] half).
* ``sgemm``: "异步拷贝与 Hopper/Blackwell 新特性", section
  "cp.async 与多级流水 sm_80+" (C = alpha·A·B + beta·C, row-major fp32).
* ``gemm_f16_nt_epilogue``: "第 6 章 · Shared Memory & Tile", section
  "6.5.4 Epilogue 融合" (activation(GEMM + bias)), with alpha, beta and a
  residual.
* ``gemm_mxfp8_nt``: "异步拷贝与 Hopper/Blackwell 新特性", section
  "Blackwell 概览 sm_100" (MXFP8: 32 elements share one 8-bit exponent
  scale), E4M3 elements and UE8M0 scales.
* ``gemm_nvfp4_nt``: the same section (NVFP4: 16 elements share one FP8
  scale, plus a tensor-level FP32 scale), E2M1 elements packed two per
  byte, UE4M3 block scales, alpha the tensor-level scale.

Every function returns the unrounded float64 result C and the tolerance
scale S = |alpha|·Σ_k |A·B| per element.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-std=c99", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into liboracle.so next to it (gcc + OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.oracle_half_to_f64.restype = dbl
            lib.oracle_half_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f64_to_half_rn.restype = ctypes.c_uint16
            lib.oracle_f64_to_half_rn.argtypes = [dbl]
            lib.oracle_half_to_f64_array.argtypes = [i64, vp, vp]
            lib.oracle_f64_to_half_rn_array.argtypes = [i64, vp, vp]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_gemm_f16_nt.restype = ctypes.c_int
            lib.oracle_gemm_f16_nt.argtypes = [i64, i64, i64, vp, vp, vp, vp]
            lib.oracle_gemm_f16_nt_sampled.restype = ctypes.c_int
            lib.oracle_gemm_f16_nt_sampled.argtypes = [i64, i64, i64, vp, vp, i64, vp, vp, vp, vp]
            lib.oracle_sgemm.restype = ctypes.c_int
            lib.oracle_sgemm.argtypes = [i64, i64, i64, dbl, vp, vp, dbl, vp, vp, vp]
            lib.oracle_activation.restype = dbl
            lib.oracle_activation.argtypes = [dbl, ctypes.c_int]
            lib.oracle_gemm_f16_nt_epilogue.restype = ctypes.c_int
            lib.oracle_gemm_f16_nt_epilogue.argtypes = [i64, i64, i64, vp, vp, dbl, vp, dbl, vp,
                                                        ctypes.c_int, vp, vp]
            lib.oracle_gemm_f16_nt_epilogue_sampled.restype = ctypes.c_int
            lib.oracle_gemm_f16_nt_epilogue_sampled.argtypes = [
                i64, i64, i64, vp, vp, dbl, vp, dbl, vp, ctypes.c_int, i64, vp, vp, vp, vp]
            u8 = ctypes.c_uint8
            lib.oracle_e4m3_to_f64.restype = dbl
            lib.oracle_e4m3_to_f64.argtypes = [u8]
            lib.oracle_ue8m0_to_f64.restype = dbl
            lib.oracle_ue8m0_to_f64.argtypes = [u8]
            lib.oracle_gemm_mxfp8_nt.restype = ctypes.c_int
            lib.oracle_gemm_mxfp8_nt.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, vp]
            lib.oracle_gemm_mxfp8_nt_sampled.restype = ctypes.c_int
            lib.oracle_gemm_mxfp8_nt_sampled.argtypes = [i64, i64, i64, vp, vp, vp, vp, i64, vp, vp,
                                                         vp, vp]
            lib.oracle_e2m1_to_f64.restype = dbl
            lib.oracle_e2m1_to_f64.argtypes = [u8]
            lib.oracle_gemm_nvfp4_nt.restype = ctypes.c_int
            lib.oracle_gemm_nvfp4_nt.argtypes = [i64, i64, i64, vp, vp, vp, vp, dbl, vp, vp]
            lib.oracle_gemm_nvfp4_nt_sampled.restype = ctypes.c_int
            lib.oracle_gemm_nvfp4_nt_sampled.argtypes = [i64, i64, i64, vp, vp, vp, vp, dbl, i64, vp,
                                                         vp, vp, vp]
            lib.oracle_sgemm_sampled.restype = ctypes.c_int
            lib.oracle_sgemm_sampled.argtypes = [i64, i64, i64, dbl, vp, vp, dbl, vp, i64, vp, vp,
                                                 vp, vp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data


def _as_half_bits(x) -> np.ndarray:
    """Accept float16 or uint16 arrays (or CPU torch tensors) as binary16 bits."""
    if hasattr(x, "numpy"):
        x = x.detach().cpu().contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float16:
        return x.view(np.uint16)
    if x.dtype == np.uint16:
        return x
    raise TypeError(f"expected float16/uint16 half data, got {x.dtype}")


def _as_f32(x) -> np.ndarray:
    if hasattr(x, "numpy"):
        x = x.detach().cpu().contiguous().numpy()
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError(f"expected float32 data, got {x.dtype}")
    return x


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def half_to_f64(bits) -> np.ndarray:
    """Decode binary16 bit patterns to float64 (exact)."""
    b = _as_half_bits(np.asarray(bits))
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_half_to_f64_array(b.size, _ptr(b), _ptr(out))
    return out


def f64_to_half_rn(x) -> np.ndarray:
    """Round float64 values to binary16 (nearest, ties to even); returns bits."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f64_to_half_rn_array(x.size, _ptr(x), _ptr(out))
    return out


def gemm_f16_nt(A, B):
    """C = A·Bᵀ in float64 for half A [M,K], B [N,K].  Returns (C, S)."""
    a, b = _as_half_bits(A), _as_half_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}^T")
    M, K = a.shape
    N = b.shape[0]
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_f16_nt(M, N, K, _ptr(a), _ptr(b), _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f16_nt failed ({rc})")
    return C, S


def gemm_f16_nt_sampled(A, B, rows, cols):
    """Entries (rows[t], cols[t]) of A·Bᵀ in float64.  Returns (C[t], S[t])."""
    a, b = _as_half_bits(A), _as_half_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}^T")
    M, K = a.shape
    N = b.shape[0]
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    C = np.zeros(r.shape, dtype=np.float64)
    S = np.zeros(r.shape, dtype=np.float64)
    rc = _load().oracle_gemm_f16_nt_sampled(M, N, K, _ptr(a), _ptr(b), r.size, _ptr(r), _ptr(c),
                                            _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f16_nt_sampled failed ({rc})")
    return C, S


def sgemm(A, B, alpha=1.0, beta=0.0, C0=None):
    """alpha·A·B + beta·C0 in float64 for fp32 row-major A [M,K], B [K,N], C0 [M,N].

    With beta == 0, C0 is not read (BLAS convention).  Returns (C, S)."""
    a, b = _as_f32(A), _as_f32(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}")
    M, K = a.shape
    N = b.shape[1]
    c0 = None
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        c0 = _as_f32(C0)
        if c0.shape != (M, N):
            raise ValueError(f"C0 shape {c0.shape} != {(M, N)}")
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_sgemm(M, N, K, float(alpha), _ptr(a), _ptr(b), float(beta), _ptr(c0),
                              _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm failed ({rc})")
    return C, S


def sgemm_sampled(A, B, rows, cols, alpha=1.0, beta=0.0, C0=None):
    """Entries (rows[t], cols[t]) of alpha·A·B + beta·C0.  Returns (C[t], S[t])."""
    a, b = _as_f32(A), _as_f32(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[0]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}")
    M, K = a.shape
    N = b.shape[1]
    c0 = None
    if beta != 0.0:
        if C0 is None:
            raise ValueError("beta != 0 needs C0")
        c0 = _as_f32(C0)
        if c0.shape != (M, N):
            raise ValueError(f"C0 shape {c0.shape} != {(M, N)}")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    C = np.zeros(r.shape, dtype=np.float64)
    S = np.zeros(r.shape, dtype=np.float64)
    rc = _load().oracle_sgemm_sampled(M, N, K, float(alpha), _ptr(a), _ptr(b), float(beta),
                                      _ptr(c0), r.size, _ptr(r), _ptr(c), _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm_sampled failed ({rc})")
    return C, S


ACTIVATIONS = {"none": 0, "relu": 1, "silu": 2, "gelu_tanh": 3}


def activation(v, act: str) -> float:
    """The activation the fused epilogue applies, in float64."""
    return float(_load().oracle_activation(float(v), ACTIVATIONS[act]))


def gemm_f16_nt_epilogue(A, B, alpha=1.0, bias=None, beta=0.0, R=None, act="none"):
    """act(alpha·A·Bᵀ + bias[n] + beta·R[m,n]) in float64 for half A [M,K],
    B [N,K], bias [N], R [M,N].  Returns (Y, S), S the pre-activation scale."""
    a, b = _as_half_bits(A), _as_half_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}^T")
    M, K = a.shape
    N = b.shape[0]
    bb = None if bias is None else _as_half_bits(bias)
    rr = None if R is None else _as_half_bits(R)
    if bb is not None and bb.shape != (N,):
        raise ValueError("bias must be [N]")
    if rr is not None and rr.shape != (M, N):
        raise ValueError("R must be [M, N]")
    Y = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_f16_nt_epilogue(M, N, K, _ptr(a), _ptr(b), float(alpha), _ptr(bb),
                                             float(beta), _ptr(rr), ACTIVATIONS[act], _ptr(Y),
                                             _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f16_nt_epilogue failed ({rc})")
    return Y, S


def gemm_f16_nt_epilogue_sampled(A, B, rows, cols, alpha=1.0, bias=None, beta=0.0, R=None,
                                 act="none"):
    """Entries (rows[t], cols[t]) of gemm_f16_nt_epilogue.  Returns (Y[t], S[t])."""
    a, b = _as_half_bits(A), _as_half_bits(B)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}^T")
    M, K = a.shape
    N = b.shape[0]
    bb = None if bias is None else _as_half_bits(bias)
    rr = None if R is None else _as_half_bits(R)
    if bb is not None and bb.shape != (N,):
        raise ValueError("bias must be [N]")
    if rr is not None and rr.shape != (M, N):
        raise ValueError("R must be [M, N]")
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    Y = np.zeros(r.shape, dtype=np.float64)
    S = np.zeros(r.shape, dtype=np.float64)
    rc = _load().oracle_gemm_f16_nt_epilogue_sampled(M, N, K, _ptr(a), _ptr(b), float(alpha),
                                                     _ptr(bb), float(beta), _ptr(rr),
                                                     ACTIVATIONS[act], r.size, _ptr(r), _ptr(c),
                                                     _ptr(Y), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_f16_nt_epilogue_sampled failed ({rc})")
    return Y, S


def _as_u8(x) -> np.ndarray:
    if hasattr(x, "numpy"):
        x = x.contiguous().cpu()
        import torch

        if x.dtype != torch.uint8:
            x = x.view(torch.uint8)
        x = x.numpy()
    return np.ascontiguousarray(x, dtype=np.uint8)


def e4m3_to_f64(codes) -> np.ndarray:
    """FP8 E4M3 codes (uint8) decoded to float64 (NaN for S.1111.111)."""
    c = _as_u8(codes)
    f = _load().oracle_e4m3_to_f64
    return np.array([f(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def ue8m0_to_f64(codes) -> np.ndarray:
    """UE8M0 scale codes decoded to float64: 2^(e-127), NaN for 0xFF."""
    c = _as_u8(codes)
    f = _load().oracle_ue8m0_to_f64
    return np.array([f(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def _mx_args(A, SA, B, SB):
    a, sa, b, sb = _as_u8(A), _as_u8(SA), _as_u8(B), _as_u8(SB)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}^T")
    M, K = a.shape
    N = b.shape[0]
    if K % 32:
        raise ValueError("K must be a multiple of the 32-element scale block")
    if sa.shape != (M, K // 32) or sb.shape != (N, K // 32):
        raise ValueError(f"scales must be [M, K/32] and [N, K/32], got {sa.shape} and {sb.shape}")
    return a, sa, b, sb, M, N, K


def gemm_mxfp8_nt(A, SA, B, SB):
    """sum_k e4m3(A[m,k]) 2^(SA[m,k/32]-127) * e4m3(B[n,k]) 2^(SB[n,k/32]-127)
    in float64 for uint8 codes A [M,K], B [N,K] and scales SA [M,K/32],
    SB [N,K/32].  Returns (C, S)."""
    a, sa, b, sb, M, N, K = _mx_args(A, SA, B, SB)
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_mxfp8_nt(M, N, K, _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_mxfp8_nt failed ({rc})")
    return C, S


def gemm_mxfp8_nt_sampled(A, SA, B, SB, rows, cols):
    """Entries (rows[t], cols[t]) of gemm_mxfp8_nt.  Returns (C[t], S[t])."""
    a, sa, b, sb, M, N, K = _mx_args(A, SA, B, SB)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    C = np.zeros(r.shape, dtype=np.float64)
    S = np.zeros(r.shape, dtype=np.float64)
    rc = _load().oracle_gemm_mxfp8_nt_sampled(M, N, K, _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), r.size,
                                              _ptr(r), _ptr(c), _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_mxfp8_nt_sampled failed ({rc})")
    return C, S


def e2m1_to_f64(nibbles) -> np.ndarray:
    """FP4 E2M1 codes (one per uint8, low 4 bits) decoded to float64."""
    c = _as_u8(nibbles)
    f = _load().oracle_e2m1_to_f64
    return np.array([f(int(v) & 0xF) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def _nv_args(A, SA, B, SB):
    a, sa, b, sb = _as_u8(A), _as_u8(SA), _as_u8(B), _as_u8(SB)
    if a.ndim != 2 or b.ndim != 2 or a.shape[1] != b.shape[1]:
        raise ValueError(f"shape mismatch {a.shape} x {b.shape}^T")
    M, K = a.shape[0], 2 * a.shape[1]
    N = b.shape[0]
    if K % 16:
        raise ValueError("K must be a multiple of the 16-element scale block")
    if sa.shape != (M, K // 16) or sb.shape != (N, K // 16):
        raise ValueError(f"scales must be [M, K/16] and [N, K/16], got {sa.shape} and {sb.shape}")
    return a, sa, b, sb, M, N, K


def gemm_nvfp4_nt(A, SA, B, SB, alpha=1.0):
    """alpha * sum_k e2m1(A[m,k]) e4m3(SA[m,k/16]) e2m1(B[n,k]) e4m3(SB[n,k/16])
    in float64; A [M,K/2], B [N,K/2] packed (element 2i in the low nibble of
    byte i), SA [M,K/16], SB [N,K/16].  Returns (C, S)."""
    a, sa, b, sb, M, N, K = _nv_args(A, SA, B, SB)
    C = np.zeros((M, N), dtype=np.float64)
    S = np.zeros((M, N), dtype=np.float64)
    rc = _load().oracle_gemm_nvfp4_nt(M, N, K, _ptr(a), _ptr(sa), _ptr(b), _ptr(sb), float(alpha),
                                      _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_nvfp4_nt failed ({rc})")
    return C, S


def gemm_nvfp4_nt_sampled(A, SA, B, SB, rows, cols, alpha=1.0):
    """Entries (rows[t], cols[t]) of gemm_nvfp4_nt.  Returns (C[t], S[t])."""
    a, sa, b, sb, M, N, K = _nv_args(A, SA, B, SB)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    c = np.ascontiguousarray(cols, dtype=np.int64)
    if r.shape != c.shape:
        raise ValueError("rows and cols differ in length")
    C = np.zeros(r.shape, dtype=np.float64)
    S = np.zeros(r.shape, dtype=np.float64)
    rc = _load().oracle_gemm_nvfp4_nt_sampled(M, N, K, _ptr(a), _ptr(sa), _ptr(b), _ptr(sb),
                                              float(alpha), r.size, _ptr(r), _ptr(c), _ptr(C), _ptr(S))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_nvfp4_nt_sampled failed ({rc})")
    return C, S
