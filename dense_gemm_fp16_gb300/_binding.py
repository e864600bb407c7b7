"""ctypes binding of libgemm.so: the C ABI of include/gemm.h under the same
names, plus tensor conveniences.  Argument marshalling only: every step of
both products runs in the library's CUDA kernels.  There is no fallback; if
the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgemm.so")

GEMM_OK = 0
GEMM_ERR_INVALID_ARG = -1
GEMM_ERR_MISALIGNED = -2
GEMM_ERR_UNSUPPORTED = -3
GEMM_ERR_CUDA = -4
GEMM_ERR_DEVICE_TIMEOUT = -5

GEMM_F16_AUTO, GEMM_F16_128x256, GEMM_F16_128x128, GEMM_F16_256x256_PAIR, GEMM_F16_GEMV = 0, 1, 2, 3, 4
GEMM_F16_SKINNY, GEMM_F16_256x256_QUAD, GEMM_F16_256x256_KSPLIT, GEMM_F16_NUM_VARIANTS = 5, 6, 7, 8
GEMM_SGEMM_AUTO, GEMM_SGEMM_128x128, GEMM_SGEMM_64x64, GEMM_SGEMM_128x64 = 0, 1, 2, 3
GEMM_F16_FLAG_STREAM_K = 1
GEMM_MXFP8_AUTO, GEMM_MXFP8_128x128, GEMM_MXFP8_256x128_PAIR, GEMM_MXFP8_128x256 = 0, 1, 2, 3
GEMM_MXFP8_256x256_PAIR, GEMM_MXFP8_NUM_VARIANTS = 4, 5
GEMM_ACT_NONE, GEMM_ACT_RELU, GEMM_ACT_SILU, GEMM_ACT_GELU_TANH = 0, 1, 2, 3
ACTIVATIONS = {"none": GEMM_ACT_NONE, "relu": GEMM_ACT_RELU, "silu": GEMM_ACT_SILU,
               "gelu_tanh": GEMM_ACT_GELU_TANH}

STATUS_NAMES = {
    GEMM_OK: "GEMM_OK",
    GEMM_ERR_INVALID_ARG: "GEMM_ERR_INVALID_ARG",
    GEMM_ERR_MISALIGNED: "GEMM_ERR_MISALIGNED",
    GEMM_ERR_UNSUPPORTED: "GEMM_ERR_UNSUPPORTED",
    GEMM_ERR_CUDA: "GEMM_ERR_CUDA",
    GEMM_ERR_DEVICE_TIMEOUT: "GEMM_ERR_DEVICE_TIMEOUT",
}


class GemmError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class _F16Config(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("grid", ctypes.c_int), ("flags", ctypes.c_int),
                ("raster", ctypes.c_int)]


class _F16Epilogue(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("residual", ctypes.c_void_p), ("activation", ctypes.c_int)]


class _MxConfig(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("grid", ctypes.c_int)]


class _SgemmConfig(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int), ("splits", ctypes.c_int)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgemm.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m dense_gemm_fp16_gb300.build` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        i, vp, f = ctypes.c_int, ctypes.c_void_p, ctypes.c_float
        lib.gemm_f16_nt.argtypes = [i, i, i, vp, vp, vp, vp]
        lib.gemm_f16_nt.restype = i
        lib.gemm_f16_nt_ex.argtypes = [i, i, i, vp, vp, vp, vp, ctypes.POINTER(_F16Config)]
        lib.gemm_f16_nt_ex.restype = i
        lib.gemm_f16_nt_fused.argtypes = [i, i, i, vp, vp, vp, ctypes.POINTER(_F16Epilogue), vp,
                                          ctypes.POINTER(_F16Config)]
        lib.gemm_f16_nt_fused.restype = i
        lib.gemm_mxfp8_nt.argtypes = [i, i, i, vp, vp, vp, vp, vp, vp]
        lib.gemm_mxfp8_nt.restype = i
        lib.gemm_mxfp8_nt_ex.argtypes = [i, i, i, vp, vp, vp, vp, vp, vp, ctypes.POINTER(_MxConfig)]
        lib.gemm_mxfp8_nt_ex.restype = i
        lib.gemm_nvfp4_nt_ex.argtypes = [i, i, i, vp, vp, vp, vp, f, vp, vp, ctypes.POINTER(_MxConfig)]
        lib.gemm_nvfp4_nt_ex.restype = i
        lib.gemm_nvfp4_nt.argtypes = [i, i, i, vp, vp, vp, vp, f, vp, vp]
        lib.gemm_nvfp4_nt.restype = i
        lib.gemm_nvfp4_scale_bytes.argtypes = [i, i]
        lib.gemm_nvfp4_scale_bytes.restype = ctypes.c_size_t
        lib.gemm_nvfp4_pack_scales.argtypes = [i, i, vp, vp, vp]
        lib.gemm_nvfp4_pack_scales.restype = i
        lib.gemm_mxfp8_scale_bytes.argtypes = [i, i]
        lib.gemm_mxfp8_scale_bytes.restype = ctypes.c_size_t
        lib.gemm_mxfp8_pack_scales.argtypes = [i, i, vp, vp, vp]
        lib.gemm_mxfp8_pack_scales.restype = i
        lib.sgemm.argtypes = [i, i, i, f, vp, vp, f, vp, vp]
        lib.sgemm.restype = i
        lib.sgemm_ex.argtypes = [i, i, i, f, vp, vp, f, vp, vp, ctypes.POINTER(_SgemmConfig)]
        lib.sgemm_ex.restype = i
        lib.gemm_last_error.argtypes = []
        lib.gemm_last_error.restype = ctypes.c_char_p
        lib.gemm_check_device_status.argtypes = [vp]
        lib.gemm_check_device_status.restype = i
        lib.gemm_f16_select.argtypes = [i, i, i, i, ctypes.POINTER(_F16Config)]
        lib.gemm_f16_select.restype = i
        lib.gemm_sgemm_select.argtypes = [i, i, i, i, ctypes.POINTER(_SgemmConfig)]
        lib.gemm_sgemm_select.restype = i
        lib.gemm_f16_nt_stream_k_noalloc.argtypes = [i, i, i, vp, vp, vp, vp]
        lib.gemm_f16_nt_stream_k_noalloc.restype = i
        lib.gemm_debug_f16_nt_skip_load.argtypes = [i, i, i, vp, vp, vp, vp, i, ctypes.c_ulonglong]
        lib.gemm_debug_f16_nt_skip_load.restype = i
        lib.gemm_debug_skinny_plan.argtypes = [i, i, i, i, ctypes.POINTER(i), ctypes.POINTER(i),
                                               ctypes.POINTER(i)]
        lib.gemm_debug_skinny_plan.restype = i
        lib.gemm_debug_skinny_parts.argtypes = [i, i, i, i]
        lib.gemm_debug_skinny_parts.restype = i
        lib.gemm_debug_last_pair_launch.argtypes = [ctypes.POINTER(i)] * 4
        lib.gemm_debug_sm_clocks.restype = i
        lib.gemm_debug_sm_clocks.argtypes = [vp, i, vp]
        lib.gemm_debug_last_pair_launch.restype = i
        lib.gemm_debug_blockscaled_skip_load.argtypes = [i, i, i, i, vp, vp, vp, vp, vp, vp,
                                                         ctypes.POINTER(_MxConfig), i,
                                                         ctypes.c_ulonglong]
        lib.gemm_debug_blockscaled_skip_load.restype = i
        lib.gemm_debug_f16_nt_stream_k_skip_publish.argtypes = [i, i, i, vp, vp, vp, vp,
                                                                ctypes.c_ulonglong]
        lib.gemm_debug_f16_nt_stream_k_skip_publish.restype = i
        _lib = lib
        return lib


def gemm_last_error() -> str:
    return load_library().gemm_last_error().decode("utf-8", "replace")


def _check(status: int) -> int:
    if status != GEMM_OK:
        raise GemmError(status, gemm_last_error())
    return status


# ---------------------------------------------------------------------------
# The C ABI, same names and argument order (pointers and streams as ints).
# ---------------------------------------------------------------------------

def gemm_f16_nt(M: int, N: int, K: int, A: int, B: int, C: int, stream: int | None = 0) -> int:
    return _check(load_library().gemm_f16_nt(M, N, K, A, B, C, stream or None))


def gemm_f16_nt_ex(M, N, K, A, B, C, stream=0, variant=GEMM_F16_AUTO, grid=0, flags=0, raster=0) -> int:
    cfg = _F16Config(variant, grid, flags, raster)
    return _check(load_library().gemm_f16_nt_ex(M, N, K, A, B, C, stream or None, ctypes.byref(cfg)))


def gemm_f16_nt_fused(M, N, K, A, B, C, alpha=1.0, beta=0.0, bias=0, residual=0,
                      activation=GEMM_ACT_NONE, stream=0, variant=GEMM_F16_AUTO, grid=0,
                      flags=0, raster=0) -> int:
    """C = act(alpha·A·Bᵀ + bias + beta·residual) rounded to half once; bias and
    residual are device pointers or 0 (absent)."""
    epi = _F16Epilogue(float(alpha), float(beta), bias or None, residual or None, int(activation))
    cfg = _F16Config(variant, grid, flags, raster)
    return _check(load_library().gemm_f16_nt_fused(M, N, K, A, B, C, ctypes.byref(epi),
                                                   stream or None, ctypes.byref(cfg)))


def gemm_mxfp8_nt(M, N, K, A, SFA, B, SFB, C, stream=0) -> int:
    """Block-scaled FP8 product; SFA/SFB in the chunk layout (pointers as ints)."""
    return _check(load_library().gemm_mxfp8_nt(M, N, K, A, SFA, B, SFB, C, stream or None))


def gemm_mxfp8_nt_ex(M, N, K, A, SFA, B, SFB, C, stream=0, variant=GEMM_MXFP8_AUTO, grid=0) -> int:
    cfg = _MxConfig(variant, grid)
    return _check(load_library().gemm_mxfp8_nt_ex(M, N, K, A, SFA, B, SFB, C, stream or None,
                                                  ctypes.byref(cfg)))


def gemm_nvfp4_nt(M, N, K, A, SFA, B, SFB, alpha, C, stream=0) -> int:
    """Block-scaled FP4 product; SFA/SFB in the NVFP4 chunk layout (pointers as ints)."""
    return _check(load_library().gemm_nvfp4_nt(M, N, K, A, SFA, B, SFB, float(alpha), C, stream or None))


def gemm_nvfp4_nt_ex(M, N, K, A, SFA, B, SFB, alpha, C, stream=0, variant=GEMM_MXFP8_AUTO, grid=0) -> int:
    cfg = _MxConfig(variant, grid)
    return _check(load_library().gemm_nvfp4_nt_ex(M, N, K, A, SFA, B, SFB, float(alpha), C,
                                                  stream or None, ctypes.byref(cfg)))


def gemm_nvfp4_scale_bytes(rows: int, K: int) -> int:
    return int(load_library().gemm_nvfp4_scale_bytes(rows, K))


def gemm_nvfp4_pack_scales(rows, K, plain, blocked, stream=0) -> int:
    return _check(load_library().gemm_nvfp4_pack_scales(rows, K, plain, blocked, stream or None))


def gemm_mxfp8_scale_bytes(rows: int, K: int) -> int:
    return int(load_library().gemm_mxfp8_scale_bytes(rows, K))


def gemm_mxfp8_pack_scales(rows, K, plain, blocked, stream=0) -> int:
    return _check(load_library().gemm_mxfp8_pack_scales(rows, K, plain, blocked, stream or None))


def gemm_f16_nt_stream_k_noalloc(M: int, N: int, K: int, A: int, B: int, C: int,
                                 stream: int | None = 0) -> int:
    """gemm_f16_nt without any allocation by the library: for callers that must
    not let it cudaMalloc (a pre-reserved memory pool, a latency-critical path,
    an allocator that owns every byte).  Uses a static 19.0 MiB array; calls
    that overlap on the GPU race on it."""
    return _check(load_library().gemm_f16_nt_stream_k_noalloc(M, N, K, A, B, C, stream or None))


def sgemm(M: int, N: int, K: int, alpha: float, A: int, B: int, beta: float, C: int,
          stream: int | None = 0) -> int:
    return _check(load_library().sgemm(M, N, K, alpha, A, B, beta, C, stream or None))


def sgemm_ex(M, N, K, alpha, A, B, beta, C, stream=0, variant=GEMM_SGEMM_AUTO, splits=0) -> int:
    cfg = _SgemmConfig(variant, splits)
    return _check(load_library().sgemm_ex(M, N, K, alpha, A, B, beta, C, stream or None,
                                          ctypes.byref(cfg)))


def gemm_check_device_status(stream: int | None = 0) -> int:
    return _check(load_library().gemm_check_device_status(stream or None))


def gemm_f16_select(M: int, N: int, K: int, sm_count: int) -> tuple[int, int, int]:
    """(variant, grid, raster) of the library's choice."""
    cfg = _F16Config(0, 0, 0, 0)
    _check(load_library().gemm_f16_select(M, N, K, sm_count, ctypes.byref(cfg)))
    return cfg.variant, cfg.grid, cfg.raster


def gemm_sgemm_select(M: int, N: int, K: int, sm_count: int) -> tuple[int, int]:
    cfg = _SgemmConfig(0, 0)
    _check(load_library().gemm_sgemm_select(M, N, K, sm_count, ctypes.byref(cfg)))
    return cfg.variant, cfg.splits


def gemm_debug_f16_nt_skip_load(M, N, K, A, B, C, stream, skip_kblock, timeout_ns) -> int:
    """Raw status of the fault-injection hook of include/gemm_testing.h."""
    return load_library().gemm_debug_f16_nt_skip_load(M, N, K, A, B, C, stream or None,
                                                      skip_kblock, timeout_ns)


def gemm_debug_blockscaled_skip_load(fmt, M, N, K, A, SFA, B, SFB, C, stream, variant, skip_kblock,
                                     timeout_ns) -> int:
    """Raw status of the block-scaled fault-injection hook (fmt 0 MXFP8, 1 NVFP4)."""
    cfg = _MxConfig(variant, 0)
    return load_library().gemm_debug_blockscaled_skip_load(fmt, M, N, K, A, SFA, B, SFB, C,
                                                           stream or None, ctypes.byref(cfg),
                                                           skip_kblock, timeout_ns)


def gemm_debug_f16_nt_stream_k_skip_publish(M, N, K, A, B, C, stream, timeout_ns) -> int:
    """Raw status of the stream-K hook whose partials are never flagged ready."""
    return load_library().gemm_debug_f16_nt_stream_k_skip_publish(M, N, K, A, B, C, stream or None,
                                                                  timeout_ns)


def gemm_debug_last_pair_launch():
    """(pairs, whole tiles, shared k-block units, scratch kind) of the last
    CTA-pair launch on this thread (scratch kind: 0 none, 1 allocated
    workspace, 2 the allocation-free entry point's static array), or None."""
    vals = [ctypes.c_int(0) for _ in range(4)]
    if load_library().gemm_debug_last_pair_launch(*[ctypes.byref(v) for v in vals]) != 0:
        return None
    return tuple(v.value for v in vals)


def gemm_debug_sm_clocks(out, ctas, stream) -> None:
    """Enqueue one clock sample per CTA into device words out[3 * ctas]:
    (SM id, SM cycle counter, global timer in ns) for each CTA."""
    _check(load_library().gemm_debug_sm_clocks(out, ctas, stream or None))


def gemm_debug_skinny_parts(M, N, K, ctas):
    """Clusters per tile the skinny variant plans (host logic only)."""
    parts = load_library().gemm_debug_skinny_parts(M, N, K, ctas)
    if parts < 0:
        raise ValueError(f"bad plan arguments M={M} N={N} K={K} ctas={ctas}")
    return parts


def gemm_debug_skinny_plan(M, N, K, ctas):
    """(shares, rows per group, groups, k-blocks per share) the skinny variant
    plans (host logic only; every slot assumed to hold a cluster of each size)."""
    rows, groups, kb = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    splits = load_library().gemm_debug_skinny_plan(M, N, K, ctas, ctypes.byref(rows), ctypes.byref(groups),
                                                   ctypes.byref(kb))
    if splits < 0:
        raise ValueError(f"bad plan arguments M={M} N={N} K={K} ctas={ctas}")
    return splits, rows.value, groups.value, kb.value


# ---------------------------------------------------------------------------
# Tensor conveniences (torch supplies device memory and the stream).
# ---------------------------------------------------------------------------

def _stream_handle(stream) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def f16_nt(A, B, C=None, stream=None, variant: int = GEMM_F16_AUTO, grid: int = 0, flags: int = 0):
    """C = A·Bᵀ for contiguous half CUDA tensors A [M,K], B [N,K]; returns C [M,N]."""
    import torch

    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("f16_nt expects float16 tensors")
    if not (A.is_cuda and B.is_cuda and A.is_contiguous() and B.is_contiguous()):
        raise ValueError("f16_nt expects contiguous CUDA tensors")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}^T")
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif C.shape != (M, N) or C.dtype != torch.float16 or not C.is_contiguous():
        raise ValueError("C must be a contiguous float16 [M, N] tensor")
    gemm_f16_nt_ex(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), _stream_handle(stream),
                   variant, grid, flags)
    return C


def f16_nt_fused(A, B, C=None, alpha: float = 1.0, bias=None, beta: float = 0.0, residual=None,
                 activation: str | int = "none", stream=None, variant: int = GEMM_F16_AUTO,
                 grid: int = 0, flags: int = 0):
    """C = act(alpha·A·Bᵀ + bias + beta·residual) for contiguous half CUDA
    tensors A [M,K], B [N,K], bias [N], residual [M,N] (residual may be C)."""
    import torch

    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise TypeError("f16_nt_fused expects float16 tensors")
    if not (A.is_cuda and B.is_cuda and A.is_contiguous() and B.is_contiguous()):
        raise ValueError("f16_nt_fused expects contiguous CUDA tensors")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[1]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}^T")
    M, K = A.shape
    N = B.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    elif C.shape != (M, N) or C.dtype != torch.float16 or not C.is_contiguous():
        raise ValueError("C must be a contiguous float16 [M, N] tensor")
    for name, t, shape in (("bias", bias, (N,)), ("residual", residual, (M, N))):
        if t is not None and (t.shape != shape or t.dtype != torch.float16 or not t.is_cuda
                              or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous float16 CUDA tensor of shape {shape}")
    act = ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)
    gemm_f16_nt_fused(M, N, K, A.data_ptr(), B.data_ptr(), C.data_ptr(), alpha, beta,
                      bias.data_ptr() if bias is not None else 0,
                      residual.data_ptr() if residual is not None else 0, act,
                      _stream_handle(stream), variant, grid, flags)
    return C


def mxfp8_pack_scales(S, stream=None):
    """Plain UE8M0 scales [rows, K/32] (uint8 CUDA tensor) -> the chunk layout."""
    import torch

    if S.dtype != torch.uint8 or not S.is_cuda or not S.is_contiguous() or S.dim() != 2:
        raise ValueError("scales must be a contiguous uint8 CUDA tensor [rows, K/32]")
    rows, ksf = S.shape
    K = 32 * ksf
    out = torch.empty(gemm_mxfp8_scale_bytes(rows, K), dtype=torch.uint8, device=S.device)
    gemm_mxfp8_pack_scales(rows, K, S.data_ptr(), out.data_ptr(), _stream_handle(stream))
    return out


def mxfp8_nt(A, SA, B, SB, C=None, stream=None, packed=False, variant=GEMM_MXFP8_AUTO, grid=0):
    """C (half) = MXFP8 product of E4M3 codes A [M,K], B [N,K] (uint8 CUDA
    tensors) with UE8M0 scales SA [M,K/32], SB [N,K/32] (or, with packed=True,
    already in the chunk layout)."""
    import torch

    for t in (A, B):
        if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError("A and B must be contiguous uint8 CUDA tensors (E4M3 codes)")
    if A.shape[1] != B.shape[1]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}^T")
    M, K = A.shape
    N = B.shape[0]
    if not packed:
        SA, SB = mxfp8_pack_scales(SA, stream), mxfp8_pack_scales(SB, stream)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    gemm_mxfp8_nt_ex(M, N, K, A.data_ptr(), SA.data_ptr(), B.data_ptr(), SB.data_ptr(), C.data_ptr(),
                     _stream_handle(stream), variant, grid)
    return C


def nvfp4_pack_scales(S, stream=None):
    """Plain E4M3 block scales [rows, K/16] (uint8 CUDA tensor) -> the NVFP4 chunk layout."""
    import torch

    if S.dtype != torch.uint8 or not S.is_cuda or not S.is_contiguous() or S.dim() != 2:
        raise ValueError("scales must be a contiguous uint8 CUDA tensor [rows, K/16]")
    rows, ksf = S.shape
    K = 16 * ksf
    out = torch.empty(gemm_nvfp4_scale_bytes(rows, K), dtype=torch.uint8, device=S.device)
    gemm_nvfp4_pack_scales(rows, K, S.data_ptr(), out.data_ptr(), _stream_handle(stream))
    return out


def nvfp4_nt(A, SA, B, SB, alpha: float = 1.0, C=None, stream=None, packed=False,
             variant=GEMM_MXFP8_AUTO, grid=0):
    """C (half) = alpha * NVFP4 product of packed E2M1 A [M,K/2], B [N,K/2]
    (uint8 CUDA tensors) with E4M3 block scales SA [M,K/16], SB [N,K/16] (or,
    with packed=True, already in the chunk layout)."""
    import torch

    for t in (A, B):
        if t.dtype != torch.uint8 or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError("A and B must be contiguous uint8 CUDA tensors (packed E2M1)")
    if A.shape[1] != B.shape[1]:
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)}^T")
    M, K = A.shape[0], 2 * A.shape[1]
    N = B.shape[0]
    if not packed:
        SA, SB = nvfp4_pack_scales(SA, stream), nvfp4_pack_scales(SB, stream)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    gemm_nvfp4_nt_ex(M, N, K, A.data_ptr(), SA.data_ptr(), B.data_ptr(), SB.data_ptr(), alpha,
                     C.data_ptr(), _stream_handle(stream), variant, grid)
    return C


def sgemm_(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None,
           variant: int = GEMM_SGEMM_AUTO):
    """In place: C = alpha·A·B + beta·C for contiguous float32 CUDA tensors."""
    import torch

    for t in (A, B, C):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("sgemm_ expects contiguous float32 CUDA tensors")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0] or C.shape != (A.shape[0], B.shape[1]):
        raise ValueError(f"shape mismatch {tuple(A.shape)} x {tuple(B.shape)} -> {tuple(C.shape)}")
    M, K = A.shape
    N = B.shape[1]
    sgemm_ex(M, N, K, float(alpha), A.data_ptr(), B.data_ptr(), float(beta), C.data_ptr(),
             _stream_handle(stream), variant)
    return C
