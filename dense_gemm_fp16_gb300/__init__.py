"""GB300-native (sm_103a) dense matrix multiplication.

Two products behind the C ABI of ``include/gemm.h`` (``libgemm.so``):

* ``gemm_f16_nt(M, N, K, A, B, C, stream)``: C = A·Bᵀ, half in, fp32
  accumulation on the tcgen05 tensor cores, half out.
* ``gemm_f16_nt_fused(..., epi, stream, cfg)``: the same product passed
  through a fused epilogue act(alpha·A·Bᵀ + bias + beta·R) before rounding.
* ``gemm_mxfp8_nt(M, N, K, A, SFA, B, SFB, C, stream)``: the block-scaled
  FP8 (MXFP8) product on the tensor cores, half out.
* ``gemm_nvfp4_nt(M, N, K, A, SFA, B, SFB, alpha, C, stream)``: the
  block-scaled FP4 (NVFP4) product, half out.
* ``sgemm(M, N, K, alpha, A, B, beta, C, stream)``: C = alpha·A·B + beta·C in
  fp32 on the CUDA cores.

This package is the thin Python binding (same names, pointers as ints) plus
tensor conveniences ``f16_nt``, ``f16_nt_fused`` and ``sgemm_``; ``workloads`` holds the seeded
synthetic inputs.  The library is built in-tree by
``python -m dense_gemm_fp16_gb300.build``; without it every call raises.
"""
from ._binding import (  # noqa: F401
    ACTIVATIONS,
    GEMM_ACT_GELU_TANH,
    GEMM_ACT_NONE,
    GEMM_ACT_RELU,
    GEMM_ACT_SILU,
    GEMM_ERR_CUDA,
    GEMM_ERR_DEVICE_TIMEOUT,
    GEMM_ERR_INVALID_ARG,
    GEMM_ERR_MISALIGNED,
    GEMM_ERR_UNSUPPORTED,
    GEMM_F16_128x128,
    GEMM_F16_128x256,
    GEMM_F16_256x256_PAIR,
    GEMM_F16_256x256_QUAD,
    GEMM_F16_256x256_KSPLIT,
    GEMM_F16_AUTO,
    GEMM_F16_FLAG_STREAM_K,
    GEMM_F16_GEMV,
    GEMM_F16_SKINNY,
    GEMM_F16_NUM_VARIANTS,
    GEMM_MXFP8_128x128,
    GEMM_MXFP8_128x256,
    GEMM_MXFP8_256x128_PAIR,
    GEMM_MXFP8_256x256_PAIR,
    GEMM_MXFP8_NUM_VARIANTS,
    GEMM_MXFP8_AUTO,
    GEMM_OK,
    GEMM_SGEMM_64x64,
    GEMM_SGEMM_128x64,
    GEMM_SGEMM_128x128,
    GEMM_SGEMM_AUTO,
    LIB_PATH,
    GemmError,
    f16_nt,
    f16_nt_fused,
    gemm_check_device_status,
    gemm_debug_f16_nt_skip_load,
    gemm_debug_skinny_plan,
    gemm_debug_skinny_parts,
    gemm_debug_last_pair_launch,
    gemm_debug_sm_clocks,
    gemm_debug_blockscaled_skip_load,
    gemm_debug_f16_nt_stream_k_skip_publish,
    gemm_f16_nt,
    gemm_f16_nt_ex,
    gemm_f16_nt_fused,
    gemm_f16_nt_stream_k_noalloc,
    gemm_mxfp8_nt,
    gemm_mxfp8_nt_ex,
    gemm_mxfp8_pack_scales,
    gemm_mxfp8_scale_bytes,
    gemm_nvfp4_nt,
    gemm_nvfp4_nt_ex,
    gemm_nvfp4_pack_scales,
    gemm_nvfp4_scale_bytes,
    gemm_f16_select,
    gemm_last_error,
    gemm_sgemm_select,
    load_library,
    mxfp8_nt,
    mxfp8_pack_scales,
    nvfp4_nt,
    nvfp4_pack_scales,
    sgemm,
    sgemm_,
    sgemm_ex,
)
