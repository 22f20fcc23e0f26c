"""moe_grouped_fp8_gb300: GB300 (sm_103a) blockwise-scaled FP8 grouped GEMM for MoE.

The compute lives in libdg.so (hand-written CUDA, C ABI in include/dg.h); `api` holds the
Python binding with the same entry-point names; `workloads` holds the seeded synthetic
inputs.  Importing the package does not load the library: the first call does, and fails
loudly if it has not been built (`moe_grouped_fp8_gb300.build.build()`).
"""
from ._lib import (DG_DEBUG_A_SCALE, DG_DEBUG_B_SCALE, DG_DEBUG_CAST_IN, DG_DEBUG_CAST_OUT, DG_DEBUG_OUT, DG_ERR_CUDA, DG_ERR_INVALID_ARG, DG_ERR_UNSUPPORTED, DG_OK, DG_OUT_BF16, DG_OUT_FP32, DG_SF_FP32,
                   DG_SF_UE8M0, DG_STATUS_BAD_INDEX, DG_STATUS_COUNT_GT_CAP, DG_STATUS_K_NOT_ALIGNED,
                   DG_STATUS_K_OVERFLOW, DG_STATUS_TIMEOUT, DG_STATUS_TOO_MANY_RUNS, DGError)

__all__ = ["DG_OK", "DG_ERR_INVALID_ARG", "DG_ERR_UNSUPPORTED", "DG_ERR_CUDA", "DG_OUT_BF16", "DG_OUT_FP32", "DG_SF_FP32", "DG_SF_UE8M0", "DG_STATUS_BAD_INDEX",
           "DG_STATUS_COUNT_GT_CAP", "DG_STATUS_K_NOT_ALIGNED", "DG_STATUS_K_OVERFLOW", "DG_STATUS_TIMEOUT",
           "DG_STATUS_TOO_MANY_RUNS", "DG_DEBUG_A_SCALE", "DG_DEBUG_B_SCALE", "DG_DEBUG_OUT", "DG_DEBUG_CAST_IN",
           "DG_DEBUG_CAST_OUT", "DGError"]
