"""ctypes declarations of libdg.so (include/dg.h).  Loading fails loudly when the library is
missing: there is no fallback implementation of any entry point."""
from __future__ import annotations

import ctypes
import os
import threading

from .build import library_path

DG_OK, DG_ERR_INVALID_ARG, DG_ERR_UNSUPPORTED, DG_ERR_CUDA = 0, 1, 2, 3
DG_SF_FP32, DG_SF_UE8M0 = 0, 1
DG_OUT_BF16, DG_OUT_FP32 = 0, 1
DG_STATUS_BAD_INDEX = 1
DG_STATUS_COUNT_GT_CAP = 2
DG_STATUS_K_NOT_ALIGNED = 4
DG_STATUS_K_OVERFLOW = 8
DG_STATUS_TIMEOUT = 16
DG_STATUS_TOO_MANY_RUNS = 32
DG_DEBUG_A_SCALE, DG_DEBUG_B_SCALE, DG_DEBUG_OUT, DG_DEBUG_CAST_IN, DG_DEBUG_CAST_OUT = 1, 2, 4, 8, 16
DG_OP_M_GROUPED_CONTIGUOUS, DG_OP_M_GROUPED_MASKED, DG_OP_K_GROUPED_WGRAD = 0, 1, 2
DG_MAX_GROUPS = 1024
DG_MAX_M_BLOCKS = 4096
DG_NOALLOC_MAX_GROUPS = 256

# name -> (restype, argtypes); every symbol include/dg.h declares
P, I64, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
SIGNATURES = {
    "dg_last_error": (ctypes.c_char_p, []),
    "dg_workspace_size": (SZ, [I32, I32, I64, I64, I64]),
    "dg_quant_per_token_1x128": (I32, [P, I64, I64, I64, P, P, I32, F32, P, I32, P]),
    "dg_quant_per_token_1x128_routed": (I32, [P, I64, I64, I64, P, P, I32, F32, P, P]),
    "dg_quant_per_channel_128": (I32, [P, I64, I64, P, I32, P, P, F32, P, P]),
    "dg_quant_per_channel_128_pair": (I32, [P, I64, P, P, P, I64, P, P, I64, P, I32, F32, P, P]),
    "dg_quant_block_128x128": (I32, [P, I32, I64, I64, P, P, I32, F32, P]),
    "dg_m_grouped_fp8_contiguous": (I32, [P, P, P, P, P, I32, P, I64, I32, I64, I64, I32, P, SZ, P, P]),
    "dg_m_grouped_fp8_masked": (I32, [P, P, P, P, P, I32, P, I32, I64, I64, I64, I32, I32, P, SZ, P, P]),
    "dg_fp8_gemm_nt": (I32, [P, P, P, P, P, P, I32, I64, I64, I64, I32, P, P]),
    "dg_fp8_gemm_nt_batched": (I32, [P, P, P, P, P, P, I32, I32, I64, I64, I64, I32, P, P]),
    "dg_m_grouped_fp8_contiguous_psum": (I32, [P, P, P, P, P, I32, P, I64, I32, I64, I64, I32, P, SZ, P, P]),
    "dg_k_grouped_fp8_wgrad_psum": (I32, [P, P, P, P, P, P, P, I32, I64, I64, I64, P, SZ, P, P]),
    "dg_quant_per_channel_128_psum": (I32, [P, I64, I64, P, I32, P, P, F32, P, P]),
    "dg_quant_per_channel_128_pair_psum": (I32, [P, I64, P, P, P, I64, P, P, I64, P, I32, F32, P, P]),
    "dg_m_grouped_bf16_masked": (I32, [P, P, P, I32, P, I32, I64, I64, I64, I32, P, P]),
    "dg_m_grouped_bf16_contiguous": (I32, [P, P, P, I32, P, I64, I32, I64, I64, P, P]),
    "dg_k_grouped_fp8_wgrad": (I32, [P, P, P, P, P, P, P, I32, I64, I64, I64, P, SZ, P, P]),
    "dg_k_grouped_fp8_wgrad_from_bf16": (I32, [P, P, P, I32, I64, I64, I64, P, P, P, P, P, P, F32, P, SZ, P, P]),
    "dg_k_grouped_fp8_wgrad_from_bf16_psum": (I32, [P, P, P, I32, I64, I64, I64, P, P, P, P, P, P, F32, P, SZ, P, P]),
    "dg_k_grouped_fp8_wgrad_noalloc": (I32, [P, P, P, P, P, P, P, I32, I64, I64, I64, P, P]),
    "dg_quant_block_128x128_fp4": (I32, [P, I32, I64, I64, P, P, F32, P]),
    "dg_m_grouped_fp8_fp4_contiguous": (I32, [P, P, P, P, P, I32, P, I64, I32, I64, I64, P, P]),
    "dg_m_grouped_fp8_fp4_masked": (I32, [P, P, P, P, P, I32, P, I32, I64, I64, I64, I32, P, P]),
    "dg_quant_per_token_1x128_packed": (I32, [P, I64, I64, P, P, I32, F32, P, I32, I64, P]),
    "dg_pack_masked_rows": (I32, [P, I32, I64, I64, P, P, P]),
    "dg_set_arg_log": (I32, [ctypes.c_char_p]),
    "dg_debug_build": (I32, []),
    "dg_debug_word": (I32, [ctypes.POINTER(ctypes.c_uint32), I32]),
}
# test hooks exported by the library (not part of include/dg.h)
TESTING_SIGNATURES = {
    "dg_testing_kgrouped_prologue": (I32, [P, P, P, I32, I64, I64, I64, P, P]),
    "dg_testing_kgrouped_host_maps": (I32, [P, P, P, I32, I64, I64, P]),
    "dg_testing_kgrouped_gemm_only": (I32, [P, P, P, P, P, P, P, I32, I64, I64, I64, P, SZ, P, P]),
    "dg_testing_mgrouped_kernel": (I32, [I32]),
    "dg_testing_mgrouped_warps": (I32, [I32]),
    "dg_testing_wait_limit_ns": (I32, [ctypes.c_uint64]),
    "dg_testing_mgrouped_store": (I32, [I32]),
    "dg_testing_mgrouped_bn": (I32, [I32]),
    "dg_testing_token_items_per_cta": (I32, [I32]),
    "dg_testing_debug_out_rows": (I32, [I64]),
    "dg_testing_debug_stop_producer": (I32, [I32]),
    "dg_testing_bf16_bn": (I32, [I32]),
}

_lock = threading.Lock()
_lib = None


class DGError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"dg error {code}: {msg}")
        self.code = code


def load() -> ctypes.CDLL:
    """The library of this process: libdg.so, or the debug build libdg_debug.so when the
    environment sets DG_DEBUG=1."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path(os.environ.get("DG_DEBUG", "0") == "1")
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
                                   "(or moe_grouped_fp8_gb300.build.build(debug=...)); there is no fallback path")
            lib = ctypes.CDLL(path)
            for name, (res, args) in {**SIGNATURES, **TESTING_SIGNATURES}.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def check(rc: int):
    if rc != DG_OK:
        raise DGError(rc, load().dg_last_error().decode())
