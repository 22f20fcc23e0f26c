"""CPU oracle for blockwise-scaled FP8 grouped GEMM — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu-baseline / reference
legs may import this package.  The product library (``moe_grouped_fp8_gb300``) never does,
and shares no code with it.  The arithmetic lives in ``oracle.c`` (plain C, fp64
accumulation, see its header for the passages of the source pages each function follows);
this module only marshals numpy arrays through ctypes.

Every function here is pinned by ``tests/test_oracle_pins.py`` against facts the pages and
the mathematics fix (exhaustive codec checks, closed forms, library special cases, the
pages' printed reference norm).  The one part left "parity unpinned" is the agreement of
the *unquantized* bf16 product with the quantized one, which the pages only bound loosely.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fexcess-precision=standard",
          "-fno-fast-math", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so beside it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_e4m3_encode.argtypes = [f32]
            lib.oracle_e4m3_encode_array.argtypes = [P, i64, P]
            lib.oracle_e4m3_decode_array.argtypes = [P, i64, P]
            lib.oracle_scale_from_amax.argtypes = [P, i64, f32, i32, P, P]
            lib.oracle_e2m1_decode.restype = ctypes.c_double
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_encode.restype = ctypes.c_uint8
            lib.oracle_e2m1_encode.argtypes = [f32]
            lib.oracle_e2m1_encode_array.argtypes = [P, i64, P]
            lib.oracle_e2m1_decode_array.argtypes = [P, i64, P]
            lib.oracle_quant_block_128x128_fp4.argtypes = [P, i32, i64, i64, f32, P, P]
            lib.oracle_gemm_contiguous_fp4.argtypes = [P, P, P, P, P, i64, i32, i64, i64, P]
            lib.oracle_gemm_masked_fp4.argtypes = [P, P, P, P, P, i32, i64, i64, i64, P]
            lib.oracle_quant_per_token_1x128.argtypes = [P, i64, i64, i64, P, i32, f32, i32, P, P, P]
            lib.oracle_quant_block_128x128.argtypes = [P, i32, i64, i64, f32, i32, P, P, P]
            lib.oracle_quant_per_channel_128.argtypes = [P, i64, i64, f32, P, P]
            lib.oracle_pack_kmajor.argtypes = [P, P, i32, i64, P]
            lib.oracle_gemm_contiguous.argtypes = [P, P, P, P, P, i64, i32, i64, i64, P]
            lib.oracle_gemm_masked.argtypes = [P, P, P, P, P, i32, i64, i64, i64, P]
            lib.oracle_gemm_batched.argtypes = [P, P, P, P, P, i64, i64, i64, i64, P]
            lib.oracle_gemm_kgrouped.argtypes = [P, P, P, P, P, P, i32, i64, i64, i64, P]
            lib.oracle_gemm_masked_bf16.argtypes = [P, P, P, i32, i64, i64, i64, P]
            lib.oracle_sizes_from_psum.argtypes = [P, i32, P]
            lib.oracle_m_indices_from_psum.argtypes = [P, i32, i64, P]
            lib.oracle_gemm_contiguous_bf16.argtypes = [P, P, P, i64, i32, i64, i64, P]
            lib.oracle_round_bf16.restype = ctypes.c_uint16
            lib.oracle_round_bf16.argtypes = [ctypes.c_double]
            lib.oracle_round_bf16_array.argtypes = [P, i64, P]
            lib.oracle_calc_diff.restype = ctypes.c_double
            lib.oracle_calc_diff.argtypes = [P, P, i64]
            lib.oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bf16_bits(x) -> np.ndarray:
    """Accept a uint16 array of bf16 bits or a torch bf16 CPU tensor."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch  # only for tensors handed in by tests
    assert x.dtype == torch.bfloat16
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------------------ codec

def e4m3_decode(codes) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode_array(_p(c), c.size, _p(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e4m3_encode_array(_p(v), v.size, _p(out))
    return out


def e2m1_decode(codes) -> np.ndarray:
    """Values of FP4 (e2m1) codes 0..15 (one code per array element, not packed)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e2m1_decode_array(_p(c), c.size, _p(out))
    return out


def e2m1_encode(values) -> np.ndarray:
    """FP4 (e2m1) codes 0..15 of fp32 values (one code per array element)."""
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    _load().oracle_e2m1_encode_array(_p(v), v.size, _p(out))
    return out


def scale_from_amax(amax, sf_zero: float, ue8m0: bool):
    a = _c(amax, np.float32)
    sf = np.empty(a.shape, np.float32)
    ue = np.empty(a.shape, np.uint8)
    _load().oracle_scale_from_amax(_p(a), a.size, sf_zero, int(ue8m0), _p(sf), _p(ue))
    return sf, ue


def ue8m0_value(ue_bytes) -> np.ndarray:
    """Value of a UE8M0 byte: 2^(byte - 127), as fp32 (exact)."""
    b = np.asarray(ue_bytes).astype(np.int32)
    return np.ldexp(np.float32(1.0), b - 127).astype(np.float32)


# ------------------------------------------------------------------------------ casts

def quant_per_token_1x128(x, sf_zero: float = 1e-30, ue8m0: bool = False, row_counts=None):
    """x: bf16 [M, K].  Returns q [M, K] uint8, sf [M, K/128] fp32, ue [M, K/128] uint8 (or
    None).  With row_counts (length G), rows r >= count of each of the G equal row groups are
    left as 0 / NaN / 0 (not cast)."""
    xb = _bf16_bits(x)
    M, K = xb.shape
    assert K % 128 == 0
    q = np.zeros((M, K), np.uint8)
    sf = np.full((M, K // 128), np.nan, np.float32)
    ue = np.zeros((M, K // 128), np.uint8) if ue8m0 else None
    rc = None if row_counts is None else _c(row_counts, np.int32)
    G = 0 if rc is None else rc.size
    _load().oracle_quant_per_token_1x128(_p(xb), M, K, K, _p(rc), G, sf_zero, int(ue8m0),
                                         _p(q), _p(sf), _p(ue))
    return q, sf, ue


def quant_block_128x128(w, sf_zero: float = 1e-30, ue8m0: bool = False):
    """w: bf16 [G, N, K].  Returns q [G, N, K], sf [G, N/128, K/128], ue (or None)."""
    wb = _bf16_bits(w)
    G, N, K = wb.shape
    assert N % 128 == 0 and K % 128 == 0
    q = np.empty((G, N, K), np.uint8)
    sf = np.empty((G, N // 128, K // 128), np.float32)
    ue = np.empty((G, N // 128, K // 128), np.uint8) if ue8m0 else None
    _load().oracle_quant_block_128x128(_p(wb), G, N, K, sf_zero, int(ue8m0), _p(q), _p(sf), _p(ue))
    return q, sf, ue


def quant_block_128x128_fp4(w, sf_zero: float = 1e-30):
    """w: bf16 [G, N, K].  FP4 weights with power-of-two block scales: returns q_packed
    [G, N, K/2] (two e2m1 codes per byte, the even element in the low nibble) and the UE8M0
    bytes [G, N/128, K/128]."""
    wb = _bf16_bits(w)
    G, N, K = wb.shape
    assert N % 128 == 0 and K % 128 == 0
    q = np.empty((G, N, K // 2), np.uint8)
    ue = np.empty((G, N // 128, K // 128), np.uint8)
    _load().oracle_quant_block_128x128_fp4(_p(wb), G, N, K, sf_zero, _p(q), _p(ue))
    return q, ue


def quant_per_channel_128(x, sf_zero: float = 1e-30):
    """x: bf16 [T, C] token-major.  Returns q [T, C] and sf [T/128, C]."""
    xb = _bf16_bits(x)
    T, C = xb.shape
    assert T % 128 == 0
    q = np.empty((T, C), np.uint8)
    sf = np.empty((T // 128, C), np.float32)
    _load().oracle_quant_per_channel_128(_p(xb), T, C, sf_zero, _p(q), _p(sf))
    return q, sf


def pack_kmajor(q, ks) -> np.ndarray:
    """q [T, C] -> flat [sum(ks) * C]: expert e's block is q[span].T, row-major."""
    q = _c(q, np.uint8)
    ks = _c(ks, np.int32)
    T, C = q.shape
    out = np.zeros(int(ks.sum()) * C, np.uint8)
    _load().oracle_pack_kmajor(_p(q), _p(ks), ks.size, C, _p(out))
    return out


# ------------------------------------------------------------------------------ GEMMs

def gemm_contiguous(qa, sfa, qb, sfb, m_indices) -> np.ndarray:
    """fp64 D [M, N]; rows not routed are NaN."""
    qa, sfa, qb, sfb = _c(qa, np.uint8), _c(sfa, np.float32), _c(qb, np.uint8), _c(sfb, np.float32)
    mi = _c(m_indices, np.int32)
    M, K = qa.shape
    G, N, _ = qb.shape
    d = np.full((M, N), np.nan, np.float64)
    _load().oracle_gemm_contiguous(_p(qa), _p(sfa), _p(qb), _p(sfb), _p(mi), M, G, N, K, _p(d))
    return d


def gemm_contiguous_fp4(qa, sfa, qb_packed, sfb, m_indices) -> np.ndarray:
    """gemm_contiguous with FP4 weights: qb_packed [G, N, K/2] packed e2m1 codes."""
    qa, sfa, qb, sfb = _c(qa, np.uint8), _c(sfa, np.float32), _c(qb_packed, np.uint8), _c(sfb, np.float32)
    mi = _c(m_indices, np.int32)
    M, K = qa.shape
    G, N, K2 = qb.shape
    assert K2 * 2 == K
    d = np.full((M, N), np.nan, np.float64)
    _load().oracle_gemm_contiguous_fp4(_p(qa), _p(sfa), _p(qb), _p(sfb), _p(mi), M, G, N, K, _p(d))
    return d


def gemm_masked_fp4(qa, sfa, qb_packed, sfb, counts) -> np.ndarray:
    """gemm_masked with FP4 weights: qb_packed [G, N, K/2] packed e2m1 codes."""
    qa, sfa, qb, sfb = _c(qa, np.uint8), _c(sfa, np.float32), _c(qb_packed, np.uint8), _c(sfb, np.float32)
    cnt = _c(counts, np.int32)
    G, cap, K = qa.shape
    N = qb.shape[1]
    assert qb.shape[2] * 2 == K
    d = np.full((G, cap, N), np.nan, np.float64)
    _load().oracle_gemm_masked_fp4(_p(qa), _p(sfa), _p(qb), _p(sfb), _p(cnt), G, cap, N, K, _p(d))
    return d


def gemm_masked(qa, sfa, qb, sfb, counts) -> np.ndarray:
    """fp64 D [G, cap, N]; rows at or past min(count, cap) are NaN."""
    qa, sfa, qb, sfb = _c(qa, np.uint8), _c(sfa, np.float32), _c(qb, np.uint8), _c(sfb, np.float32)
    cnt = _c(counts, np.int32)
    G, cap, K = qa.shape
    N = qb.shape[1]
    d = np.full((G, cap, N), np.nan, np.float64)
    _load().oracle_gemm_masked(_p(qa), _p(sfa), _p(qb), _p(sfb), _p(cnt), G, cap, N, K, _p(d))
    return d


def gemm_batched(qa, sfa, qb, sfb, c=None) -> np.ndarray:
    """fp64 D [B, M, N] = c + per-entry products (plain GEMM: B = 1); qa [B, M, K],
    sfa [B, M, K/128] fp32 values, qb [B, N, K], sfb [B, N/128, K/128], c [B, M, N] or None."""
    qa, sfa, qb, sfb = _c(qa, np.uint8), _c(sfa, np.float32), _c(qb, np.uint8), _c(sfb, np.float32)
    B, M, K = qa.shape
    N = qb.shape[1]
    cc = None if c is None else _c(c, np.float64)
    d = np.empty((B, M, N), np.float64)
    _load().oracle_gemm_batched(_p(qa), _p(sfa), _p(qb), _p(sfb), _p(cc), B, M, N, K, _p(d))
    return d


def gemm_masked_bf16(a, b, counts) -> np.ndarray:
    """BF16 masked GEMM in fp64: D [G, cap, N]; rows at or past min(count, cap) are NaN."""
    a, b = _bf16_bits(a), _bf16_bits(b)
    cnt = _c(counts, np.int32)
    G, cap, K = a.shape
    N = b.shape[1]
    d = np.full((G, cap, N), np.nan, np.float64)
    _load().oracle_gemm_masked_bf16(_p(a), _p(b), _p(cnt), G, cap, N, K, _p(d))
    return d


def gemm_contiguous_bf16(a, b, m_indices) -> np.ndarray:
    """BF16 contiguous GEMM in fp64: D [M, N]; rows not routed are NaN."""
    a, b = _bf16_bits(a), _bf16_bits(b)
    mi = _c(m_indices, np.int32)
    M, K = a.shape
    G, N, _ = b.shape
    d = np.full((M, N), np.nan, np.float64)
    _load().oracle_gemm_contiguous_bf16(_p(a), _p(b), _p(mi), M, G, N, K, _p(d))
    return d


def sizes_from_psum(psum) -> np.ndarray:
    """K_e from inclusive prefix sums (k-grouped psum layout)."""
    ps = _c(psum, np.int32)
    ks = np.empty_like(ps)
    _load().oracle_sizes_from_psum(_p(ps), ps.size, _p(ks))
    return ks


def m_indices_from_psum(psum, M) -> np.ndarray:
    """Per-row expert of the contiguous psum layout (-1 = unrouted)."""
    ps = _c(psum, np.int32)
    mi = np.empty(M, np.int32)
    _load().oracle_m_indices_from_psum(_p(ps), ps.size, M, _p(mi))
    return mi


def gemm_kgrouped(a_packed, sfa, b_packed, sfb, ks, N, H, K_cap=None, c=None) -> np.ndarray:
    """fp64 D [G, N, H] = C + A_e^T B_e per expert; experts not computed are NaN (or C)."""
    ap, bp = _c(a_packed, np.uint8), _c(b_packed, np.uint8)
    sfa, sfb = _c(sfa, np.float32), _c(sfb, np.float32)
    ks = _c(ks, np.int32)
    G = ks.size
    if K_cap is None:
        K_cap = int(ks.sum())
    cc = None if c is None else _c(c, np.float32)
    d = np.full((G, N, H), np.nan, np.float64)
    _load().oracle_gemm_kgrouped(_p(ap), _p(sfa), _p(bp), _p(sfb), _p(cc), _p(ks), G, K_cap, N, H, _p(d))
    return d


# ------------------------------------------------------------------------------ comparison

def round_bf16(v) -> np.ndarray:
    """fp64 -> bf16 bits (uint16), one round-to-nearest-even."""
    a = _c(v, np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().oracle_round_bf16_array(_p(a), a.size, _p(out))
    return out


def bf16_bits_to_f64(bits) -> np.ndarray:
    b = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def calc_diff(x, y) -> float:
    """1 - 2 sum(x y) / sum(x^2 + y^2) in fp64 (0 when both are all zero)."""
    a, b = _c(x, np.float64).ravel(), _c(y, np.float64).ravel()
    assert a.size == b.size
    return float(_load().oracle_calc_diff(_p(a), _p(b), a.size))


def num_threads() -> int:
    return int(_load().oracle_num_threads())
