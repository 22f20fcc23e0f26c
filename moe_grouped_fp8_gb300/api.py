"""Python binding of libdg.so: the same entry points as include/dg.h, taking torch tensors.

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
PyTorch provides device memory and the current stream.  Each function checks tensor dtypes,
devices and sizes against the C ABI's layouts before the call, then raises DGError on a
non-zero return code.
"""
from __future__ import annotations

import ctypes

import torch

from ._lib import DG_OP_K_GROUPED_WGRAD, DG_OUT_BF16, DG_OUT_FP32, DG_SF_FP32, DGError, check, load

__all__ = [
    "dg_quant_per_token_1x128", "dg_quant_per_token_1x128_routed", "dg_quant_per_channel_128", "dg_quant_per_channel_128_pair",
    "dg_quant_block_128x128", "dg_quant_block_128x128_fp4", "dg_m_grouped_fp8_fp4_contiguous", "dg_m_grouped_fp8_fp4_masked",
    "dg_m_grouped_fp8_contiguous", "dg_m_grouped_fp8_masked", "dg_k_grouped_fp8_wgrad", "dg_fp8_gemm_nt",
    "dg_fp8_gemm_nt_batched",
    "dg_k_grouped_fp8_wgrad_noalloc", "dg_k_grouped_fp8_wgrad_from_bf16", "dg_k_grouped_fp8_wgrad_from_bf16_psum",
    "dg_workspace_size", "dg_last_error", "sfa_padded_rows", "empty_sfa", "kgrouped_workspace", "DGError",
]


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(cond, msg):
    if not cond:
        raise ValueError(msg)


def _dev(*ts):
    for t in ts:
        if t is not None:
            _need(t.is_cuda, "all tensors must be CUDA tensors")


def _sf_dtype(fmt):
    return torch.float32 if fmt == DG_SF_FP32 else torch.uint8


def sfa_padded_rows(M: int, sf_format: int) -> int:
    """Row count Mp of the MN-major per-token scale layout [K/128][Mp]."""
    return (M + 3) // 4 * 4 if sf_format == DG_SF_FP32 else (M + 15) // 16 * 16


def empty_sfa(M: int, K: int, sf_format: int, device) -> torch.Tensor:
    return torch.empty((K // 128, sfa_padded_rows(M, sf_format)), dtype=_sf_dtype(sf_format), device=device)


def dg_last_error() -> str:
    return load().dg_last_error().decode()


def dg_workspace_size(op: int, G: int, M: int = 0, N: int = 0, K: int = 0) -> int:
    return int(load().dg_workspace_size(op, G, M, N, K))


def kgrouped_workspace(G: int, device) -> torch.Tensor:
    return torch.empty(dg_workspace_size(DG_OP_K_GROUPED_WGRAD, G), dtype=torch.uint8, device=device)


def _token_cast_shapes(x, q, sfa, sf_format):
    _need(x.dim() == 2 and x.dtype == torch.bfloat16 and x.stride(1) == 1, "x must be a 2-D bf16 row-major view")
    M, K = x.shape
    _need(q.is_contiguous() and q.numel() == M * K and q.element_size() == 1, "q must be a contiguous 1-byte [M, K]")
    _need(sfa.is_contiguous() and sfa.dtype == _sf_dtype(sf_format)
          and sfa.numel() >= (K // 128) * sfa_padded_rows(M, sf_format), "sfa has the wrong dtype or size")
    return M, K


def dg_quant_per_token_1x128(x, q, sfa, sf_format=DG_SF_FP32, sf_zero=1e-30, row_counts=None, stream=None):
    """x bf16 [M, K] (row stride >= K) -> q e4m3/uint8 [M, K], sfa [K/128][Mp]."""
    _dev(x, q, sfa, row_counts)
    M, K = _token_cast_shapes(x, q, sfa, sf_format)
    G = 0
    if row_counts is not None:
        _need(row_counts.dtype == torch.int32 and row_counts.is_contiguous(), "row_counts must be int32")
        G = row_counts.numel()
    check(load().dg_quant_per_token_1x128(_p(x), M, K, x.stride(0), _p(q), _p(sfa), sf_format, sf_zero,
                                          _p(row_counts), G, _s(stream)))


def dg_quant_per_token_1x128_routed(x, q, sfa, m_indices, sf_format=DG_SF_FP32, sf_zero=1e-30, stream=None):
    """dg_quant_per_token_1x128 over the rows with m_indices >= 0 only (int32 [M]); the other rows
    of q and sfa are left as they were."""
    _dev(x, q, sfa, m_indices)
    M, K = _token_cast_shapes(x, q, sfa, sf_format)
    _need(m_indices.dtype == torch.int32 and m_indices.is_contiguous() and m_indices.numel() == M,
          "m_indices must be int32 [M]")
    check(load().dg_quant_per_token_1x128_routed(_p(x), M, K, x.stride(0), _p(q), _p(sfa), sf_format, sf_zero,
                                                 _p(m_indices), _s(stream)))


def dg_quant_per_token_1x128_packed(x, q, sfa, row_counts, sf_format=DG_SF_FP32, sf_zero=1e-30, stream=None):
    """The masked cast from packed rows: x bf16 [G*cap, K] holds each group's valid rows packed at
    its front, group after group; q e4m3/uint8 [G, cap, K] (or [G*cap, K]), sfa [K/128][Mp]
    (Mp from G*cap) receive them at the masked positions; row_counts int32 [G]."""
    _dev(x, q, sfa, row_counts)
    _need(row_counts.dtype == torch.int32 and row_counts.is_contiguous(), "row_counts must be int32")
    G = row_counts.numel()
    qq = q.view(-1, q.shape[-1])
    _need(G >= 1 and qq.shape[0] % G == 0, "q rows must be G x cap")
    cap = qq.shape[0] // G
    M, K = _token_cast_shapes(x, qq, sfa, sf_format)
    _need(M == G * cap, "x must have G x cap rows")
    check(load().dg_quant_per_token_1x128_packed(_p(x), K, x.stride(0), _p(qq), _p(sfa), sf_format, sf_zero,
                                                 _p(row_counts), G, cap, _s(stream)))


def dg_pack_masked_rows(src, counts, dst, stream=None):
    """src [G, cap, ...] (contiguous) -> dst (capacity G*cap rows of the same row size): each
    group's first clamp(count, 0, cap) rows, packed group after group; counts int32 [G]."""
    _dev(src, counts, dst)
    _need(src.is_contiguous() and dst.is_contiguous() and src.dim() >= 2, "contiguous src [G, cap, ...] and dst")
    G, cap = src.shape[0], src.shape[1]
    _need(counts.dtype == torch.int32 and counts.numel() == G, "counts must be int32 [G]")
    row_bytes = src[0, 0].numel() * src.element_size() if cap > 0 else 0
    _need(dst.numel() * dst.element_size() >= G * cap * row_bytes, "dst must hold G x cap rows")
    check(load().dg_pack_masked_rows(_p(src), G, cap, row_bytes, _p(counts), _p(dst), _s(stream)))


def dg_quant_per_channel_128(x, ks, q_packed, sf, sf_zero=1e-30, status=None, stream=None, _fn="dg_quant_per_channel_128"):
    """x bf16 [K_cap, C] token-major -> q_packed [K_cap*C] per-expert K-major, sf fp32 [K_cap/128][C]."""
    _dev(x, ks, q_packed, sf, status)
    _need(x.dim() == 2 and x.dtype == torch.bfloat16 and x.is_contiguous(), "x must be contiguous bf16 [K_cap, C]")
    K_cap, C = x.shape
    _need(ks.dtype == torch.int32 and ks.is_contiguous(), "ks must be int32")
    _need(q_packed.is_contiguous() and q_packed.numel() >= K_cap * C and q_packed.element_size() == 1, "q_packed size")
    _need(sf.is_contiguous() and sf.dtype == torch.float32 and sf.numel() >= (K_cap // 128) * C, "sf size")
    check(getattr(load(), _fn)(_p(x), K_cap, C, _p(ks), ks.numel(), _p(q_packed), _p(sf), sf_zero, _p(status),
                               _s(stream)))


def dg_quant_per_channel_128_psum(x, psum, q_packed, sf, sf_zero=1e-30, status=None, stream=None):
    """dg_quant_per_channel_128 with expert spans as inclusive prefix sums psum int32 [G]."""
    dg_quant_per_channel_128(x, psum, q_packed, sf, sf_zero, status, stream, _fn="dg_quant_per_channel_128_psum")


def dg_quant_per_channel_128_pair(x_a, x_b, ks, q_a, sf_a, q_b, sf_b, sf_zero=1e-30, status=None, stream=None,
                                  _fn="dg_quant_per_channel_128_pair"):
    """Both wgrad operands in one launch: same results as two dg_quant_per_channel_128 calls."""
    _dev(x_a, x_b, ks, q_a, sf_a, q_b, sf_b, status)
    for x, q, sf in ((x_a, q_a, sf_a), (x_b, q_b, sf_b)):
        _need(x.dim() == 2 and x.dtype == torch.bfloat16 and x.is_contiguous(), "x must be contiguous bf16 [K_cap, C]")
        _need(q.is_contiguous() and q.numel() >= x.numel() and q.element_size() == 1, "q size")
        _need(sf.is_contiguous() and sf.dtype == torch.float32 and sf.numel() >= x.numel() // 128, "sf size")
    _need(x_a.shape[0] == x_b.shape[0], "both operands need the same K_cap")
    _need(ks.dtype == torch.int32 and ks.is_contiguous(), "ks must be int32")
    check(getattr(load(), _fn)(_p(x_a), x_a.shape[1], _p(q_a), _p(sf_a), _p(x_b), x_b.shape[1], _p(q_b), _p(sf_b),
                               x_a.shape[0], _p(ks), ks.numel(), sf_zero, _p(status), _s(stream)))


def dg_quant_per_channel_128_pair_psum(x_a, x_b, psum, q_a, sf_a, q_b, sf_b, sf_zero=1e-30, status=None, stream=None):
    """dg_quant_per_channel_128_pair with expert spans as inclusive prefix sums psum int32 [G]."""
    dg_quant_per_channel_128_pair(x_a, x_b, psum, q_a, sf_a, q_b, sf_b, sf_zero, status, stream,
                                  _fn="dg_quant_per_channel_128_pair_psum")


def dg_quant_block_128x128(w, q, sfb, sf_format=DG_SF_FP32, sf_zero=1e-30, stream=None):
    """w bf16 [G, N, K] -> q [G, N, K], sfb [G][N/128][K/128]."""
    _dev(w, q, sfb)
    _need(w.dim() == 3 and w.dtype == torch.bfloat16 and w.is_contiguous(), "w must be contiguous bf16 [G, N, K]")
    G, N, K = w.shape
    _need(q.is_contiguous() and q.numel() == G * N * K and q.element_size() == 1, "q size")
    _need(sfb.is_contiguous() and sfb.dtype == _sf_dtype(sf_format)
          and sfb.numel() >= G * (N // 128) * (K // 128), "sfb has the wrong dtype or size")
    check(load().dg_quant_block_128x128(_p(w), G, N, K, _p(q), _p(sfb), sf_format, sf_zero, _s(stream)))


def dg_quant_block_128x128_fp4(w, q_packed, sfb, sf_zero=1e-30, stream=None):
    """w bf16 [G, N, K] -> FP4 codes q_packed uint8 [G, N, K/2] (two per byte, the even element in the
    low nibble) and UE8M0 block scales sfb uint8 [G][N/128][K/128]."""
    _dev(w, q_packed, sfb)
    _need(w.dim() == 3 and w.dtype == torch.bfloat16 and w.is_contiguous(), "w must be contiguous bf16 [G, N, K]")
    G, N, K = w.shape
    _need(q_packed.is_contiguous() and q_packed.dtype == torch.uint8 and q_packed.numel() == G * N * K // 2,
          "q_packed must be uint8 [G, N, K/2]")
    _need(sfb.is_contiguous() and sfb.dtype == torch.uint8 and sfb.numel() >= G * (N // 128) * (K // 128),
          "sfb must be uint8 [G][N/128][K/128]")
    check(load().dg_quant_block_128x128_fp4(_p(w), G, N, K, _p(q_packed), _p(sfb), sf_zero, _s(stream)))


def _out_code(d):
    if d.dtype == torch.bfloat16:
        return DG_OUT_BF16
    _need(d.dtype == torch.float32, "d must be bf16 or fp32")
    return DG_OUT_FP32


def dg_m_grouped_fp8_contiguous(a, sfa, b, sfb, d, m_indices, sf_format=DG_SF_FP32, status=None, workspace=None,
                                stream=None, _psum=False):
    """a [M, K] e4m3, b [G, N, K] e4m3, d [M, N] bf16/fp32, m_indices int32 [M]."""
    _dev(a, sfa, b, sfb, d, m_indices, status)
    M, K = a.shape
    G, N, K2 = b.shape
    _need(K == K2 and tuple(d.shape) == (M, N) and d.is_contiguous() and a.is_contiguous() and b.is_contiguous(),
          "shapes")
    if _psum:
        _need(m_indices.dtype == torch.int32 and m_indices.numel() == G, "psum must be int32 [G]")
    else:
        _need(m_indices.dtype == torch.int32 and m_indices.numel() == M, "m_indices must be int32 [M]")
    _need(sfa.dtype == _sf_dtype(sf_format) and sfb.dtype == _sf_dtype(sf_format), "scale dtype")
    _need(sfa.numel() >= (K // 128) * sfa_padded_rows(M, sf_format), "sfa size")
    _need(sfb.numel() >= G * (N // 128) * (K // 128), "sfb size")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    fn = load().dg_m_grouped_fp8_contiguous_psum if _psum else load().dg_m_grouped_fp8_contiguous
    check(fn(_p(a), _p(sfa), _p(b), _p(sfb), _p(d), _out_code(d), _p(m_indices), M, G, N, K, sf_format, _p(workspace),
             ws_bytes, _p(status), _s(stream)))


def dg_m_grouped_fp8_contiguous_psum(a, sfa, b, sfb, d, psum, sf_format=DG_SF_FP32, status=None, workspace=None,
                                     stream=None):
    """dg_m_grouped_fp8_contiguous routed by psum int32 [G]: expert e owns rows
    [round_up(psum[e-1], 128), psum[e])."""
    dg_m_grouped_fp8_contiguous(a, sfa, b, sfb, d, psum, sf_format, status, workspace, stream, _psum=True)


def dg_fp8_gemm_nt(a, sfa, b, sfb, d, c=None, sf_format=DG_SF_FP32, status=None, stream=None):
    """Plain FP8 GEMM: d [M, N] = c + a [M, K] . b [N, K]^T (c optional fp32, may be d)."""
    _dev(a, sfa, b, sfb, d, c, status)
    _need(a.dim() == 2 and b.dim() == 2 and a.shape[1] == b.shape[1], "a [M, K], b [N, K]")
    M, K = a.shape
    N = b.shape[0]
    _need(tuple(d.shape) == (M, N) and a.is_contiguous() and b.is_contiguous() and d.is_contiguous(), "d [M, N]")
    _need(sfa.dtype == _sf_dtype(sf_format) and sfb.dtype == _sf_dtype(sf_format), "scale dtype")
    _need(sfa.numel() >= (K // 128) * sfa_padded_rows(M, sf_format), "sfa size")
    _need(sfb.numel() >= (N // 128) * (K // 128), "sfb size")
    if c is not None:
        _need(c.dtype == torch.float32 and tuple(c.shape) == (M, N) and c.is_contiguous(), "c fp32 [M, N]")
    check(load().dg_fp8_gemm_nt(_p(a), _p(sfa), _p(b), _p(sfb), _p(c), _p(d), _out_code(d), M, N, K, sf_format,
                                _p(status), _s(stream)))


def dg_fp8_gemm_nt_batched(a, sfa, b, sfb, d, c=None, sf_format=DG_SF_FP32, status=None, stream=None):
    """Batched FP8 GEMM: d [B, M, N] = c + a [B, M, K] . b [B, N, K]^T per batch entry."""
    _dev(a, sfa, b, sfb, d, c, status)
    _need(a.dim() == 3 and b.dim() == 3 and a.shape[0] == b.shape[0] and a.shape[2] == b.shape[2], "shapes")
    Bt, M, K = a.shape
    N = b.shape[1]
    _need(tuple(d.shape) == (Bt, M, N) and a.is_contiguous() and b.is_contiguous() and d.is_contiguous(),
          "d [B, M, N]")
    _need(sfa.dtype == _sf_dtype(sf_format) and sfb.dtype == _sf_dtype(sf_format), "scale dtype")
    _need(sfa.numel() >= (K // 128) * sfa_padded_rows(Bt * M, sf_format), "sfa size")
    _need(sfb.numel() >= Bt * (N // 128) * (K // 128), "sfb size")
    if c is not None:
        _need(c.dtype == torch.float32 and tuple(c.shape) == (Bt, M, N) and c.is_contiguous(), "c fp32 [B, M, N]")
    check(load().dg_fp8_gemm_nt_batched(_p(a), _p(sfa), _p(b), _p(sfb), _p(c), _p(d), _out_code(d), Bt, M, N, K,
                                        sf_format, _p(status), _s(stream)))


def dg_m_grouped_fp8_fp4_contiguous(a, sfa, b_packed, sfb, d, m_indices, status=None, stream=None):
    """a [M, K] e4m3 with UE8M0 sfa, b_packed [G, N, K/2] FP4 codes with UE8M0 sfb, d [M, N] bf16/fp32,
    m_indices int32 [M]."""
    _dev(a, sfa, b_packed, sfb, d, m_indices, status)
    M, K = a.shape
    G, N, K2 = b_packed.shape
    _need(K == 2 * K2 and tuple(d.shape) == (M, N) and d.is_contiguous() and a.is_contiguous()
          and b_packed.is_contiguous(), "shapes")
    _need(m_indices.dtype == torch.int32 and m_indices.numel() == M, "m_indices must be int32 [M]")
    _need(sfa.dtype == torch.uint8 and sfb.dtype == torch.uint8, "UE8M0 scales are uint8")
    _need(sfa.numel() >= (K // 128) * sfa_padded_rows(M, 1), "sfa size")
    _need(sfb.numel() >= G * (N // 128) * (K // 128), "sfb size")
    check(load().dg_m_grouped_fp8_fp4_contiguous(_p(a), _p(sfa), _p(b_packed), _p(sfb), _p(d), _out_code(d),
                                                 _p(m_indices), M, G, N, K, _p(status), _s(stream)))


def dg_m_grouped_fp8_fp4_masked(a, sfa, b_packed, sfb, d, counts, expected_m=0, status=None, stream=None):
    """a [G, cap, K] e4m3 with UE8M0 sfa, b_packed [G, N, K/2] FP4 codes with UE8M0 sfb,
    d [G, cap, N] bf16/fp32, counts int32 [G]."""
    _dev(a, sfa, b_packed, sfb, d, counts, status)
    G, cap, K = a.shape
    G2, N, K2 = b_packed.shape
    _need(G == G2 and K == 2 * K2 and tuple(d.shape) == (G, cap, N), "shapes")
    _need(a.is_contiguous() and b_packed.is_contiguous() and d.is_contiguous(), "contiguity")
    _need(counts.dtype == torch.int32 and counts.numel() == G, "counts must be int32 [G]")
    _need(sfa.dtype == torch.uint8 and sfb.dtype == torch.uint8, "UE8M0 scales are uint8")
    _need(sfa.numel() >= (K // 128) * sfa_padded_rows(G * cap, 1), "sfa size")
    _need(sfb.numel() >= G * (N // 128) * (K // 128), "sfb size")
    check(load().dg_m_grouped_fp8_fp4_masked(_p(a), _p(sfa), _p(b_packed), _p(sfb), _p(d), _out_code(d), _p(counts),
                                             G, cap, N, K, int(expected_m), _p(status), _s(stream)))


def dg_m_grouped_fp8_masked(a, sfa, b, sfb, d, counts, expected_m=0, sf_format=DG_SF_FP32, status=None,
                            workspace=None, stream=None):
    """a [G, cap, K] e4m3, b [G, N, K] e4m3, d [G, cap, N] bf16/fp32, counts int32 [G]."""
    _dev(a, sfa, b, sfb, d, counts, status)
    G, cap, K = a.shape
    G2, N, K2 = b.shape
    _need(G == G2 and K == K2 and tuple(d.shape) == (G, cap, N), "shapes")
    _need(a.is_contiguous() and b.is_contiguous() and d.is_contiguous(), "contiguity")
    _need(counts.dtype == torch.int32 and counts.numel() == G, "counts must be int32 [G]")
    _need(sfa.dtype == _sf_dtype(sf_format) and sfb.dtype == _sf_dtype(sf_format), "scale dtype")
    _need(sfa.numel() >= (K // 128) * sfa_padded_rows(G * cap, sf_format), "sfa size")
    _need(sfb.numel() >= G * (N // 128) * (K // 128), "sfb size")
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    check(load().dg_m_grouped_fp8_masked(_p(a), _p(sfa), _p(b), _p(sfb), _p(d), _out_code(d), _p(counts), G, cap, N,
                                         K, int(expected_m), sf_format, _p(workspace), ws_bytes, _p(status),
                                         _s(stream)))


def dg_m_grouped_bf16_masked(a, b, d, counts, expected_m=0, status=None, stream=None):
    """a [G, cap, K] bf16, b [G, N, K] bf16, d [G, cap, N] bf16/fp32, counts int32 [G]."""
    _dev(a, b, d, counts, status)
    G, cap, K = a.shape
    G2, N, K2 = b.shape
    _need(G == G2 and K == K2 and tuple(d.shape) == (G, cap, N), "shapes")
    _need(a.dtype == torch.bfloat16 and b.dtype == torch.bfloat16, "a and b must be bf16")
    _need(a.is_contiguous() and b.is_contiguous() and d.is_contiguous(), "contiguity")
    _need(counts.dtype == torch.int32 and counts.numel() == G, "counts must be int32 [G]")
    check(load().dg_m_grouped_bf16_masked(_p(a), _p(b), _p(d), _out_code(d), _p(counts), G, cap, N, K,
                                          int(expected_m), _p(status), _s(stream)))


def dg_m_grouped_bf16_contiguous(a, b, d, m_indices, status=None, stream=None):
    """a [M, K] bf16, b [G, N, K] bf16, d [M, N] bf16/fp32, m_indices int32 [M] (-1 = padding)."""
    _dev(a, b, d, m_indices, status)
    M, K = a.shape
    G, N, K2 = b.shape
    _need(K == K2 and tuple(d.shape) == (M, N), "shapes")
    _need(a.dtype == torch.bfloat16 and b.dtype == torch.bfloat16, "a and b must be bf16")
    _need(a.is_contiguous() and b.is_contiguous() and d.is_contiguous(), "contiguity")
    _need(m_indices.dtype == torch.int32 and m_indices.numel() == M, "m_indices must be int32 [M]")
    check(load().dg_m_grouped_bf16_contiguous(_p(a), _p(b), _p(d), _out_code(d), _p(m_indices), M, G, N, K,
                                              _p(status), _s(stream)))


def dg_k_grouped_fp8_wgrad(a_packed, sfa, b_packed, sfb, c, d, ks, K_cap, workspace, status=None, stream=None,
                           _fn="dg_k_grouped_fp8_wgrad"):
    """D_e = C_e + A_e^T B_e.  a_packed/b_packed: per-expert K-major codes; sfa [K_cap/128][N],
    sfb [K_cap/128][H]; c (or None, may be d) and d fp32 [G, N, H]; ks int32 [G]."""
    _dev(a_packed, sfa, b_packed, sfb, c, d, ks, workspace, status)
    G, N, H = d.shape
    _need(d.dtype == torch.float32 and d.is_contiguous(), "d must be contiguous fp32 [G, N, H]")
    _need(c is None or (tuple(c.shape) == tuple(d.shape) and c.dtype == torch.float32 and c.is_contiguous()), "c")
    _need(ks.dtype == torch.int32 and ks.numel() == G, "ks must be int32 [G]")
    _need(sfa.dtype == torch.float32 and sfa.numel() >= (K_cap // 128) * N, "sfa")
    _need(sfb.dtype == torch.float32 and sfb.numel() >= (K_cap // 128) * H, "sfb")
    _need(a_packed.numel() >= K_cap * N and b_packed.numel() >= K_cap * H, "packed operand size")
    ws_bytes = workspace.numel() * workspace.element_size()
    check(getattr(load(), _fn)(_p(a_packed), _p(sfa), _p(b_packed), _p(sfb), _p(c), _p(d), _p(ks), G, K_cap, N, H,
                               _p(workspace), ws_bytes, _p(status), _s(stream)))


def dg_k_grouped_fp8_wgrad_from_bf16(grad_y, act, ks, a_packed, sfa, b_packed, sfb, c, d, workspace, sf_zero=1e-30,
                                     status=None, stream=None, _fn="dg_k_grouped_fp8_wgrad_from_bf16"):
    """The whole wgrad from bf16: per-channel casts and packs of grad_y [K_cap, N] and act
    [K_cap, H] into a_packed/sfa and b_packed/sfb (caller buffers, as dg_quant_per_channel_128_pair
    fills them), then D_e = C_e + A_e^T B_e (c may be None or d) -- two launches."""
    _dev(grad_y, act, ks, a_packed, sfa, b_packed, sfb, c, d, workspace, status)
    G, N, H = d.shape
    _need(grad_y.dim() == 2 and act.dim() == 2 and grad_y.shape[0] == act.shape[0], "grad_y [K_cap, N], act [K_cap, H]")
    K_cap = grad_y.shape[0]
    _need(grad_y.shape[1] == N and act.shape[1] == H, "grad_y / act columns must match d's N and H")
    _need(grad_y.dtype == torch.bfloat16 and act.dtype == torch.bfloat16 and grad_y.is_contiguous()
          and act.is_contiguous(), "grad_y and act must be contiguous bf16")
    _need(d.dtype == torch.float32 and d.is_contiguous(), "d must be contiguous fp32 [G, N, H]")
    _need(c is None or (tuple(c.shape) == tuple(d.shape) and c.dtype == torch.float32 and c.is_contiguous()), "c")
    _need(ks.dtype == torch.int32 and ks.numel() == G, "ks must be int32 [G]")
    _need(sfa.dtype == torch.float32 and sfa.numel() >= (K_cap // 128) * N, "sfa")
    _need(sfb.dtype == torch.float32 and sfb.numel() >= (K_cap // 128) * H, "sfb")
    _need(a_packed.numel() >= K_cap * N and b_packed.numel() >= K_cap * H, "packed operand size")
    ws_bytes = workspace.numel() * workspace.element_size()
    check(getattr(load(), _fn)(_p(grad_y), _p(act), _p(ks), G, K_cap, N, H, _p(a_packed), _p(sfa), _p(b_packed),
                               _p(sfb), _p(c), _p(d), sf_zero, _p(workspace), ws_bytes, _p(status), _s(stream)))


def dg_k_grouped_fp8_wgrad_from_bf16_psum(grad_y, act, psum, a_packed, sfa, b_packed, sfb, c, d, workspace,
                                          sf_zero=1e-30, status=None, stream=None):
    """dg_k_grouped_fp8_wgrad_from_bf16 with expert spans as inclusive prefix sums psum int32 [G]."""
    dg_k_grouped_fp8_wgrad_from_bf16(grad_y, act, psum, a_packed, sfa, b_packed, sfb, c, d, workspace, sf_zero,
                                     status, stream, _fn="dg_k_grouped_fp8_wgrad_from_bf16_psum")


def dg_k_grouped_fp8_wgrad_psum(a_packed, sfa, b_packed, sfb, c, d, psum, K_cap, workspace, status=None, stream=None):
    """dg_k_grouped_fp8_wgrad with expert spans as inclusive prefix sums psum int32 [G]."""
    dg_k_grouped_fp8_wgrad(a_packed, sfa, b_packed, sfb, c, d, psum, K_cap, workspace, status, stream,
                           _fn="dg_k_grouped_fp8_wgrad_psum")


def dg_k_grouped_fp8_wgrad_noalloc(a_packed, sfa, b_packed, sfb, c, d, ks, K_cap, status=None, stream=None):
    """dg_k_grouped_fp8_wgrad for callers that cannot allocate device memory: no workspace
    argument; the library's built-in descriptor scratch (at most DG_NOALLOC_MAX_GROUPS experts)
    is shared by all calls, so calls that may overlap on the GPU must be serialised."""
    _dev(a_packed, sfa, b_packed, sfb, c, d, ks, status)
    G, N, H = d.shape
    _need(d.dtype == torch.float32 and d.is_contiguous(), "d must be contiguous fp32 [G, N, H]")
    _need(c is None or (tuple(c.shape) == tuple(d.shape) and c.dtype == torch.float32 and c.is_contiguous()), "c")
    _need(ks.dtype == torch.int32 and ks.numel() == G, "ks must be int32 [G]")
    _need(sfa.dtype == torch.float32 and sfa.numel() >= (K_cap // 128) * N, "sfa")
    _need(sfb.dtype == torch.float32 and sfb.numel() >= (K_cap // 128) * H, "sfb")
    _need(a_packed.numel() >= K_cap * N and b_packed.numel() >= K_cap * H, "packed operand size")
    check(load().dg_k_grouped_fp8_wgrad_noalloc(_p(a_packed), _p(sfa), _p(b_packed), _p(sfb), _p(c), _p(d), _p(ks),
                                                G, K_cap, N, H, _p(status), _s(stream)))


# ---- debug aids

def dg_set_arg_log(path: str | None) -> None:
    """Append one line per entry-point call (name and arguments) to `path`; None stops it."""
    check(load().dg_set_arg_log(None if not path else str(path).encode()))


def dg_debug_build() -> bool:
    """True when the loaded library is the debug build (kernels check their computed indices)."""
    return bool(load().dg_debug_build())


def dg_debug_word(clear: bool = True) -> int:
    """Waits for the current device, then returns the DG_DEBUG_* bits the debug build's index
    checks raised since the last clear (always 0 for the release build)."""
    w = ctypes.c_uint32(0)
    check(load().dg_debug_word(ctypes.byref(w), 1 if clear else 0))
    return int(w.value)
