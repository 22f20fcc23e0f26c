"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI binding, run the
oracle on the same bf16 bytes on the host, and compare (codes and scales bit-exact; outputs
by calc_diff and max error, with the thresholds of the acceptance criteria)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_SF_FP32, _lib, api

# Acceptance thresholds: calc_diff <= 2e-5 for bf16 outputs and <= 1e-6 for fp32 outputs, and
# max |err| <= 1e-2 * max |ref| on the valid elements.
CALC_DIFF_BF16 = 2e-5
CALC_DIFF_FP32 = 1e-6
MAX_ERR_REL = 1e-2
SENTINEL_BF16 = 0xFFFF  # an all-ones NaN pattern never produced by the kernels
SENTINEL_F32 = 0xFFFFFFFF


def sync():
    torch.cuda.synchronize()


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int32).cpu().numpy().view(np.uint32)


def sentinel_like(shape, dtype, device="cuda"):
    if dtype == torch.bfloat16:
        return torch.full(shape, -1, dtype=torch.int16, device=device).view(torch.bfloat16)
    return torch.full(shape, -1, dtype=torch.int32, device=device).view(torch.float32)


def out_bits(d: torch.Tensor) -> np.ndarray:
    return bf16_bits(d) if d.dtype == torch.bfloat16 else f32_bits(d)


def sentinel_value(dtype):
    return SENTINEL_BF16 if dtype == torch.bfloat16 else SENTINEL_F32


def to_f64(d: torch.Tensor) -> np.ndarray:
    return d.detach().double().cpu().numpy()


# ------------------------------------------------------------------------------ GPU side

def gpu_quant_tokens(x: torch.Tensor, fmt: int, sf_zero: float = 1e-30, row_counts=None):
    M, K = x.shape
    q = torch.zeros(M, K, dtype=torch.uint8, device=x.device)
    sfa = api.empty_sfa(M, K, fmt, x.device)
    sfa.zero_()
    api.dg_quant_per_token_1x128(x, q, sfa, fmt, sf_zero, row_counts)
    return q, sfa


def gpu_quant_blocks(w: torch.Tensor, fmt: int, sf_zero: float = 1e-30):
    G, N, K = w.shape
    q = torch.empty(G, N, K, dtype=torch.uint8, device=w.device)
    sfb = torch.empty(G, N // 128, K // 128, dtype=torch.float32 if fmt == DG_SF_FP32 else torch.uint8,
                      device=w.device)
    api.dg_quant_block_128x128(w, q, sfb, fmt, sf_zero)
    return q, sfb


def gpu_quant_channels(x: torch.Tensor, ks_dev: torch.Tensor, sf_zero: float = 1e-30, status=None):
    K_cap, C = x.shape
    qp = torch.zeros(K_cap * C, dtype=torch.uint8, device=x.device)
    sf = torch.zeros(K_cap // 128, C, dtype=torch.float32, device=x.device)
    api.dg_quant_per_channel_128(x, ks_dev, qp, sf, sf_zero, status)
    return qp, sf


def sfa_rows(sfa: torch.Tensor, M: int) -> np.ndarray:
    """[K/128][Mp] layout -> natural [M][K/128] (fp32 values or UE8M0 bytes)."""
    return sfa[:, :M].t().contiguous().cpu().numpy()


# ------------------------------------------------------------------------------ comparisons

def assert_close(gpu: np.ndarray, ref: np.ndarray, fp32_out: bool, what: str = ""):
    gpu = np.asarray(gpu, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    assert gpu.size == ref.size
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    if gpu.size == 0:
        return 0.0
    diff = oracle.calc_diff(gpu, ref)
    tol = CALC_DIFF_FP32 if fp32_out else CALC_DIFF_BF16
    assert diff <= tol, f"{what}: calc_diff {diff:.3e} > {tol:.0e}"
    max_ref = np.abs(ref).max()
    err = np.abs(gpu - ref).max()
    assert err <= MAX_ERR_REL * max_ref + 1e-300, f"{what}: max err {err:.3e} > 1e-2 * {max_ref:.3e}"
    return diff


def ref_out(d64: np.ndarray, fp32_out: bool) -> np.ndarray:
    """The oracle's fp64 result rounded to the output dtype (bf16: one RNE rounding)."""
    if fp32_out:
        return d64.astype(np.float32).astype(np.float64)
    return oracle.bf16_bits_to_f64(oracle.round_bf16(d64))


def set_mgrouped_kernel(which: str) -> None:
    """Test hook: the m-grouped kernel of later UE8M0-scale calls ("auto", "promotion" per-128-K fp32
    promotion, "mx" the block-scaled MMA kernel)."""
    lib = _lib.load()
    _lib.check(lib.dg_testing_mgrouped_kernel({"auto": 0, "promotion": 1, "mx": 2}[which]))


def set_mgrouped_warps(warps: int) -> None:
    """Test hook: promotion warps of 128 x 256 tiles (0 automatic, 8 or 16)."""
    lib = _lib.load()
    _lib.check(lib.dg_testing_mgrouped_warps(int(warps)))


def set_token_items_per_cta(items: int):
    """Testing hook: items per CTA of the per-token casts (0 restores the automatic choice)."""
    lib = _lib.load()
    _lib.check(lib.dg_testing_token_items_per_cta(int(items)))


def set_mgrouped_store(which: str) -> None:
    """Test hook: how the m-grouped kernel stores tiles ("auto"; TMA stores issued by "thread0" of
    the promotion warps; "direct" owner-thread stores)."""
    lib = _lib.load()
    _lib.check(lib.dg_testing_mgrouped_store({"auto": 0, "thread0": 1, "direct": 3}[which]))


def set_mgrouped_bn(bn: int) -> None:
    """Test hook: the single-CTA tile width (0 automatic, 128, or 256 where N allows)."""
    lib = _lib.load()
    _lib.check(lib.dg_testing_mgrouped_bn(int(bn)))
