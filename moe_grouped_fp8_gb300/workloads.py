"""Seeded synthetic inputs shaped like the workloads of the source pages.

This module is the only code that the CUDA path's tests and the CPU oracle share.  It holds
no quantization, scaling or GEMM arithmetic: only random draws (bf16 tensors, expert routing)
and the layout bookkeeping that turns per-expert counts into routing tensors.

Recipes (all seeded; the same bytes feed the GPU and, copied to the host, the oracle):

* masked repro ("Fix cross-expert output overwrites in SM90 masked GEMM", reproduction):
  G=8, cap=32, N=K=256, counts [0,1,16,31,32,1,32,32], A and B ~ randn bf16, seed 29.
* k-grouped wgrad ("Non-deterministic numerical problem of k_grouped_fp8_gemm_nt_contiguous",
  repro listing): Ks=[256,128,128,256], grad_y = randn*1e-7 and act = randn*0.4 (bf16,
  [768, 2048] each), channel 0 of grad_y zeroed inside every 128-token expert, seed 0.
* contiguous prefill: G=32, N=4096, K=7168, 8192 tokens routed top-1 with Zipf(s=1.1)
  expert probabilities over a seeded permutation of the experts; each expert's segment is
  padded to a multiple of 128 rows with m_indices = -1; B = randn*0.02.  Seed 1003.
* masked decode (the largest shape of the #469 performance table): G=32, cap=4096,
  N=6144, K=7168, counts ~ Poisson(192) clipped to [0, cap].  Seed 1004.
* many-expert UE8M0 contiguous ("SM120 m_grouped_fp8 contiguous kernel ... graph replay",
  environment): G=288, w13 N=512 K=4096 and w2 N=4096 K=256, T = 288*E tokens drawn
  multinomially over uniform experts for E in {1, 32, 113}; the buffer holds
  T + 288*127 rows so that any draw fits.  Seed 1005.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 128  # segment alignment of the contiguous layout and the K granularity


def randn_bf16(shape, seed: int, scale: float = 1.0, device="cpu") -> torch.Tensor:
    """randn * scale drawn in fp32 from a seeded torch generator on `device`, rounded once
    to bf16."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    x = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


# ------------------------------------------------------------------------------ routing

def zipf_counts(T: int, G: int, s: float, seed: int) -> np.ndarray:
    """Top-1 routing of T tokens with p(rank r) ~ r^-s, ranks assigned to experts by a
    seeded permutation.  Returns counts[G] (sum T)."""
    rng = np.random.default_rng(seed)
    p = np.arange(1, G + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    perm = rng.permutation(G)
    probs = np.empty(G)
    probs[perm] = p
    return rng.multinomial(T, probs).astype(np.int32)


def poisson_counts(G: int, lam: float, cap: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return np.clip(rng.poisson(lam, G), 0, cap).astype(np.int32)


def multinomial_counts(T: int, G: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.multinomial(T, np.full(G, 1.0 / G)).astype(np.int32)


def contiguous_psum(counts, align: int = BLOCK) -> np.ndarray:
    """The expert segments of contiguous_m_indices as per-expert end rows: expert e's rows start
    at the previous end rounded up to `align` and end at start + counts[e]."""
    psum = np.empty(len(counts), np.int32)
    start = 0
    for e, c in enumerate(np.asarray(counts, np.int64)):
        psum[e] = start + c
        start += (int(c) + align - 1) // align * align
    return psum


def contiguous_m_indices(counts, m_max: int | None = None, align: int = BLOCK) -> np.ndarray:
    """Stack expert segments in expert order, each padded to a multiple of `align` rows with
    -1; the buffer is m_max rows (default: the padded total), tail rows -1."""
    counts = np.asarray(counts, np.int64)
    padded = (counts + align - 1) // align * align
    total = int(padded.sum())
    if m_max is None:
        m_max = total
    assert m_max >= total, (m_max, total)
    mi = np.full(m_max, -1, np.int32)
    off = 0
    for e, (c, p) in enumerate(zip(counts, padded)):
        mi[off:off + c] = e
        off += int(p)
    return mi


def contiguous_capacity(T: int, G: int, align: int = BLOCK) -> int:
    """Rows a contiguous buffer needs so that any routing of T tokens over G experts fits."""
    return T + G * (align - 1)


# ------------------------------------------------------------------------------ workloads

@dataclass
class Masked:
    G: int
    cap: int
    N: int
    K: int
    counts: np.ndarray
    seed: int
    a_scale: float = 1.0
    b_scale: float = 1.0
    name: str = "masked"
    expected_m: int = 0  # the caller's hint of rows per group (what a decode step passes)

    def draw(self, device="cpu"):
        a = randn_bf16((self.G, self.cap, self.K), self.seed, self.a_scale, device)
        b = randn_bf16((self.G, self.N, self.K), self.seed + 1, self.b_scale, device)
        return a, b

    @property
    def valid_rows(self) -> int:
        return int(np.clip(self.counts, 0, self.cap).sum())

    @property
    def flops(self) -> float:
        return 2.0 * self.valid_rows * self.N * self.K


@dataclass
class Contiguous:
    G: int
    N: int
    K: int
    counts: np.ndarray
    m_max: int
    seed: int
    a_scale: float = 1.0
    b_scale: float = 1.0
    ue8m0: bool = False
    name: str = "contiguous"

    @property
    def m_indices(self) -> np.ndarray:
        return contiguous_m_indices(self.counts, self.m_max)

    def draw(self, device="cpu"):
        a = randn_bf16((self.m_max, self.K), self.seed, self.a_scale, device)
        b = randn_bf16((self.G, self.N, self.K), self.seed + 1, self.b_scale, device)
        return a, b

    @property
    def valid_rows(self) -> int:
        return int(np.asarray(self.counts).sum())

    @property
    def flops(self) -> float:
        return 2.0 * self.valid_rows * self.N * self.K


@dataclass
class KGrouped:
    ks: list
    N: int
    H: int
    seed: int
    gy_scale: float = 1e-7
    act_scale: float = 0.4
    zero_channel_in_128_experts: bool = True
    name: str = "kgrouped"

    @property
    def T(self) -> int:
        return int(sum(self.ks))

    @property
    def offsets(self) -> list:
        out, o = [], 0
        for k in self.ks:
            out.append(o)
            o += k
        return out

    def draw(self, device="cpu"):
        """grad_y [T, N] and act [T, H], bf16, token-major (the repro's draw order)."""
        gy = randn_bf16((self.T, self.N), self.seed, self.gy_scale, device)
        act = randn_bf16((self.T, self.H), self.seed + 1, self.act_scale, device)
        if self.zero_channel_in_128_experts:
            for o, k in zip(self.offsets, self.ks):
                if k == BLOCK:
                    gy[o:o + k, 0] = 0
        return gy, act

    @property
    def flops(self) -> float:
        return 2.0 * self.T * self.N * self.H


def masked_repro() -> Masked:
    return Masked(G=8, cap=32, N=256, K=256,
                  counts=np.array([0, 1, 16, 31, 32, 1, 32, 32], np.int32), seed=29)


def kgrouped_repro() -> KGrouped:
    return KGrouped(ks=[256, 128, 128, 256], N=2048, H=2048, seed=0)


def contiguous_prefill() -> Contiguous:
    G, T = 32, 8192
    counts = zipf_counts(T, G, 1.1, 1003)
    return Contiguous(G=G, N=4096, K=7168, counts=counts, m_max=contiguous_capacity(T, G),
                      seed=1003, b_scale=0.02)


def masked_decode() -> Masked:
    G, cap = 32, 4096
    return Masked(G=G, cap=cap, N=6144, K=7168, counts=poisson_counts(G, 192.0, cap, 1004),
                  seed=1004, b_scale=0.02, expected_m=192)


# Reduced cases for profiler captures: the per-expert shapes above with 8 experts, so that the
# inputs still exceed L2 (weights 235 / 352 MB) while a capture holds well under a few GB.
def contiguous_prefill_g8() -> Contiguous:
    G, T = 8, 2048
    counts = zipf_counts(T, G, 1.1, 1003)
    return Contiguous(G=G, N=4096, K=7168, counts=counts, m_max=contiguous_capacity(T, G),
                      seed=1003, b_scale=0.02, name="contiguous_prefill_g8")


def masked_decode_g8() -> Masked:
    G, cap = 8, 1024
    return Masked(G=G, cap=cap, N=6144, K=7168, counts=poisson_counts(G, 192.0, cap, 1004),
                  seed=1004, b_scale=0.02, expected_m=192, name="masked_decode_g8")


# Compute-bound shapes for the tensor-peak measurement: every expert holds the prefill's full
# 4096-token batch (no padding rows, no empty experts), N=4096, K=7168, 8 experts.
def contiguous_balanced() -> Contiguous:
    G, per = 8, 4096
    return Contiguous(G=G, N=4096, K=7168, counts=np.full(G, per, np.int32), m_max=G * per, seed=1006,
                      b_scale=0.02, name="contiguous_balanced")


def contiguous_balanced_ue8m0() -> Contiguous:
    """contiguous_balanced with UE8M0 scales on both operands (the scale format of the many-expert
    shapes on a compute-bound shape)."""
    G, per = 8, 4096
    return Contiguous(G=G, N=4096, K=7168, counts=np.full(G, per, np.int32), m_max=G * per, seed=1006,
                      b_scale=0.02, ue8m0=True, name="contiguous_balanced_ue8m0")


def masked_balanced() -> Masked:
    G, cap = 8, 4096
    return Masked(G=G, cap=cap, N=4096, K=7168, counts=np.full(G, cap, np.int32), seed=1007, b_scale=0.02,
                  expected_m=cap, name="masked_balanced")


def many_expert(E: int, which: str = "w13", seed: int = 1005) -> Contiguous:
    G = 288
    N, K = (512, 4096) if which == "w13" else (4096, 256)
    T = G * E
    counts = multinomial_counts(T, G, seed + E)
    return Contiguous(G=G, N=N, K=K, counts=counts, m_max=contiguous_capacity(T, G), seed=seed,
                      ue8m0=True, name=f"many_expert_{which}_E{E}")
