"""Guard regions around every output buffer: each output of each kernel family is a view into a
larger allocation whose bytes before and after it hold a fill pattern; after the call the pattern
must be intact (no store lands outside the buffer the layout defines).  Shapes have ragged
tails: rows that are not multiples of 128, counts at 0, 1, cap and past cap, the last expert
full."""
import numpy as np
import pytest
import torch

from moe_grouped_fp8_gb300 import DG_SF_FP32, DG_SF_UE8M0, _lib, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import gpu_quant_blocks, gpu_quant_tokens, sync

pytestmark = pytest.mark.gpu

GUARD = 4096   # bytes on each side (keeps every view 1024-byte aligned)
FILL = 0xA5


class Guarded:
    """`n` elements of `dtype` between two guard regions."""

    def __init__(self, shape, dtype):
        self.shape = tuple(shape)
        self.dtype = dtype
        esz = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = int(np.prod(self.shape)) * esz
        body = (self.nbytes + 1023) // 1024 * 1024
        self.base = torch.full((2 * GUARD + body,), FILL, dtype=torch.uint8, device="cuda")
        self.tail = GUARD + self.nbytes
        self.t = self.base[GUARD:GUARD + self.nbytes].view(dtype).view(self.shape)

    def check(self, what):
        sync()
        b = self.base.cpu().numpy()
        assert np.all(b[:GUARD] == FILL), f"{what}: bytes written before the buffer"
        assert np.all(b[self.tail:] == FILL), f"{what}: bytes written past the end of the buffer"


def test_guards_token_casts():
    for fmt in (DG_SF_FP32, DG_SF_UE8M0):
        M, K = 301, 384
        x = wl.randn_bf16((M, K), 1, 0.5, "cuda")
        q = Guarded((M, K), torch.uint8)
        sfa = Guarded((api.empty_sfa(M, K, fmt, "cpu").numel(),), api.empty_sfa(M, K, fmt, "cpu").dtype)
        api.dg_quant_per_token_1x128(x, q.t, sfa.t, fmt)
        q.check("plain cast q"), sfa.check("plain cast sfa")
        G, cap = 5, 41
        xm = wl.randn_bf16((G * cap, K), 2, 0.5, "cuda")
        cnt = torch.tensor([0, 41, 1, 60, 40], dtype=torch.int32, device="cuda")
        for packed in (False, True):
            q = Guarded((G * cap, K), torch.uint8)
            sfa = Guarded((api.empty_sfa(G * cap, K, fmt, "cpu").numel(),), api.empty_sfa(G * cap, K, fmt, "cpu").dtype)
            if packed:
                api.dg_quant_per_token_1x128_packed(xm, q.t, sfa.t, cnt, fmt)
            else:
                api.dg_quant_per_token_1x128(xm, q.t, sfa.t, fmt, row_counts=cnt)
            q.check(f"masked cast q packed={packed}"), sfa.check(f"masked cast sfa packed={packed}")
        mi = torch.tensor(wl.contiguous_m_indices([130, 0, 9], 401), dtype=torch.int32, device="cuda")
        xr = wl.randn_bf16((401, K), 3, 0.5, "cuda")
        q = Guarded((401, K), torch.uint8)
        sfa = Guarded((api.empty_sfa(401, K, fmt, "cpu").numel(),), api.empty_sfa(401, K, fmt, "cpu").dtype)
        api.dg_quant_per_token_1x128_routed(xr, q.t, sfa.t, mi, fmt)
        q.check("routed cast q"), sfa.check("routed cast sfa")


def test_guards_block_and_channel_casts():
    w = wl.randn_bf16((3, 256, 384), 4, 0.5, "cuda")
    for fmt in (DG_SF_FP32, DG_SF_UE8M0):
        q = Guarded((3, 256, 384), torch.uint8)
        sfb = Guarded((3, 2, 3), torch.float32 if fmt == DG_SF_FP32 else torch.uint8)
        api.dg_quant_block_128x128(w, q.t, sfb.t, fmt)
        q.check("block cast q"), sfb.check("block cast sfb")
    q = Guarded((3, 256, 192), torch.uint8)
    sfb = Guarded((3, 2, 3), torch.uint8)
    api.dg_quant_block_128x128_fp4(w, q.t, sfb.t)
    q.check("fp4 block cast q"), sfb.check("fp4 block cast sfb")
    K_cap, C = 768, 192
    x = wl.randn_bf16((K_cap, C), 5, 0.5, "cuda")
    ks = torch.tensor([256, 0, 128, 384], dtype=torch.int32, device="cuda")
    qp = Guarded((K_cap * C,), torch.uint8)
    sf = Guarded((K_cap // 128, C), torch.float32)
    api.dg_quant_per_channel_128(x, ks, qp.t, sf.t)
    qp.check("channel cast codes"), sf.check("channel cast scales")


@pytest.mark.parametrize("K", [512, 7168])
@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
def test_guards_masked_gemm(K, fmt):
    """Owner-thread stores (short K), staged TMA stores with owner tails (long K, fp32 scales), the
    block-scaled kernel (long K, UE8M0); counts past cap are clamped."""
    G, cap, N = 4, 201, 512
    a = wl.randn_bf16((G * cap, K), 6, 1.0, "cuda")
    b = wl.randn_bf16((G, N, K), 7, 1.0, "cuda")
    qa, sfa = gpu_quant_tokens(a, fmt)
    qb, sfb = gpu_quant_blocks(b, fmt)
    cnt = torch.tensor([201, 77, 0, 300], dtype=torch.int32, device="cuda")
    for out in (torch.bfloat16, torch.float32):
        d = Guarded((G, cap, N), out)
        api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d.t, cnt, 0, fmt)
        d.check(f"masked GEMM K={K} out={out}")
    pk = Guarded((G * cap, N), torch.bfloat16)
    d = Guarded((G, cap, N), torch.bfloat16)
    api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d.t, cnt, 0, fmt)
    api.dg_pack_masked_rows(d.t, cnt, pk.t)
    pk.check("pack masked rows")


def test_guards_contiguous_dense_batched_fp4_bf16():
    counts = [130, 0, 257, 5]
    M = wl.contiguous_capacity(sum(counts), len(counts))
    K, N = 1024, 384
    a = wl.randn_bf16((M, K), 8, 1.0, "cuda")
    b = wl.randn_bf16((4, N, K), 9, 1.0, "cuda")
    qa, sfa = gpu_quant_tokens(a, DG_SF_FP32)
    qb, sfb = gpu_quant_blocks(b, DG_SF_FP32)
    mi = torch.tensor(wl.contiguous_m_indices(counts, M), dtype=torch.int32, device="cuda")
    d = Guarded((M, N), torch.bfloat16)
    api.dg_m_grouped_fp8_contiguous(qa, sfa, qb, sfb, d.t, mi)
    d.check("contiguous GEMM")
    d = Guarded((M, N), torch.bfloat16)
    api.dg_m_grouped_fp8_contiguous_psum(qa, sfa, qb, sfb, d.t,
                                         torch.tensor(wl.contiguous_psum(counts), dtype=torch.int32, device="cuda"))
    d.check("contiguous psum GEMM")
    # plain GEMM with C in place, ragged M
    a = wl.randn_bf16((301, K), 10, 1.0, "cuda")
    qa, sfa = gpu_quant_tokens(a, DG_SF_FP32)
    d = Guarded((301, N), torch.float32)
    d.t.copy_(wl.randn_bf16((301, N), 11, 1.0, "cuda").float())
    api.dg_fp8_gemm_nt(qa, sfa, qb[0], sfb[0:1], d.t, d.t)
    d.check("plain GEMM, C in place")
    # batched
    a = wl.randn_bf16((3 * 70, K), 12, 1.0, "cuda")
    qa, sfa = gpu_quant_tokens(a, DG_SF_FP32)
    d = Guarded((3, 70, N), torch.bfloat16)
    api.dg_fp8_gemm_nt_batched(qa.view(3, 70, K), sfa, qb[:3], sfb[:3], d.t)
    d.check("batched GEMM")
    # FP8 x FP4 contiguous (N % 256 == 0)
    N4 = 256
    b4 = wl.randn_bf16((4, N4, K), 13, 1.0, "cuda")
    qb4 = torch.empty(4, N4, K // 2, dtype=torch.uint8, device="cuda")
    sb4 = torch.empty(4, N4 // 128, K // 128, dtype=torch.uint8, device="cuda")
    api.dg_quant_block_128x128_fp4(b4, qb4, sb4)
    a = wl.randn_bf16((M, K), 14, 1.0, "cuda")
    qa, sfa = gpu_quant_tokens(a, DG_SF_UE8M0)
    d = Guarded((M, N4), torch.bfloat16)
    api.dg_m_grouped_fp8_fp4_contiguous(qa, sfa, qb4, sb4, d.t, mi)
    d.check("FP8 x FP4 contiguous GEMM")
    # BF16 masked and contiguous
    ab = wl.randn_bf16((3, 90, 512), 15, 1.0, "cuda")
    bb = wl.randn_bf16((3, 256, 512), 16, 1.0, "cuda")
    for bn in (128, 256):
        _lib.check(_lib.load().dg_testing_bf16_bn(bn))
        try:
            d = Guarded((3, 90, 256), torch.bfloat16)
            api.dg_m_grouped_bf16_masked(ab, bb, d.t, torch.tensor([90, 0, 33], dtype=torch.int32, device="cuda"))
            d.check(f"BF16 masked GEMM, {bn}-column tiles")
        finally:
            _lib.check(_lib.load().dg_testing_bf16_bn(0))
    ac = wl.randn_bf16((M, 512), 17, 1.0, "cuda")
    bc = wl.randn_bf16((4, 256, 512), 18, 1.0, "cuda")
    d = Guarded((M, 256), torch.bfloat16)
    api.dg_m_grouped_bf16_contiguous(ac, bc, d.t, mi)
    d.check("BF16 contiguous GEMM")


def test_guards_kgrouped():
    kg = wl.kgrouped_repro()
    gy, act = kg.draw("cuda")
    G, N, H, K_cap = len(kg.ks), kg.N, kg.H, kg.T
    ks = torch.tensor(kg.ks, dtype=torch.int32, device="cuda")
    ap = Guarded((K_cap * N,), torch.uint8)
    bp = Guarded((K_cap * H,), torch.uint8)
    sa = Guarded((K_cap // 128, N), torch.float32)
    sb = Guarded((K_cap // 128, H), torch.float32)
    d = Guarded((G, N, H), torch.float32)
    d.t.zero_()
    api.dg_k_grouped_fp8_wgrad_from_bf16(gy, act, ks, ap.t, sa.t, bp.t, sb.t, d.t, d.t,
                                         api.kgrouped_workspace(G, "cuda"))
    for g_, what in ((ap, "packed A"), (bp, "packed B"), (sa, "A scales"), (sb, "B scales"), (d, "wgrad D")):
        g_.check(f"k-grouped {what}")
