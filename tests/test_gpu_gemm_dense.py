"""GPU parity of the plain and batched FP8 GEMMs (the pages' adjacent-path checks of ordinary
GEMM layouts, output dtypes and accumulation, and batched GEMM, in "Fix cross-expert output
overwrites in SM90 masked GEMM", validation) against the oracle's fp64 GEMM on the oracle's own
casts of the same bf16 bytes."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_SF_FP32, DG_SF_UE8M0, DGError, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import assert_close, gpu_quant_blocks, gpu_quant_tokens, out_bits, ref_out, sync, to_f64

pytestmark = pytest.mark.gpu


def quantized(a, b, fmt):
    """Device casts of a [R, K] and b [G, N, K], checked code-exact against the oracle's casts."""
    ue = fmt == DG_SF_UE8M0
    qa, sfa = gpu_quant_tokens(a.cuda(), fmt)
    qb, sfb = gpu_quant_blocks(b.cuda(), fmt)
    sync()
    oqa, osfa, _ = oracle.quant_per_token_1x128(a, ue8m0=ue)
    oqb, osfb, _ = oracle.quant_block_128x128(b, ue8m0=ue)
    np.testing.assert_array_equal(qa.cpu().numpy(), oqa)
    np.testing.assert_array_equal(qb.cpu().numpy(), oqb)
    return qa, sfa, qb, sfb, oqa, osfa, oqb, osfb


def dense_case(M, N, K, fmt=DG_SF_FP32, out=torch.bfloat16, accumulate=None, calls=1, seed=0):
    """accumulate: None, "c" (a separate fp32 C) or "inplace" (C is D)."""
    a = wl.randn_bf16((M, K), 700 + seed, 1.5)
    b = wl.randn_bf16((1, N, K), 701 + seed, 0.02)
    qa, sfa, qb, sfb, oqa, osfa, oqb, osfb = quantized(a, b, fmt)
    c_host = None
    c = None
    d = torch.empty(M, N, dtype=out, device="cuda")
    if accumulate is not None:
        c_host = torch.randn(M, N, dtype=torch.float32, generator=torch.Generator().manual_seed(702 + seed)) * 4
        if accumulate == "inplace":
            d.copy_(c_host.cuda())
            c = d
        else:
            c = c_host.cuda()
    first = None
    for i in range(calls):
        if accumulate == "inplace" and i > 0:
            d.copy_(c_host.cuda())
        api.dg_fp8_gemm_nt(qa, sfa, qb.view(N, K), sfb.view(N // 128, K // 128), d, c=c, sf_format=fmt)
        if calls > 1:
            bits = out_bits(d)
            if first is None:
                first = bits
            else:
                assert np.array_equal(bits, first), f"call {i} differs bitwise from call 0"
    sync()
    ref = oracle.gemm_batched(oqa[None], osfa[None], oqb, osfb,
                              None if c_host is None else c_host.double().numpy()[None])[0]
    fp32 = out == torch.float32
    assert_close(to_f64(d), ref_out(ref, fp32), fp32, "plain GEMM")
    return d


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (37, 384, 640), (300, 1024, 256), (1029, 256, 384)])
def test_plain_gemm(M, N, K, fmt):
    dense_case(M, N, K, fmt, seed=M)


@pytest.mark.parametrize("accumulate", ["c", "inplace"])
@pytest.mark.parametrize("M,N,K", [(130, 384, 512), (513, 256, 256)])
def test_plain_gemm_fp32_accumulate(M, N, K, accumulate):
    """D = C + A . B^T in fp32, with C a separate buffer or D itself."""
    dense_case(M, N, K, out=torch.float32, accumulate=accumulate, seed=M + 1)


@pytest.mark.parametrize("out,accumulate", [(torch.bfloat16, None), (torch.float32, None), (torch.float32, "c"),
                                          (torch.float32, "inplace")])
def test_plain_gemm_ue8m0_long_k(out, accumulate):
    """UE8M0 scales with K = 2304 (18 blocks) and N % 256 == 0: the block-scaled MMA kernel, bf16 and
    fp32 outputs, C added separately and in place, repeated calls bitwise equal."""
    dense_case(261, 768, 2304, DG_SF_UE8M0, out=out, accumulate=accumulate, calls=3, seed=17)


def test_plain_gemm_fp32_out_and_repeat_bitwise():
    dense_case(200, 512, 768, out=torch.float32, calls=8, seed=5)
    dense_case(200, 1024, 768, out=torch.bfloat16, calls=8, seed=6)


def test_plain_gemm_empty_and_argument_errors():
    qa = torch.zeros(0, 128, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(0, 128, DG_SF_FP32, "cuda")
    qb = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    sfb = torch.ones(1, 1, dtype=torch.float32, device="cuda")
    api.dg_fp8_gemm_nt(qa, sfa, qb, sfb, torch.empty(0, 128, dtype=torch.bfloat16, device="cuda"))
    qa = torch.zeros(8, 128, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(8, 128, DG_SF_FP32, "cuda")
    d = torch.empty(8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(DGError):  # accumulation needs fp32 output
        api.dg_fp8_gemm_nt(qa, sfa, qb, sfb, d, c=torch.zeros(8, 128, dtype=torch.float32, device="cuda"))
    sync()


@pytest.mark.parametrize("fmt,out,accumulate", [(DG_SF_FP32, torch.bfloat16, False), (DG_SF_UE8M0, torch.bfloat16, False),
                                                (DG_SF_FP32, torch.float32, True)])
@pytest.mark.parametrize("Bt,M,N,K", [(1, 64, 256, 256), (5, 130, 384, 384), (3, 7, 1024, 512)])
def test_batched_gemm(Bt, M, N, K, fmt, out, accumulate):
    a = wl.randn_bf16((Bt, M, K), 710 + M, 1.5)
    b = wl.randn_bf16((Bt, N, K), 711 + M, 0.02)
    qa, sfa, qb, sfb, oqa, osfa, oqb, osfb = quantized(a.view(Bt * M, K), b, fmt)
    c_host = (torch.randn(Bt, M, N, dtype=torch.float32, generator=torch.Generator().manual_seed(712)) * 4
              if accumulate else None)
    d = torch.empty(Bt, M, N, dtype=out, device="cuda")
    api.dg_fp8_gemm_nt_batched(qa.view(Bt, M, K), sfa, qb, sfb, d,
                               c=None if c_host is None else c_host.cuda(), sf_format=fmt)
    sync()
    ref = oracle.gemm_batched(oqa.reshape(Bt, M, K), osfa.reshape(Bt, M, K // 128), oqb, osfb,
                              None if c_host is None else c_host.double().numpy())
    fp32 = out == torch.float32
    assert_close(to_f64(d), ref_out(ref, fp32), fp32, "batched GEMM")


@pytest.mark.slow
def test_plain_gemm_determinism_10000_calls():
    """10,000 in-place accumulating calls from the same C: each bitwise equal to the first."""
    M, N, K = 300, 512, 384
    a = wl.randn_bf16((M, K), 730, 1.5)
    b = wl.randn_bf16((1, N, K), 731, 0.02)
    qa, sfa, qb, sfb, *_ = quantized(a, b, DG_SF_FP32)
    c0 = torch.randn(M, N, dtype=torch.float32, device="cuda")
    d = c0.clone()
    api.dg_fp8_gemm_nt(qa, sfa, qb.view(N, K), sfb.view(N // 128, K // 128), d, c=d)
    first = d.clone()
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(10000):
        d.copy_(c0)
        api.dg_fp8_gemm_nt(qa, sfa, qb.view(N, K), sfb.view(N // 128, K // 128), d, c=d)
        bad += (d.view(torch.int32) != first.view(torch.int32)).any().to(torch.int64)
    sync()
    assert bad.item() == 0, f"{bad.item()} of 10000 calls differ"
