"""GPU parity of the FP4-weight path (the FP8 x FP4 form of m_grouped_fp8_fp4_gemm_nt_contiguous,
"SM120 m_grouped_fp8 contiguous kernel: illegal memory access at CUDA graph replay"): the FP4
weight cast bit-exact against the oracle, and the contiguous and masked GEMMs with FP4 weights
against the oracle's fp64 GEMMs on the same codes and scales (calc_diff <= 2e-5 for bf16 out,
<= 1e-6 for fp32 out), with rows that are not valid left untouched."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_ERR_UNSUPPORTED, DG_SF_UE8M0, DGError, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import (assert_close, gpu_quant_tokens, out_bits, ref_out, sentinel_like, sentinel_value, sync,
                         to_f64)

pytestmark = pytest.mark.gpu


def gpu_quant_fp4(w):
    G, N, K = w.shape
    q = torch.empty(G, N, K // 2, dtype=torch.uint8, device=w.device)
    sfb = torch.empty(G, N // 128, K // 128, dtype=torch.uint8, device=w.device)
    api.dg_quant_block_128x128_fp4(w, q, sfb)
    return q, sfb


@pytest.mark.parametrize("G,N,K", [(2, 256, 512), (1, 128, 128), (3, 384, 1024)])
def test_fp4_weight_cast_bit_exact(G, N, K):
    w = wl.randn_bf16((G, N, K), 900 + K, 0.02)
    w[0, :128, :128] = 0                                  # a zero block: sf_zero rounded up
    w[-1, -128:, -128:] *= 3e4                            # a block of large values
    q, sfb = gpu_quant_fp4(w.cuda())
    sync()
    oq, oue = oracle.quant_block_128x128_fp4(w)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    np.testing.assert_array_equal(sfb.cpu().numpy(), oue)


def fp4_operands(a, b):
    """GPU casts (per-token UE8M0 activations, FP4 weights) and the oracle's own casts."""
    M, K = a.shape
    qa, sfa = gpu_quant_tokens(a.cuda(), DG_SF_UE8M0)
    qb, sfb = gpu_quant_fp4(b.cuda())
    oqa, osfa, _ = oracle.quant_per_token_1x128(a, ue8m0=True)
    oqb, oue = oracle.quant_block_128x128_fp4(b)
    sync()
    np.testing.assert_array_equal(qa.cpu().numpy(), oqa)
    np.testing.assert_array_equal(qb.cpu().numpy(), oqb)
    return qa, sfa, qb, sfb, oqa, osfa, oqb, oracle.ue8m0_value(oue)


def contiguous_fp4_case(counts, N, K, out=torch.bfloat16, calls=1, seed=0):
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    M, G = mi.size, len(counts)
    a = wl.randn_bf16((M, K), 910 + seed, 1.5)
    b = wl.randn_bf16((G, N, K), 911 + seed, 0.02)
    qa, sfa, qb, sfb, oqa, osfa, oqb, osfb = fp4_operands(a, b)
    d = sentinel_like((M, N), out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mi_dev = torch.tensor(mi, device="cuda")
    first = None
    for i in range(calls):
        api.dg_m_grouped_fp8_fp4_contiguous(qa, sfa, qb, sfb, d, mi_dev, status)
        if calls > 1:
            bits = out_bits(d)
            if first is None:
                first = bits
            else:
                assert np.array_equal(bits, first), f"call {i} differs bitwise"
    sync()
    assert status.item() == 0
    ref = oracle.gemm_contiguous_fp4(oqa, osfa, oqb, osfb, mi)
    valid = mi >= 0
    fp32 = out == torch.float32
    assert_close(to_f64(d)[valid], ref_out(ref[valid], fp32), fp32, "fp8 x fp4 contiguous")
    assert np.all(out_bits(d)[~valid] == sentinel_value(out)), "a padding row was written"


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_fp4_contiguous_ragged(out):
    contiguous_fp4_case([130, 0, 1, 128, 257], 512, 512, out=out)


def test_fp4_contiguous_long_k_repeat_bitwise():
    contiguous_fp4_case([200, 33, 128], 256, 4096, calls=3, seed=1)


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_fp4_masked(out):
    G, cap, N, K = 3, 200, 256, 384
    counts = np.array([200, 77, 0], np.int32)
    a = wl.randn_bf16((G, cap, K), 920, 2.0)
    b = wl.randn_bf16((G, N, K), 921, 0.02)
    qa, sfa, qb, sfb, oqa, osfa, oqb, osfb = fp4_operands(a.view(G * cap, K), b)
    d = sentinel_like((G, cap, N), out)
    cnt = torch.tensor(counts, device="cuda")
    api.dg_m_grouped_fp8_fp4_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 64)
    sync()
    ref = oracle.gemm_masked_fp4(oqa.reshape(G, cap, K), osfa.reshape(G, cap, K // 128), oqb, osfb, counts)
    valid = np.arange(cap)[None, :] < counts[:, None]
    fp32 = out == torch.float32
    assert_close(to_f64(d)[valid], ref_out(ref[valid], fp32), fp32, "fp8 x fp4 masked")
    assert np.all(out_bits(d)[~valid] == sentinel_value(out)), "a row at or past its count was written"


def test_fp4_graph_replay_with_changed_routing():
    """Cast + FP8 x FP4 GEMM captured once, replayed with m_indices re-drawn in place."""
    G, N, K, E = 16, 512, 512, 20
    T = G * E
    m_max = wl.contiguous_capacity(T, G)
    a = wl.randn_bf16((m_max, K), 930, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), 931, 0.02, device="cuda")
    qa = torch.empty(m_max, K, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(m_max, K, DG_SF_UE8M0, "cuda")
    qb, sfb = gpu_quant_fp4(b)
    mi_dev = torch.full((m_max,), -1, dtype=torch.int32, device="cuda")
    d = torch.empty(m_max, N, dtype=torch.bfloat16, device="cuda")

    def step():
        api.dg_quant_per_token_1x128_routed(a, qa, sfa, mi_dev, DG_SF_UE8M0)
        api.dg_m_grouped_fp8_fp4_contiguous(qa, sfa, qb, sfb, d, mi_dev)

    mi_dev.copy_(torch.from_numpy(wl.contiguous_m_indices(wl.multinomial_counts(T, G, 1), m_max)))
    step()
    sync()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    sync()
    oqb, oue = oracle.quant_block_128x128_fp4(b.cpu())
    osfb = oracle.ue8m0_value(oue)
    for it in range(10):
        mi = wl.contiguous_m_indices(wl.multinomial_counts(T, G, 100 + it), m_max)
        mi_dev.copy_(torch.from_numpy(mi))
        d.view(torch.int16).fill_(-1)
        g.replay()
        sync()
        bits = out_bits(d)
        assert np.all(bits[mi < 0] == 0xFFFF), f"replay {it}: padding row written"
        rows = np.unique(np.random.default_rng(it).choice(np.nonzero(mi >= 0)[0], 24, replace=False))
        oqa, osfa, _ = oracle.quant_per_token_1x128(a[torch.from_numpy(rows).cuda()].cpu(), ue8m0=True)
        ref = oracle.gemm_contiguous_fp4(oqa, osfa, oqb, osfb, mi[rows])
        assert_close(to_f64(d)[rows], ref_out(ref, False), False, f"replay {it}")


def test_fp4_determinism_1000_calls():
    counts = [130, 0, 1, 128, 257]
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    M, G, N, K = mi.size, len(counts), 512, 2048
    a = wl.randn_bf16((M, K), 940, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), 941, 0.02, device="cuda")
    qa, sfa = gpu_quant_tokens(a, DG_SF_UE8M0)
    qb, sfb = gpu_quant_fp4(b)
    mi_dev = torch.tensor(mi, device="cuda")
    d = torch.zeros(M, N, dtype=torch.bfloat16, device="cuda")
    api.dg_m_grouped_fp8_fp4_contiguous(qa, sfa, qb, sfb, d, mi_dev)
    first = d.clone()
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(1000):
        api.dg_m_grouped_fp8_fp4_contiguous(qa, sfa, qb, sfb, d, mi_dev)
        bad += (d.view(torch.int16) != first.view(torch.int16)).any().to(torch.int64)
    sync()
    assert bad.item() == 0


def test_fp4_needs_n_multiple_of_256():
    qa = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(128, 128, DG_SF_UE8M0, "cuda")
    qb = torch.zeros(1, 384, 64, dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(1, 3, 1, dtype=torch.uint8, device="cuda")
    d = torch.empty(128, 384, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(DGError) as e:
        api.dg_m_grouped_fp8_fp4_contiguous(qa, sfa, qb, sfb, d, torch.zeros(128, dtype=torch.int32, device="cuda"))
    assert e.value.code == DG_ERR_UNSUPPORTED


@pytest.mark.slow
def test_fp4_decode_shape_full_size_whole_expert():
    """The decode shape with FP4 weights (G=32, cap=4096, N=6144, K=7168, Poisson(192) counts,
    UE8M0 scales on both operands): one full-size launch; every valid row x every output column of
    the largest expert against the oracle's FP4 GEMM, and every padding row untouched."""
    w = wl.masked_decode()
    G, cap, N, K = w.G, w.cap, w.N, w.K
    a, b = w.draw(device="cuda")
    cnt = torch.tensor(w.counts, device="cuda")
    qa, sfa = gpu_quant_tokens(a.view(G * cap, K), DG_SF_UE8M0, row_counts=cnt)
    qb, sfb = gpu_quant_fp4(b)
    d = sentinel_like((G, cap, N), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_m_grouped_fp8_fp4_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 192, status)
    sync()
    assert status.item() == 0
    rows = torch.arange(cap, device="cuda")[None, :]
    assert bool((d.view(torch.int16)[rows >= cnt[:, None]] == -1).all()), "padding rows written"
    g = int(np.argmax(w.counts))
    c = int(w.counts[g])
    oqb, oue = oracle.quant_block_128x128_fp4(b[g:g + 1].cpu())
    np.testing.assert_array_equal(qb[g].cpu().numpy(), oqb[0])
    oqa, osfa, _ = oracle.quant_per_token_1x128(a[g, :c].cpu(), ue8m0=True)
    ref = oracle.gemm_masked_fp4(oqa.reshape(1, c, K), osfa.reshape(1, c, K // 128), oqb, oracle.ue8m0_value(oue),
                                 [c])
    assert_close(to_f64(d[g, :c]), ref_out(ref[0], False), False, f"fp4 decode expert {g} whole")
