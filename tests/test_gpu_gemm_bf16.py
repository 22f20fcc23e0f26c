"""GPU parity of the BF16 m-grouped GEMMs (masked and contiguous) against the oracle's fp64
BF16 GEMM on the same bf16 bytes ("Fix cross-expert output overwrites in SM90 masked GEMM", #469:
the reproduction runs m_grouped_bf16_gemm_nt_masked and checks the valid rows against
bmm(a.double(), b.double().mT) rounded to bf16 with calc_diff < 1e-5)."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_STATUS_BAD_INDEX, DG_STATUS_COUNT_GT_CAP, _lib, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import assert_close, out_bits, ref_out, sentinel_like, sentinel_value, sync, to_f64

pytestmark = pytest.mark.gpu

PAGES_CALC_DIFF = 1e-5  # the reproduction's own threshold


def masked_bf16_case(a, b, counts, out=torch.bfloat16, calls=1, expected_m=0):
    G, cap, K = a.shape
    N = b.shape[1]
    ad, bd = a.cuda(), b.cuda()
    cnt = torch.tensor(np.asarray(counts, np.int32), device="cuda")
    d = sentinel_like((G, cap, N), out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = None
    for i in range(calls):
        api.dg_m_grouped_bf16_masked(ad, bd, d, cnt, expected_m, status)
        if calls > 1:
            bits = out_bits(d)
            if first is None:
                first = bits
            else:
                assert np.array_equal(bits, first), f"call {i} differs bitwise from call 0"
    sync()
    ref = oracle.gemm_masked_bf16(a, b, counts)
    v = np.clip(np.asarray(counts), 0, cap)
    valid = np.arange(cap)[None, :] < v[:, None]
    fp32 = out == torch.float32
    if valid.any():
        assert_close(to_f64(d)[valid], ref_out(ref[valid], fp32), fp32, "bf16 masked valid rows")
    assert np.all(out_bits(d)[~valid] == sentinel_value(out)), "a row at or past its expert's count was written"
    return d, status, ref, valid


def test_pages_reproduction_bf16_16_calls():
    """G=8, cap=32, N=K=256, counts [0,1,16,31,32,1,32,32], seed 29 (the reproduction's shape and
    counts, our seeded generator): 16 bitwise-identical calls, calc_diff < 1e-5 on the valid rows,
    every padding row keeps its sentinel."""
    w = wl.masked_repro()
    a, b = w.draw()
    d, _, ref, valid = masked_bf16_case(a, b, w.counts, calls=16, expected_m=32)
    diff = oracle.calc_diff(to_f64(d)[valid], oracle.bf16_bits_to_f64(oracle.round_bf16(ref[valid])))
    assert diff < PAGES_CALC_DIFF, f"calc_diff {diff:.3e}"


CAPS = [1, 7, 8, 9, 16, 31, 33, 64, 96, 127, 128, 129, 200, 257]


@pytest.mark.parametrize("cap", CAPS)
def test_bf16_capacity_panel(cap):
    rng = np.random.default_rng(100 + cap)
    G, N, K = 4, 256, 192
    counts = rng.integers(0, cap + 1, G)
    counts[rng.integers(0, G)] = cap
    counts[rng.integers(0, G)] = 0
    masked_bf16_case(wl.randn_bf16((G, cap, K), 300 + cap), wl.randn_bf16((G, N, K), 400 + cap), counts)


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_bf16_masked_output_dtypes_and_k_not_multiple_of_128(out):
    G, cap, N, K = 3, 200, 384, 320
    masked_bf16_case(wl.randn_bf16((G, cap, K), 11, 2.0), wl.randn_bf16((G, N, K), 12, 0.05), [200, 77, 129], out)


def test_bf16_masked_counts_clamped_and_flagged():
    G, cap, N, K = 3, 48, 128, 128
    _, status, _, _ = masked_bf16_case(wl.randn_bf16((G, cap, K), 31), wl.randn_bf16((G, N, K), 32), [-5, 1000, 20])
    assert status.item() & DG_STATUS_COUNT_GT_CAP


def test_bf16_masked_all_empty_and_single_expert():
    masked_bf16_case(wl.randn_bf16((3, 64, 128), 23), wl.randn_bf16((3, 128, 128), 24), [0, 0, 0])
    masked_bf16_case(wl.randn_bf16((1, 130, 256), 21), wl.randn_bf16((1, 128, 256), 22), [130])


def contiguous_bf16_case(a, b, m_indices, out=torch.bfloat16, calls=1):
    M, K = a.shape
    G, N, _ = b.shape
    mi = torch.tensor(np.asarray(m_indices, np.int32), device="cuda")
    d = sentinel_like((M, N), out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = None
    for i in range(calls):
        api.dg_m_grouped_bf16_contiguous(a.cuda(), b.cuda(), d, mi, status)
        if calls > 1:
            bits = out_bits(d)
            if first is None:
                first = bits
            else:
                assert np.array_equal(bits, first), f"call {i} differs bitwise"
    sync()
    ref = oracle.gemm_contiguous_bf16(a, b, m_indices)
    mi_np = np.asarray(m_indices)
    block_e = mi_np[(np.arange(M) // 128) * 128]
    valid = (mi_np >= 0) & (mi_np == block_e)
    fp32 = out == torch.float32
    if valid.any():
        assert_close(to_f64(d)[valid], ref_out(ref[valid], fp32), fp32, "bf16 contiguous routed rows")
    assert np.all(out_bits(d)[~valid] == sentinel_value(out)), "a padding row was written"
    return d, status


@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_bf16_contiguous_ragged_segments(out):
    counts = [130, 0, 1, 128, 257]
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    contiguous_bf16_case(wl.randn_bf16((mi.size, 384), 51, 1.5), wl.randn_bf16((5, 256, 384), 52, 0.05), mi, out, calls=4)


def test_bf16_contiguous_bad_indices_flagged_and_skipped():
    mi = np.full(256, -1, np.int32)
    mi[0:10] = 0
    mi[10:12] = 7                                      # >= G: flagged, not written
    mi[129:140] = 1                                    # block 1 headed by -1: skipped
    a, b = wl.randn_bf16((256, 128), 91), wl.randn_bf16((2, 128, 128), 92)
    d = sentinel_like((256, 128), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_m_grouped_bf16_contiguous(a.cuda(), b.cuda(), d, torch.tensor(mi, device="cuda"), status)
    sync()
    assert status.item() & DG_STATUS_BAD_INDEX
    ref = oracle.gemm_contiguous_bf16(a, b, np.where(mi >= 2, -1, mi))
    assert_close(to_f64(d)[:10], ref_out(ref[:10], False), False, "rows of expert 0")
    bits = out_bits(d)
    assert np.all(bits[10:] == sentinel_value(torch.bfloat16))


def set_bf16_bn(bn: int) -> None:
    """Test hook: the BF16 GEMM's tile width for later calls (0 automatic, 128, 256)."""
    _lib.check(_lib.load().dg_testing_bf16_bn(int(bn)))


@pytest.mark.parametrize("layout", ["masked", "contiguous"])
def test_bf16_tile_widths_bitwise_equal(layout):
    """128 x 256 tiles (the automatic choice for bf16 output with N % 256 == 0 on calls with enough
    tiles) and 128 x 128 tiles write the same bits: every output element sums the same K-ordered
    products either way."""
    outs = []
    for bn in (256, 128):
        set_bf16_bn(bn)
        try:
            if layout == "masked":
                d, _, _, _ = masked_bf16_case(wl.randn_bf16((4, 200, 320), 61), wl.randn_bf16((4, 512, 320), 62, 0.05),
                                              [200, 77, 0, 130])
            else:
                counts = [130, 0, 257, 5]
                mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
                d, _ = contiguous_bf16_case(wl.randn_bf16((mi.size, 1024), 63, 1.0),
                                            wl.randn_bf16((4, 256, 1024), 64, 0.05), mi)
            outs.append(out_bits(d))
        finally:
            set_bf16_bn(0)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.slow
def test_bf16_masked_decode_shape_sampled():
    """G=32, cap=4096, N=6144, K=7168 (the FP8 decode shape with bf16 operands), counts ~ Poisson(192):
    the full launch, checked on sampled rows of every expert against the oracle row by row."""
    w = wl.masked_decode()
    G, cap, N, K = w.G, w.cap, w.N, w.K
    a, b = w.draw(device="cuda")
    cnt = torch.tensor(w.counts, device="cuda")
    d = sentinel_like((G, cap, N), torch.bfloat16)
    api.dg_m_grouped_bf16_masked(a, b, d, cnt, 192)
    sync()
    rng = np.random.default_rng(5)
    for g in range(0, G, 3):
        c = int(min(max(w.counts[g], 0), cap))
        if c == 0:
            continue
        rows = np.unique(rng.integers(0, c, 4))
        cols = slice(128 * (g % (N // 128)), 128 * (g % (N // 128)) + 128)
        ref = oracle.gemm_masked_bf16(a[g:g + 1, rows].cpu(), b[g:g + 1, cols].cpu(), [len(rows)])
        assert_close(to_f64(d[g, rows, cols]), ref_out(ref[0], False), False, f"expert {g}")
        assert np.all(out_bits(d[g, c:]) == sentinel_value(torch.bfloat16))
