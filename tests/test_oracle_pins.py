"""Pins for the CPU oracle: facts fixed by the source pages and by the mathematics, so that a
plausible mistake anywhere in the oracle (a dropped scale, a transposed operand, a wrong
rounding tie, a missing C term, a packing index swap) fails at least one test here.

None of these tests re-type an oracle formula and compare it with itself: each one uses an
independent route (exhaustive enumeration, an exact integer computation, a library routine
such as torch's e4m3 conversion or numpy's matmul, a closed form, or a value printed on the
pages)."""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32_1E30 = float(np.float32(1e-30))


def bf16_from_f64(vals) -> torch.Tensor:
    """Values that are exactly representable in bf16 -> a bf16 tensor (checked exact)."""
    t = torch.tensor(np.asarray(vals, np.float64), dtype=torch.float64).to(torch.bfloat16)
    assert torch.equal(t.double(), torch.tensor(np.asarray(vals, np.float64)))
    return t


def e4m3_grid():
    """All finite e4m3 values, from the format definition (not from the oracle)."""
    vals = [0.0]
    for m in range(1, 8):
        vals.append(m * 2.0 ** -9)
    for e in range(1, 16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            vals.append((1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


# ---------------------------------------------------------------------------------- codec

def test_decode_matches_format_definition_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.e4m3_decode(codes)
    # the format definition, value by value
    assert dec[0x00] == 0.0 and not math.copysign(1, dec[0x00]) < 0
    assert dec[0x01] == 2.0 ** -9 and dec[0x07] == 7 * 2.0 ** -9 and dec[0x08] == 2.0 ** -6
    assert dec[0x38] == 1.0 and dec[0x7E] == 448.0 and dec[0xFE] == -448.0
    assert math.isnan(dec[0x7F]) and math.isnan(dec[0xFF])
    assert dec[0x80] == 0.0 and math.copysign(1, dec[0x80]) < 0
    pos = dec[:0x7F]
    assert np.all(np.diff(pos) > 0), "non-negative codes must increase with the code"
    np.testing.assert_array_equal(pos, e4m3_grid())
    # library routine: torch's own e4m3 -> fp32 decode
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    np.testing.assert_array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(dec[ok], ref[ok])


def test_encode_roundtrip_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    dec = oracle.e4m3_decode(codes)
    keep = ~np.isnan(dec)
    enc = oracle.e4m3_encode(dec[keep].astype(np.float32))
    np.testing.assert_array_equal(enc, codes[keep])


def test_encode_midpoints_tie_to_even():
    grid = e4m3_grid()
    lo, hi = grid[:-1], grid[1:]
    mid = (lo + hi) / 2  # at most 5 significant bits: exact in fp32
    assert np.all(mid.astype(np.float32).astype(np.float64) == mid)
    enc = oracle.e4m3_encode(mid.astype(np.float32))
    idx = np.arange(len(lo))
    even = np.where(idx % 2 == 0, idx, idx + 1)
    np.testing.assert_array_equal(enc, even.astype(np.uint8))
    np.testing.assert_array_equal(oracle.e4m3_encode(-mid.astype(np.float32)), even.astype(np.uint8) | 0x80)
    # just off the midpoint rounds to the nearer neighbour
    below = np.nextafter(mid.astype(np.float32), np.float32(-1))
    above = np.nextafter(mid.astype(np.float32), np.float32(1000))
    np.testing.assert_array_equal(oracle.e4m3_encode(below), idx.astype(np.uint8))
    np.testing.assert_array_equal(oracle.e4m3_encode(above), (idx + 1).astype(np.uint8))


def test_encode_matches_torch_below_saturation():
    rng = np.random.default_rng(7)
    parts = [rng.uniform(-463.9, 463.9, 400_000), rng.normal(0, 1e-2, 200_000),
             rng.normal(0, 3e-3, 200_000), np.ldexp(rng.uniform(-1, 1, 200_000), rng.integers(-14, 9, 200_000))]
    y = np.concatenate(parts).astype(np.float32)
    ours = oracle.e4m3_encode(y)
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_encode_saturates_and_nan():
    big = np.array([448, 448.0001, 463.99, 464, 479, 480, 1e6, np.inf], np.float32)
    np.testing.assert_array_equal(oracle.e4m3_encode(big), np.full(big.size, 0x7E, np.uint8))
    np.testing.assert_array_equal(oracle.e4m3_encode(-big), np.full(big.size, 0xFE, np.uint8))
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F
    np.testing.assert_array_equal(oracle.e4m3_encode(np.array([0.0, -0.0], np.float32)), [0x00, 0x80])


# ---------------------------------------------------------------------------------- scales

def test_scale_rule_closed_cases():
    amax = np.array([0.0, 0.0, 0.0, 448.0, 224.0, 449.0, 1.0], np.float32)
    sf, _ = oracle.scale_from_amax(amax, 1.0, False)
    assert sf[0] == 1.0 and sf[3] == 1.0 and sf[4] == 0.5
    assert sf[5] == np.float32(449.0) / np.float32(448.0)
    assert sf[6] == np.float32(1.0) / np.float32(448.0)
    # zero amax takes sf_zero, then the 1e-30 floor applies
    for sz, want in [(1e-4, np.float32(1e-4)), (1e-8, np.float32(1e-8)), (1e-30, np.float32(1e-30)),
                     (0.0, np.float32(1e-30)), (1e-40, np.float32(1e-30))]:
        s, _ = oracle.scale_from_amax(np.zeros(1, np.float32), sz, False)
        assert s[0] == want, (sz, s[0])
    # a tiny non-zero amax is floored too
    s, _ = oracle.scale_from_amax(np.array([1e-36], np.float32), 1.0, False)
    assert s[0] == np.float32(1e-30)


def test_ue8m0_rounds_up_to_power_of_two():
    rng = np.random.default_rng(3)
    amax = np.concatenate([np.ldexp(rng.uniform(0.5, 1, 50_000), rng.integers(-60, 60, 50_000)),
                           [448.0, 224.0, 896.0, 449.0, 447.0, 0.0]]).astype(np.float32)
    sf32, _ = oracle.scale_from_amax(amax, 1e-30, False)
    sf2, ue = oracle.scale_from_amax(amax, 1e-30, True)
    np.testing.assert_array_equal(oracle.ue8m0_value(ue), sf2)
    m, _ = np.frexp(sf2.astype(np.float64))
    assert np.all(m == 0.5), "UE8M0 scales are powers of two"
    assert np.all(sf2 >= sf32) and np.all(sf2 < 2 * sf32.astype(np.float64))
    exact = (np.frexp(sf32.astype(np.float64))[0] == 0.5)
    np.testing.assert_array_equal(sf2[exact], sf32[exact])
    assert ue[-6] == 127 and ue[-5] == 126 and ue[-4] == 128 and ue[-3] == 128 and ue[-2] == 127


# ---------------------------------------------------------------------------------- casts

def dequant_err_bound(x, sf):
    """RNE onto e4m3 after scaling: |decode(q) sf - x| <= half an e4m3 ulp, i.e.
    <= 2^-4 |x| in the normal range and <= 2^-10 sf in the subnormal range, plus fp32
    rounding of the reciprocal and the product."""
    return (np.maximum(2.0 ** -4 * np.abs(x), 2.0 ** -10 * sf)) * (1 + 1e-6) + 1e-300


@pytest.mark.parametrize("ue8m0", [False, True])
def test_per_token_cast_pins(ue8m0):
    M, K = 7, 512
    x = wl.randn_bf16((M, K), 11, 3.0)
    x[2, 128:256] = 0                                  # all-zero block
    grid = e4m3_grid()
    rng = np.random.default_rng(5)
    row = rng.choice(np.concatenate([grid, -grid]), 128)
    row[17] = 448.0                                    # amax 448 -> sf 1, codes exact
    x[4, 256:384] = bf16_from_f64(row)
    q, sf, ue = oracle.quant_per_token_1x128(x, sf_zero=0.25, ue8m0=ue8m0)
    assert sf[2, 1] == 0.25 and np.all(q[2, 128:256] == 0)
    assert sf[4, 2] == 1.0
    np.testing.assert_array_equal(oracle.e4m3_decode(q[4, 256:384]), row)
    xf = x.double().numpy()
    deq = oracle.e4m3_decode(q) * np.repeat(sf.astype(np.float64), 128, axis=1)
    assert np.all(np.abs(deq - xf) <= dequant_err_bound(xf, np.repeat(sf.astype(np.float64), 128, axis=1)))
    # every non-zero block uses its full range: max |q| hits 448 exactly for fp32 scales
    amax_code = np.abs(oracle.e4m3_decode(q)).reshape(M, K // 128, 128).max(-1)
    if not ue8m0:
        nz = np.abs(xf).reshape(M, K // 128, 128).max(-1) > 0
        assert np.all(amax_code[nz] == 448.0)
    else:
        np.testing.assert_array_equal(oracle.ue8m0_value(ue), sf)
        assert np.all(amax_code <= 448.0)


def test_per_token_cast_row_counts_leave_other_rows():
    x = wl.randn_bf16((4 * 6, 256), 2)
    q, sf, _ = oracle.quant_per_token_1x128(x, row_counts=[0, 6, 3, 9])
    rows = np.arange(24)
    cast = ((rows // 6 == 1) | ((rows // 6 == 2) & (rows % 6 < 3)) | (rows // 6 == 3))
    assert np.all(np.isnan(sf[~cast])) and np.all(q[~cast] == 0)
    assert not np.any(np.isnan(sf[cast]))
    q_all, sf_all, _ = oracle.quant_per_token_1x128(x)
    np.testing.assert_array_equal(q[cast], q_all[cast])
    np.testing.assert_array_equal(sf[cast], sf_all[cast])


def test_per_token_cast_matches_torch_library_conversion():
    """The cast steps in torch ops (amax, fp32 divide, reciprocal, multiply, torch's own
    e4m3 conversion); the conversion is the library routine pinning the oracle encode."""
    x = wl.randn_bf16((33, 1024), 21, 5.0)
    q, sf, _ = oracle.quant_per_token_1x128(x)
    xv = x.float().view(33, 8, 128)
    amax = xv.abs().amax(-1)
    s = (amax / 448.0).clamp_min(1e-30)
    tq = (xv * (1.0 / s).unsqueeze(-1)).to(torch.float8_e4m3fn).view(torch.uint8).view(33, 1024)
    np.testing.assert_array_equal(sf, s.numpy())
    np.testing.assert_array_equal(q, tq.numpy())


@pytest.mark.parametrize("ue8m0", [False, True])
def test_block_cast_pins(ue8m0):
    G, N, K = 2, 256, 384
    w = wl.randn_bf16((G, N, K), 4, 0.02)
    w[1, 128:256, 0:128] = 0
    w[0, 5, 130] = 448.0 * 0.02 * 50                  # one large element dominates block (0,0,1)
    q, sf, ue = oracle.quant_block_128x128(w, sf_zero=2.0, ue8m0=ue8m0)
    assert sf[1, 1, 0] == 2.0 and np.all(q[1, 128:256, 0:128] == 0)
    big = np.float32(448.0 * 0.02 * 50)
    expect = np.float32(float(torch.tensor(big).to(torch.bfloat16).float()) / np.float32(448.0))
    if not ue8m0:
        assert sf[0, 0, 1] == expect
        assert q[0, 5, 130] == 0x7E
    wf = w.double().numpy()
    sfe = np.repeat(np.repeat(sf.astype(np.float64), 128, 1), 128, 2)
    deq = oracle.e4m3_decode(q) * sfe
    assert np.all(np.abs(deq - wf) <= dequant_err_bound(wf, sfe))
    # the scale of a block is the block's own amax: other blocks are unaffected
    w2 = w.clone()
    w2[0, 0:128, 256:384] *= 4
    q2, sf2, _ = oracle.quant_block_128x128(w2, sf_zero=2.0, ue8m0=ue8m0)
    mask = np.ones_like(sf, bool)
    mask[0, 0, 2] = False
    np.testing.assert_array_equal(sf2[mask], sf[mask])


def test_per_channel_cast_and_pack():
    ks = [256, 128, 0, 128, 256]
    T, C = sum(ks), 192
    x = wl.randn_bf16((T, C), 8, 1e-7)
    x[256:384, 0] = 0                                  # zero channel inside the 128-token expert
    q, sf = oracle.quant_per_channel_128(x, sf_zero=1e-4)
    assert sf.shape == (T // 128, C)
    assert sf[2, 0] == np.float32(1e-4) and np.all(q[256:384, 0] == 0)
    xf = x.double().numpy()
    sfe = np.repeat(sf.astype(np.float64), 128, 0)
    assert np.all(np.abs(oracle.e4m3_decode(q) * sfe - xf) <= dequant_err_bound(xf, sfe))
    packed = oracle.pack_kmajor(q, ks)
    assert packed.size == T * C
    # independent route: numpy transpose of each expert's span
    o = 0
    for k in ks:
        blk = packed[o * C:(o + k) * C].reshape(C, k)
        np.testing.assert_array_equal(blk, q[o:o + k].T)
        o += k


# ---------------------------------------------------------------------------------- GEMMs

def grid_operand(shape, seed):
    """bf16 values on the e4m3 grid with a 448 in every 128-wide block along the last axis:
    every 1x128 and 128x128 scale is exactly 1 and the codes are the values themselves."""
    rng = np.random.default_rng(seed)
    grid = e4m3_grid()
    grid = grid[grid <= 64]
    v = rng.choice(np.concatenate([grid, -grid]), shape)
    v.reshape(-1, 128)[:, rng.integers(0, 128)] = 448.0
    return bf16_from_f64(v), v


def test_contiguous_exact_integer_closed_form():
    G, N, K = 3, 128, 256
    counts = [5, 0, 130]
    mi = wl.contiguous_m_indices(counts, 512)
    M = mi.size
    a, av = grid_operand((M, K), 1)
    b, bv = grid_operand((G, N, K), 2)
    qa, sfa, _ = oracle.quant_per_token_1x128(a)
    qb, sfb, _ = oracle.quant_block_128x128(b)
    assert np.all(sfa == 1.0) and np.all(sfb == 1.0)
    d = oracle.gemm_contiguous(qa, sfa, qb, sfb, mi)
    ai = (av * 2 ** 9).astype(np.int64)                # e4m3 values are multiples of 2^-9
    bi = (bv * 2 ** 9).astype(np.int64)
    for m in range(M):
        e = mi[m]
        if e < 0:
            assert np.all(np.isnan(d[m]))
            continue
        exact = (ai[m][None, :] * bi[e]).sum(-1)     # int64, exact
        np.testing.assert_array_equal(d[m], exact.astype(np.float64) * 2.0 ** -18)


def test_contiguous_block_integer_formulation_random_scales():
    """Second formulation: D = sum_kb sfa sfb (sum_{k in kb} qa qb), inner sums exact int64."""
    G, N, K = 2, 256, 512
    counts = [130, 77]
    mi = wl.contiguous_m_indices(counts, 512)
    a = wl.randn_bf16((mi.size, K), 3, 2.0)
    b = wl.randn_bf16((G, N, K), 4, 0.02)
    qa, sfa, _ = oracle.quant_per_token_1x128(a)
    qb, sfb, _ = oracle.quant_block_128x128(b)
    d = oracle.gemm_contiguous(qa, sfa, qb, sfb, mi)
    ia = np.rint(oracle.e4m3_decode(qa) * 2 ** 9).astype(np.int64)
    ib = np.rint(oracle.e4m3_decode(qb) * 2 ** 9).astype(np.int64)
    for m in np.nonzero(mi >= 0)[0][::7]:
        e = mi[m]
        part = (ia[m].reshape(1, K // 128, 128) * ib[e].reshape(N, K // 128, 128)).sum(-1)  # [N, KB]
        scl = sfa[m].astype(np.float64)[None, :] * np.repeat(sfb[e].astype(np.float64), 128, 0)
        terms = part * 2.0 ** -18 * scl
        ref = terms.sum(-1)
        # fp64 summation error is bounded relative to sum |terms| (cancellation-safe)
        assert np.all(np.abs(d[m] - ref) <= 1e-13 * np.abs(terms).sum(-1) + 1e-300)


@pytest.mark.parametrize("G,M_list", [(1, [0]), (1, [1]), (2, [2, 127]), (3, [128, 0, 129]), (3, [1, 129, 2])])
def test_masked_brute_force_equals_batched_matmul(G, M_list):
    cap = max(max(M_list), 1)
    N, K = 128, 256
    a = wl.randn_bf16((G, cap, K), 10 + G)
    b = wl.randn_bf16((G, N, K), 20 + G)
    qa, sfa, _ = oracle.quant_per_token_1x128(a.view(G * cap, K))
    qb, sfb, _ = oracle.quant_block_128x128(b)
    d = oracle.gemm_masked(qa.reshape(G, cap, K), sfa.reshape(G, cap, K // 128), qb, sfb, M_list)
    xa = (oracle.e4m3_decode(qa) * np.repeat(sfa.astype(np.float64), 128, 1)).reshape(G, cap, K)
    xb = oracle.e4m3_decode(qb) * np.repeat(np.repeat(sfb.astype(np.float64), 128, 1), 128, 2)
    full = np.matmul(xa, xb.transpose(0, 2, 1))       # library batched GEMM
    for g, cnt in enumerate(M_list):
        np.testing.assert_allclose(d[g, :cnt], full[g, :cnt], rtol=1e-10, atol=1e-12)
        assert np.all(np.isnan(d[g, cnt:]))


def test_masked_counts_clamped_and_all_empty():
    G, cap, N, K = 3, 5, 128, 128
    a = wl.randn_bf16((G, cap, K), 1)
    b = wl.randn_bf16((G, N, K), 2)
    qa, sfa, _ = oracle.quant_per_token_1x128(a.view(G * cap, K))
    qb, sfb, _ = oracle.quant_block_128x128(b)
    qa, sfa = qa.reshape(G, cap, K), sfa.reshape(G, cap, 1)
    d = oracle.gemm_masked(qa, sfa, qb, sfb, [0, 0, 0])
    assert np.all(np.isnan(d))
    d1 = oracle.gemm_masked(qa, sfa, qb, sfb, [-3, 99, 2])
    assert np.all(np.isnan(d1[0])) and not np.any(np.isnan(d1[1])) and np.all(np.isnan(d1[2, 2:]))
    d2 = oracle.gemm_masked(qa, sfa, qb, sfb, [0, cap, 2])
    np.testing.assert_array_equal(d1[1], d2[1])


def test_contiguous_single_expert_is_plain_matmul():
    M, N, K = 129, 256, 384
    a = wl.randn_bf16((M, K), 31)
    b = wl.randn_bf16((1, N, K), 32, 0.02)
    qa, sfa, _ = oracle.quant_per_token_1x128(a, ue8m0=True)
    qb, sfb, _ = oracle.quant_block_128x128(b, ue8m0=True)
    d = oracle.gemm_contiguous(qa, sfa, qb, sfb, np.zeros(M, np.int32))
    xa = oracle.e4m3_decode(qa) * np.repeat(sfa.astype(np.float64), 128, 1)
    xb = oracle.e4m3_decode(qb[0]) * np.repeat(np.repeat(sfb[0].astype(np.float64), 128, 0), 128, 1)
    np.testing.assert_allclose(d, xa @ xb.T, rtol=1e-10, atol=1e-12)
    # and the quantized product tracks the bf16 product to e4m3 precision
    ref = a.double().numpy() @ b[0].double().numpy().T
    assert oracle.calc_diff(d, ref) < 2e-3


def test_group_independence():
    G, cap, N, K = 3, 40, 128, 256
    a = wl.randn_bf16((G, cap, K), 41)
    b = wl.randn_bf16((G, N, K), 42)
    counts = [40, 17, 33]

    def run(a, b):
        qa, sfa, _ = oracle.quant_per_token_1x128(a.view(G * cap, K))
        qb, sfb, _ = oracle.quant_block_128x128(b)
        return oracle.gemm_masked(qa.reshape(G, cap, K), sfa.reshape(G, cap, 2), qb, sfb, counts)

    d0 = run(a, b)
    a2, b2 = a.clone(), b.clone()
    a2[1] *= 3
    b2[2] = wl.randn_bf16((N, K), 99)
    d1 = run(a2, b2)
    np.testing.assert_array_equal(d1[0], d0[0])
    assert not np.array_equal(d1[1, :17], d0[1, :17])
    # contiguous: perturbing expert 1's rows leaves expert 0's rows bitwise unchanged
    mi = wl.contiguous_m_indices([100, 60], 300)
    ac = wl.randn_bf16((300, K), 43)
    bc = wl.randn_bf16((2, N, K), 44)
    qb, sfb, _ = oracle.quant_block_128x128(bc)
    qa, sfa, _ = oracle.quant_per_token_1x128(ac)
    dc0 = oracle.gemm_contiguous(qa, sfa, qb, sfb, mi)
    ac2 = ac.clone()
    ac2[128:188] *= -2
    qa2, sfa2, _ = oracle.quant_per_token_1x128(ac2)
    dc1 = oracle.gemm_contiguous(qa2, sfa2, qb, sfb, mi)
    np.testing.assert_array_equal(dc1[:100], dc0[:100])


def kgrouped_operands(ks, N, H, seed, gy_scale=1.0, act_scale=1.0, sf_zero=1e-30, zero_ch=False):
    T = sum(ks)
    gy = wl.randn_bf16((T, N), seed, gy_scale)
    act = wl.randn_bf16((T, H), seed + 1, act_scale)
    if zero_ch:
        o = 0
        for k in ks:
            if k == 128:
                gy[o:o + k, 0] = 0
            o += k
    qa, sfa = oracle.quant_per_channel_128(gy, sf_zero)
    qb, sfb = oracle.quant_per_channel_128(act, sf_zero)
    return gy, act, qa, sfa, qb, sfb


def test_kgrouped_equals_matmul_and_per_expert_sum():
    ks = [256, 0, 128, 384]
    N, H = 128, 256
    gy, act, qa, sfa, qb, sfb = kgrouped_operands(ks, N, H, 51)
    ap, bp = oracle.pack_kmajor(qa, ks), oracle.pack_kmajor(qb, ks)
    c = np.random.default_rng(0).normal(size=(len(ks), N, H)).astype(np.float32)
    d = oracle.gemm_kgrouped(ap, sfa, bp, sfb, ks, N, H, c=c)
    xa = oracle.e4m3_decode(qa) * np.repeat(sfa.astype(np.float64), 128, 0)   # [T, N]
    xb = oracle.e4m3_decode(qb) * np.repeat(sfb.astype(np.float64), 128, 0)   # [T, H]
    o = 0
    for e, k in enumerate(ks):
        ref = c[e].astype(np.float64) + xa[o:o + k].T @ xb[o:o + k]          # library GEMM, unpacked
        np.testing.assert_allclose(d[e], ref, rtol=1e-10, atol=1e-12)
        # the same expert alone (its own span, scales and pack) gives the same block
        de = oracle.gemm_kgrouped(oracle.pack_kmajor(qa[o:o + k], [k]), sfa[o // 128:(o + k) // 128],
                                  oracle.pack_kmajor(qb[o:o + k], [k]), sfb[o // 128:(o + k) // 128],
                                  [k], N, H, c=c[e:e + 1])
        np.testing.assert_array_equal(de[0], d[e])
        o += k
    np.testing.assert_array_equal(d[1], c[1].astype(np.float64))              # K_e = 0 -> D_e = C_e
    d0 = oracle.gemm_kgrouped(ap, sfa, bp, sfb, ks, N, H)                     # c = NULL
    np.testing.assert_array_equal(d0[1], np.zeros((N, H)))


def test_kgrouped_invalid_expert_stops_the_walk():
    ks = [128, 100, 128]
    N, H = 128, 128
    T = 128 + 128 + 128
    qa = np.ones((T, N), np.uint8)
    sf = np.ones((T // 128, N), np.float32)
    ap = np.ones(T * N, np.uint8)
    d = oracle.gemm_kgrouped(ap, sf, ap, sf, ks, N, H, K_cap=T)
    assert not np.any(np.isnan(d[0])) and np.all(np.isnan(d[1])) and np.all(np.isnan(d[2]))
    d2 = oracle.gemm_kgrouped(ap, sf, ap, sf, [128, 128, 256], N, H, K_cap=T)  # overflows K_cap
    assert not np.any(np.isnan(d2[1])) and np.all(np.isnan(d2[2]))


def test_kgrouped_sf_zero_invariance_bitwise():
    """An all-zero channel has zero codes, so the output is bitwise independent of sf_val
    (the #365 repro sweeps sf_val over 1, 1e-4, 1e-8, 1e-30)."""
    ks = [256, 128, 128, 256]
    N, H = 128, 128
    outs = []
    for sz in [1.0, 1e-4, 1e-8, 1e-30]:
        gy, act, qa, sfa, qb, sfb = kgrouped_operands(ks, N, H, 60, 1e-7, 0.4, sz, zero_ch=True)
        assert np.all(qa[128 * 2:128 * 3, 0] == 0)
        d = oracle.gemm_kgrouped(oracle.pack_kmajor(qa, ks), sfa, oracle.pack_kmajor(qb, ks), sfb, ks, N, H)
        outs.append(d)
    for d in outs[1:]:
        np.testing.assert_array_equal(d.view(np.uint64), outs[0].view(np.uint64))
    assert np.all(outs[0][1, 0] == 0) and np.all(outs[0][2, 0] == 0)


@pytest.mark.slow
def test_kgrouped_repro_matches_printed_reference_norm():
    """The pages print the reference wgrad's largest per-expert norm as 1.311e-03."""
    golden = {}
    with open(os.path.join(GOLDEN, "kgrouped_repro_reference_norm.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                golden[k] = float(v)
    w = wl.kgrouped_repro()
    gy, act = w.draw()
    qa, sfa = oracle.quant_per_channel_128(gy)
    qb, sfb = oracle.quant_per_channel_128(act)
    d = oracle.gemm_kgrouped(oracle.pack_kmajor(qa, w.ks), sfa, oracle.pack_kmajor(qb, w.ks), sfb,
                             w.ks, w.N, w.H)
    norms = np.sqrt((d.reshape(4, -1) ** 2).sum(1))
    assert abs(norms.max() - golden["reference_max_norm"]) / golden["reference_max_norm"] < 0.01
    closed128 = math.sqrt(w.N * w.H * 128) * 1e-7 * 0.4
    assert abs(norms[1] - closed128) / closed128 < 0.01 and abs(norms[2] - closed128) / closed128 < 0.01


# ---------------------------------------------------------------------------------- comparison

def test_round_bf16_nearest_even():
    rng = np.random.default_rng(9)
    v = np.concatenate([rng.normal(0, 1, 100_000) * np.ldexp(1.0, rng.integers(-130, 120, 100_000)),
                        [0.0, -0.0, 1.0, 3.0e38, 3.5e38, 1e-45]])
    r = oracle.bf16_bits_to_f64(oracle.round_bf16(v))
    # neighbours from the bf16 bit pattern (truncation toward zero and the next code)
    f = v.astype(np.float32)
    ok = np.isfinite(f) & (np.abs(v) < 3.38e38)
    t = (f[ok].view(np.uint32) & 0xFFFF0000).view(np.float32).astype(np.float64)
    nxt = ((f[ok].view(np.uint32) & 0xFFFF0000) + 0x10000).view(np.float32).astype(np.float64)
    dv = np.abs(v[ok] - r[ok])
    assert np.all(dv <= np.abs(v[ok] - t)) and np.all(dv <= np.abs(v[ok] - nxt))
    # ties go to the even code
    one = 1.0 + 2.0 ** -8                               # halfway between 1 and 1+2^-7
    assert oracle.round_bf16([one])[0] == 0x3F80
    assert oracle.round_bf16([1.0 + 3 * 2.0 ** -8])[0] == 0x3F82
    assert oracle.round_bf16([3.5e38])[0] == 0x7F80      # overflow -> inf


def test_calc_diff_closed_forms():
    rng = np.random.default_rng(1)
    x = rng.normal(size=1000)
    assert oracle.calc_diff(x, x) == 0.0
    assert abs(oracle.calc_diff(x, np.zeros_like(x)) - 1.0) < 1e-15
    assert abs(oracle.calc_diff(x, -x) - 2.0) < 1e-15
    eps = 1e-3
    want = eps ** 2 / (2 + 2 * eps + eps ** 2)
    assert abs(oracle.calc_diff(x, (1 + eps) * x) - want) < 1e-12


# ---------------------------------------------------------------------------- BF16 grouped GEMM
# "Fix cross-expert output overwrites in SM90 masked GEMM" (#469), reproduction: the reference
# of m_grouped_bf16_gemm_nt_masked is bmm(a.double(), b.double().mT) on the valid rows.

def _bf16(shape, seed, scale=1.0):
    return wl.randn_bf16(shape, seed, scale)


@pytest.mark.parametrize("G,cap,N,K", [(3, 7, 5, 9), (2, 33, 16, 40)])
def test_bf16_masked_equals_batched_matmul_on_valid_rows(G, cap, N, K):
    a, b = _bf16((G, cap, K), 71), _bf16((G, N, K), 72)
    counts = np.array([cap, 0, 3][:G], np.int32)
    d = oracle.gemm_masked_bf16(a, b, counts)
    ref = np.einsum("grk,gnk->grn", a.double().numpy(), b.double().numpy())   # library routine
    for g in range(G):
        v = int(np.clip(counts[g], 0, cap))
        np.testing.assert_allclose(d[g, :v], ref[g, :v], rtol=1e-12, atol=1e-12)
        assert np.all(np.isnan(d[g, v:])), "rows past the count must stay untouched"


def test_bf16_masked_counts_clamped():
    a, b = _bf16((2, 4, 8), 73), _bf16((2, 3, 8), 74)
    d = oracle.gemm_masked_bf16(a, b, np.array([-3, 99], np.int32))
    assert np.all(np.isnan(d[0])) and not np.any(np.isnan(d[1]))


def test_bf16_products_exact_closed_form():
    """One nonzero K term per output: D is the exact product of two bf16 values; a permutation
    matrix as B permutes A's columns (a transposed operand or a wrong index fails here)."""
    G, cap, K = 1, 4, 8
    a = _bf16((G, cap, K), 75)
    perm = np.random.default_rng(3).permutation(K)
    b = torch.zeros((G, K, K), dtype=torch.bfloat16)
    b[0, np.arange(K), perm] = 1.0                    # row n of B selects A column perm[n]
    d = oracle.gemm_masked_bf16(a, b, np.array([cap], np.int32))
    np.testing.assert_array_equal(d[0], a[0].double().numpy()[:, perm])


def test_bf16_contiguous_routing():
    M, G, N, K = 10, 3, 6, 12
    a, b = _bf16((M, K), 76), _bf16((G, N, K), 77)
    mi = np.array([0, 0, 2, -1, 1, 7, 2, 2, -1, 0], np.int32)
    d = oracle.gemm_contiguous_bf16(a, b, mi)
    an, bn = a.double().numpy(), b.double().numpy()
    for m in range(M):
        if 0 <= mi[m] < G:
            np.testing.assert_allclose(d[m], bn[mi[m]] @ an[m], rtol=1e-12, atol=1e-12)
        else:
            assert np.all(np.isnan(d[m]))


# ---------------------------------------------------------------------------- psum layouts

def test_sizes_from_psum_inverts_cumsum():
    ks = np.array([256, 0, 128, 384, 0, 128], np.int32)
    np.testing.assert_array_equal(oracle.sizes_from_psum(np.cumsum(ks).astype(np.int32)), ks)


@pytest.mark.parametrize("counts", [[130, 0, 1, 128, 257], [0, 0, 5], [128, 256, 1], [300]])
def test_m_indices_from_psum_matches_the_padded_layout(counts):
    """The psum reading reproduces, row for row, the 128-aligned segments of the m_indices layout."""
    M = wl.contiguous_capacity(sum(counts), len(counts))
    np.testing.assert_array_equal(oracle.m_indices_from_psum(wl.contiguous_psum(counts), M),
                                  wl.contiguous_m_indices(counts, m_max=M))


def test_m_indices_from_psum_stops_at_the_first_bad_entry():
    M = 1024
    base = wl.contiguous_psum([130, 50, 10])           # [130, 306, 394]
    for bad, e in ([130, 100, 394], 1), ([130, 306, 2000], 2), ([130, 200, 394], 1):
        mi = oracle.m_indices_from_psum(np.array(bad, np.int32), M)
        good = oracle.m_indices_from_psum(base, M)
        first_row_of_e = {1: 256, 2: 384}[e]
        np.testing.assert_array_equal(mi[:first_row_of_e], good[:first_row_of_e])
        assert np.all(mi[first_row_of_e:] == -1)


# ------------------------------------------------------------------------------ plain / batched GEMM

def _random_codes(rng, shape):
    q = rng.integers(0, 256, shape, dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0          # no NaN codes
    return q


def test_batched_gemm_matches_numpy_einsum_and_adds_c():
    """The plain/batched oracle GEMM equals numpy's einsum over torch-decoded operands with the
    block scales expanded (an independent route), C is added as given, and B = 1 is a plain GEMM."""
    rng = np.random.default_rng(7)
    Bt, M, N, K = 3, 5, 256, 384
    qa, qb = _random_codes(rng, (Bt, M, K)), _random_codes(rng, (Bt, N, K))
    sfa = rng.uniform(0.5, 2.0, (Bt, M, K // 128)).astype(np.float32)
    sfb = rng.uniform(0.5, 2.0, (Bt, N // 128, K // 128)).astype(np.float32)
    c = rng.standard_normal((Bt, M, N))
    dec = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    A = dec[qa] * np.repeat(sfa.astype(np.float64), 128, axis=2)
    B = dec[qb] * np.repeat(np.repeat(sfb.astype(np.float64), 128, axis=1), 128, axis=2)
    prod = np.einsum("bmk,bnk->bmn", A, B)
    got = oracle.gemm_batched(qa, sfa, qb, sfb, c)
    np.testing.assert_allclose(got, c + prod, rtol=0, atol=1e-9 * np.abs(prod).max())
    np.testing.assert_allclose(oracle.gemm_batched(qa, sfa, qb, sfb), prod, rtol=0, atol=1e-9 * np.abs(prod).max())
    one = oracle.gemm_batched(qa[:1], sfa[:1], qb[:1], sfb[:1])
    np.testing.assert_array_equal(one[0], oracle.gemm_batched(qa, sfa, qb, sfb)[0])


def test_batched_gemm_equals_masked_at_full_counts_and_contiguous_single_expert():
    """Batched GEMM = masked GEMM with every count = capacity; a plain GEMM = the contiguous
    GEMM with every row routed to expert 0 (bitwise: same fp64 sums in the same order)."""
    rng = np.random.default_rng(8)
    Bt, M, N, K = 2, 7, 128, 256
    qa, qb = _random_codes(rng, (Bt, M, K)), _random_codes(rng, (Bt, N, K))
    sfa = rng.uniform(0.5, 2.0, (Bt, M, K // 128)).astype(np.float32)
    sfb = rng.uniform(0.5, 2.0, (Bt, N // 128, K // 128)).astype(np.float32)
    got = oracle.gemm_batched(qa, sfa, qb, sfb)
    np.testing.assert_array_equal(got, oracle.gemm_masked(qa, sfa, qb, sfb, np.full(Bt, M, np.int32)))
    cont = oracle.gemm_contiguous(qa[0], sfa[0], qb[:1], sfb[:1], np.zeros(M, np.int32))
    np.testing.assert_array_equal(got[0], cont)


# ------------------------------------------------------------------------------ FP4 (e2m1) weights

def e2m1_grid():
    """The non-negative e2m1 values by code 0..7, from the format definition (exponent bias 1,
    one mantissa bit, subnormal at exponent 0), not from the oracle."""
    vals = []
    for e in range(4):
        for m in range(2):
            vals.append(m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
    return np.array(vals)


def test_e2m1_decode_matches_format_definition():
    grid = e2m1_grid()
    np.testing.assert_array_equal(grid, [0, 0.5, 1, 1.5, 2, 3, 4, 6])
    got = oracle.e2m1_decode(np.arange(16, dtype=np.uint8))
    np.testing.assert_array_equal(got[:8], grid)
    np.testing.assert_array_equal(got[8:], -grid)
    assert math.copysign(1.0, got[8]) == -1.0            # code 8 is -0


def test_e2m1_encode_roundtrip_midpoints_and_saturation():
    grid = e2m1_grid()
    codes = np.arange(16, dtype=np.uint8)
    vals = oracle.e2m1_decode(codes)
    np.testing.assert_array_equal(oracle.e2m1_encode(vals.astype(np.float32)), codes)
    mids = (grid[:-1] + grid[1:]) / 2                  # ties go to the even code
    got = oracle.e2m1_encode(mids.astype(np.float32))
    want = np.array([c if c % 2 == 0 else c + 1 for c in range(7)], np.uint8)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(oracle.e2m1_encode(-mids.astype(np.float32)), want | 8)
    big = np.array([6.0, 6.5, 7.0, 1e30, np.inf], np.float32)
    np.testing.assert_array_equal(oracle.e2m1_encode(big), 7)
    np.testing.assert_array_equal(oracle.e2m1_encode(-big), 15)
    # brute force: every other value goes to the nearest grid point
    rng = np.random.default_rng(5)
    y = rng.uniform(-7, 7, 20000).astype(np.float32)
    q = oracle.e2m1_encode(y)
    dec = oracle.e2m1_decode(q)
    full = np.concatenate([grid, -grid])
    nearest = np.abs(np.abs(y.astype(np.float64))[:, None] - grid[None, :]).min(axis=1)
    sat = np.abs(y) >= 6
    np.testing.assert_array_equal(np.abs(np.abs(y[~sat]) - np.abs(dec[~sat])), nearest[~sat])
    assert np.all(np.sign(dec[dec != 0]) == np.sign(y[dec != 0]))
    assert set(np.unique(dec)) <= set(full)


def _unpack_fp4(q_packed):
    lo, hi = q_packed & 0xF, q_packed >> 4
    out = np.empty(q_packed.shape[:-1] + (q_packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2], out[..., 1::2] = lo, hi
    return out


def test_fp4_block_cast_pins():
    """Zero blocks take sf_zero rounded up to a power of two with zero codes; a block whose amax is
    6 * 2^k gets the scale 2^k and reproduces grid values exactly; every code is the nearest
    e2m1 value of x / sf (brute force over the grid); the even element sits in the low nibble."""
    grid = e2m1_grid()
    G, N, K = 2, 128, 256
    rng = np.random.default_rng(9)
    w = np.zeros((G, N, K))
    w[0, :, :128] = rng.choice(np.concatenate([grid, -grid]), (128, 128)) * 4.0   # amax 24 = 6 * 2^2
    w[0, 0, 0] = 24.0
    w[1] = rng.standard_normal((N, K)) * 0.3                                      # block (1, 0, *)
    wt = bf16_from_f64(np.asarray(torch.tensor(w).to(torch.bfloat16).double()))
    q, ue = oracle.quant_block_128x128_fp4(wt, sf_zero=1e-30)
    assert q.shape == (G, N, K // 2) and ue.shape == (G, 1, 2)
    codes = _unpack_fp4(q)
    assert ue[0, 0, 0] == 127 + 2
    np.testing.assert_array_equal(oracle.e2m1_decode(codes[0, :, :128]) * 4.0, w[0, :, :128])
    # the zero block: sf_zero = 1e-30 rounds up to 2^-99
    assert ue[0, 0, 1] == 127 - 99 and np.all(codes[0, :, 128:] == 0)
    # random block: scale = 2^ceil(log2(amax / 6)) in fp32, codes nearest to x / sf
    wf = wt.double().numpy()
    for kb in range(2):
        blk = wf[1, :, kb * 128:(kb + 1) * 128]
        amax = np.float32(np.abs(blk).max())
        sf = np.float32(amax / np.float32(6.0))
        e = int(np.frexp(sf)[1]) - 1 + (0 if np.frexp(sf)[0] == 0.5 else 1)
        assert ue[1, 0, kb] == 127 + e
        y = blk / 2.0 ** e
        dec = oracle.e2m1_decode(codes[1, :, kb * 128:(kb + 1) * 128])
        nearest = np.abs(np.abs(y)[..., None] - grid).min(axis=-1)
        np.testing.assert_array_equal(np.abs(np.abs(y) - np.abs(dec)), nearest)
    # packing: element 2i in the low nibble, 2i + 1 in the high nibble
    np.testing.assert_array_equal(q & 0xF, codes[..., 0::2])
    np.testing.assert_array_equal(q >> 4, codes[..., 1::2])


def test_fp4_gemms_equal_the_fp8_gemms_on_the_same_values():
    """Every e2m1 value is an e4m3 value, so the FP4-weight GEMMs must equal the (pinned) FP8 GEMMs
    fed the e4m3 codes of the same weight values, bit for bit; and numpy's einsum."""
    rng = np.random.default_rng(13)
    G, N, K, M = 3, 128, 256, 7
    q4 = rng.integers(0, 16, (G, N, K), dtype=np.uint8)
    packed = (q4[..., 0::2] | (q4[..., 1::2] << 4)).astype(np.uint8)
    q8 = oracle.e4m3_encode(oracle.e2m1_decode(q4).astype(np.float32))
    np.testing.assert_array_equal(oracle.e4m3_decode(q8), oracle.e2m1_decode(q4))
    qa = _random_codes(rng, (M, K))
    sfa = rng.uniform(0.5, 2.0, (M, K // 128)).astype(np.float32)
    sfb = np.ldexp(np.float32(1.0), rng.integers(-4, 4, (G, N // 128, K // 128))).astype(np.float32)
    mi = np.array([0, 2, -1, 1, 2, 0, 5], np.int32)
    got = oracle.gemm_contiguous_fp4(qa, sfa, packed, sfb, mi)
    want = oracle.gemm_contiguous(qa, sfa, q8, sfb, mi)
    np.testing.assert_array_equal(got, want)
    A = oracle.e4m3_decode(qa) * np.repeat(sfa.astype(np.float64), 128, axis=1)
    B = oracle.e2m1_decode(q4) * np.repeat(np.repeat(sfb.astype(np.float64), 128, axis=1), 128, axis=2)
    for m in range(M):
        if 0 <= mi[m] < G:
            np.testing.assert_allclose(got[m], B[mi[m]] @ A[m], rtol=1e-12, atol=1e-12 * np.abs(B).max())
        else:
            assert np.all(np.isnan(got[m]))
    cap = 3
    qam = _random_codes(rng, (G, cap, K))
    sfam = rng.uniform(0.5, 2.0, (G, cap, K // 128)).astype(np.float32)
    counts = np.array([3, 0, 2], np.int32)
    np.testing.assert_array_equal(oracle.gemm_masked_fp4(qam, sfam, packed, sfb, counts),
                                  oracle.gemm_masked(qam, sfam, q8, sfb, counts))


# Plumbing that computes nothing the path does (compilation, thread count).
_NOT_ARITHMETIC = {"build", "num_threads"}


def test_every_exported_oracle_function_has_a_pin():
    """Each public function of the oracle is called by at least one test in this file, so none
    is left unpinned (a function that nothing pins must be pinned or removed)."""
    import inspect
    src = open(__file__).read()
    public = [n for n, f in vars(oracle).items()
              if inspect.isfunction(f) and not n.startswith("_") and f.__module__ == oracle.__name__]
    missing = [n for n in public if n not in _NOT_ARITHMETIC and f"oracle.{n}(" not in src]
    assert not missing, f"oracle functions without a pin: {missing}"
