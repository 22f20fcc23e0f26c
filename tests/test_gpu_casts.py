"""GPU parity of the three cast kernels against the oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_SF_FP32, DG_SF_UE8M0, DG_STATUS_K_NOT_ALIGNED, DG_STATUS_K_OVERFLOW
from moe_grouped_fp8_gb300 import api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import gpu_quant_blocks, gpu_quant_channels, gpu_quant_tokens, set_token_items_per_cta, sfa_rows, sync

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("M,K,scale", [(1, 128, 1.0), (37, 256, 3.0), (300, 1024, 1e-3), (1029, 7168, 0.02)])
def test_per_token_codes_and_scales_bit_exact(fmt, M, K, scale):
    x = wl.randn_bf16((M, K), 100 + M, scale)
    x[0, :128] = 0                                     # all-zero block -> sf_zero
    if M > 3:
        x[3, 128 % K:128 % K + 5] = 448 * scale * 30    # dominant element
    q, sfa = gpu_quant_tokens(x.cuda(), fmt, sf_zero=0.5)
    sync()
    oq, osf, oue = oracle.quant_per_token_1x128(x, sf_zero=0.5, ue8m0=(fmt == DG_SF_UE8M0))
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    got = sfa_rows(sfa, M)
    if fmt == DG_SF_FP32:
        np.testing.assert_array_equal(got.view(np.uint32), osf.view(np.uint32))
    else:
        np.testing.assert_array_equal(got, oue)


FINITE_MAGNITUDES = np.arange(1, 0x7F80, dtype=np.uint32)  # every finite positive bf16, subnormals included


def magnitude_blocks(mags: np.ndarray, size: int, seed: int) -> np.ndarray:
    """bf16 bits [n, size]: block i holds +-mags[i] once and mags[i] * u (|u| < 1, truncated to
    bf16) elsewhere, so mags[i] is its amax."""
    n = mags.size
    v = (mags.astype(np.uint32) << 16).view(np.float32)
    rng = np.random.default_rng(seed)
    blk = (v[:, None] * rng.uniform(-1.0, 1.0, (n, size)).astype(np.float32)).astype(np.float32)
    bits = (blk.view(np.uint32) >> 16).astype(np.uint16)
    pos = (np.arange(n) * 37) % size
    bits[np.arange(n), pos] = mags.astype(np.uint16) | np.where(rng.random(n) < 0.5, 0x8000, 0).astype(np.uint16)
    return bits


def as_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def every_bf16_magnitude_blocks(seed: int) -> torch.Tensor:
    """Rows of 64 1x128 blocks, one per finite bf16 magnitude (the last block repeats 1.0)."""
    mags = np.concatenate([FINITE_MAGNITUDES, np.full((-FINITE_MAGNITUDES.size) % 64, 0x3F80, np.uint32)])
    return as_bf16(magnitude_blocks(mags, 128, seed).reshape(mags.size // 64, 64 * 128))


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
def test_per_token_every_bf16_magnitude_as_block_amax(fmt):
    """Each finite bf16 magnitude is the amax of one block, so every scale (and its reciprocal)
    the cast can form from bf16 input is checked against the oracle's IEEE arithmetic."""
    x = every_bf16_magnitude_blocks(61)
    M = x.shape[0]
    q, sfa = gpu_quant_tokens(x.cuda(), fmt, sf_zero=0.25)
    sync()
    oq, osf, oue = oracle.quant_per_token_1x128(x, sf_zero=0.25, ue8m0=(fmt == DG_SF_UE8M0))
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    got = sfa_rows(sfa, M)
    if fmt == DG_SF_FP32:
        np.testing.assert_array_equal(got.view(np.uint32), osf.view(np.uint32))
    else:
        np.testing.assert_array_equal(got, oue)


def test_per_token_strided_input_and_row_counts():
    G, cap, K = 5, 40, 512
    x = wl.randn_bf16((G, cap, K + 64), 7)             # padded rows: ldx = K + 64
    xd = x.cuda().view(G * cap, K + 64)[:, :K]
    counts = torch.tensor([0, 40, 13, 99, 1], dtype=torch.int32)
    q, sfa = gpu_quant_tokens(xd, DG_SF_FP32, row_counts=counts.cuda())
    sync()
    oq, osf, _ = oracle.quant_per_token_1x128(x.view(G * cap, K + 64)[:, :K].contiguous(), row_counts=counts.numpy())
    live = np.zeros(G * cap, bool)
    for g, c in enumerate(np.clip(counts.numpy(), 0, cap)):
        live[g * cap:g * cap + c] = True
    qn = q.cpu().numpy()
    np.testing.assert_array_equal(qn[live], oq[live])
    assert np.all(qn[~live] == 0), "rows past the count must not be written"
    got = sfa_rows(sfa, G * cap)
    np.testing.assert_array_equal(got[live], osf[live])
    assert np.all(got[~live] == 0)


def test_per_channel_every_bf16_magnitude_as_column_amax():
    """Each finite bf16 magnitude is the amax of one (128-token block, column) pair of the
    per-channel cast, over three experts; codes, pack and scales bit-exact."""
    mags = np.concatenate([FINITE_MAGNITUDES, np.full(1, 0x3F80, np.uint32)])  # 32640 = 255 * 128
    C, TB = 128, mags.size // 128
    bits = magnitude_blocks(mags, 128, 62).reshape(TB, C, 128).transpose(0, 2, 1).reshape(TB * 128, C)
    x = as_bf16(bits)
    ks = [128 * 100, 128 * 100, 128 * 55]
    qp, sf = gpu_quant_channels(x.cuda(), torch.tensor(ks, dtype=torch.int32, device="cuda"), 0.125)
    sync()
    oq, osf = oracle.quant_per_channel_128(x, 0.125)
    np.testing.assert_array_equal(qp.cpu().numpy(), oracle.pack_kmajor(oq, ks))
    np.testing.assert_array_equal(sf.cpu().numpy().view(np.uint32), osf.view(np.uint32))


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
def test_block_sampled_bf16_magnitudes_as_block_amax(fmt):
    """Every 16th finite bf16 magnitude plus the 32 smallest and largest as the amax of one
    128x128 weight block each."""
    mags = np.unique(np.concatenate([FINITE_MAGNITUDES[::16], FINITE_MAGNITUDES[:32], FINITE_MAGNITUDES[-32:]]))
    mags = np.concatenate([mags, np.full((-mags.size) % 16, 0x3F80, np.uint32)])
    NB, KB = mags.size // 16, 16
    bits = magnitude_blocks(mags, 128 * 128, 63).reshape(NB, KB, 128, 128).transpose(0, 2, 1, 3)
    w = as_bf16(bits.reshape(1, NB * 128, KB * 128))
    q, sfb = gpu_quant_blocks(w.cuda(), fmt, sf_zero=4.0)
    sync()
    oq, osf, oue = oracle.quant_block_128x128(w, sf_zero=4.0, ue8m0=(fmt == DG_SF_UE8M0))
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    if fmt == DG_SF_FP32:
        np.testing.assert_array_equal(sfb.cpu().numpy().view(np.uint32), osf.view(np.uint32))
    else:
        np.testing.assert_array_equal(sfb.cpu().numpy(), oue)


def masked_cast_case(G, cap, K, counts, fmt, seed):
    x = wl.randn_bf16((G, cap, K), seed)
    counts = np.asarray(counts, np.int32)
    q, sfa = gpu_quant_tokens(x.cuda().view(G * cap, K), fmt, row_counts=torch.tensor(counts, device="cuda"))
    sync()
    ue = fmt == DG_SF_UE8M0
    oq, osf, oue = oracle.quant_per_token_1x128(x.view(G * cap, K), ue8m0=ue, row_counts=counts)
    live = (np.arange(cap)[None, :] < np.clip(counts, 0, cap)[:, None]).reshape(-1)
    qn = q.cpu().numpy()
    np.testing.assert_array_equal(qn[live], oq[live])
    assert np.all(qn[~live] == 0), "rows past the count must not be written"
    got = sfa_rows(sfa, G * cap)
    ref = oue if ue else osf
    np.testing.assert_array_equal(got[live].view(np.uint8), ref[live].view(np.uint8))
    assert np.all(got[~live] == 0)


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("G,cap,K", [(300, 5, 384), (6, 1000, 2048), (1100, 2, 128), (1, 77, 7168)])
def test_per_token_masked_groups(fmt, G, cap, K):
    """Valid rows of many groups (one index space walked by resident CTAs, several passes for the
    6 x 1000 case) and more groups than that walk takes (1100: one CTA row per group)."""
    rng = np.random.default_rng(G * 7 + cap)
    counts = rng.integers(-2, cap + 3, G)
    counts[0] = 0
    counts[-1] = cap
    masked_cast_case(G, cap, K, counts, fmt, 500 + G)


def routed_cast_case(counts, K, fmt, m_max=None, seed=3):
    mi = wl.contiguous_m_indices(counts, m_max=m_max)
    M = mi.size
    x = wl.randn_bf16((M, K), seed, 2.0)
    q = torch.full((M, K), 0xA5, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(M, K, fmt, "cuda")
    sfa.view(torch.uint8).fill_(0x5A)
    api.dg_quant_per_token_1x128_routed(x.cuda(), q, sfa, torch.tensor(mi, device="cuda"), fmt, 0.5)
    sync()
    ue = fmt == DG_SF_UE8M0
    oq, osf, oue = oracle.quant_per_token_1x128(x, sf_zero=0.5, ue8m0=ue)
    live = mi >= 0
    qn = q.cpu().numpy()
    np.testing.assert_array_equal(qn[live], oq[live])
    assert np.all(qn[~live] == 0xA5), "a padding row was written"
    got = sfa_rows(sfa, M)
    ref = oue if ue else osf
    np.testing.assert_array_equal(got[live].view(np.uint8), ref[live].view(np.uint8))
    assert np.all(got[~live].view(np.uint8) == 0x5A), "a padding row's scale was written"


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("counts,K", [([130, 0, 1, 128, 257], 384), ([3, 300, 0, 0, 45], 7168),
                                      ([1] * 40, 256), ([700], 65536)])
def test_per_token_routed_skips_padding_rows(fmt, counts, K):
    """Routed rows (m_indices >= 0) bit-exact against the oracle; padding rows inside expert
    segments and past the last segment keep the buffers' previous bytes."""
    routed_cast_case(counts, K, fmt, m_max=wl.contiguous_capacity(sum(counts), len(counts)))


@pytest.mark.parametrize("items", [1, 56, 64, 300, 5000])
def test_per_token_any_chunk_size(items):
    """The CTA chunk size (items per CTA) only changes the grid: plain, masked and routed casts
    stay bit-exact for chunks of one item up to several rows."""
    set_token_items_per_cta(items)
    try:
        x = wl.randn_bf16((301, 7168), 71, 0.5)
        q, sfa = gpu_quant_tokens(x.cuda(), DG_SF_FP32)
        sync()
        oq, osf, _ = oracle.quant_per_token_1x128(x)
        np.testing.assert_array_equal(q.cpu().numpy(), oq)
        np.testing.assert_array_equal(sfa_rows(sfa, 301).view(np.uint32), osf.view(np.uint32))
        masked_cast_case(7, 33, 384, [0, 33, 5, 40, 1, 17, 32], DG_SF_UE8M0, 72)
        routed_cast_case([130, 0, 1, 128, 9], 256, DG_SF_FP32, m_max=700)
    finally:
        set_token_items_per_cta(0)


def test_per_token_routed_all_padding_and_empty():
    routed_cast_case([0, 0, 0], 256, DG_SF_FP32, m_max=300)
    x = torch.zeros(0, 128, dtype=torch.bfloat16, device="cuda")
    api.dg_quant_per_token_1x128_routed(x, torch.zeros(0, 128, dtype=torch.uint8, device="cuda"),
                                        api.empty_sfa(0, 128, DG_SF_FP32, "cuda"),
                                        torch.zeros(0, dtype=torch.int32, device="cuda"))
    sync()


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("G,N,K,scale", [(1, 128, 128, 1.0), (3, 256, 384, 0.02), (2, 512, 1024, 5.0)])
def test_block_codes_and_scales_bit_exact(fmt, G, N, K, scale):
    w = wl.randn_bf16((G, N, K), 200 + G, scale)
    w[0, :128, :128] = 0
    q, sfb = gpu_quant_blocks(w.cuda(), fmt, sf_zero=2.0)
    sync()
    oq, osf, oue = oracle.quant_block_128x128(w, sf_zero=2.0, ue8m0=(fmt == DG_SF_UE8M0))
    np.testing.assert_array_equal(q.cpu().numpy(), oq)
    if fmt == DG_SF_FP32:
        np.testing.assert_array_equal(sfb.cpu().numpy().view(np.uint32), osf.view(np.uint32))
    else:
        np.testing.assert_array_equal(sfb.cpu().numpy(), oue)


@pytest.mark.parametrize("sf_zero", [1.0, 1e-4, 1e-8, 1e-30])
@pytest.mark.parametrize("ks,C", [([256, 128, 128, 256], 2048), ([128, 0, 384, 128], 192), ([640], 64)])
def test_per_channel_codes_pack_and_scales_bit_exact(ks, C, sf_zero):
    T = sum(ks)
    K_cap = T + 256                                     # capacity beyond sum(ks) is left untouched
    x = wl.randn_bf16((K_cap, C), 300 + C, 1e-7)
    o = 0
    for k in ks:
        if k == 128:
            x[o:o + k, 0] = 0
        o += k
    qp, sf = gpu_quant_channels(x.cuda(), torch.tensor(ks, dtype=torch.int32, device="cuda"), sf_zero)
    sync()
    oq, osf = oracle.quant_per_channel_128(x[:T], sf_zero)
    packed = oracle.pack_kmajor(oq, ks)
    qpn = qp.cpu().numpy()
    np.testing.assert_array_equal(qpn[:T * C], packed)
    assert np.all(qpn[T * C:] == 0)
    sfn = sf.cpu().numpy()
    np.testing.assert_array_equal(sfn[:T // 128].view(np.uint32), osf.view(np.uint32))
    assert np.all(sfn[T // 128:] == 0)


def test_per_channel_bad_ks_sets_status_and_stops():
    C = 128
    x = wl.randn_bf16((512, C), 5).cuda()
    for ks, bit, good in [([128, 100, 128], DG_STATUS_K_NOT_ALIGNED, 128), ([256, 512, 128], DG_STATUS_K_OVERFLOW, 256)]:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        qp, sf = gpu_quant_channels(x, torch.tensor(ks, dtype=torch.int32, device="cuda"), status=status)
        sync()
        assert status.item() & bit
        sfn = sf.cpu().numpy()
        assert np.all(sfn[:good // 128] > 0) and np.all(sfn[good // 128:] == 0)


def test_cast_matches_oracle_on_every_code_midpoint():
    """Device encode on values at every e4m3 midpoint (ties to even), with every scale exactly 1."""
    grid = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    vals = np.concatenate([grid.astype(np.float32), mids, -mids])
    n = (vals.size + 127) // 128 * 128
    row = np.zeros(n, np.float32)
    row[:vals.size] = vals
    row = row.reshape(-1, 128)
    row[:, 0] = 448.0                                    # every block has amax 448 -> sf = 1 exactly
    x = torch.from_numpy(row).to(torch.bfloat16)
    assert torch.equal(x.float(), torch.from_numpy(row)), "midpoints are bf16-exact"
    q, sfa = gpu_quant_tokens(x.cuda(), DG_SF_FP32)
    sync()
    oq, osf, _ = oracle.quant_per_token_1x128(x)
    assert np.all(osf == 1.0)
    np.testing.assert_array_equal(q.cpu().numpy(), oq)


@pytest.mark.parametrize("ks,Ca,Cb", [([256, 128, 128, 256], 2048, 2048), ([128, 0, 384], 192, 64)])
def test_per_channel_pair_equals_two_single_calls(ks, Ca, Cb):
    from moe_grouped_fp8_gb300 import api
    T = sum(ks)
    K_cap = T + 128
    xa = wl.randn_bf16((K_cap, Ca), 7, 1e-7)
    xb = wl.randn_bf16((K_cap, Cb), 8, 0.4)
    xa[128:256, 0] = 0
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    qa1, sa1 = gpu_quant_channels(xa.cuda(), ks_dev, 1e-4)
    qb1, sb1 = gpu_quant_channels(xb.cuda(), ks_dev, 1e-4)
    qa2 = torch.zeros_like(qa1)
    qb2 = torch.zeros_like(qb1)
    sa2 = torch.zeros_like(sa1)
    sb2 = torch.zeros_like(sb1)
    api.dg_quant_per_channel_128_pair(xa.cuda(), xb.cuda(), ks_dev, qa2, sa2, qb2, sb2, sf_zero=1e-4)
    sync()
    for one, two in ((qa1, qa2), (qb1, qb2), (sa1, sa2), (sb1, sb2)):
        assert torch.equal(one.view(torch.uint8), two.view(torch.uint8))
    oq, osf = oracle.quant_per_channel_128(xb[:T], 1e-4)
    np.testing.assert_array_equal(qb2.cpu().numpy()[:T * Cb], oracle.pack_kmajor(oq, ks))
    np.testing.assert_array_equal(sb2.cpu().numpy()[:T // 128].view(np.uint32), osf.view(np.uint32))


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("counts,cap,K", [([3, 40, 0, 17, 40], 40, 384), ([0, 0, 0], 16, 256),
                                          ([300, -2, 1, 129, 0, 257], 257, 7168), ([1] * 40, 8, 128)])
def test_per_token_packed_equals_masked_cast(fmt, counts, cap, K):
    """The cast from packed rows writes the same codes and scales, at the same masked positions,
    as the masked cast of the same rows scattered into [G, cap, K] (itself pinned to the oracle
    above); rows past the counts stay untouched, and rows of x past the packed ones are not read."""
    G = len(counts)
    M = G * cap
    v = np.clip(counts, 0, cap)
    x = wl.randn_bf16((M, K), 91, 0.5)
    x[torch.from_numpy(np.arange(cap)[None, :].repeat(G, 0).ravel() >= np.repeat(v, cap))] = float("nan")
    rows = np.concatenate([np.arange(g * cap, g * cap + v[g]) for g in range(G)]).astype(np.int64)
    packed = torch.full((M, K), float("nan"), dtype=torch.bfloat16)  # NaN rows past the packed ones
    packed[: len(rows)] = x[torch.from_numpy(rows)]
    cnt = torch.tensor(np.asarray(counts, np.int32), device="cuda")
    outs = []
    for packed_in in (False, True):
        q = torch.full((M, K), 0xA5, dtype=torch.uint8, device="cuda")
        sfa = api.empty_sfa(M, K, fmt, "cuda")
        sfa.view(torch.uint8).fill_(0x5A)
        if packed_in:
            api.dg_quant_per_token_1x128_packed(packed.cuda(), q, sfa, cnt, fmt)
        else:
            api.dg_quant_per_token_1x128(x.cuda(), q, sfa, fmt, row_counts=cnt)
        sync()
        outs.append((q.cpu().numpy(), sfa.view(torch.uint8).cpu().numpy()))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])
    if len(rows):
        oq, osf, _ = oracle.quant_per_token_1x128(x[torch.from_numpy(rows)], ue8m0=fmt == DG_SF_UE8M0)
        np.testing.assert_array_equal(outs[1][0][rows], oq)


@pytest.mark.parametrize("counts,cap,width,dtype", [([5, 0, 130, 64], 130, 6144, torch.bfloat16),
                                                    ([0, 0], 4, 256, torch.float32),
                                                    ([3, -1, 9, 2000], 16, 8, torch.bfloat16),
                                                    ([191] * 32, 256, 6144, torch.bfloat16)])
def test_pack_masked_rows(counts, cap, width, dtype):
    """Each group's first clamp(count, 0, cap) rows land packed, group after group, byte for byte;
    dst past them is untouched."""
    G = len(counts)
    v = np.clip(counts, 0, cap)
    src = wl.randn_bf16((G, cap, width), 92, 1.0).to(dtype)
    dst = torch.full((G * cap, width), -1, dtype=torch.int16 if dtype == torch.bfloat16 else torch.int32,
                     device="cuda").view(dtype)
    api.dg_pack_masked_rows(src.cuda(), torch.tensor(np.asarray(counts, np.int32), device="cuda"), dst)
    sync()
    got = dst.cpu().contiguous().view(torch.uint8).numpy().reshape(G * cap, -1)
    want = torch.cat([src[g, : v[g]] for g in range(G)]).contiguous().view(torch.uint8).numpy().reshape(-1, got.shape[1])
    n = int(v.sum())
    np.testing.assert_array_equal(got[:n], want)
    assert np.all(got[n:] == 0xFF)


@pytest.mark.slow
def test_packed_cast_and_row_packing_at_decode_size():
    """At the decode size (G=32, cap=4096, K=7168, N=6144, Poisson(192) counts): the packed cast
    equals the masked cast of the same rows bitwise, and the row packing of a [32, 4096, 6144] bf16
    buffer equals the valid rows gathered by index."""
    w = wl.masked_decode()
    G, cap, K, N = w.G, w.cap, w.K, w.N
    counts = np.asarray(w.counts, np.int32)
    v = np.clip(counts, 0, cap)
    rows = torch.from_numpy(np.concatenate([np.arange(g * cap, g * cap + v[g]) for g in range(G)])).cuda()
    x = wl.randn_bf16((G * cap, K), 93, 1.0, "cuda")
    packed = torch.empty_like(x)
    packed[: rows.numel()] = x[rows]
    cnt = torch.tensor(counts, device="cuda")
    outs = []
    for packed_in in (False, True):
        q = torch.zeros(G * cap, K, dtype=torch.uint8, device="cuda")
        sfa = api.empty_sfa(G * cap, K, DG_SF_FP32, "cuda")
        sfa.zero_()
        if packed_in:
            api.dg_quant_per_token_1x128_packed(packed, q, sfa, cnt, DG_SF_FP32)
        else:
            api.dg_quant_per_token_1x128(x, q, sfa, DG_SF_FP32, row_counts=cnt)
        outs.append((q, sfa))
    sync()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    del x, packed, outs
    d = wl.randn_bf16((G, cap, N), 94, 1.0, "cuda")
    dst = torch.full((G * cap, N), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    api.dg_pack_masked_rows(d, cnt, dst)
    sync()
    n = rows.numel()
    assert torch.equal(dst[:n].view(torch.int16), d.view(G * cap, N)[rows].view(torch.int16))
    assert bool((dst[n:].view(torch.int16) == -1).all())
