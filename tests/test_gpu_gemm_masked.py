"""GPU parity of the m-grouped masked FP8 GEMM against the oracle (cast -> GEMM on the device,
the oracle's own cast -> fp64 GEMM on the host, from the same bf16 bytes)."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_SF_FP32, DG_SF_UE8M0, DG_STATUS_COUNT_GT_CAP, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import (assert_close, gpu_quant_blocks, gpu_quant_tokens, out_bits, ref_out, sentinel_like,
                         sentinel_value, set_mgrouped_bn, set_mgrouped_kernel, set_mgrouped_store, set_mgrouped_warps, sync,
                         to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["auto", "promotion", "mx"], autouse=True)
def ue8m0_kernel(request):
    """Calls with UE8M0 scales run on the kernel the library picks, then forced onto the promotion
    kernel and onto the block-scaled MMA kernel (where N % 256 == 0); fp32-scale cases and full-size
    cases run once, on the library's choice."""
    if request.param != "auto":
        cs = getattr(request.node, "callspec", None)
        fmt = cs.params.get("fmt") if cs is not None else None
        if request.node.get_closest_marker("slow") or (fmt != DG_SF_UE8M0 and not request.node.get_closest_marker("ue8m0")):
            pytest.skip("one kernel for this case")
    set_mgrouped_kernel(request.param)
    yield request.param
    set_mgrouped_kernel("auto")


def masked_case(a, b, counts, fmt=DG_SF_FP32, out=torch.bfloat16, expected_m=0, calls=1):
    """Run the device path `calls` times into one sentinel-filled output and check it."""
    G, cap, K = a.shape
    N = b.shape[1]
    ad, bd = a.cuda(), b.cuda()
    cnt = torch.tensor(np.asarray(counts, np.int32), device="cuda")
    qa, sfa = gpu_quant_tokens(ad.view(G * cap, K), fmt)
    qb, sfb = gpu_quant_blocks(bd, fmt)
    d = sentinel_like((G, cap, N), out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = None
    for i in range(calls):
        api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, expected_m, fmt, status)
        if calls > 1:
            bits = out_bits(d)
            if first is None:
                first = bits
            else:
                assert np.array_equal(bits, first), f"call {i} differs bitwise from call 0"
    sync()
    ue = fmt == DG_SF_UE8M0
    oqa, osfa, _ = oracle.quant_per_token_1x128(a.view(G * cap, K), ue8m0=ue)
    oqb, osfb, _ = oracle.quant_block_128x128(b, ue8m0=ue)
    np.testing.assert_array_equal(qa.cpu().numpy(), oqa)
    np.testing.assert_array_equal(qb.cpu().numpy(), oqb)
    ref = oracle.gemm_masked(oqa.reshape(G, cap, K), osfa.reshape(G, cap, K // 128), oqb, osfb, counts)
    v = np.clip(np.asarray(counts), 0, cap)
    valid = np.arange(cap)[None, :] < v[:, None]
    fp32 = out == torch.float32
    if valid.any():
        assert_close(to_f64(d)[valid], ref_out(ref[valid], fp32), fp32, "masked valid rows")
    assert np.all(out_bits(d)[~valid] == sentinel_value(out)), "a row at or past its expert's count was written"
    return d, status


def test_pages_boundary_repro_16_calls():
    """G=8, cap=32, N=K=256, counts [0,1,16,31,32,1,32,32], seed 29; 16 calls, all bitwise equal;
    valid rows within tolerance; every padding row keeps its sentinel."""
    w = wl.masked_repro()
    a, b = w.draw()
    masked_case(a, b, w.counts, calls=16, expected_m=32)


CAPS = [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 96, 127, 128, 129, 160, 200, 255, 256, 257]


@pytest.mark.parametrize("cap", CAPS)
def test_capacity_panel(cap):
    rng = np.random.default_rng(cap)
    G, N, K = 4, 256, 256
    counts = rng.integers(0, cap + 1, G)
    counts[rng.integers(0, G)] = cap                  # one full expert
    counts[rng.integers(0, G)] = 0                    # one empty expert
    a = wl.randn_bf16((G, cap, K), 1000 + cap)
    b = wl.randn_bf16((G, N, K), 2000 + cap)
    masked_case(a, b, counts)


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_formats_and_output_dtypes(fmt, out):
    G, cap, N, K = 3, 200, 384, 512
    a = wl.randn_bf16((G, cap, K), 11, 2.0)
    b = wl.randn_bf16((G, N, K), 12, 0.02)
    masked_case(a, b, [200, 77, 129], fmt=fmt, out=out)


def test_odd_blocks_and_narrow_tiles():
    """Groups of 5 and 4 m-blocks (partial last blocks), N = 640 (five 128-column tiles)."""
    G, cap, N, K = 2, 640, 640, 256
    a = wl.randn_bf16((G, cap, K), 97)
    b = wl.randn_bf16((G, N, K), 98, 0.05)
    masked_case(a, b, [640, 385])


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("K", [384, 4224])
def test_wide_tiles_promotion_warps_bitwise_equal(ue8m0_kernel, fmt, K):
    """N = 1024: 128 x 256 tiles of the promotion kernel, promoted by 16 warps (64 accumulators per
    thread, the default) or by 8 (128 each); both pass the oracle check and give the same bits, with
    owner-thread stores (K = 384) and staged TMA stores (K = 4224, 33 blocks)."""
    if ue8m0_kernel != "auto":
        pytest.skip("a property of the promotion kernel, forced below")
    set_mgrouped_kernel("promotion")
    G, cap, N = 3, 300, 1024
    a = wl.randn_bf16((G, cap, K), 15, 2.0)
    b = wl.randn_bf16((G, N, K), 16, 0.02)
    outs = []
    try:
        for warps in (16, 8):
            set_mgrouped_warps(warps)
            d, _ = masked_case(a, b, [300, 77, 129], fmt=fmt)
            outs.append(out_bits(d))
    finally:
        set_mgrouped_warps(0)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
def test_tile_widths_bitwise_equal(ue8m0_kernel, fmt):
    """The promotion kernel on 128- and 256-column tiles: both pass the oracle check, same bits."""
    if ue8m0_kernel != "auto":
        pytest.skip("a property of the promotion kernel, forced below")
    G, cap, N, K = 3, 260, 512, 640
    a = wl.randn_bf16((G, cap, K), 19, 2.0)
    b = wl.randn_bf16((G, N, K), 20, 0.02)
    outs = []
    set_mgrouped_kernel("promotion")
    try:
        for bn in (128, 256):
            set_mgrouped_bn(bn)
            d, _ = masked_case(a, b, [260, 9, 131], fmt=fmt)
            outs.append(out_bits(d))
    finally:
        set_mgrouped_bn(0)
    assert np.array_equal(outs[0], outs[1])


def test_single_expert_and_all_empty():
    a = wl.randn_bf16((1, 130, 256), 21)
    b = wl.randn_bf16((1, 128, 256), 22)
    masked_case(a, b, [130])
    a3 = wl.randn_bf16((3, 64, 256), 23)
    b3 = wl.randn_bf16((3, 128, 256), 24)
    masked_case(a3, b3, [0, 0, 0])


def test_expected_m_does_not_change_result():
    w = wl.masked_repro()
    a, b = w.draw()
    d1, _ = masked_case(a, b, w.counts, expected_m=1)
    d2, _ = masked_case(a, b, w.counts, expected_m=4096)
    assert np.array_equal(out_bits(d1), out_bits(d2))


@pytest.mark.parametrize("N,out", [(512, torch.bfloat16), (1024, torch.bfloat16), (384, torch.float32)])
def test_store_paths_bitwise_equal(N, out):
    """Tile stores by TMA (issued by thread 0 of the promotion warps) or from registers by each
    row's owner thread: each passes the oracle check (valid rows, untouched padding rows) and both
    give the same bits, on 128- and 256-column tiles, with partial tiles that need owner-thread
    tails."""
    G, cap, K = 3, 300, 512
    a = wl.randn_bf16((G, cap, K), 17, 1.5)
    b = wl.randn_bf16((G, N, K), 18, 0.02)
    outs = []
    try:
        for which in ("thread0", "direct"):
            set_mgrouped_store(which)
            d, _ = masked_case(a, b, [300, 77, 133], out=out, calls=2)
            outs.append(out_bits(d))
    finally:
        set_mgrouped_store("auto")
    assert np.array_equal(outs[0], outs[1])


def test_counts_out_of_range_are_clamped_and_flagged():
    G, cap, N, K = 3, 48, 128, 256
    a = wl.randn_bf16((G, cap, K), 31)
    b = wl.randn_bf16((G, N, K), 32)
    _, status = masked_case(a, b, [-5, 1000, 20])
    assert status.item() & DG_STATUS_COUNT_GT_CAP


def test_group_independence_bitwise():
    G, cap, N, K = 3, 160, 256, 384
    a = wl.randn_bf16((G, cap, K), 41)
    b = wl.randn_bf16((G, N, K), 42)
    counts = [160, 100, 33]
    d0, _ = masked_case(a, b, counts)
    a2, b2 = a.clone(), b.clone()
    a2[1] *= -3
    b2[2] = wl.randn_bf16((N, K), 43)
    d1, _ = masked_case(a2, b2, counts)
    assert np.array_equal(out_bits(d0)[0], out_bits(d1)[0])


@pytest.mark.slow
def test_decode_shape_full_size_sampled():
    """G=32, cap=4096, N=6144, K=7168, counts ~ Poisson(192): the full-size launch, checked on
    sampled rows x column blocks that the oracle computes one by one."""
    w = wl.masked_decode()
    G, cap, N, K = w.G, w.cap, w.N, w.K
    a, b = w.draw(device="cuda")
    cnt = torch.tensor(w.counts, device="cuda")
    qa, sfa = gpu_quant_tokens(a.view(G * cap, K), DG_SF_FP32, row_counts=cnt)
    qb, sfb = gpu_quant_blocks(b, DG_SF_FP32)
    d = sentinel_like((G, cap, N), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 192, DG_SF_FP32, status)
    sync()
    assert status.item() == 0
    rng = np.random.default_rng(5)
    groups = [g for g in range(G) if w.counts[g] > 0]
    gpu_vals, ref_vals = [], []
    for g in rng.choice(groups, 6, replace=False):
        c = int(w.counts[g])
        rows = np.unique(np.concatenate([[0, c - 1], rng.integers(0, c, 4)]))
        for nb in rng.choice(N // 128, 2, replace=False):
            wb = b[g, nb * 128:(nb + 1) * 128].cpu()
            oqb, osfb, _ = oracle.quant_block_128x128(wb.unsqueeze(0))
            np.testing.assert_array_equal(qb[g, nb * 128:(nb + 1) * 128].cpu().numpy(), oqb[0])
            for r in rows:
                oqa, osfa, _ = oracle.quant_per_token_1x128(a[g, r:r + 1].cpu())
                ref = oracle.gemm_masked(oqa.reshape(1, 1, K), osfa.reshape(1, 1, K // 128), oqb, osfb, [1])
                gpu_vals.append(to_f64(d[g, r, nb * 128:(nb + 1) * 128]))
                ref_vals.append(ref_out(ref[0, 0], False))
    assert_close(np.concatenate(gpu_vals), np.concatenate(ref_vals), False, "decode sampled")
    rows = torch.arange(cap, device="cuda")[None, :]
    pad = rows >= cnt[:, None]
    assert bool((d.view(torch.int16)[pad] == -1).all()), "padding rows written"
    # the whole of the largest expert: every valid row x every output column
    g = int(np.argmax(w.counts))
    c = int(w.counts[g])
    oqb, osfb, _ = oracle.quant_block_128x128(b[g:g + 1].cpu())
    np.testing.assert_array_equal(qb[g].cpu().numpy(), oqb[0])
    oqa, osfa, _ = oracle.quant_per_token_1x128(a[g, :c].cpu())
    ref = oracle.gemm_masked(oqa.reshape(1, c, K), osfa.reshape(1, c, K // 128), oqb, osfb, [c])
    assert_close(to_f64(d[g, :c]), ref_out(ref[0], False), False, f"decode expert {g} whole")


def test_graph_replay_with_changed_counts():
    """Cast (row counts) + GEMM captured once; 24 replays with the counts re-drawn in place
    (including all-zero, full and over-capacity values): valid rows match the oracle on samples,
    rows at or past each count keep their sentinel."""
    G, cap, N, K = 12, 320, 512, 384
    a = wl.randn_bf16((G, cap, K), 81, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), 82, 0.02, device="cuda")
    qa = torch.empty(G * cap, K, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(G * cap, K, DG_SF_FP32, "cuda")
    qb, sfb = gpu_quant_blocks(b, DG_SF_FP32)
    cnt = torch.zeros(G, dtype=torch.int32, device="cuda")
    d = sentinel_like((G, cap, N), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        api.dg_quant_per_token_1x128(a.view(G * cap, K), qa, sfa, DG_SF_FP32, row_counts=cnt)
        api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 96, DG_SF_FP32, status)

    cnt.copy_(torch.full((G,), 100, dtype=torch.int32))
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
    oqb, osfb, _ = oracle.quant_block_128x128(b.cpu())
    rng = np.random.default_rng(83)
    for it in range(24):
        counts = rng.poisson(96, G).astype(np.int32)
        if it == 5:
            counts[:] = 0
        if it == 9:
            counts[:] = cap
        if it == 13:
            counts[::3] = cap + 50                        # clamped to cap and flagged
        cnt.copy_(torch.from_numpy(counts))
        d.view(torch.int16).fill_(-1)
        status.zero_()
        g.replay()
        sync()
        v = np.clip(counts, 0, cap)
        valid = np.arange(cap)[None, :] < v[:, None]
        assert np.all(out_bits(d)[~valid] == sentinel_value(torch.bfloat16)), f"replay {it}: padding row written"
        assert bool(status.item()) == bool(np.any(counts > cap)), f"replay {it}: status {status.item()}"
        for e in rng.choice(G, 3, replace=False):
            if v[e] == 0:
                continue
            rows = np.unique(rng.integers(0, v[e], 4))
            oqa, osfa, _ = oracle.quant_per_token_1x128(a[int(e), torch.from_numpy(rows).cuda()].cpu())
            ref = oracle.gemm_masked(oqa[None], osfa[None], oqb[int(e):int(e) + 1], osfb[int(e):int(e) + 1], [len(rows)])
            assert_close(to_f64(d[int(e), torch.from_numpy(rows).cuda()]), ref_out(ref[0], False), False,
                         f"replay {it} expert {e}")


def test_graph_replay_packed_rows_in_and_out():
    """The packed movement around the masked call, captured once: packed cast -> GEMM -> packing of
    the output's valid rows, replayed 12 times with re-drawn counts (each replay's packed rows
    re-written in place).  The packed output equals the masked output's valid rows bitwise, and
    sampled rows match the oracle."""
    G, cap, N, K = 9, 256, 256, 512
    src = wl.randn_bf16((G * cap, K), 84, 1.0)
    b = wl.randn_bf16((G, N, K), 85, 0.02, device="cuda")
    x_pk = torch.empty(G * cap, K, dtype=torch.bfloat16, device="cuda")
    qa = torch.empty(G * cap, K, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(G * cap, K, DG_SF_FP32, "cuda")
    qb, sfb = gpu_quant_blocks(b, DG_SF_FP32)
    cnt = torch.full((G,), 100, dtype=torch.int32, device="cuda")
    d = sentinel_like((G, cap, N), torch.bfloat16)
    d_pk = sentinel_like((G * cap, N), torch.bfloat16)

    def step():
        api.dg_quant_per_token_1x128_packed(x_pk, qa, sfa, cnt, DG_SF_FP32)
        api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 100, DG_SF_FP32)
        api.dg_pack_masked_rows(d, cnt, d_pk)

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
    oqb, osfb, _ = oracle.quant_block_128x128(b.cpu())
    rng = np.random.default_rng(86)
    for it in range(12):
        counts = rng.integers(0, cap + 1, G).astype(np.int32)
        if it == 3:
            counts[:] = 0
        if it == 7:
            counts[::2] = cap + 9
        v = np.clip(counts, 0, cap)
        n = int(v.sum())
        rows = torch.from_numpy(rng.permutation(G * cap)[:n])  # any rows serve as this step's tokens
        x_pk[:n].copy_(src[rows].cuda())
        cnt.copy_(torch.from_numpy(counts))
        d.view(torch.int16).fill_(-1)
        d_pk.view(torch.int16).fill_(-1)
        g.replay()
        sync()
        valid = np.arange(cap)[None, :] < v[:, None]
        dm = out_bits(d)
        assert np.all(dm[~valid] == sentinel_value(torch.bfloat16)), f"replay {it}: padding row written"
        pk = out_bits(d_pk)
        np.testing.assert_array_equal(pk[:n], dm[valid])
        assert np.all(pk[n:] == sentinel_value(torch.bfloat16))
        off = np.concatenate([[0], np.cumsum(v)])
        for e in rng.choice(G, 2, replace=False):
            if v[e] == 0:
                continue
            r = np.unique(rng.integers(0, v[e], 3))
            xr = src[rows[torch.from_numpy(off[e] + r)]]
            oqa, osfa, _ = oracle.quant_per_token_1x128(xr)
            ref = oracle.gemm_masked(oqa[None], osfa[None], oqb[int(e):int(e) + 1], osfb[int(e):int(e) + 1], [len(r)])
            assert_close(to_f64(d[int(e), torch.from_numpy(r).cuda()]), ref_out(ref[0], False), False,
                         f"replay {it} expert {e}")


@pytest.mark.slow
def test_determinism_10000_calls():
    """The pages' reproduction shape (G=8, cap=32, N=K=256, its counts): 10,000 calls, each
    bitwise equal to the first; and 2,000 on a 128 x 256-tile shape with partial blocks."""
    for (G, cap, N, K, counts, iters) in [(8, 32, 256, 256, [0, 1, 16, 31, 32, 1, 32, 32], 10000),
                                          (4, 300, 1024, 768, [300, 7, 129, 0], 2000)]:
        a = wl.randn_bf16((G, cap, K), 37, 1.0, device="cuda")
        b = wl.randn_bf16((G, N, K), 38, 0.02, device="cuda")
        qa, sfa = gpu_quant_tokens(a.view(G * cap, K), DG_SF_FP32)
        qb, sfb = gpu_quant_blocks(b, DG_SF_FP32)
        cnt = torch.tensor(counts, dtype=torch.int32, device="cuda")
        d = torch.zeros(G, cap, N, dtype=torch.bfloat16, device="cuda")
        api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 0, DG_SF_FP32)
        first = d.clone()
        bad = torch.zeros((), dtype=torch.int64, device="cuda")
        for _ in range(iters):
            api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 0, DG_SF_FP32)
            bad += (d.view(torch.int16) != first.view(torch.int16)).any().to(torch.int64)
        sync()
        assert bad.item() == 0, f"{bad.item()} of {iters} calls differ"
