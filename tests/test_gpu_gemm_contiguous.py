"""GPU parity of the m-grouped contiguous FP8 GEMM (m_indices routing, -1 padding rows), including
CUDA-graph replay with the expert distribution re-drawn in place between replays."""
import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_SF_FP32, DG_SF_UE8M0, DG_STATUS_BAD_INDEX, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import (assert_close, gpu_quant_blocks, gpu_quant_tokens, out_bits, ref_out, sentinel_like,
                         sentinel_value, set_mgrouped_kernel, set_mgrouped_store, set_mgrouped_warps, sync, to_f64)

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


def contiguous_case(a, b, m_indices, fmt=DG_SF_FP32, out=torch.bfloat16, calls=1):
    M, K = a.shape
    G, N, _ = b.shape
    qa, sfa = gpu_quant_tokens(a.cuda(), fmt)
    qb, sfb = gpu_quant_blocks(b.cuda(), fmt)
    mi = torch.tensor(np.asarray(m_indices, np.int32), device="cuda")
    d = sentinel_like((M, N), out)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = None
    for i in range(calls):
        api.dg_m_grouped_fp8_contiguous(qa, sfa, qb, sfb, d, mi, fmt, status)
        if calls > 1:
            bits = out_bits(d)
            if first is None:
                first = bits
            else:
                assert np.array_equal(bits, first), f"call {i} differs bitwise"
    sync()
    ue = fmt == DG_SF_UE8M0
    oqa, osfa, _ = oracle.quant_per_token_1x128(a, ue8m0=ue)
    oqb, osfb, _ = oracle.quant_block_128x128(b, ue8m0=ue)
    np.testing.assert_array_equal(qa.cpu().numpy(), oqa)
    ref = oracle.gemm_contiguous(oqa, osfa, oqb, osfb, m_indices)
    mi_np = np.asarray(m_indices)
    # rows written: routed rows whose 128-row block is headed by the same expert
    block_e = mi_np[(np.arange(M) // 128) * 128]
    valid = (mi_np >= 0) & (mi_np == block_e)
    fp32 = out == torch.float32
    if valid.any():
        assert_close(to_f64(d)[valid], ref_out(ref[valid], fp32), fp32, "contiguous routed rows")
    assert np.all(out_bits(d)[~valid] == sentinel_value(out)), "a padding row was written"
    return d, status


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_small_ragged_segments(fmt, out):
    counts = [130, 0, 1, 128, 257]
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    a = wl.randn_bf16((mi.size, 384), 51, 1.5)
    b = wl.randn_bf16((5, 256, 384), 52, 0.02)
    contiguous_case(a, b, mi, fmt, out)


def test_wide_tiles_ragged_segments():
    """N = 1024: 128 x 256 tiles on ragged segments, repeated calls bitwise identical."""
    counts = [130, 0, 257, 1]
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    a = wl.randn_bf16((mi.size, 256), 57, 1.0)
    b = wl.randn_bf16((4, 1024, 256), 58, 0.02)
    contiguous_case(a, b, mi, calls=4)


def test_single_expert_plain_gemm_and_repeat_bitwise():
    mi = np.zeros(300, np.int32)
    mi[290:] = -1
    a = wl.randn_bf16((300, 256), 61)
    b = wl.randn_bf16((1, 512, 256), 62)
    contiguous_case(a, b, mi, calls=8)


def test_all_padding_and_ragged_last_block():
    mi = np.full(200, -1, np.int32)
    a = wl.randn_bf16((200, 128), 71)
    b = wl.randn_bf16((2, 128, 128), 72)
    contiguous_case(a, b, mi)
    mi2 = np.full(200, -1, np.int32)
    mi2[128:133] = 1                                   # ragged final block (rows 128..199 of a 256 block)
    contiguous_case(a, b, mi2)


def test_odd_runs_and_narrow_tiles():
    """Runs of 5, 1, 3 and 1 m-blocks and N = 640 (five 128-column tiles)."""
    counts = [640, 1, 0, 300, 128]
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    a = wl.randn_bf16((mi.size, 256), 95)
    b = wl.randn_bf16((5, 640, 256), 96, 0.05)
    contiguous_case(a, b, mi)


@pytest.mark.parametrize("N", [512, 1024])
def test_store_paths_bitwise_equal(N):
    """The two store paths (TMA stores issued by thread 0, owner-thread stores) on ragged m_indices
    segments (TMA store extent from the row ballots): same bits."""
    counts = [130, 0, 1, 128, 257, 9]
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    a = wl.randn_bf16((mi.size, 384), 61, 1.5)
    b = wl.randn_bf16((len(counts), N, 384), 62, 0.02)
    outs = []
    try:
        for which in ("thread0", "direct"):
            set_mgrouped_store(which)
            d, _ = contiguous_case(a, b, mi, calls=2)
            outs.append(out_bits(d))
    finally:
        set_mgrouped_store("auto")
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fmt", [DG_SF_FP32, DG_SF_UE8M0])
def test_promotion_warps_bitwise_equal(ue8m0_kernel, fmt):
    """128 x 256 tiles of the promotion kernel promoted by 16 warps (64 accumulators each) or by 8
    (128 each): each passes the oracle check and both give the same bits, with both store paths."""
    if ue8m0_kernel != "auto":
        pytest.skip("a property of the promotion kernel, forced below")
    set_mgrouped_kernel("promotion")
    counts = [130, 0, 1, 128, 257, 9]
    mi = wl.contiguous_m_indices(counts, m_max=wl.contiguous_capacity(sum(counts), len(counts)))
    for K in (384, 4224):                               # owner-thread stores / staged TMA stores
        a = wl.randn_bf16((mi.size, K), 63, 1.5)
        b = wl.randn_bf16((len(counts), 1024, K), 64, 0.02)
        outs = []
        try:
            for warps in (16, 8):
                set_mgrouped_warps(warps)
                d, _ = contiguous_case(a, b, mi, fmt=fmt)
                outs.append(out_bits(d))
        finally:
            set_mgrouped_warps(0)
        assert np.array_equal(outs[0], outs[1]), f"K={K}"



def test_segments_out_of_expert_order():
    mi = np.full(512, -1, np.int32)
    mi[0:70] = 2
    mi[128:256] = 0
    mi[256:300] = 1
    a = wl.randn_bf16((512, 256), 81)
    b = wl.randn_bf16((3, 256, 256), 82)
    contiguous_case(a, b, mi)


def test_bad_indices_flagged_and_skipped():
    mi = np.full(256, -1, np.int32)
    mi[0:10] = 0
    mi[10:12] = 7                                      # >= G: bad and not written
    mi[128] = -9                                       # < -1: bad block head -> block skipped
    mi[129:140] = 1
    a = wl.randn_bf16((256, 128), 91)
    b = wl.randn_bf16((2, 128, 128), 92)
    qa, sfa = gpu_quant_tokens(a.cuda(), DG_SF_FP32)
    qb, sfb = gpu_quant_blocks(b.cuda(), DG_SF_FP32)
    d = sentinel_like((256, 128), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_m_grouped_fp8_contiguous(qa, sfa, qb, sfb, d, torch.tensor(mi, device="cuda"), DG_SF_FP32, status)
    sync()
    assert status.item() & DG_STATUS_BAD_INDEX
    bits = out_bits(d)
    assert np.all(bits[10:12] == 0xFFFF) and np.all(bits[128:] == 0xFFFF)
    oqa, osfa, _ = oracle.quant_per_token_1x128(a)
    oqb, osfb, _ = oracle.quant_block_128x128(b)
    ok = np.full(256, -1, np.int32)
    ok[0:10] = 0
    ref = oracle.gemm_contiguous(oqa, osfa, oqb, osfb, ok)
    assert_close(to_f64(d)[:10], ref_out(ref[:10], False), False, "rows before the bad ones")


def test_psum_layout_bitwise_equals_m_indices():
    """Routing by per-expert end rows: the same rows, bitwise the same results as the m_indices
    call; the oracle routes by its own reading of psum."""
    counts = [130, 0, 1, 128, 257]
    M = wl.contiguous_capacity(sum(counts), len(counts))
    mi = wl.contiguous_m_indices(counts, m_max=M)
    psum = wl.contiguous_psum(counts)
    a, b = wl.randn_bf16((M, 384), 53, 1.5), wl.randn_bf16((5, 256, 384), 54, 0.02)
    d_mi, _ = contiguous_case(a, b, mi)
    qa, sfa = gpu_quant_tokens(a.cuda(), DG_SF_FP32)
    qb, sfb = gpu_quant_blocks(b.cuda(), DG_SF_FP32)
    d = sentinel_like((M, 256), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_m_grouped_fp8_contiguous_psum(qa, sfa, qb, sfb, d, torch.tensor(psum, device="cuda"), DG_SF_FP32, status)
    sync()
    assert status.item() == 0
    assert np.array_equal(out_bits(d), out_bits(d_mi))
    routed = oracle.m_indices_from_psum(psum, M)
    oqa, osfa, _ = oracle.quant_per_token_1x128(a)
    oqb, osfb, _ = oracle.quant_block_128x128(b)
    ref = oracle.gemm_contiguous(oqa, osfa, oqb, osfb, routed)
    ok = routed >= 0
    assert_close(to_f64(d)[ok], ref_out(ref[ok], False), False, "psum routed rows")
    assert np.all(out_bits(d)[~ok] == 0xFFFF)


def test_psum_bad_entry_flagged_and_walk_stops():
    psum = np.array([130, 100, 394], np.int32)           # expert 1 ends before expert 0
    M, K, N = 512, 256, 128
    a, b = wl.randn_bf16((M, K), 55), wl.randn_bf16((3, N, K), 56)
    qa, sfa = gpu_quant_tokens(a.cuda(), DG_SF_FP32)
    qb, sfb = gpu_quant_blocks(b.cuda(), DG_SF_FP32)
    d = sentinel_like((M, N), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_m_grouped_fp8_contiguous_psum(qa, sfa, qb, sfb, d, torch.tensor(psum, device="cuda"), DG_SF_FP32, status)
    sync()
    assert status.item() & DG_STATUS_BAD_INDEX
    routed = oracle.m_indices_from_psum(psum, M)
    assert np.all(routed[130:] == -1)
    bits = out_bits(d)
    assert np.all(bits[130:] == 0xFFFF)
    oqa, osfa, _ = oracle.quant_per_token_1x128(a)
    oqb, osfb, _ = oracle.quant_block_128x128(b)
    ref = oracle.gemm_contiguous(oqa, osfa, oqb, osfb, routed)
    assert_close(to_f64(d)[:130], ref_out(ref[:130], False), False, "expert 0")


def replay_case(G, N, K, E, replays, check_every, seed, mode="m_indices"):
    """Capture cast + GEMM once; replay with routing re-drawn in place (same buffers), routed by
    m_indices or by psum (the modes of the pages' graph-mutation test); "routed" also casts only
    the rows whose m_indices entry is >= 0 (the routed cast reads the same re-drawn tensor)."""
    T = G * E
    m_max = wl.contiguous_capacity(T, G)
    a = wl.randn_bf16((m_max, K), seed, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), seed + 1, 0.02, device="cuda")
    fmt = DG_SF_UE8M0
    qa = torch.empty(m_max, K, dtype=torch.uint8, device="cuda")
    sfa = api.empty_sfa(m_max, K, fmt, "cuda")
    qb, sfb = gpu_quant_blocks(b, fmt)
    psum_mode = mode == "psum"
    routed_cast = mode == "routed"
    mi_dev = torch.full((G if psum_mode else m_max,), -1, dtype=torch.int32, device="cuda")
    d = torch.empty(m_max, N, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def routing(counts):
        return wl.contiguous_psum(counts) if psum_mode else wl.contiguous_m_indices(counts, m_max)

    def step():
        if routed_cast:
            api.dg_quant_per_token_1x128_routed(a, qa, sfa, mi_dev, fmt)
        else:
            api.dg_quant_per_token_1x128(a, qa, sfa, fmt)
        if psum_mode:
            api.dg_m_grouped_fp8_contiguous_psum(qa, sfa, qb, sfb, d, mi_dev, fmt, status)
        else:
            api.dg_m_grouped_fp8_contiguous(qa, sfa, qb, sfb, d, mi_dev, fmt, status)

    mi_dev.copy_(torch.from_numpy(routing(wl.multinomial_counts(T, G, seed))))
    step()                                             # eager warm-up before capture
    sync()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    sync()
    qcache = {}                                        # expert -> oracle codes/scales of its weights

    def oracle_weights(experts):
        for e in experts:
            if e not in qcache:
                q, sf, _ = oracle.quant_block_128x128(b[e:e + 1].cpu(), ue8m0=True)
                qcache[e] = (q[0], sf[0])
        return (np.stack([qcache[e][0] for e in experts]), np.stack([qcache[e][1] for e in experts]))

    checked = 0
    for it in range(replays):
        counts = wl.multinomial_counts(T, G, seed + 1 + it)
        if it == replays // 2:
            counts = np.zeros(G, np.int32)             # an all-empty phase
        r_np = routing(counts)
        mi_dev.copy_(torch.from_numpy(r_np))           # same pointer, new values
        mi_np = oracle.m_indices_from_psum(r_np, m_max) if psum_mode else r_np
        d.view(torch.int16).fill_(-1)
        g.replay()
        if it % check_every == 0 or it == replays // 2:
            sync()
            assert status.item() == 0
            bits = out_bits(d)
            assert np.all(bits[mi_np < 0] == 0xFFFF), f"replay {it}: padding row written"
            rows = np.nonzero(mi_np >= 0)[0]
            if rows.size:
                pick = np.unique(np.random.default_rng(it).choice(rows, min(24, rows.size), replace=False))
                experts = sorted(set(int(e) for e in mi_np[pick]))
                oqb, osfb = oracle_weights(experts)
                local = np.array([experts.index(int(e)) for e in mi_np[pick]], np.int32)
                oqa, osfa, _ = oracle.quant_per_token_1x128(a[torch.from_numpy(pick).cuda()].cpu(), ue8m0=True)
                ref = oracle.gemm_contiguous(oqa, osfa, oqb, osfb, local)
                assert_close(to_f64(d)[pick], ref_out(ref, False), False, f"replay {it}")
            checked += 1
    assert checked >= replays // check_every


@pytest.mark.ue8m0
@pytest.mark.parametrize("mode", ["m_indices", "psum", "routed"])
def test_graph_replay_with_changed_routing_small(mode):
    replay_case(G=16, N=256, K=256, E=20, replays=30, check_every=3, seed=7, mode=mode)


@pytest.mark.slow
@pytest.mark.parametrize("which,E", [("w13", 1), ("w13", 32), ("w13", 113), ("w2", 1), ("w2", 32), ("w2", 113)])
def test_many_expert_ue8m0_graph_replay(which, E):
    """G=288 many-expert shapes, UE8M0 scales, 100 replays with re-drawn routing (every 10th
    replay checked against the oracle on sampled rows)."""
    N, K = (512, 4096) if which == "w13" else (4096, 256)
    replay_case(G=288, N=N, K=K, E=E, replays=100, check_every=10, seed=1005 + E)


@pytest.mark.slow
def test_prefill_shape_full_size_sampled():
    """G=32, N=4096, K=7168, 8192 Zipf-routed tokens: the full-size launch, sampled rows."""
    w = wl.contiguous_prefill()
    M, K, N = w.m_max, w.K, w.N
    a, b = w.draw(device="cuda")
    mi = w.m_indices
    qa, sfa = gpu_quant_tokens(a, DG_SF_FP32)
    qb, sfb = gpu_quant_blocks(b, DG_SF_FP32)
    d = sentinel_like((M, N), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_m_grouped_fp8_contiguous(qa, sfa, qb, sfb, d, torch.from_numpy(mi).cuda(), DG_SF_FP32, status)
    sync()
    assert status.item() == 0
    rng = np.random.default_rng(3)
    rows = rng.choice(np.nonzero(mi >= 0)[0], 24, replace=False)
    gpu_vals, ref_vals = [], []
    for nb in rng.choice(N // 128, 2, replace=False):
        for r in rows:
            e = int(mi[r])
            oqb, osfb, _ = oracle.quant_block_128x128(b[e:e + 1, nb * 128:(nb + 1) * 128].cpu())
            oqa, osfa, _ = oracle.quant_per_token_1x128(a[r:r + 1].cpu())
            ref = oracle.gemm_contiguous(oqa, osfa, oqb, osfb, np.zeros(1, np.int32))
            gpu_vals.append(to_f64(d[r, nb * 128:(nb + 1) * 128]))
            ref_vals.append(ref_out(ref[0], False))
    assert_close(np.concatenate(gpu_vals), np.concatenate(ref_vals), False, "prefill sampled")
    pad = torch.from_numpy(mi < 0).cuda()
    assert bool((d.view(torch.int16)[pad] == -1).all()), "padding rows written"
    # the whole of the largest expert: every one of its rows x every output column
    e = int(np.argmax(w.counts))
    rows = np.nonzero(mi == e)[0]
    oqb, osfb, _ = oracle.quant_block_128x128(b[e:e + 1].cpu())
    np.testing.assert_array_equal(qb[e].cpu().numpy(), oqb[0])
    oqa, osfa, _ = oracle.quant_per_token_1x128(a[torch.from_numpy(rows).cuda()].cpu())
    ref = oracle.gemm_contiguous(oqa, osfa, oqb, osfb, np.zeros(rows.size, np.int32))
    assert_close(to_f64(d[torch.from_numpy(rows).cuda()]), ref_out(ref, False), False, f"prefill expert {e} whole")


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["m_indices", "psum"])
def test_block_scaled_determinism_10000_calls(mode):
    """UE8M0 scales, N = 1024, K = 2048 (the block-scaled MMA kernel) on ragged segments routed by
    m_indices or psum: 10,000 calls, each bitwise equal to the first."""
    counts = [130, 0, 1, 128, 257, 9]
    G, N, K = len(counts), 1024, 2048
    m_max = wl.contiguous_capacity(sum(counts), G)
    a = wl.randn_bf16((m_max, K), 57, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), 58, 0.02, device="cuda")
    qa, sfa = gpu_quant_tokens(a, DG_SF_UE8M0)
    qb, sfb = gpu_quant_blocks(b, DG_SF_UE8M0)
    route = wl.contiguous_psum(counts) if mode == "psum" else wl.contiguous_m_indices(counts, m_max)
    r = torch.tensor(route, dtype=torch.int32, device="cuda")
    fn = api.dg_m_grouped_fp8_contiguous_psum if mode == "psum" else api.dg_m_grouped_fp8_contiguous
    d = torch.zeros(m_max, N, dtype=torch.bfloat16, device="cuda")
    fn(qa, sfa, qb, sfb, d, r, DG_SF_UE8M0)
    first = d.clone()
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(10000):
        fn(qa, sfa, qb, sfb, d, r, DG_SF_UE8M0)
        bad += (d.view(torch.int16) != first.view(torch.int16)).any().to(torch.int64)
    sync()
    assert bad.item() == 0, f"{bad.item()} of 10000 calls differ"


@pytest.mark.slow
@pytest.mark.parametrize("mode", ["m_indices", "psum"])
def test_determinism_10000_calls(mode):
    """Ragged segments routed by m_indices or psum: 10,000 calls, each bitwise equal to the first."""
    counts = [130, 0, 1, 128, 257, 9]
    G, N, K = len(counts), 1024, 512
    m_max = wl.contiguous_capacity(sum(counts), G)
    a = wl.randn_bf16((m_max, K), 47, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), 48, 0.02, device="cuda")
    qa, sfa = gpu_quant_tokens(a, DG_SF_UE8M0)
    qb, sfb = gpu_quant_blocks(b, DG_SF_UE8M0)
    route = wl.contiguous_psum(counts) if mode == "psum" else wl.contiguous_m_indices(counts, m_max)
    r = torch.tensor(route, dtype=torch.int32, device="cuda")
    fn = api.dg_m_grouped_fp8_contiguous_psum if mode == "psum" else api.dg_m_grouped_fp8_contiguous
    d = torch.zeros(m_max, N, dtype=torch.bfloat16, device="cuda")
    fn(qa, sfa, qb, sfb, d, r, DG_SF_UE8M0)
    first = d.clone()
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(10000):
        fn(qa, sfa, qb, sfb, d, r, DG_SF_UE8M0)
        bad += (d.view(torch.int16) != first.view(torch.int16)).any().to(torch.int64)
    sync()
    assert bad.item() == 0, f"{bad.item()} of 10000 calls differ"
