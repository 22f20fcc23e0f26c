"""GPU parity of the k-grouped wgrad FP8 GEMM (D_e = C_e + A_e^T B_e) against the oracle.

The first test compares, byte for byte, the per-expert TMA descriptors that the device
prologue builds with descriptors encoded on the host for the same layout; it launches no TMA,
and the GEMM tests below rely on it."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import DG_STATUS_K_NOT_ALIGNED, DG_STATUS_K_OVERFLOW, api
from moe_grouped_fp8_gb300 import _lib
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import assert_close, f32_bits, gpu_quant_channels, sync

pytestmark = pytest.mark.gpu


def test_prologue_descriptors_match_host_encoding():
    lib = _lib.load()
    for ks, N, H in [([256, 0, 128, 384], 256, 384), ([256, 128, 128, 256], 2048, 2048), ([128] * 40, 128, 128),
                     ([128, 1024, 512], 128, 256)]:
        G = len(ks)
        K_cap = sum(ks) + 128
        ap = torch.empty(K_cap * N, dtype=torch.uint8, device="cuda")
        bp = torch.empty(K_cap * H, dtype=torch.uint8, device="cuda")
        ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
        ws = torch.zeros(G * 256, dtype=torch.uint8, device="cuda")
        _lib.check(lib.dg_testing_kgrouped_prologue(ctypes.c_void_p(ap.data_ptr()), ctypes.c_void_p(bp.data_ptr()),
                                                    ctypes.c_void_p(ks_dev.data_ptr()), G, K_cap, N, H,
                                                    ctypes.c_void_p(ws.data_ptr()),
                                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
        sync()
        host = np.zeros(G * 256, np.uint8)
        ks_np = np.array(ks, np.int32)
        _lib.check(lib.dg_testing_kgrouped_host_maps(ctypes.c_void_p(ap.data_ptr()), ctypes.c_void_p(bp.data_ptr()),
                                                     ks_np.ctypes.data_as(ctypes.c_void_p), G, N, H,
                                                     host.ctypes.data_as(ctypes.c_void_p)))
        dev = ws.cpu().numpy()
        for e, k in enumerate(ks):
            if k > 0:
                np.testing.assert_array_equal(dev[e * 256:(e + 1) * 256], host[e * 256:(e + 1) * 256],
                                              err_msg=f"expert {e} (K_e={k}, N={N}, H={H})")


def kgrouped_case(ks, N, H, c_mode="alias", sf_zero=1e-30, seed=0, gy_scale=1.0, act_scale=1.0, zero_ch=False,
                  calls=1, K_cap=None):
    """c_mode: 'none' (c = NULL), 'separate' (random C), 'alias' (c = d, zero-initialised),
    'alias_random' (c = d, initialised with the random C of 'separate')."""
    G = len(ks)
    T = sum(ks)
    K_cap = T if K_cap is None else K_cap
    gy = wl.randn_bf16((K_cap, N), seed, gy_scale)
    act = wl.randn_bf16((K_cap, H), seed + 1, act_scale)
    if zero_ch:
        o = 0
        for k in ks:
            if k == 128:
                gy[o:o + k, 0] = 0
            o += k
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    ap, sfa = gpu_quant_channels(gy.cuda(), ks_dev, sf_zero)
    bp, sfb = gpu_quant_channels(act.cuda(), ks_dev, sf_zero)
    ws = api.kgrouped_workspace(G, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    c_host = None
    if c_mode in ("separate", "alias_random"):
        c_host = torch.from_numpy(np.random.default_rng(seed).normal(0, 1e-3, (G, N, H)).astype(np.float32))
    first = None
    for i in range(calls):
        if c_mode == "alias_random":
            d = c_host.cuda()
            c = d
        else:
            d = torch.zeros(G, N, H, dtype=torch.float32, device="cuda")
            c = None if c_mode == "none" else (d if c_mode == "alias" else c_host.cuda())
        api.dg_k_grouped_fp8_wgrad(ap, sfa, bp, sfb, c, d, ks_dev, K_cap, ws, status)
        if calls > 1:
            if first is None:
                first = d.clone()
            else:
                assert torch.equal(d.view(torch.int32), first.view(torch.int32)), f"call {i} differs bitwise"
    sync()
    oqa, osfa = oracle.quant_per_channel_128(gy[:T], sf_zero)
    oqb, osfb = oracle.quant_per_channel_128(act[:T], sf_zero)
    ref = oracle.gemm_kgrouped(oracle.pack_kmajor(oqa, ks), osfa, oracle.pack_kmajor(oqb, ks), osfb, ks, N, H,
                               c=None if c_host is None else c_host.numpy())
    got = d.double().cpu().numpy()
    for e in range(G):
        if ks[e] == 0:
            want = np.zeros((N, H)) if c_host is None else c_host[e].double().numpy()
            np.testing.assert_array_equal(got[e], want)
        else:
            assert_close(got[e], ref[e].astype(np.float32), True, f"expert {e}")
    return d, status


@pytest.mark.parametrize("c_mode", ["alias", "alias_random", "none", "separate"])
def test_small_with_empty_expert(c_mode):
    kgrouped_case([256, 0, 128, 384], 256, 384, c_mode=c_mode, seed=3)


def test_aliased_and_separate_accumulator_bitwise_equal():
    """D = C + result with C aliasing D (the tile is added into D where it lies) and with C in its
    own buffer (C loaded and added before the store): the same fp32 bits, for every expert."""
    d_alias, _ = kgrouped_case([256, 128, 0, 384], 384, 512, c_mode="alias_random", seed=5)
    d_sep, _ = kgrouped_case([256, 128, 0, 384], 384, 512, c_mode="separate", seed=5)
    assert torch.equal(d_alias.view(torch.int32), d_sep.view(torch.int32))


def test_pages_wgrad_repro_full():
    """Ks=[256,128,128,256], N=H=2048, grad_y=randn*1e-7 with a zeroed channel in the 128-token
    experts, act=randn*0.4, out passed as both c and d."""
    w = wl.kgrouped_repro()
    d, status = kgrouped_case(w.ks, w.N, w.H, "alias", seed=w.seed, gy_scale=w.gy_scale, act_scale=w.act_scale,
                              zero_ch=True)
    assert status.item() == 0
    norms = torch.linalg.vector_norm(d.view(4, -1), dim=1).cpu().numpy()
    assert abs(norms.max() - 1.311e-3) / 1.311e-3 < 0.01, norms


def test_sf_zero_invariance_bitwise():
    outs = []
    for sz in [1.0, 1e-4, 1e-8, 1e-30]:
        d, _ = kgrouped_case([256, 128, 128, 256], 256, 256, "alias", sf_zero=sz, seed=9, gy_scale=1e-7,
                             act_scale=0.4, zero_ch=True)
        outs.append(f32_bits(d))
    for o in outs[1:]:
        np.testing.assert_array_equal(o, outs[0])


def test_repeat_calls_bitwise_identical():
    kgrouped_case([256, 128, 128, 256], 512, 512, "alias", seed=13, gy_scale=1e-7, act_scale=0.4, zero_ch=True,
                  calls=50)


def test_capacity_beyond_sum_of_ks():
    kgrouped_case([128, 256], 128, 256, "separate", seed=17, K_cap=1024)


def test_psum_layout_bitwise_equals_ks():
    """Spans given as inclusive prefix sums (use_psum_layout): the pair cast and the wgrad give
    bitwise the results of the ks calls; the oracle recovers K_e by its own reading of psum."""
    ks = [256, 0, 128, 384]
    G, N, H = len(ks), 256, 384
    T = sum(ks)
    psum = np.cumsum(ks).astype(np.int32)
    gy, act = wl.randn_bf16((T, N), 61, 1e-3).cuda(), wl.randn_bf16((T, H), 62, 0.4).cuda()
    outs = []
    for fn_cast, fn_gemm, spans in ((api.dg_quant_per_channel_128_pair, api.dg_k_grouped_fp8_wgrad, ks),
                                    (api.dg_quant_per_channel_128_pair_psum, api.dg_k_grouped_fp8_wgrad_psum, psum)):
        sp = torch.tensor(np.asarray(spans, np.int32), device="cuda")
        ap = torch.zeros(T * N, dtype=torch.uint8, device="cuda")
        bp = torch.zeros(T * H, dtype=torch.uint8, device="cuda")
        sfa = torch.zeros(T // 128, N, device="cuda")
        sfb = torch.zeros(T // 128, H, device="cuda")
        fn_cast(gy, act, sp, ap, sfa, bp, sfb)
        d = torch.full((G, N, H), 0.5, dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        fn_gemm(ap, sfa, bp, sfb, d, d, sp, T, api.kgrouped_workspace(G, "cuda"), status)
        sync()
        assert status.item() == 0
        outs.append((ap.clone(), sfa.clone(), d.clone()))
    for x, y in zip(outs[0], outs[1]):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))
    ks_o = oracle.sizes_from_psum(psum)
    oqa, osfa = oracle.quant_per_channel_128(gy.cpu(), 1e-30)
    oqb, osfb = oracle.quant_per_channel_128(act.cpu(), 1e-30)
    c = np.full((G, N, H), 0.5, np.float32)
    ref = oracle.gemm_kgrouped(oracle.pack_kmajor(oqa, ks_o), osfa, oracle.pack_kmajor(oqb, ks_o), osfb, ks_o, N, H,
                               c=c)
    got = outs[1][2].double().cpu().numpy()
    for e in range(G):
        assert_close(got[e], ref[e].astype(np.float32), True, f"expert {e}")


def test_psum_decreasing_entry_stops_the_walk():
    psum = np.array([128, 384, 256, 512], np.int32)     # K_2 = -128
    G, N, H, K_cap = 4, 128, 128, 512
    gy, act = wl.randn_bf16((K_cap, N), 63).cuda(), wl.randn_bf16((K_cap, H), 64).cuda()
    sp = torch.tensor(psum, device="cuda")
    ap = torch.zeros(K_cap * N, dtype=torch.uint8, device="cuda")
    bp = torch.zeros(K_cap * H, dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(K_cap // 128, N, device="cuda")
    sfb = torch.zeros(K_cap // 128, H, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_quant_per_channel_128_pair_psum(gy, act, sp, ap, sfa, bp, sfb, status=status)
    d = torch.zeros(G, N, H, dtype=torch.float32, device="cuda")
    api.dg_k_grouped_fp8_wgrad_psum(ap, sfa, bp, sfb, None, d, sp, K_cap, api.kgrouped_workspace(G, "cuda"), status)
    sync()
    assert status.item() & DG_STATUS_K_NOT_ALIGNED
    ks_o = oracle.sizes_from_psum(psum)
    assert ks_o[2] < 0
    got = d.double().cpu().numpy()
    assert np.all(got[2:] == 0), "experts from the bad one on are not computed"
    oqa, osfa = oracle.quant_per_channel_128(gy[:384].cpu(), 1e-30)
    oqb, osfb = oracle.quant_per_channel_128(act[:384].cpu(), 1e-30)
    ref = oracle.gemm_kgrouped(oracle.pack_kmajor(oqa, ks_o[:2]), osfa, oracle.pack_kmajor(oqb, ks_o[:2]), osfb,
                               ks_o[:2], N, H)
    for e in range(2):
        assert_close(got[e], ref[e].astype(np.float32), True, f"expert {e}")


def test_bad_ks_flagged_and_walk_stops():
    ks = [128, 100, 128]
    G, N, H, K_cap = 3, 128, 128, 512
    gy = wl.randn_bf16((K_cap, N), 1).cuda()
    act = wl.randn_bf16((K_cap, H), 2).cuda()
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    ap, sfa = gpu_quant_channels(gy, ks_dev)
    bp, sfb = gpu_quant_channels(act, ks_dev)
    d = torch.full((G, N, H), 7.0, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    api.dg_k_grouped_fp8_wgrad(ap, sfa, bp, sfb, None, d, ks_dev, K_cap, api.kgrouped_workspace(G, "cuda"), status)
    sync()
    assert status.item() & DG_STATUS_K_NOT_ALIGNED
    dn = d.cpu().numpy()
    assert not np.any(dn[0] == 7.0) and np.all(dn[1] == 7.0) and np.all(dn[2] == 7.0)
    status.zero_()
    ks2 = torch.tensor([256, 384, 128], dtype=torch.int32, device="cuda")
    api.dg_k_grouped_fp8_wgrad(ap, sfa, bp, sfb, None, d, ks2, K_cap, api.kgrouped_workspace(G, "cuda"), status)
    sync()
    assert status.item() & DG_STATUS_K_OVERFLOW


@pytest.mark.slow
def test_determinism_10000_calls():
    """10,000 calls on identical operands, each bitwise equal to the first (the #365 harness with
    the bitwise check of its follow-up comment), and 2,500 for each other sf_val of the repro."""
    w = wl.kgrouped_repro()
    gy, act = w.draw(device="cuda")
    ks_dev = torch.tensor(w.ks, dtype=torch.int32, device="cuda")
    for sz in [1.0, 1e-4, 1e-8, 1e-30]:
        ap, sfa = gpu_quant_channels(gy, ks_dev, sz)
        bp, sfb = gpu_quant_channels(act, ks_dev, sz)
        ws = api.kgrouped_workspace(4, "cuda")
        out = torch.zeros(4, w.N, w.H, device="cuda")
        api.dg_k_grouped_fp8_wgrad(ap, sfa, bp, sfb, out, out, ks_dev, w.T, ws)
        first = out.clone()
        bad = torch.zeros((), dtype=torch.int64, device="cuda")
        iters = 10000 if sz == 1.0 else 2500
        for _ in range(iters):
            out.zero_()
            api.dg_k_grouped_fp8_wgrad(ap, sfa, bp, sfb, out, out, ks_dev, w.T, ws)
            bad += (out.view(torch.int32) != first.view(torch.int32)).any().to(torch.int64)
        sync()
        assert bad.item() == 0, f"sf_val={sz}: {bad.item()} calls differ"


def _fused_vs_two_calls(ks_or_psum, K_cap, N, H, c_mode, psum=False, seed=21, gy_scale=1.0, act_scale=1.0):
    """The fused call and the pair cast + wgrad sequence on the same inputs: packed codes,
    scales, output and status bitwise equal."""
    G = len(ks_or_psum)
    gy = wl.randn_bf16((K_cap, N), seed, gy_scale).cuda()
    act = wl.randn_bf16((K_cap, H), seed + 1, act_scale).cuda()
    spans = torch.tensor(ks_or_psum, dtype=torch.int32, device="cuda")
    c_sep = (torch.from_numpy(np.random.default_rng(seed).normal(0, 1e-3, (G, N, H)).astype(np.float32)).cuda()
             if c_mode == "separate" else None)
    outs = []
    for fused in (False, True):
        ap = torch.zeros(K_cap * N, dtype=torch.uint8, device="cuda")
        bp = torch.zeros(K_cap * H, dtype=torch.uint8, device="cuda")
        sfa = torch.zeros(K_cap // 128, N, dtype=torch.float32, device="cuda")
        sfb = torch.zeros(K_cap // 128, H, dtype=torch.float32, device="cuda")
        d = torch.zeros(G, N, H, dtype=torch.float32, device="cuda")
        c = None if c_mode == "none" else (d if c_mode == "alias" else c_sep)
        ws = api.kgrouped_workspace(G, "cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            fn = api.dg_k_grouped_fp8_wgrad_from_bf16_psum if psum else api.dg_k_grouped_fp8_wgrad_from_bf16
            fn(gy, act, spans, ap, sfa, bp, sfb, c, d, ws, status=status)
        else:
            cast = api.dg_quant_per_channel_128_pair_psum if psum else api.dg_quant_per_channel_128_pair
            cast(gy, act, spans, ap, sfa, bp, sfb, status=status)
            gemm = api.dg_k_grouped_fp8_wgrad_psum if psum else api.dg_k_grouped_fp8_wgrad
            gemm(ap, sfa, bp, sfb, c, d, spans, K_cap, ws, status)
        sync()
        outs.append([t.cpu().numpy().view(np.uint8) for t in (ap, bp, sfa, sfb, d)] + [status.item()])
    for i, what in enumerate(["a_packed", "b_packed", "sfa", "sfb", "d"]):
        np.testing.assert_array_equal(outs[0][i], outs[1][i], err_msg=what)
    assert outs[0][5] == outs[1][5]
    return outs[1][5]


@pytest.mark.parametrize("ks,K_cap,N,H,c_mode", [([256, 0, 128, 384], 768, 256, 384, "alias"),
                                                 ([128, 256], 1024, 128, 256, "separate"),
                                                 ([256, 128, 128, 256], 768, 2048, 2048, "alias"),
                                                 ([384, 128], 512, 256, 128, "none")])
def test_from_bf16_bitwise_equals_cast_then_wgrad(ks, K_cap, N, H, c_mode):
    """Casts + descriptors in one launch, then the GEMM: the same bits as the two public calls
    (which the tests above hold to the oracle)."""
    assert _fused_vs_two_calls(ks, K_cap, N, H, c_mode, gy_scale=1e-3, act_scale=0.4) == 0


def test_from_bf16_psum_and_bad_spans():
    assert _fused_vs_two_calls([256, 256, 384, 768], 768, 256, 256, "alias", psum=True) == 0
    st = _fused_vs_two_calls([128, 100, 128], 512, 128, 128, "alias")        # K_e not a multiple of 128
    assert st & DG_STATUS_K_NOT_ALIGNED
    st = _fused_vs_two_calls([256, 512, 128], 512, 128, 256, "alias")        # spans past K_cap
    assert st & DG_STATUS_K_OVERFLOW


def test_fused_graph_replay_with_changed_ks():
    """dg_k_grouped_fp8_wgrad_from_bf16 captured once; 12 replays with the expert spans re-drawn in
    place (including empty experts), each checked against the oracle (C = D = 0 before a replay)."""
    G, N, H, K_cap = 5, 256, 128, 1280
    gy = wl.randn_bf16((K_cap, N), 91, 1e-3)
    act = wl.randn_bf16((K_cap, H), 92, 0.4)
    gyd, actd = gy.cuda(), act.cuda()
    ks_dev = torch.tensor([256, 256, 256, 256, 256], dtype=torch.int32, device="cuda")
    ap = torch.empty(K_cap * N, dtype=torch.uint8, device="cuda")
    bp = torch.empty(K_cap * H, dtype=torch.uint8, device="cuda")
    sfa = torch.empty(K_cap // 128, N, dtype=torch.float32, device="cuda")
    sfb = torch.empty(K_cap // 128, H, dtype=torch.float32, device="cuda")
    d = torch.zeros(G, N, H, dtype=torch.float32, device="cuda")
    ws = api.kgrouped_workspace(G, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        api.dg_k_grouped_fp8_wgrad_from_bf16(gyd, actd, ks_dev, ap, sfa, bp, sfb, d, d, ws, status=status)

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
    rng = np.random.default_rng(93)
    for it in range(12):
        blocks = rng.multinomial(K_cap // 128 - rng.integers(0, 3), np.full(G, 1.0 / G))
        if it == 4:
            blocks[1] = 0
            blocks[3] = 0
        ks = (blocks * 128).astype(np.int32)
        ks_dev.copy_(torch.from_numpy(ks))
        d.zero_()
        g.replay()
        sync()
        assert status.item() == 0
        T = int(ks.sum())
        oqa, osfa = oracle.quant_per_channel_128(gy[:T])
        oqb, osfb = oracle.quant_per_channel_128(act[:T])
        ref = oracle.gemm_kgrouped(oracle.pack_kmajor(oqa, ks), osfa, oracle.pack_kmajor(oqb, ks), osfb, list(ks), N, H)
        got = d.double().cpu().numpy()
        for e in range(G):
            if ks[e] == 0:
                assert np.all(got[e] == 0), f"replay {it}: empty expert {e} written"
            else:
                assert_close(got[e], ref[e].astype(np.float32), True, f"replay {it} expert {e}")
