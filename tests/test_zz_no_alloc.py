"""The allocation-free k-grouped entry point (dg_k_grouped_fp8_wgrad_noalloc) against the workspace
entry point (dg_k_grouped_fp8_wgrad) on the same operands, and against the oracle.

It serves callers that cannot allocate device memory at call time: runtimes that carve all device
memory into a fixed arena at start-up, serving loops that must not pay cudaMalloc's implicit
synchronisation, and C code without a device allocator of its own.  Both entry points run the same
kernels with the same descriptors, so their outputs must be bitwise equal.  The calls come in a row
with different expert layouts, so later calls run on a scratch array that still holds an earlier
call's descriptors.  This file is collected last; it also passes when run alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from moe_grouped_fp8_gb300 import _lib, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import CALC_DIFF_FP32, MAX_ERR_REL, gpu_quant_channels, sync

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _operands(ks, N, H, seed):
    T = sum(ks)
    gy = wl.randn_bf16((T, N), seed, 1e-3)
    act = wl.randn_bf16((T, H), seed + 1, 0.4)
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    ap, sfa = gpu_quant_channels(gy.cuda(), ks_dev)
    bp, sfb = gpu_quant_channels(act.cuda(), ks_dev)
    return dict(gy=gy, act=act, ap=ap, sfa=sfa, bp=bp, sfb=sfb, ks=ks_dev, T=T)


def _c_of(mode, G, N, H, seed):
    if mode == "none":
        return None
    return torch.from_numpy(np.random.default_rng(seed).normal(0, 1e-3, (G, N, H)).astype(np.float32)).cuda()


def _reference_call(o, c_mode, c, G, N, H):
    """The workspace entry point on fresh buffers: d starts as C when C aliases D."""
    d = c.clone() if c_mode == "alias" else torch.zeros(G, N, H, device="cuda")
    cc = d if c_mode == "alias" else c
    api.dg_k_grouped_fp8_wgrad(o["ap"], o["sfa"], o["bp"], o["sfb"], cc, d, o["ks"], o["T"],
                               api.kgrouped_workspace(G, "cuda"))
    return d


def _noalloc_call(o, c_mode, c, G, N, H, via_api):
    d = c.clone() if c_mode == "alias" else torch.full((G, N, H), 3.0, device="cuda")
    cc = d if c_mode == "alias" else c
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if via_api:
        api.dg_k_grouped_fp8_wgrad_noalloc(o["ap"], o["sfa"], o["bp"], o["sfb"], cc, d, o["ks"], o["T"], status)
    else:
        lib = _lib.load()
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = lib.dg_k_grouped_fp8_wgrad_noalloc(_p(o["ap"]), _p(o["sfa"]), _p(o["bp"]), _p(o["sfb"]), _p(cc), _p(d),
                                                _p(o["ks"]), G, o["T"], N, H, _p(status), stream)
        assert rc == 0, lib.dg_last_error()
    sync()
    assert status.item() == 0
    return d


def test_noalloc_bitwise_equal_to_workspace_entry_point_on_consecutive_calls():
    """Four calls in a row (four expert layouts; C separate, absent and aliasing D; through the C ABI
    and through the Python binding): each bitwise equal to the workspace entry point's result."""
    N, H = 256, 384
    calls = [([256, 128, 0, 384], "separate", False), ([128, 512, 128], "none", False),
             ([0, 256, 128, 128, 0], "alias", True), ([384, 128], "separate", True)]
    for i, (ks, c_mode, via_api) in enumerate(calls):
        G = len(ks)
        o = _operands(ks, N, H, seed=40 + 2 * i)
        c = _c_of(c_mode, G, N, H, seed=i)
        ref = _reference_call(o, c_mode, c, G, N, H)
        got = _noalloc_call(o, c_mode, c, G, N, H, via_api)
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), f"call {i} ({c_mode}) differs bitwise"


def test_noalloc_matches_the_oracle():
    """One call against the oracle's casts, packs and fp64 k-grouped GEMM on the same bf16 inputs."""
    ks, N, H = [256, 0, 128, 384], 256, 384
    G = len(ks)
    o = _operands(ks, N, H, seed=61)
    c = _c_of("separate", G, N, H, seed=62)
    got = _noalloc_call(o, "separate", c, G, N, H, via_api=False).double().cpu().numpy()
    qa, sa = oracle.quant_per_channel_128(o["gy"])
    qb, sb = oracle.quant_per_channel_128(o["act"])
    ref = oracle.gemm_kgrouped(oracle.pack_kmajor(qa, ks), sa, oracle.pack_kmajor(qb, ks), sb, ks, N, H,
                               c=c.cpu().numpy())
    assert np.all(np.isfinite(got))
    diff = oracle.calc_diff(got, ref)
    assert diff <= CALC_DIFF_FP32, f"calc_diff {diff:.3e}"
    assert np.abs(got - ref).max() <= MAX_ERR_REL * np.abs(ref).max()


def test_noalloc_at_the_expert_limit():
    """G = DG_NOALLOC_MAX_GROUPS: most experts empty, live experts at high indices up to the last
    slot of the array (descriptors 2 * 255 and 2 * 255 + 1); bitwise equal to the workspace entry."""
    G = _lib.DG_NOALLOC_MAX_GROUPS
    ks = [0] * G
    for e, k in ((3, 128), (200, 256), (254, 128), (255, 384)):
        ks[e] = k
    N, H = 128, 256
    o = _operands(ks, N, H, seed=71)
    c = _c_of("separate", G, N, H, seed=72)
    ref = _reference_call(o, "separate", c, G, N, H)
    got = _noalloc_call(o, "separate", c, G, N, H, via_api=False)
    assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
    assert torch.equal(got[0].view(torch.int32), c[0].view(torch.int32))   # empty expert: D_e = C_e


def test_noalloc_rejects_too_many_experts():
    lib = _lib.load()
    G = _lib.DG_NOALLOC_MAX_GROUPS + 1
    buf = torch.zeros(1024, dtype=torch.float32, device="cuda")
    rc = lib.dg_k_grouped_fp8_wgrad_noalloc(_p(buf), _p(buf), _p(buf), _p(buf), None, _p(buf), _p(buf), G, 128, 128,
                                            128, None, None)
    assert rc == _lib.DG_ERR_UNSUPPORTED
    assert "at most" in lib.dg_last_error().decode()
