"""The allocation-free k-grouped entry point (dg_k_grouped_fp8_wgrad_noalloc), called through the
C ABI, against the workspace entry point (dg_k_grouped_fp8_wgrad) on the same operands.

It serves callers that cannot allocate device memory at call time (a fixed device-memory arena
planned at start-up, no cudaMalloc in a latency-critical loop, C code without a device
allocator of its own).  The test makes two calls in a row with different expert layouts, so
the second call runs on a scratch array that still holds the first call's descriptors; this
file is collected last, and it also passes when run alone in a fresh process.
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
    gy = wl.randn_bf16((T, N), seed, 1e-3).cuda()
    act = wl.randn_bf16((T, H), seed + 1, 0.4).cuda()
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    ap, sfa = gpu_quant_channels(gy, ks_dev)
    bp, sfb = gpu_quant_channels(act, ks_dev)
    return ap, sfa, bp, sfb, ks_dev, T


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    lib = _lib.load()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    N, H = 256, 384
    # call 1 uses four experts, call 2 another layout: the scratch keeps call 1's descriptors
    for call, ks in enumerate([[256, 128, 0, 384], [128, 512, 128]]):
        G = len(ks)
        ap, sfa, bp, sfb, ks_dev, T = _operands(ks, N, H, seed=40 + call)
        c = torch.from_numpy(np.random.default_rng(call).normal(0, 1e-3, (G, N, H)).astype(np.float32)).cuda()
        d_ref = torch.zeros(G, N, H, device="cuda")
        api.dg_k_grouped_fp8_wgrad(ap, sfa, bp, sfb, c, d_ref, ks_dev, T, api.kgrouped_workspace(G, "cuda"))
        d = torch.full((G, N, H), 3.0, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        rc = lib.dg_k_grouped_fp8_wgrad_noalloc(_p(ap), _p(sfa), _p(bp), _p(sfb), _p(c), _p(d), _p(ks_dev), G, T, N,
                                                H, _p(status), stream)
        assert rc == 0, lib.dg_last_error()
        sync()
        assert status.item() == 0
        got, ref = d.double().cpu().numpy(), d_ref.double().cpu().numpy()
        assert np.all(np.isfinite(got))
        diff = oracle.calc_diff(got, ref)
        assert diff <= CALC_DIFF_FP32, f"call {call}: calc_diff {diff:.3e}"
        assert np.abs(got - ref).max() <= MAX_ERR_REL * np.abs(ref).max(), f"call {call}: max error"


def test_noalloc_rejects_too_many_experts():
    lib = _lib.load()
    G = _lib.DG_NOALLOC_MAX_GROUPS + 1
    buf = torch.zeros(1024, dtype=torch.float32, device="cuda")
    rc = lib.dg_k_grouped_fp8_wgrad_noalloc(_p(buf), _p(buf), _p(buf), _p(buf), None, _p(buf), _p(buf), G, 128, 128,
                                            128, None, None)
    assert rc == _lib.DG_ERR_UNSUPPORTED
    assert "at most" in lib.dg_last_error().decode()
