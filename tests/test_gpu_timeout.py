"""The kernels' bounded waits, made to run out.  Through a test hook the limit of the work waits
is set to a few nanoseconds, far below a TMA load's latency, so some wait in every CTA gives up:
the call must still return (the kernels drain what they issued, free tensor memory and exit), the
status word must carry DG_STATUS_TIMEOUT, and once the default limit is back the next call must be
bitwise identical to a clean run on the same inputs (the context and the library are unharmed)."""
import numpy as np
import pytest
import torch

from moe_grouped_fp8_gb300 import DG_SF_FP32, DG_STATUS_TIMEOUT, _lib, api
from moe_grouped_fp8_gb300 import workloads as wl

from gpu_helpers import gpu_quant_blocks, gpu_quant_channels, gpu_quant_tokens, out_bits, set_mgrouped_store, sync

pytestmark = pytest.mark.gpu

SHORT_NS = 4


def set_wait_limit(ns: int):
    _lib.check(_lib.load().dg_testing_wait_limit_ns(ns))


def run_with_short_waits(call):
    """call(status) once with the short limit; returns the status word."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    set_wait_limit(SHORT_NS)
    try:
        call(status)
        sync()
    finally:
        set_wait_limit(0)
    return int(status.item())


@pytest.mark.parametrize("store", ["thread0", "direct"])
@pytest.mark.parametrize("N", [512, 1024])
def test_masked_gemm_times_out_and_recovers(store, N):
    G, cap, K = 4, 256, 4096
    a = wl.randn_bf16((G, cap, K), 301, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), 302, 0.02, device="cuda")
    counts = torch.tensor([256, 130, 0, 77], dtype=torch.int32, device="cuda")
    qa, sfa = gpu_quant_tokens(a.view(G * cap, K), DG_SF_FP32)
    qb, sfb = gpu_quant_blocks(b, DG_SF_FP32)
    d = torch.zeros(G, cap, N, dtype=torch.bfloat16, device="cuda")

    def call(status=None):
        api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, counts, 64, DG_SF_FP32, status)

    set_mgrouped_store(store)
    try:
        call()
        sync()
        clean = out_bits(d)
        st = run_with_short_waits(call)
        assert st & DG_STATUS_TIMEOUT, f"status {st}"
        d.zero_()
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        call(status)
        sync()
    finally:
        set_mgrouped_store("auto")
    assert status.item() == 0
    assert np.array_equal(out_bits(d), clean), "the call after the timeout differs from a clean run"


def test_kgrouped_wgrad_times_out_and_recovers():
    ks = [256, 128, 384]
    T, N, H = sum(ks), 512, 768
    gy = wl.randn_bf16((T, N), 311, 1e-3, device="cuda")
    act = wl.randn_bf16((T, H), 312, 0.4, device="cuda")
    ks_dev = torch.tensor(ks, dtype=torch.int32, device="cuda")
    ap, sa = gpu_quant_channels(gy, ks_dev)
    bp, sb = gpu_quant_channels(act, ks_dev)
    c = torch.randn(len(ks), N, H, device="cuda") * 1e-3
    d = torch.zeros(len(ks), N, H, device="cuda")
    ws = api.kgrouped_workspace(len(ks), "cuda")

    def call(status=None):
        api.dg_k_grouped_fp8_wgrad(ap, sa, bp, sb, c, d, ks_dev, T, ws, status)

    call()
    sync()
    clean = d.clone()
    st = run_with_short_waits(call)
    assert st & DG_STATUS_TIMEOUT, f"status {st}"
    d.zero_()
    call()
    sync()
    assert torch.equal(d.view(torch.int32), clean.view(torch.int32))


def test_bf16_gemm_times_out_and_recovers():
    G, cap, N, K = 3, 256, 512, 2048
    a = wl.randn_bf16((G, cap, K), 321, 1.0, device="cuda")
    b = wl.randn_bf16((G, N, K), 322, 0.02, device="cuda")
    counts = torch.tensor([256, 100, 3], dtype=torch.int32, device="cuda")
    d = torch.zeros(G, cap, N, dtype=torch.bfloat16, device="cuda")

    def call(status=None):
        api.dg_m_grouped_bf16_masked(a, b, d, counts, 64, status=status)

    call()
    sync()
    clean = out_bits(d)
    st = run_with_short_waits(call)
    assert st & DG_STATUS_TIMEOUT, f"status {st}"
    d.zero_()
    call()
    sync()
    assert np.array_equal(out_bits(d), clean)
