"""Runs one call of every kernel family on small seeded inputs and saves the output bytes, so that
tests/test_gpu_debug_build.py can compare the debug build (DG_DEBUG=1 in the environment: the
binding loads libdg_debug.so) with the release build bit for bit.

    python tests/debug_build_cases.py OUT.npz

Saved: every case's output bytes; "word", the debug word after the in-bounds cases (the debug
build must raise no bit on them); for the planted case (the test hook narrows the output rows
the store checks allow to the first group's), "planted_out" and "planted_word"; and for the
injected producer stall, "stall_status" and the output of the clean call after it.
"""
from __future__ import annotations

import sys

import numpy as np
import torch

from moe_grouped_fp8_gb300 import DG_SF_FP32, DG_SF_UE8M0, _lib, api
from moe_grouped_fp8_gb300 import workloads as wl

dev = "cuda"
out: dict[str, np.ndarray] = {}


def keep(name, *ts):
    for i, t in enumerate(ts):
        out[f"{name}.{i}"] = t.detach().contiguous().view(torch.uint8).cpu().numpy().ravel()


def sentinel(shape, dtype):
    if dtype == torch.bfloat16:
        return torch.full(shape, -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
    return torch.full(shape, -1, dtype=torch.int32, device=dev).view(torch.float32)


def tokens(x, fmt, row_counts=None):
    M, K = x.shape
    q = torch.zeros(M, K, dtype=torch.uint8, device=dev)
    sfa = api.empty_sfa(M, K, fmt, dev)
    sfa.zero_()
    api.dg_quant_per_token_1x128(x, q, sfa, fmt, 1e-30, row_counts)
    return q, sfa


def blocks(w, fmt):
    G, N, K = w.shape
    q = torch.zeros(G, N, K, dtype=torch.uint8, device=dev)
    sfb = torch.zeros(G, N // 128, K // 128, dtype=torch.float32 if fmt == DG_SF_FP32 else torch.uint8, device=dev)
    api.dg_quant_block_128x128(w, q, sfb, fmt, 1e-30)
    return q, sfb


def masked(G, cap, N, K, counts, fmt, seed, out_dtype=torch.bfloat16):
    a = wl.randn_bf16((G * cap, K), seed, 1.0, dev)
    b = wl.randn_bf16((G, N, K), seed + 1, 1.0, dev)
    qa, sfa = tokens(a, fmt)
    qb, sfb = blocks(b, fmt)
    d = sentinel((G, cap, N), out_dtype)
    cnt = torch.tensor(counts, dtype=torch.int32, device=dev)
    api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 0, fmt)
    return d


def main(path):
    torch.manual_seed(0)
    # ---- casts
    for fmt in (DG_SF_FP32, DG_SF_UE8M0):
        x = wl.randn_bf16((301, 384), 11, 0.5, dev)
        keep(f"tok{fmt}", *tokens(x, fmt))
        xm = wl.randn_bf16((5 * 40, 384), 12, 0.5, dev)
        keep(f"tokmask{fmt}", *tokens(xm, fmt, torch.tensor([3, 40, 0, 17, 40], dtype=torch.int32, device=dev)))
        mi = torch.tensor(wl.contiguous_m_indices([130, 0, 1, 9], 700), dtype=torch.int32, device=dev)
        xr = wl.randn_bf16((700, 256), 13, 0.5, dev)
        q = torch.zeros(700, 256, dtype=torch.uint8, device=dev)
        sfa = api.empty_sfa(700, 256, fmt, dev)
        sfa.zero_()
        api.dg_quant_per_token_1x128_routed(xr, q, sfa, mi, fmt)
        keep(f"tokroute{fmt}", q, sfa)
        keep(f"block{fmt}", *blocks(wl.randn_bf16((3, 256, 384), 14, 0.5, dev), fmt))
        xp = wl.randn_bf16((5 * 40, 384), 16, 0.5, dev)
        q = torch.zeros(200, 384, dtype=torch.uint8, device=dev)
        sfa = api.empty_sfa(200, 384, fmt, dev)
        sfa.zero_()
        api.dg_quant_per_token_1x128_packed(xp, q, sfa, torch.tensor([3, 40, 0, 17, 40], dtype=torch.int32, device=dev),
                                            fmt)
        keep(f"tokpacked{fmt}", q, sfa)
    w4 = wl.randn_bf16((2, 256, 512), 15, 0.5, dev)
    q4 = torch.zeros(2, 256, 256, dtype=torch.uint8, device=dev)
    s4 = torch.zeros(2, 2, 4, dtype=torch.uint8, device=dev)
    api.dg_quant_block_128x128_fp4(w4, q4, s4)
    keep("block_fp4", q4, s4)

    # ---- m-grouped masked: long K (staged stores + owner tails), short K (owner-thread stores),
    # UE8M0 long K (block-scaled MMA kernel), fp32 output
    d = masked(4, 200, 512, 7168, [200, 77, 0, 130], DG_SF_FP32, 21)
    keep("masked_long", d)
    pk = torch.zeros(800, 512, dtype=torch.bfloat16, device=dev)
    api.dg_pack_masked_rows(d, torch.tensor([200, 77, 0, 130], dtype=torch.int32, device=dev), pk)
    keep("pack_rows", pk)
    keep("masked_short", masked(4, 200, 512, 512, [200, 77, 0, 130], DG_SF_FP32, 22))
    keep("masked_mx", masked(3, 140, 512, 4096, [140, 1, 129], DG_SF_UE8M0, 23))
    keep("masked_f32", masked(3, 100, 384, 1024, [100, 37, 64], DG_SF_UE8M0, 24, torch.float32))

    # ---- m-grouped contiguous (m_indices with padding, and prefix sums), 128-column tiles
    counts = [130, 0, 257, 5]
    M = wl.contiguous_capacity(sum(counts), len(counts))
    a = wl.randn_bf16((M, 1024), 31, 1.0, dev)
    b = wl.randn_bf16((4, 384, 1024), 32, 1.0, dev)
    qa, sfa = tokens(a, DG_SF_FP32)
    qb, sfb = blocks(b, DG_SF_FP32)
    mi = torch.tensor(wl.contiguous_m_indices(counts, M), dtype=torch.int32, device=dev)
    d = sentinel((M, 384), torch.bfloat16)
    api.dg_m_grouped_fp8_contiguous(qa, sfa, qb, sfb, d, mi)
    keep("contig", d)
    ps = torch.tensor(wl.contiguous_psum(counts), dtype=torch.int32, device=dev)
    d = sentinel((M, 384), torch.bfloat16)
    api.dg_m_grouped_fp8_contiguous_psum(qa, sfa, qb, sfb, d, ps)
    keep("contig_psum", d)

    # ---- plain GEMM with C, batched GEMM
    a = wl.randn_bf16((300, 1024), 41, 1.0, dev)
    b = wl.randn_bf16((1, 256, 1024), 42, 1.0, dev)
    qa, sfa = tokens(a, DG_SF_FP32)
    qb, sfb = blocks(b, DG_SF_FP32)
    c = wl.randn_bf16((300, 256), 43, 1.0, dev).float()
    d = sentinel((300, 256), torch.float32)
    api.dg_fp8_gemm_nt(qa, sfa, qb.view(256, 1024), sfb, d, c)
    keep("dense_c", d)
    a = wl.randn_bf16((3 * 70, 512), 44, 1.0, dev)
    b = wl.randn_bf16((3, 256, 512), 45, 1.0, dev)
    qa, sfa = tokens(a, DG_SF_UE8M0)
    qb, sfb = blocks(b, DG_SF_UE8M0)
    d = sentinel((3, 70, 256), torch.bfloat16)
    api.dg_fp8_gemm_nt_batched(qa.view(3, 70, 512), sfa, qb, sfb, d, None, DG_SF_UE8M0)
    keep("batched", d)

    # ---- FP8 x FP4 masked, BF16 masked
    a = wl.randn_bf16((2 * 150, 1024), 51, 1.0, dev)
    qa, sfa = tokens(a, DG_SF_UE8M0)
    b = wl.randn_bf16((2, 256, 1024), 52, 1.0, dev)
    qb = torch.zeros(2, 256, 512, dtype=torch.uint8, device=dev)
    sb = torch.zeros(2, 2, 8, dtype=torch.uint8, device=dev)
    api.dg_quant_block_128x128_fp4(b, qb, sb)
    d = sentinel((2, 150, 256), torch.bfloat16)
    api.dg_m_grouped_fp8_fp4_masked(qa.view(2, 150, 1024), sfa, qb, sb, d,
                                    torch.tensor([150, 61], dtype=torch.int32, device=dev))
    keep("fp4_masked", d)
    a = wl.randn_bf16((3, 90, 512), 53, 1.0, dev)
    b = wl.randn_bf16((3, 256, 512), 54, 1.0, dev)
    d = sentinel((3, 90, 256), torch.bfloat16)
    api.dg_m_grouped_bf16_masked(a, b, d, torch.tensor([90, 0, 33], dtype=torch.int32, device=dev))
    keep("bf16_masked", d)

    # ---- k-grouped wgrad from bf16 (per-channel casts + packs, descriptors, GEMM)
    kg = wl.kgrouped_repro()
    gy, act = kg.draw(dev)
    G, N, H, K_cap = len(kg.ks), kg.N, kg.H, kg.T
    ks = torch.tensor(kg.ks, dtype=torch.int32, device=dev)
    ap = torch.zeros(K_cap * N, dtype=torch.uint8, device=dev)
    bp = torch.zeros(K_cap * H, dtype=torch.uint8, device=dev)
    sa = torch.zeros(K_cap // 128, N, dtype=torch.float32, device=dev)
    sb = torch.zeros(K_cap // 128, H, dtype=torch.float32, device=dev)
    d = torch.zeros(G, N, H, dtype=torch.float32, device=dev)
    api.dg_k_grouped_fp8_wgrad_from_bf16(gy, act, ks, ap, sa, bp, sb, None, d, api.kgrouped_workspace(G, dev))
    keep("kgrouped", ap, sa, bp, sb, d)

    out["word"] = np.array([api.dg_debug_word(clear=True)], np.uint32)

    # ---- planted: the store checks allow the first group's rows only (short K: every row is
    # stored by its owner thread); no access leaves the buffers either way
    lib = _lib.load()
    _lib.check(lib.dg_testing_debug_out_rows(200))
    try:
        out["planted_out"] = masked(4, 200, 512, 512, [200, 77, 0, 130], DG_SF_FP32, 22).view(torch.uint8).cpu() \
            .numpy().ravel()
    finally:
        _lib.check(lib.dg_testing_debug_out_rows(0))
    out["planted_word"] = np.array([api.dg_debug_word(clear=True)], np.uint32)

    # ---- injected stall (debug build): CTA 0's producer stops before its 5th stage load; with a
    # 50 ms wait limit the call returns with DG_STATUS_TIMEOUT set, and the next call (hook off,
    # default limit) is clean
    G, cap, N, K = 4, 200, 512, 7168
    a = wl.randn_bf16((G * cap, K), 21, 1.0, dev)
    b = wl.randn_bf16((G, N, K), 22, 1.0, dev)
    qa, sfa = tokens(a, DG_SF_FP32)
    qb, sfb = blocks(b, DG_SF_FP32)
    cnt = torch.tensor([200, 77, 0, 130], dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    _lib.check(lib.dg_testing_wait_limit_ns(50_000_000))
    _lib.check(lib.dg_testing_debug_stop_producer(5))
    try:
        d = sentinel((G, cap, N), torch.bfloat16)
        api.dg_m_grouped_fp8_masked(qa.view(G, cap, K), sfa, qb, sfb, d, cnt, 0, DG_SF_FP32, status)
        torch.cuda.synchronize()
    finally:
        _lib.check(lib.dg_testing_debug_stop_producer(0))
        _lib.check(lib.dg_testing_wait_limit_ns(0))
    out["stall_status"] = np.array([int(status.item())], np.int32)
    keep("after_stall", masked(4, 200, 512, 7168, [200, 77, 0, 130], DG_SF_FP32, 21))
    out["debug_build"] = np.array([int(api.dg_debug_build())], np.int32)
    torch.cuda.synchronize()
    np.savez(path, **out)


if __name__ == "__main__":
    main(sys.argv[1])
