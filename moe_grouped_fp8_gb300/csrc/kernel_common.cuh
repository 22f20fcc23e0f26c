// kernel_common.cuh - small device helpers shared by the grouped-GEMM kernels: CTA-wide scans,
// the uniform OR-barrier of the promotion warps, run lookup, drain waits, UE8M0 decoding.
#pragma once

#include <cstdint>

#include "debug.cuh"
#include "ptx.cuh"

namespace dg {

__device__ __forceinline__ float ue8m0_to_float(uint8_t b) {
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(b) << 23);
}

// K_e of expert e from per-expert sizes ks, or (psum != 0) from inclusive prefix sums
// (K_e = psum[e] - psum[e-1], psum[-1] = 0); a negative difference reads as a bad K_e.
__device__ __forceinline__ long long expert_k(const int32_t* ks, int e, int psum) {
    return psum ? static_cast<long long>(ks[e]) - (e > 0 ? ks[e - 1] : 0) : static_cast<long long>(ks[e]);
}

// Exclusive prefix sum of one int per thread over a CTA of NT threads (all must call).
template <int NT>
__device__ int cta_excl_scan(int v, int* scratch, int* total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) scratch[wid] = incl;
    __syncthreads();
    int pre = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const int w = scratch[i];
        pre += (i < wid) ? w : 0;
        tot += w;
    }
    __syncthreads();
    *total = tot;
    return pre + incl - v;
}

// OR-reduction at named barrier `id` over `n` threads: every participant gets the same answer.
__device__ __forceinline__ bool bar_or(uint32_t id, uint32_t n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Largest r with prefix[r] <= t (prefix non-decreasing, prefix[0] = 0 <= t, R >= 1).
__device__ __forceinline__ int find_run(const int* prefix, int R, int t) {
    int lo = 0, hi = R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Wait used when draining copies in flight on the way out: bounded, ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return;
    }
}

// 1-D bulk copy global -> shared, completing on an mbarrier (sizes and addresses 16-byte aligned).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Wait until at most N of this thread's committed bulk store groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

}  // namespace dg
