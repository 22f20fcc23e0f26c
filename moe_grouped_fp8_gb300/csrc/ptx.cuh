// ptx.cuh - thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor),
// tcgen05 (tensor memory allocation, MMA, loads) and the bounded waits every kernel uses.
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (type only)

#include "dg.h"

namespace dg {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void status_or(int32_t* status, int bits) {
    if (status != nullptr && bits != 0) atomicOr(reinterpret_cast<int*>(status), bits);
}

// ------------------------------------------------------------------------------- dependent launch
// Kernels launched with programmatic stream serialization: `pdl_trigger` lets the next kernel in
// the stream be scheduled as soon as resources allow (it still waits for this one); `pdl_wait`
// blocks until every earlier kernel of the stream has finished and its memory is visible, and is
// called before a kernel's first global-memory access.  Both are no-ops without such a launch.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Context of the bounded waits: a wait that exceeds `limit_ns` ORs DG_STATUS_TIMEOUT into
// the caller's status word and raises the CTA's abort flag, which every other bounded wait
// of the CTA polls; the roles then leave their loops and the kernel returns normally.
struct WaitCtx {
    int32_t* status;
    volatile int* abort_flag;  // shared memory
    uint64_t limit_ns;
};

static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*w.abort_flag) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            status_or(w.status, DG_STATUS_TIMEOUT);
            *w.abort_flag = 1;
            return false;
        }
    }
}

// Returns false when the wait gave up (timeout, or another role of the CTA timed out).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, w);
}

// The same wait with its slow path inlined: for kernels that change their register limit with
// setmaxnreg, whose code may not call functions compiled for another limit.
__device__ __forceinline__ bool mbar_wait_inl(uint64_t* bar, uint32_t parity, const WaitCtx& w) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*w.abort_flag) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            status_or(w.status, DG_STATUS_TIMEOUT);
            *w.abort_flag = 1;
            return false;
        }
    }
}

// Named barrier over `nthreads` threads (id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Per-thread register limit of the executing warpgroup (all four warps execute the same form):
// `dec` returns registers to the CTA's pool, `inc` waits until the pool can grant them.
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg count");
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
    static_assert(N % 8 == 0 && N >= 24 && N <= 256, "setmaxnreg count");
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// ------------------------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const void* tm) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* tm, uint64_t* bar, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* tm, uint64_t* bar, int32_t x, int32_t y,
                                            int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const void* tm, const void* src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}

__device__ __forceinline__ void tma_store_3d(const void* tm, const void* src, int32_t x, int32_t y, int32_t z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
                 : "memory");
}

// A 128-byte line into L2 (a hint: no completion, no value returned).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

// Tile prefetches into L2 (no shared memory, no completion): a later load of the same box hits L2.
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tm, int32_t x, int32_t y, int32_t z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Generic-proxy shared-memory writes -> visible to the async proxy (TMA store, MMA).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// A tensor map written in global memory by an earlier launch: acquire it for the TMA unit.
__device__ __forceinline__ void tmap_acquire(const void* gtm) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(gtm))
                 : "memory");
}

// ------------------------------------------------------------------------------- tcgen05

// Warp-wide.  Writes the TMEM base address of `ncols` columns (power of two >= 32) to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the 128-byte
// swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked contiguously.
//   bits  0-13 start address >> 4        bits 16-29 leading byte offset >> 4 (unused here)
//   bits 32-45 stride byte offset >> 4   bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0: atoms are 1024-byte aligned)   bits 61-63 swizzle (2 = 128B)
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f8f6f4 with e4m3 A and B (both K-major) and
// an fp32 accumulator: bits 4-5 D format (1 = f32), 7-9 A format (0 = e4m3), 10-12 B format
// (0 = e4m3), 15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, M x N x 32 (e4m3).  Issued by one thread.
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of tcgen05.mma.kind::mxf8f6f4 (block-scaled) with e4m3 A, e4m3 or e2m1 B
// (both K-major), an fp32 accumulator and UE8M0 scale factors: bits 4-5 B scale-factor id, 7-9 A
// format (0 = e4m3), 10-12 B format (0 = e4m3, 5 = e2m1), 15/16 A/B major (0 = K), 17-22 N >> 3, 23 scale type
// (1 = UE8M0), 24-28 M >> 4, 29-30 A scale-factor id, 31 K size (0 = dense K 32).  The scale-factor
// ids pick the byte of each 32-bit tensor-memory word that holds a row's scale (id i: bits 8i..8i+7).
// Operand formats of kind::mxf8f6f4 (bits 7-9 for A, 10-12 for B): e4m3 = 0, e2m1 = 5.
constexpr uint32_t MXF_E4M3 = 0u, MXF_E2M1 = 5u;
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3_ue8m0(int M, int N, uint32_t sfa_id = 0, uint32_t sfb_id = 0,
                                                             uint32_t b_fmt = MXF_E4M3) {
    return ((sfb_id & 3u) << 4) | (MXF_E4M3 << 7) | ((b_fmt & 7u) << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24) | ((sfa_id & 3u) << 29);
}

// D[tmem] (+)= (A . 2^sfa)[smem] * (B . 2^sfb)[smem]^T, M x N x 32 (e4m3) with one UE8M0 scale per
// row of A and of B for the instruction's 32-element K block (scale_vec::1X), read from tensor
// memory at sfa_tmem / sfb_tmem.  Issued by one thread.
__device__ __forceinline__ void umma_mxf8_1x(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Shared-memory descriptor of a 32-row x 16-byte matrix stored without swizzle, rows contiguous
// (8-row core matrices 128 bytes apart: stride byte offset 128, one core matrix along K so the
// leading byte offset is unused), the source form of tcgen05.cp.32x128b.
__device__ __forceinline__ uint64_t sdesc_rows16(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>(128u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    return d;  // layout bits 61-63 = 0: no swizzle
}

// Copy 32 rows x 128 bits from shared memory into tensor-memory lanes 0-31, columns taddr ..
// taddr + 3, replicated into each of the four 32-lane quarters.  Issued by one thread; ordered
// before later tcgen05.mma of the same thread.
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Instruction descriptor of tcgen05.mma.kind::f16 with bf16 A and B (both K-major) and an fp32
// accumulator: bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
// 15/16 A/B major (0 = K), 17-22 N >> 3, 24-28 M >> 4.  A and B always share the bf16 type.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, M x N x 16 (bf16 x bf16 -> fp32).  Issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives lane (base + i).
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// A warp's 32 TMEM lanes x W consecutive columns (W = 16 or 32), by array size.
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[16]) { tmem_ld_x16(taddr, r); }
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[32]) { tmem_ld_x32(taddr, r); }

// tcgen05.wait::ld naming the 16 registers of an earlier tmem_ld_x16 (see the 32-register form).
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// tcgen05.wait::ld that also names the 32 registers of an earlier tcgen05.ld as in/out operands,
// so the compiler cannot move any use of them above the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// (y0, y1) = (x0 * s, x1 * s): one packed fp32 multiply, each lane rounded to nearest.
__device__ __forceinline__ void fmul2(float& y0, float& y1, float x0, float x1, float s) {
    asm("{\n\t.reg .b64 d, a, b;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %4};\n\t"
        "mul.rn.f32x2 d, a, b;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(y0), "=f"(y1)
        : "f"(x0), "f"(x1), "f"(s));
}

// Hardware reciprocal approximation (at most 1 ulp from 1/x for normal x).
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// acc0 += s * v0 and acc1 += s * v1 as one packed fp32 FMA; each lane rounds exactly like fmaf.
__device__ __forceinline__ void ffma2(float& acc0, float& acc1, float s, float v0, float v1) {
    asm("{\n\t.reg .b64 d, a, b;\n\t"
        "mov.b64 a, {%2, %3};\n\t"
        "mov.b64 b, {%4, %4};\n\t"
        "mov.b64 d, {%0, %1};\n\t"
        "fma.rn.f32x2 d, a, b, d;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "f"(v0), "f"(v1), "f"(s));
}

}  // namespace dg
