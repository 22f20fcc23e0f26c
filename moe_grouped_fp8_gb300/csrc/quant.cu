// quant.cu - FP8 (e4m3) cast kernels: 1x128 per-token, 128x128 per-block, and per-channel over
// 128 tokens with the per-expert K-major pack.  All three are HBM-bound single-pass kernels:
// one read of the bf16 input, one write of the codes and the scales.
//
// Scale rule (per-channel cast listing of "Non-deterministic numerical problem of
// k_grouped_fp8_gemm_nt_contiguous", applied along K or over a 128x128 tile for the other two
// casts): sf = amax / 448 in fp32; sf == 0 -> sf_zero; sf = max(sf, 1e-30); UE8M0 rounds sf up
// to a power of two.  Codes: e4m3(x * (1/sf)), an IEEE fp32 reciprocal and product, then
// round-to-nearest-even with saturation to +-448.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "host_common.hpp"
#include "cast_common.cuh"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace dg {
namespace {

// ---------------------------------------------------------------------------------------
// 1x128 per-token cast.  An item is one (row, 128-column block); a half-warp handles one item
// (16 lanes x 8 bf16) and a warp takes TOKEN_ITEMS_PER_HW items per half-warp per pass, so
// several 16-byte loads are in flight per thread.  Item indices advance incrementally by the
// items a pass covers (no division in the loop).  Three launch shapes share the item code:
//   rows:    one CTA per chunk of rows_per_cta rows of one row group; it returns at once when
//            the chunk lies past the group's count (groups on the grid's x axis: the chunks that
//            hold rows are dispatched first).  Used without row counts, for more groups than
//            the walk below keeps in shared memory, and for small masked inputs;
//   masked:  a grid of resident CTAs walks one index space of the valid rows only (the rows under
//            each group's count, numbered group after group): every CTA forms the prefix of the
//            clamped counts, then casts an equal share of the valid (row, 128-block) items, mapping
//            each row to its group and row.  No CTA is launched for rows past the counts, which in
//            decode (192 rows of a 4096-row capacity) are 95% of the grid above, and the shares
//            differ by at most one item;
//   routed:  CTA x owns rows_per_cta rows and compacts those whose m_indices entry is >= 0.
// rows_per_cta gives the rows and routed CTAs about TOKEN_ITEMS_PER_CTA items each.
// ---------------------------------------------------------------------------------------
constexpr int TOKEN_ITEMS_PER_HW = 4;
constexpr int TOKEN_ITEMS_PER_CTA = 512;
constexpr int TOKEN_MIN_ITEMS_PER_CTA = 128;
constexpr int TOKEN_CTAS_PER_SM = 4;  // resident 256-thread CTAs at the kernels' register counts
constexpr int TOKEN_PER_WARP = 2 * TOKEN_ITEMS_PER_HW;
constexpr int TOKEN_WALK_MAX_GROUPS = 1024; // groups whose prefix the masked walk keeps
// Below this many (row, block) items of capacity the per-group grid is faster: the pages'
// reproduction shape (8 x 32 rows, K = 256) casts in 2.4 us on 8 CTAs against 4.4 us on the walk's
// 4 CTAs, several passes each; from the 8-expert decode case up the two are equal or the walk wins.
constexpr int64_t TOKEN_WALK_MIN_ITEMS = 65536;

__device__ __forceinline__ uint4 token_load(const uint16_t* x, int64_t ldx, bool live, int64_t m, int kb, int sub) {
    return live ? __ldg(reinterpret_cast<const uint4*>(x + m * ldx + static_cast<int64_t>(kb) * 128) + sub)
                : make_uint4(0, 0, 0, 0);
}

// amax over the item (all 32 lanes take part in the shuffles), then codes and scale if live.
template <bool UE8M0>
__device__ __forceinline__ void token_item(const uint4& raw, bool live, int64_t m, int kb, int sub, int64_t K,
                                           uint8_t* __restrict__ q, void* sfa, int64_t Mp, float sf_zero) {
    float f[8];
    bf16x8_to_float(raw, f);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (!live || !DG_CHECKED(m < Mp, DG_DEBUG_CAST_OUT)) return;
    float sf, r;
    uint8_t byte = 0;
    block_scale<UE8M0>(amax, sf_zero, sf, r, byte);
    *reinterpret_cast<uint2*>(q + m * K + static_cast<int64_t>(kb) * 128 + sub * 8) = e4m3x8(f, r);
    if (sub == 0) {
        if constexpr (UE8M0)
            static_cast<uint8_t*>(sfa)[kb * Mp + m] = byte;
        else
            static_cast<float*>(sfa)[kb * Mp + m] = sf;
    }
}

// Items [first, end) of a CTA's rows (item i = row i / KB, block i % KB; the default range is
// every item of `nrows` rows): row i is m_base + i, or m_base + s_rows[i] (LIST), in q and sfa and,
// unless XPACK, in x; with XPACK row i is read from row x_base + i of x.
template <bool UE8M0, bool LIST, bool XPACK = false>
__device__ __forceinline__ void token_rows(const uint16_t* __restrict__ x, int64_t K, int64_t ldx,
                                           uint8_t* __restrict__ q, void* sfa, int64_t M, int64_t Mp,
                                           float sf_zero, int64_t m_base, const int* s_rows, int nrows,
                                           int first = 0, int end = -1, int64_t x_base = 0) {
    const int KBi = static_cast<int>(K / 128);
    const int items = end < 0 ? nrows * KBi : end;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hw = lane >> 4, sub = lane & 15;
    const int step = (blockDim.x >> 5) * TOKEN_PER_WARP;
    const int step_m = step / KBi, step_kb = step - step_m * KBi;
    int it[TOKEN_ITEMS_PER_HW], mr[TOKEN_ITEMS_PER_HW], kb[TOKEN_ITEMS_PER_HW];
#pragma unroll
    for (int j = 0; j < TOKEN_ITEMS_PER_HW; ++j) {
        it[j] = first + warp * TOKEN_PER_WARP + 2 * j + hw;
        mr[j] = it[j] / KBi;
        kb[j] = it[j] - mr[j] * KBi;
    }
    for (int base = first + warp * TOKEN_PER_WARP; base < items; base += step) {
        uint4 raw[TOKEN_ITEMS_PER_HW];
        int64_t m[TOKEN_ITEMS_PER_HW];
        bool live[TOKEN_ITEMS_PER_HW];
#pragma unroll
        for (int j = 0; j < TOKEN_ITEMS_PER_HW; ++j) {
            live[j] = it[j] < items;
            m[j] = m_base + (LIST ? (live[j] ? s_rows[mr[j]] : 0) : mr[j]);
            const int64_t xm = XPACK ? x_base + mr[j] : m[j];
            live[j] = live[j] && DG_CHECKED(xm >= 0 && xm < M, DG_DEBUG_CAST_IN);
            raw[j] = token_load(x, ldx, live[j], xm, kb[j], sub);
        }
#pragma unroll
        for (int j = 0; j < TOKEN_ITEMS_PER_HW; ++j) {
            token_item<UE8M0>(raw[j], live[j], m[j], kb[j], sub, K, q, sfa, Mp, sf_zero);
            it[j] += step;
            mr[j] += step_m;
            kb[j] += step_kb;
            if (kb[j] >= KBi) {
                kb[j] -= KBi;
                ++mr[j];
            }
        }
    }
}

template <bool UE8M0>
__global__ void __launch_bounds__(256) k_quant_token_1x128(const uint16_t* __restrict__ x, int64_t K, int64_t ldx,
                                                           uint8_t* __restrict__ q, void* sfa, int64_t M, int64_t Mp,
                                                           float sf_zero, const int32_t* __restrict__ row_counts,
                                                           int64_t rpg, int64_t rows_per_cta, int group_in_x) {
    pdl_trigger();
    pdl_wait();
    const int64_t g = group_in_x ? blockIdx.x : blockIdx.y;
    const int64_t chunk = group_in_x ? blockIdx.y : blockIdx.x;
    int64_t lim = rpg;
    if (row_counts != nullptr) {
        lim = row_counts[g];
        lim = lim < 0 ? 0 : (lim > rpg ? rpg : lim);
    }
    const int64_t r_begin = chunk * rows_per_cta;
    if (r_begin >= lim) return;
    const int64_t r_end = min(lim, r_begin + rows_per_cta);
    token_rows<UE8M0, false>(x, K, ldx, q, sfa, M, Mp, sf_zero, g * rpg + r_begin, nullptr,
                             static_cast<int>(r_end - r_begin));
}

// Exclusive prefix of the counts clamped to [0, cap] into s_prefix[0..G] (s_prefix[G] = the
// total), for a CTA of 256 threads (all must call); thread t sums a contiguous slice of groups.
__device__ __forceinline__ int valid_prefix(const int32_t* __restrict__ counts, int G, int64_t cap, int* s_prefix,
                                            int* s_scan) {
    const int t = threadIdx.x;
    const int ch = (G + 255) / 256;
    const int lo = min(G, t * ch), hi = min(G, lo + ch);
    int sum = 0;
    for (int g = lo; g < hi; ++g) {
        const int64_t c = counts[g];
        sum += static_cast<int>(c < 0 ? 0 : (c > cap ? cap : c));
    }
    int total = 0;
    int p = cta_excl_scan<256>(sum, s_scan, &total);
    for (int g = lo; g < hi; ++g) {
        s_prefix[g] = p;
        const int64_t c = counts[g];
        p += static_cast<int>(c < 0 ? 0 : (c > cap ? cap : c));
    }
    if (t == 0) s_prefix[G] = total;
    __syncthreads();
    return total;
}

// XPACK: x holds the valid rows packed at its front, group after group (valid row f is row f of x).
template <bool UE8M0, bool XPACK>
__global__ void __launch_bounds__(256) k_quant_token_masked(const uint16_t* __restrict__ x, int64_t K, int64_t ldx,
                                                            uint8_t* __restrict__ q, void* sfa, int64_t M, int64_t Mp,
                                                            float sf_zero, const int32_t* __restrict__ row_counts,
                                                            int G, int64_t rpg) {
    __shared__ int s_prefix[TOKEN_WALK_MAX_GROUPS + 1];
    __shared__ int s_rows[256];
    __shared__ int s_scan[8];
    pdl_trigger();
    pdl_wait();
    const int t = threadIdx.x;
    const int total = valid_prefix(row_counts, G, rpg, s_prefix, s_scan);
    // this CTA's equal share of the valid (row, 128-block) items, taken in runs of at most 256 rows
    const int KBi = static_cast<int>(K / 128);
    const int64_t items = static_cast<int64_t>(total) * KBi;
    int64_t i0 = items * blockIdx.x / gridDim.x;
    const int64_t i1 = items * (blockIdx.x + 1) / gridDim.x;
    while (i0 < i1) {
        const int64_t r0 = i0 / KBi;
        const int64_t r_end = min(r0 + 256, (i1 + KBi - 1) / KBi);
        const int64_t e1 = min(i1, r_end * KBi);
        const int n = static_cast<int>(r_end - r0);
        if (t < n) {
            const int f = static_cast<int>(r0) + t;
            const int g = find_run(s_prefix, G, f);  // the group whose valid rows hold f
            s_rows[t] = static_cast<int>(g * rpg) + (f - s_prefix[g]);
        }
        __syncthreads();
        token_rows<UE8M0, true, XPACK>(x, K, ldx, q, sfa, M, Mp, sf_zero, 0, s_rows, n,
                                       static_cast<int>(i0 - r0 * KBi), static_cast<int>(e1 - r0 * KBi), r0);
        __syncthreads();
        i0 = e1;
    }
}

template <bool UE8M0>
__global__ void __launch_bounds__(256) k_quant_token_routed(const uint16_t* __restrict__ x, int64_t K, int64_t ldx,
                                                            uint8_t* __restrict__ q, void* sfa, int64_t Mp,
                                                            float sf_zero, const int32_t* __restrict__ m_indices,
                                                            int64_t M, int rows_per_cta) {
    __shared__ int s_rows[256];
    __shared__ int s_scan[8];
    pdl_trigger();
    pdl_wait();
    const int64_t m_base = static_cast<int64_t>(blockIdx.x) * rows_per_cta;
    const int t = threadIdx.x;
    const bool v = t < rows_per_cta && m_base + t < M && m_indices[m_base + t] >= 0;
    int nrows = 0;
    const int pos = cta_excl_scan<256>(v ? 1 : 0, s_scan, &nrows);
    if (v) s_rows[pos] = t;
    __syncthreads();
    if (nrows == 0) return;
    token_rows<UE8M0, true>(x, K, ldx, q, sfa, M, Mp, sf_zero, m_base, s_rows, nrows);
}

// ---------------------------------------------------------------------------------------
// Packing of a masked buffer's valid rows: row r < min(max(count_g, 0), cap) of group g of a
// [G, cap] array of rows moves to row prefix_g + r of dst (prefix_g = the valid rows of the groups
// before g), e.g. the GEMM's [G, cap, N] output before one copy to the host.  A CTA takes an equal
// share of the valid rows; each warp copies whole rows, 16 bytes per lane, four in flight.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_pack_masked_rows(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                          int64_t row_bytes, const int32_t* __restrict__ counts,
                                                          int G, int64_t cap) {
    __shared__ int s_prefix[TOKEN_WALK_MAX_GROUPS + 1];
    __shared__ int s_scan[8];
    pdl_trigger();
    pdl_wait();
    const int total = valid_prefix(counts, G, cap, s_prefix, s_scan);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t f0 = static_cast<int64_t>(total) * blockIdx.x / gridDim.x;
    const int64_t f1 = static_cast<int64_t>(total) * (blockIdx.x + 1) / gridDim.x;
    const int64_t chunks = row_bytes / 16;
    for (int64_t f = f0 + warp; f < f1; f += blockDim.x >> 5) {
        const int g = find_run(s_prefix, G, static_cast<int>(f));
        const int64_t srow = static_cast<int64_t>(g) * cap + (f - s_prefix[g]);
        if (!DG_CHECKED(g >= 0 && g < G && srow < static_cast<int64_t>(G) * cap, DG_DEBUG_CAST_IN)) continue;
        const uint4* s = reinterpret_cast<const uint4*>(src + srow * row_bytes);
        uint4* d = reinterpret_cast<uint4*>(dst + f * row_bytes);
        for (int64_t c = lane; c < chunks; c += 32 * 4) {
            uint4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c + 32 * u < chunks) v[u] = __ldg(s + c + 32 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c + 32 * u < chunks) d[c + 32 * u] = v[u];
        }
    }
}

// ---------------------------------------------------------------------------------------
// 128x128 per-block cast.  One CTA (256 threads) per block; thread t holds 16-byte column
// chunk (t % 16) of rows (t / 16) + 16 j, j < 8, so each warp load covers two full 256-byte
// row segments.
// ---------------------------------------------------------------------------------------
template <bool UE8M0>
__global__ void __launch_bounds__(256) k_quant_block_128x128(const uint16_t* __restrict__ w, int G, int64_t N,
                                                             int64_t K, uint8_t* __restrict__ q, void* sfb,
                                                             float sf_zero) {
    pdl_trigger();
    pdl_wait();
    const int64_t NB = N / 128, KB = K / 128;
    const int64_t blk = blockIdx.x;
    const int64_t kb = blk % KB;
    const int64_t nb = (blk / KB) % NB;
    const int64_t g = blk / (KB * NB);
    if (!DG_CHECKED(g < G, DG_DEBUG_CAST_IN)) return;  // the whole CTA
    const int t = threadIdx.x;
    const int c = t & 15, r0 = t >> 4;
    const uint16_t* base = w + (g * N + nb * 128) * K + kb * 128;

    uint4 raw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        raw[j] = __ldg(reinterpret_cast<const uint4*>(base + static_cast<int64_t>(r0 + 16 * j) * K) + c);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float f[8];
        bf16x8_to_float(raw[j], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float s_amax[8];
    if ((t & 31) == 0) s_amax[t >> 5] = amax;
    __syncthreads();
    amax = s_amax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, s_amax[i]);

    float sf, r;
    uint8_t byte = 0;
    block_scale<UE8M0>(amax, sf_zero, sf, r, byte);
    uint8_t* qb = q + (g * N + nb * 128) * K + kb * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float f[8];
        bf16x8_to_float(raw[j], f);
        *reinterpret_cast<uint2*>(qb + static_cast<int64_t>(r0 + 16 * j) * K + c * 8) = e4m3x8(f, r);
    }
    if (t == 0) {
        const int64_t si = (g * NB + nb) * KB + kb;
        if constexpr (UE8M0)
            static_cast<uint8_t*>(sfb)[si] = byte;
        else
            static_cast<float*>(sfb)[si] = sf;
    }
}

// ---------------------------------------------------------------------------------------
// 128x128 per-block cast of FP4 (e2m1) weights, the weight operand of the FP8 x FP4 m-grouped
// GEMM ("SM120 m_grouped_fp8 contiguous kernel: illegal memory access at CUDA graph replay",
// #444: m_grouped_fp8_fp4_gemm_nt_contiguous, weights with 2^k scales).  The FP8 block cast's
// rule with e2m1's maximum 6 in place of 448: sf = amax / 6 (IEEE division), zero -> sf_zero,
// >= 1e-30, rounded up to a power of two (UE8M0); codes e2m1(x * (1/sf)) with round-to-nearest-
// even and saturation.  Two codes per byte along K, the even element in the low nibble.  The
// thread layout is the FP8 block cast's.
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_quant_block_128x128_fp4(const uint16_t* __restrict__ w, int G, int64_t N,
                                                                 int64_t K, uint8_t* __restrict__ q,
                                                                 uint8_t* __restrict__ sfb, float sf_zero) {
    pdl_trigger();
    pdl_wait();
    const int64_t NB = N / 128, KB = K / 128;
    const int64_t blk = blockIdx.x;
    const int64_t kb = blk % KB;
    const int64_t nb = (blk / KB) % NB;
    const int64_t g = blk / (KB * NB);
    if (!DG_CHECKED(g < G, DG_DEBUG_CAST_IN)) return;  // the whole CTA
    const int t = threadIdx.x;
    const int c = t & 15, r0 = t >> 4;
    const uint16_t* base = w + (g * N + nb * 128) * K + kb * 128;

    uint4 raw[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        raw[j] = __ldg(reinterpret_cast<const uint4*>(base + static_cast<int64_t>(r0 + 16 * j) * K) + c);
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float f[8];
        bf16x8_to_float(raw[j], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    __shared__ float s_amax[8];
    if ((t & 31) == 0) s_amax[t >> 5] = amax;
    __syncthreads();
    amax = s_amax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, s_amax[i]);

    float sf = __fdiv_rn(amax, 6.0f);
    if (sf == 0.0f) sf = sf_zero;
    sf = fmaxf(sf, 1e-30f);
    uint8_t byte = 0;
    sf = ue8m0_round_up(sf, &byte);
    const float r = __frcp_rn(sf);
    // 16 consecutive bytes of a packed row hold 32 codes; this thread's 8 values are 4 bytes
    uint8_t* qb = q + ((g * N + nb * 128) * K + kb * 128) / 2;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        float f[8];
        bf16x8_to_float(raw[j], f);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_fp4x2_storage_t two = __nv_cvt_float2_to_fp4x2(
                make_float2(__fmul_rn(f[2 * i], r), __fmul_rn(f[2 * i + 1], r)), __NV_E2M1, cudaRoundNearest);
            word |= static_cast<uint32_t>(two) << (8 * i);
        }
        *reinterpret_cast<uint32_t*>(qb + static_cast<int64_t>(r0 + 16 * j) * (K / 2) + c * 4) = word;
    }
    if (t == 0) sfb[(g * NB + nb) * KB + kb] = byte;
}

// One or two operands cast per launch (the two operands of a k-grouped wgrad share ks).
__global__ void __launch_bounds__(256) k_quant_channel_128(const ChannelOperand op0, const ChannelOperand op1,
                                                           int nblk0, int64_t K_cap, const int32_t* __restrict__ ks,
                                                           int psum, int G, float sf_zero, int32_t* status) {
    channel_cast_cta(op0, op1, nblk0, K_cap, ks, psum, G, sf_zero, status, static_cast<int>(blockIdx.x),
                     static_cast<int>(blockIdx.y));
}

}  // namespace
}  // namespace dg

using namespace dg;

namespace {

int check_token_args(const void* x, int64_t M, int64_t K, int64_t ldx, const uint8_t* q, const void* sfa,
                     int sf_format) {
    DG_CHECK_ARG(M >= 0 && K > 0 && K % 128 == 0, "need M >= 0 and K a positive multiple of 128 (M=%lld K=%lld)",
                 (long long)M, (long long)K);
    DG_CHECK_ARG(ldx >= K && (ldx * 2) % 16 == 0, "ldx must be >= K and ldx*2 a multiple of 16 (ldx=%lld)",
                 (long long)ldx);
    DG_CHECK_ARG(sf_format == DG_SF_FP32 || sf_format == DG_SF_UE8M0, "bad sf_format %d", sf_format);
    DG_CHECK_SUPPORTED(K / 128 < (1ll << 24), "K too large (K=%lld)", (long long)K);
    if (M == 0) return DG_OK;
    DG_CHECK_ARG(x && q && sfa, "null pointer argument");
    DG_CHECK_ARG(aligned16(x) && ((reinterpret_cast<uintptr_t>(q) & 7u) == 0), "x must be 16-byte and q 8-byte aligned");
    return DG_OK;
}

int64_t token_mp(int64_t M, int sf_format) {
    return (sf_format == DG_SF_FP32) ? (M + 3) / 4 * 4 : (M + 15) / 16 * 16;
}

}  // namespace

namespace {
std::atomic<int> g_token_items{0};  // items per CTA of the per-token casts; 0 = TOKEN_ITEMS_PER_CTA

// Rows per CTA.  Masked calls launch a CTA for every chunk up to the capacity, most of them
// empty in decode, so their chunks stay large (TOKEN_ITEMS_PER_CTA items).  Otherwise the chunks
// shrink (to 128 items at least) until the grid is about four waves of resident CTAs, which
// trims the last partial wave on small inputs.
int token_rows_per_cta(int64_t KB, int64_t rows, bool masked, int64_t cap_rows) {
    int64_t want = g_token_items.load(std::memory_order_relaxed);
    if (want <= 0) {
        want = TOKEN_ITEMS_PER_CTA;
        int sms = 0;
        if (!masked && device_sm_count(&sms) == DG_OK && sms > 0) {
            const int64_t waves = rows * KB / (4ll * TOKEN_CTAS_PER_SM * sms);
            want = std::max<int64_t>(TOKEN_MIN_ITEMS_PER_CTA, std::min<int64_t>(want, waves));
        }
    }
    const int64_t r = KB >= want ? 1 : want / KB;
    return static_cast<int>(r < cap_rows ? r : cap_rows);
}
}  // namespace

extern "C" int dg_testing_token_items_per_cta(int items) {
    DG_CHECK_ARG(items >= 0 && items <= (1 << 20), "items per CTA out of range (%d)", items);
    g_token_items.store(items, std::memory_order_relaxed);
    return DG_OK;
}

extern "C" int dg_quant_per_token_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, void* sfa,
                                        int sf_format, float sf_zero, const int32_t* row_counts, int G,
                                        void* stream) {
    DG_ARG_LOG(x, M, K, ldx, q, sfa, sf_format, sf_zero, row_counts, G, stream);
    if (int rc = check_token_args(x, M, K, ldx, q, sfa, sf_format)) return rc;
    if (M == 0) return DG_OK;
    int64_t rpg = M;
    if (row_counts != nullptr) {
        DG_CHECK_ARG(G >= 1 && M % G == 0, "row_counts needs G >= 1 dividing M (M=%lld G=%d)", (long long)M, G);
        rpg = M / G;
    }
    const int64_t groups = row_counts != nullptr ? G : 1;
    const bool ue = sf_format == DG_SF_UE8M0;
    const bool hooked = g_token_items.load(std::memory_order_relaxed) > 0;
    if (row_counts != nullptr && G <= TOKEN_WALK_MAX_GROUPS && M < (1ll << 31) && M * (K / 128) < (1ll << 40) &&
        (M * (K / 128) >= TOKEN_WALK_MIN_ITEMS || hooked)) {
        // the walk over valid rows: two CTAs per resident slot share the valid items equally (or,
        // through the test hook, a grid of about that many items per CTA over the capacity; the
        // hook also keeps small inputs on the walk, so that tests reach it at every size)
        int sms = 0;
        if (int rc = device_sm_count(&sms)) return rc;
        int64_t grid = std::min<int64_t>(2ll * TOKEN_CTAS_PER_SM * sms,
                                         (M * (K / 128) + TOKEN_MIN_ITEMS_PER_CTA - 1) / TOKEN_MIN_ITEMS_PER_CTA);
        const int64_t want = g_token_items.load(std::memory_order_relaxed);
        if (want > 0) grid = std::max<int64_t>(1, std::min<int64_t>(65535, M * (K / 128) / want));
        return launch_pdl(ue ? k_quant_token_masked<true, false> : k_quant_token_masked<false, false>,
                          dim3(static_cast<unsigned>(grid)), dim3(256), 0, static_cast<cudaStream_t>(stream),
                          static_cast<const uint16_t*>(x), K, ldx, q, sfa, M, token_mp(M, sf_format), sf_zero,
                          row_counts, G, rpg);
    }
    const int64_t rows_per_cta = token_rows_per_cta(K / 128, M, row_counts != nullptr, 1ll << 30);
    const int64_t chunks = (rpg + rows_per_cta - 1) / rows_per_cta;
    // groups on x (fastest dispatch) when there are several and the chunks fit the y axis
    const int group_in_x = groups > 1 && chunks < 65536 ? 1 : 0;
    DG_CHECK_SUPPORTED(group_in_x || (chunks < (1ll << 31) && groups < 65536), "too many rows or groups");
    const dim3 grid = group_in_x ? dim3(static_cast<unsigned>(groups), static_cast<unsigned>(chunks))
                                 : dim3(static_cast<unsigned>(chunks), static_cast<unsigned>(groups));
    return launch_pdl(ue ? k_quant_token_1x128<true> : k_quant_token_1x128<false>, grid, dim3(256), 0,
                      static_cast<cudaStream_t>(stream), static_cast<const uint16_t*>(x), K, ldx, q, sfa, M,
                      token_mp(M, sf_format), sf_zero, row_counts, rpg, rows_per_cta, group_in_x);
}

extern "C" int dg_quant_per_token_1x128_routed(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                               void* sfa, int sf_format, float sf_zero, const int32_t* m_indices,
                                               void* stream) {
    DG_ARG_LOG(x, M, K, ldx, q, sfa, sf_format, sf_zero, m_indices, stream);
    if (int rc = check_token_args(x, M, K, ldx, q, sfa, sf_format)) return rc;
    if (M == 0) return DG_OK;
    DG_CHECK_ARG(m_indices != nullptr, "m_indices must not be NULL");
    const int rows_per_cta = token_rows_per_cta(K / 128, M, false, 256);
    const int64_t gx = (M + rows_per_cta - 1) / rows_per_cta;
    DG_CHECK_SUPPORTED(gx < (1ll << 31), "too many rows");
    const bool ue = sf_format == DG_SF_UE8M0;
    return launch_pdl(ue ? k_quant_token_routed<true> : k_quant_token_routed<false>, dim3(static_cast<unsigned>(gx)),
                      dim3(256), 0, static_cast<cudaStream_t>(stream), static_cast<const uint16_t*>(x), K, ldx, q,
                      sfa, token_mp(M, sf_format), sf_zero, m_indices, M, rows_per_cta);
}

extern "C" int dg_quant_per_token_1x128_packed(const void* x, int64_t K, int64_t ldx, uint8_t* q, void* sfa,
                                               int sf_format, float sf_zero, const int32_t* row_counts, int G,
                                               int64_t cap, void* stream) {
    DG_ARG_LOG(x, K, ldx, q, sfa, sf_format, sf_zero, row_counts, G, cap, stream);
    DG_CHECK_ARG(G >= 1 && G <= TOKEN_WALK_MAX_GROUPS && cap >= 0, "need 1 <= G <= %d and cap >= 0 (G=%d cap=%lld)",
                 TOKEN_WALK_MAX_GROUPS, G, (long long)cap);
    const int64_t M = static_cast<int64_t>(G) * cap;
    if (int rc = check_token_args(x, M, K, ldx, q, sfa, sf_format)) return rc;
    if (M == 0) return DG_OK;
    DG_CHECK_ARG(row_counts != nullptr, "row_counts must not be NULL");
    DG_CHECK_SUPPORTED(M < (1ll << 31) && M * (K / 128) < (1ll << 40), "too many rows (G x cap = %lld)", (long long)M);
    int sms = 0;
    if (int rc = device_sm_count(&sms)) return rc;
    int64_t grid = std::min<int64_t>(2ll * TOKEN_CTAS_PER_SM * sms,
                                     (M * (K / 128) + TOKEN_MIN_ITEMS_PER_CTA - 1) / TOKEN_MIN_ITEMS_PER_CTA);
    const int64_t want = g_token_items.load(std::memory_order_relaxed);
    if (want > 0) grid = std::max<int64_t>(1, std::min<int64_t>(65535, M * (K / 128) / want));
    const bool ue = sf_format == DG_SF_UE8M0;
    return launch_pdl(ue ? k_quant_token_masked<true, true> : k_quant_token_masked<false, true>,
                      dim3(static_cast<unsigned>(grid)), dim3(256), 0, static_cast<cudaStream_t>(stream),
                      static_cast<const uint16_t*>(x), K, ldx, q, sfa, M, token_mp(M, sf_format), sf_zero, row_counts,
                      G, cap);
}

extern "C" int dg_pack_masked_rows(const void* src, int G, int64_t cap, int64_t row_bytes, const int32_t* counts,
                                   void* dst, void* stream) {
    DG_ARG_LOG(src, G, cap, row_bytes, counts, dst, stream);
    DG_CHECK_ARG(G >= 1 && G <= TOKEN_WALK_MAX_GROUPS && cap >= 0, "need 1 <= G <= %d and cap >= 0 (G=%d cap=%lld)",
                 TOKEN_WALK_MAX_GROUPS, G, (long long)cap);
    DG_CHECK_ARG(row_bytes > 0 && row_bytes % 16 == 0, "row_bytes must be a positive multiple of 16 (%lld)",
                 (long long)row_bytes);
    const int64_t M = static_cast<int64_t>(G) * cap;
    if (M == 0) return DG_OK;
    DG_CHECK_ARG(src && dst && counts, "null pointer argument");
    DG_CHECK_ARG(aligned16(src) && aligned16(dst), "src and dst must be 16-byte aligned");
    DG_CHECK_SUPPORTED(M < (1ll << 31), "too many rows (G x cap = %lld)", (long long)M);
    int sms = 0;
    if (int rc = device_sm_count(&sms)) return rc;
    const int64_t grid = std::min<int64_t>(2ll * TOKEN_CTAS_PER_SM * sms, (M + 7) / 8);
    return launch_pdl(k_pack_masked_rows, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                      static_cast<cudaStream_t>(stream), static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst),
                      row_bytes, counts, G, cap);
}

extern "C" int dg_quant_block_128x128(const void* w, int G, int64_t N, int64_t K, uint8_t* q, void* sfb,
                                      int sf_format, float sf_zero, void* stream) {
    DG_ARG_LOG(w, G, N, K, q, sfb, sf_format, sf_zero, stream);
    DG_CHECK_ARG(G >= 0 && N >= 0 && K >= 0 && N % 128 == 0 && K % 128 == 0,
                 "need N and K multiples of 128 (G=%d N=%lld K=%lld)", G, (long long)N, (long long)K);
    DG_CHECK_ARG(sf_format == DG_SF_FP32 || sf_format == DG_SF_UE8M0, "bad sf_format %d", sf_format);
    const int64_t blocks = static_cast<int64_t>(G) * (N / 128) * (K / 128);
    if (blocks == 0) return DG_OK;
    DG_CHECK_ARG(w && q && sfb, "null pointer argument");
    DG_CHECK_ARG(aligned16(w) && ((reinterpret_cast<uintptr_t>(q) & 7u) == 0), "w must be 16-byte and q 8-byte aligned");
    DG_CHECK_SUPPORTED(blocks < (1ll << 31), "too many 128x128 blocks");
    auto s = static_cast<cudaStream_t>(stream);
    const auto* wp = static_cast<const uint16_t*>(w);
    const dim3 grid(static_cast<unsigned>(blocks));
    if (sf_format == DG_SF_UE8M0)
        return launch_pdl(k_quant_block_128x128<true>, grid, dim3(256), 0, s, wp, G, N, K, q, sfb, sf_zero);
    return launch_pdl(k_quant_block_128x128<false>, grid, dim3(256), 0, s, wp, G, N, K, q, sfb, sf_zero);
}

extern "C" int dg_quant_block_128x128_fp4(const void* w, int G, int64_t N, int64_t K, uint8_t* q_packed,
                                          uint8_t* sfb, float sf_zero, void* stream) {
    DG_ARG_LOG(w, G, N, K, q_packed, sfb, sf_zero, stream);
    DG_CHECK_ARG(G >= 0 && N >= 0 && K >= 0 && N % 128 == 0 && K % 128 == 0,
                 "need N and K multiples of 128 (G=%d N=%lld K=%lld)", G, (long long)N, (long long)K);
    const int64_t blocks = static_cast<int64_t>(G) * (N / 128) * (K / 128);
    if (blocks == 0) return DG_OK;
    DG_CHECK_ARG(w && q_packed && sfb, "null pointer argument");
    DG_CHECK_ARG(aligned16(w) && ((reinterpret_cast<uintptr_t>(q_packed) & 3u) == 0),
                 "w must be 16-byte and q_packed 4-byte aligned");
    DG_CHECK_SUPPORTED(blocks < (1ll << 31), "too many 128x128 blocks");
    return launch_pdl(k_quant_block_128x128_fp4, dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                      static_cast<cudaStream_t>(stream), static_cast<const uint16_t*>(w), G, N, K, q_packed, sfb,
                      sf_zero);
}

namespace dg {
namespace {

int quant_channel(const void* x, int64_t K_cap, int64_t C, const int32_t* ks, int psum, int G, uint8_t* q_packed,
                  float* sf, float sf_zero, int32_t* status, void* stream) {
    DG_CHECK_ARG(K_cap >= 0 && K_cap % 128 == 0, "K_cap must be a multiple of 128 (%lld)", (long long)K_cap);
    DG_CHECK_ARG(C > 0 && C % CH_COLS == 0, "C must be a positive multiple of %d (%lld)", CH_COLS, (long long)C);
    DG_CHECK_ARG(G >= 1 && G <= DG_MAX_GROUPS, "G must be in [1, %d] (%d)", DG_MAX_GROUPS, G);
    if (K_cap == 0) return DG_OK;
    DG_CHECK_ARG(x && ks && q_packed && sf, "null pointer argument");
    DG_CHECK_ARG(aligned16(x) && aligned16(q_packed), "x and q_packed must be 16-byte aligned");
    DG_CHECK_SUPPORTED(K_cap / 128 < 65536, "K_cap too large");
    dim3 grid(static_cast<unsigned>(C / CH_COLS), static_cast<unsigned>(K_cap / 128));
    const ChannelOperand op{static_cast<const uint16_t*>(x), C, q_packed, sf};
    return launch_pdl(k_quant_channel_128, grid, dim3(256), 0, static_cast<cudaStream_t>(stream), op, op,
                      static_cast<int>(C / CH_COLS), K_cap, ks, psum, G, sf_zero, status);
}

int quant_channel_pair(const void* x_a, int64_t C_a, uint8_t* q_a, float* sf_a, const void* x_b, int64_t C_b,
                       uint8_t* q_b, float* sf_b, int64_t K_cap, const int32_t* ks, int psum, int G, float sf_zero,
                       int32_t* status, void* stream) {
    DG_CHECK_ARG(K_cap >= 0 && K_cap % 128 == 0, "K_cap must be a multiple of 128 (%lld)", (long long)K_cap);
    DG_CHECK_ARG(C_a > 0 && C_a % CH_COLS == 0 && C_b > 0 && C_b % CH_COLS == 0,
                 "C_a and C_b must be positive multiples of %d", CH_COLS);
    DG_CHECK_ARG(G >= 1 && G <= DG_MAX_GROUPS, "G must be in [1, %d] (%d)", DG_MAX_GROUPS, G);
    if (K_cap == 0) return DG_OK;
    DG_CHECK_ARG(x_a && q_a && sf_a && x_b && q_b && sf_b && ks, "null pointer argument");
    DG_CHECK_ARG(aligned16(x_a) && aligned16(q_a) && aligned16(x_b) && aligned16(q_b),
                 "x and q buffers must be 16-byte aligned");
    DG_CHECK_SUPPORTED(K_cap / 128 < 65536 && (C_a + C_b) / CH_COLS < (1ll << 31), "sizes too large");
    const ChannelOperand op0{static_cast<const uint16_t*>(x_a), C_a, q_a, sf_a};
    const ChannelOperand op1{static_cast<const uint16_t*>(x_b), C_b, q_b, sf_b};
    const int nblk0 = static_cast<int>(C_a / CH_COLS);
    dim3 grid(static_cast<unsigned>(nblk0 + C_b / CH_COLS), static_cast<unsigned>(K_cap / 128));
    return launch_pdl(k_quant_channel_128, grid, dim3(256), 0, static_cast<cudaStream_t>(stream), op0, op1, nblk0,
                      K_cap, ks, psum, G, sf_zero, status);
}

}  // namespace
}  // namespace dg

extern "C" int dg_quant_per_channel_128(const void* x, int64_t K_cap, int64_t C, const int32_t* ks, int G,
                                        uint8_t* q_packed, float* sf, float sf_zero, int32_t* status,
                                        void* stream) {
    DG_ARG_LOG(x, K_cap, C, ks, G, q_packed, sf, sf_zero, status, stream);
    return quant_channel(x, K_cap, C, ks, 0, G, q_packed, sf, sf_zero, status, stream);
}

extern "C" int dg_quant_per_channel_128_psum(const void* x, int64_t K_cap, int64_t C, const int32_t* psum, int G,
                                             uint8_t* q_packed, float* sf, float sf_zero, int32_t* status,
                                             void* stream) {
    DG_ARG_LOG(x, K_cap, C, psum, G, q_packed, sf, sf_zero, status, stream);
    return quant_channel(x, K_cap, C, psum, 1, G, q_packed, sf, sf_zero, status, stream);
}

extern "C" int dg_quant_per_channel_128_pair(const void* x_a, int64_t C_a, uint8_t* q_a, float* sf_a, const void* x_b,
                                             int64_t C_b, uint8_t* q_b, float* sf_b, int64_t K_cap,
                                             const int32_t* ks, int G, float sf_zero, int32_t* status,
                                             void* stream) {
    DG_ARG_LOG(x_a, C_a, q_a, sf_a, x_b, C_b, q_b, sf_b, K_cap, ks, G, sf_zero, status, stream);
    return quant_channel_pair(x_a, C_a, q_a, sf_a, x_b, C_b, q_b, sf_b, K_cap, ks, 0, G, sf_zero, status, stream);
}

extern "C" int dg_quant_per_channel_128_pair_psum(const void* x_a, int64_t C_a, uint8_t* q_a, float* sf_a,
                                                  const void* x_b, int64_t C_b, uint8_t* q_b, float* sf_b,
                                                  int64_t K_cap, const int32_t* psum, int G, float sf_zero,
                                                  int32_t* status, void* stream) {
    DG_ARG_LOG(x_a, C_a, q_a, sf_a, x_b, C_b, q_b, sf_b, K_cap, psum, G, sf_zero, status, stream);
    return quant_channel_pair(x_a, C_a, q_a, sf_a, x_b, C_b, q_b, sf_b, K_cap, psum, 1, G, sf_zero, status, stream);
}

namespace dg {
int debug_word_quant(uint32_t* out, bool clear) { return debug_word_local(out, clear); }
}  // namespace dg
