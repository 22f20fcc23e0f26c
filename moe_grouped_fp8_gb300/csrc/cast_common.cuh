// cast_common.cuh - device code shared by the FP8 casts (quant.cu) and the fused cast +
// descriptor launch of the k-grouped call (kgrouped.cu): the scale rule and its fast exact
// form, the e4m3 packing, the expert lookup over ks, and one CTA of the per-channel cast.
//
// Scale rule (per-channel cast listing of "Non-deterministic numerical problem of
// k_grouped_fp8_gemm_nt_contiguous", applied along K or over a 128x128 tile for the other two
// casts): sf = amax / 448 in fp32; sf == 0 -> sf_zero; sf = max(sf, 1e-30); UE8M0 rounds sf up
// to a power of two.  Codes: e4m3(x * (1/sf)), an IEEE fp32 reciprocal and product, then
// round-to-nearest-even with saturation to +-448.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kernel_common.cuh"
#include "ptx.cuh"

namespace dg {
namespace {

__device__ __forceinline__ float scale_rule(float amax, float sf_zero) {
    float sf = __fdiv_rn(amax, 448.0f);
    if (sf == 0.0f) sf = sf_zero;
    return fmaxf(sf, 1e-30f);
}

// Round a positive normal fp32 scale up to a power of two; *byte = its biased exponent.
__device__ __forceinline__ float ue8m0_round_up(float sf, uint8_t* byte) {
    uint32_t b = __float_as_uint(sf);
    uint32_t e = (b >> 23) & 0xFFu;
    if (b & 0x7FFFFFu) e += 1;
    *byte = static_cast<uint8_t>(e);
    return __uint_as_float(e << 23);
}

// The scale of a block and its reciprocal: bit-identical to scale_rule, ue8m0_round_up and
// __frcp_rn, with fewer instructions on the common path.  When amax lies in [1e-27, FLT_MAX] the
// clamps of scale_rule are inactive and the quotient is normal, so amax / 448 is formed by
// Markstein's FMA-corrected division (the product with the rounded reciprocal of 448, its exact
// residual, one corrective FMA), and 1/sf is exact from the exponent for UE8M0 scales (a power of
// two) or one Newton-Raphson step from the hardware approximation for fp32 scales.  Both shortcuts
// were checked in exact rational arithmetic for every finite bf16 amax on that path (the cast's
// amax is a bf16 value), the reciprocal for every start within 1 ulp of 1/sf.  Every other amax
// (zero, tiny, inf, NaN) takes the IEEE operations.
template <bool UE8M0>
__device__ __forceinline__ void block_scale(float amax, float sf_zero, float& sf, float& r, uint8_t& byte) {
    constexpr float kInv448 = 1.0f / 448.0f;
    if (amax >= 1e-27f && amax <= 3.40282347e38f) {
        const float q0 = __fmul_rn(amax, kInv448);
        sf = __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), kInv448, q0);
        if constexpr (UE8M0) {
            const uint32_t b = __float_as_uint(sf);
            const uint32_t e = (b >> 23) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
            byte = static_cast<uint8_t>(e);
            sf = __uint_as_float(e << 23);
            r = __uint_as_float((254u - e) << 23);
        } else {
            const float y = rcp_approx(sf);
            r = __fmaf_rn(__fmaf_rn(-sf, y, 1.0f), y, y);
        }
    } else {
        sf = scale_rule(amax, sf_zero);
        if constexpr (UE8M0) sf = ue8m0_round_up(sf, &byte);
        r = __frcp_rn(sf);
    }
}

// Codes of 8 values scaled by r, as two little-endian words (value i in byte i).
__device__ __forceinline__ uint2 e4m3x8(const float (&f)[8], float r) {
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        float p[4];
        fmul2(p[0], p[1], f[4 * h], f[4 * h + 1], r);
        fmul2(p[2], p[3], f[4 * h + 2], f[4 * h + 3], r);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(p[0], p[1]), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(p[2], p[3]), __NV_SATFINITE, __NV_E4M3);
        w[h] = lo | (hi << 16);
    }
    return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// ---------------------------------------------------------------------------------------
// Per-channel cast over 128-token blocks + per-expert K-major pack.  CTA = (64-column block,
// 128-token block).  Thread t holds columns 8 (t % 8) .. +8 of the four consecutive tokens
// 4 (t / 8) .. +4; codes are transposed through shared memory (4 tokens packed per 32-bit word)
// and written as 128-byte column runs of the expert's [C, K_e] block.
// ---------------------------------------------------------------------------------------
constexpr int CH_COLS = 64;
constexpr int CH_PITCH = 132;  // bytes per transposed column row (128 tokens + 4 pad)

// Expert lookup for token `tok`: returns the expert index with its token offset and K_e, or
// -1 when the token lies past the last valid expert.  Warp 0 walks ks in chunks of blockDim.x
// experts (32 at a time, with warp shuffles only) and stops after the chunk that holds the token or
// the first bad expert (K_e < 0, K_e % 128 != 0, or a span past K_cap); *bad_bits gets the
// DG_STATUS_* bits of every bad expert in the chunks it walked.  One CTA barrier publishes the
// answer.
__device__ int find_expert(const int32_t* __restrict__ ks, int psum, int G, int64_t K_cap, int64_t tok,
                           int64_t* o_out, int64_t* k_out, int* bad_bits) {
    __shared__ long long s_o, s_k;
    __shared__ int s_found, s_bad;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int chunk = static_cast<int>(blockDim.x);
        long long carry = 0, o_f = 0, k_f = 0;
        int found = -1, first_bad = 0x7fffffff, bits = 0;
        for (int c0 = 0; c0 < G; c0 += chunk) {
            for (int base = c0; base < G && base < c0 + chunk; base += 32) {
                const int e = base + lane;
                const long long k = e < G ? expert_k(ks, e, psum) : 0;
                int bad = (e < G && (k < 0 || (k % 128) != 0)) ? DG_STATUS_K_NOT_ALIGNED : 0;
                const long long kk = bad ? 0 : k;
                long long incl = kk;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                const long long o_e = carry + incl - kk;  // exclusive prefix of valid K_e
                if (e < G && !bad && o_e + kk > K_cap) bad = DG_STATUS_K_OVERFLOW;
                bits |= __reduce_or_sync(0xffffffffu, static_cast<unsigned>(bad));
                const unsigned bad_lanes = __ballot_sync(0xffffffffu, bad != 0);
                if (bad_lanes != 0 && first_bad == 0x7fffffff) first_bad = base + __ffs(bad_lanes) - 1;
                const unsigned hit = __ballot_sync(
                    0xffffffffu, e < G && e < first_bad && kk > 0 && tok >= o_e && tok < o_e + kk);
                if (hit != 0) {
                    const int src = __ffs(hit) - 1;
                    found = base + src;
                    o_f = __shfl_sync(0xffffffffu, o_e, src);
                    k_f = __shfl_sync(0xffffffffu, kk, src);
                }
                carry += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (found >= 0 || first_bad != 0x7fffffff) break;
        }
        if (lane == 0) {
            s_found = found;
            s_o = o_f;
            s_k = k_f;
            s_bad = bits;
        }
    }
    __syncthreads();
    *bad_bits = s_bad;
    const int f = s_found;
    if (f >= 0) {
        *o_out = s_o;
        *k_out = s_k;
    }
    return f;
}

// One or two operands cast in the same launch (the two operands of a k-grouped wgrad share ks):
// column blocks [0, nblk0) belong to op0, the rest to op1.
struct ChannelOperand {
    const uint16_t* x;  // bf16 [K_cap, C]
    int64_t C;
    uint8_t* q;         // packed codes
    float* sf;          // [K_cap/128][C]
};

// The work of one CTA (256 threads) of the per-channel cast: column block bx, 128-token block by.
__device__ __forceinline__ void channel_cast_cta(const ChannelOperand& op0, const ChannelOperand& op1, int nblk0,
                                                 int64_t K_cap, const int32_t* __restrict__ ks, int psum, int G,
                                                 float sf_zero, int32_t* status, int bx, int by) {
    __shared__ float s_part[8][CH_COLS];
    __shared__ float s_r[CH_COLS];
    __shared__ __align__(16) uint8_t s_t[CH_COLS * CH_PITCH];

    const bool second = static_cast<int>(bx) >= nblk0;
    const ChannelOperand& op = second ? op1 : op0;
    const uint16_t* __restrict__ x = op.x;
    const int64_t C = op.C;
    const int64_t tb = by;
    const int64_t c0 = static_cast<int64_t>(second ? bx - nblk0 : bx) * CH_COLS;
    const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
    const int c = t & 7;          // 8-column chunk
    const int rb = (t >> 3) * 4;  // first of 4 consecutive tokens

    pdl_trigger();
    // Before waiting on the previous kernel of the stream: this CTA's bf16 rows (one 128-byte line
    // each) into L2, so that the loads after the wait hit L2 (the wgrad step 32.2 -> 31.3 us, its
    // casts following the previous step's GEMM).  A hint only; L2 is the coherence point, so a line
    // the previous kernel writes afterwards is never served stale.
    if (c == 0) {
#pragma unroll
        for (int j = 0; j < 4; ++j) prefetch_l2(x + (tb * 128 + rb + j) * C + c0);
    }
    pdl_wait();
    // the bf16 loads do not depend on the expert lookup: issue them first (rows < K_cap exist)
    uint4 raw[4];
    const bool in_ok = DG_CHECKED(tb * 128 + 128 <= K_cap && c0 + CH_COLS <= C, DG_DEBUG_CAST_IN);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        raw[j] = in_ok ? __ldg(reinterpret_cast<const uint4*>(x + (tb * 128 + rb + j) * C + c0) + c)
                       : make_uint4(0, 0, 0, 0);
    int64_t o_e = 0, k_e = 0;
    int bad = 0;
    const int e = find_expert(ks, psum, G, K_cap, tb * 128, &o_e, &k_e, &bad);
    if (bx == 0 && by == 0 && threadIdx.x == 0) status_or(status, bad);
    if (e < 0) return;
    uint8_t* __restrict__ qp = op.q;
    float* __restrict__ sf_out = op.sf;
    float f[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) bf16x8_to_float(raw[j], f[j]);
    float cm[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        cm[i] = fmaxf(fmaxf(fabsf(f[0][i]), fabsf(f[1][i])), fmaxf(fabsf(f[2][i]), fabsf(f[3][i])));
        cm[i] = fmaxf(cm[i], __shfl_xor_sync(0xffffffffu, cm[i], 8));
        cm[i] = fmaxf(cm[i], __shfl_xor_sync(0xffffffffu, cm[i], 16));
    }
    if (lane < 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) s_part[wid][c * 8 + i] = cm[i];
    }
    __syncthreads();
    if (t < CH_COLS) {
        float amax = s_part[0][t];
#pragma unroll
        for (int w = 1; w < 8; ++w) amax = fmaxf(amax, s_part[w][t]);
        float sf, r;
        uint8_t unused;
        block_scale<false>(amax, sf_zero, sf, r, unused);
        if (DG_CHECKED(in_ok, DG_DEBUG_CAST_OUT)) sf_out[tb * C + c0 + t] = sf;
        s_r[t] = r;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float r = s_r[c * 8 + i];
        float p[4];
        fmul2(p[0], p[1], f[0][i], f[1][i], r);
        fmul2(p[2], p[3], f[2][i], f[3][i], r);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(p[0], p[1]), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(p[2], p[3]), __NV_SATFINITE, __NV_E4M3);
        *reinterpret_cast<uint32_t*>(&s_t[(c * 8 + i) * CH_PITCH + rb]) = lo | (hi << 16);
    }
    __syncthreads();
    // column `col` of this CTA -> 128 consecutive bytes of row (c0 + col) of expert e's block
    uint8_t* dst_base = qp + o_e * C + (tb * 128 - o_e);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int s = t + 256 * u;
        const int col = s >> 3, piece = s & 7;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(&s_t[col * CH_PITCH + piece * 16]);
        uint4 v = make_uint4(src[0], src[1], src[2], src[3]);
        // the expert's [C, K_e] block lies inside the K_cap x C packed buffer
        if (DG_CHECKED(in_ok && o_e + k_e <= K_cap && tb * 128 + 128 <= o_e + k_e, DG_DEBUG_CAST_OUT))
            *reinterpret_cast<uint4*>(dst_base + (c0 + col) * k_e + piece * 16) = v;
    }
}

}  // namespace
}  // namespace dg
