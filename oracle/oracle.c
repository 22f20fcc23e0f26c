/*
 * oracle.c - plain, slow CPU reference for blockwise-scaled FP8 (e4m3) grouped GEMM.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link or call this
 * file. It shares no code, header, table or constant generator with the CUDA kernels;
 * the only thing both sides share is the seeded input generator, which holds none of the
 * arithmetic below.
 *
 * What it computes, and where the source pages fix it (page titles are those of the
 * DeepGEMM issue/PR pages this project is built from):
 *
 *  - "Non-deterministic numerical problem of k_grouped_fp8_gemm_nt_contiguous" (#365),
 *    repro listing `_per_channel_cast_to_fp8`: per-channel scale = amax over 128 tokens / 448
 *    in fp32; a zero scale is replaced by `sf_val`; the scale is clamped below at 1e-30;
 *    codes = e4m3(x * (1/sf)), i.e. an fp32 reciprocal, an fp32 multiply, then rounding to
 *    e4m3.  `_pack_kmajor`: expert e's codes are written transposed, as a [C, K_e] row-major
 *    block at element offset prefix_e * C.  The k-grouped GEMM computes
 *    D_e = C_e + A_e^T B_e over each expert's token span (the repro passes `out` as both c
 *    and d; the reference loop skips empty experts).
 *  - "Fix cross-expert output overwrites in SM90 masked GEMM" (#469), reproduction section:
 *    masked D[g, r, :] = A[g, r, :] B[g]^T only for r < masked_m[g]; references are fp64
 *    matmuls rounded to bf16, and FP8 references use the actual quantized inputs and scales.
 *  - "SM120 m_grouped_fp8 contiguous kernel: illegal memory access at CUDA graph replay"
 *    (#444), description: m-grouped contiguous rows routed by m_indices; UE8M0 power-of-two
 *    scale factors on both operands; the kernel's name, m_grouped_fp8_fp4_gemm_nt_contiguous,
 *    gives FP8 activations with FP4 weights as the second operand form.
 *
 * Readings where the pages leave a step open (each is listed in the design notes):
 *  - the 1x128 per-token and 128x128 per-block casts reuse the per-channel rules exactly,
 *    with the 128-element block taken along K, or over the 128x128 tile;
 *  - e4m3 conversion is round-to-nearest-even with saturation to +-448 (NaN -> 0x7F);
 *  - UE8M0 rounds the fp32 scale UP to the next power of two (the mantissa is dropped and
 *    the exponent bumped when any mantissa bit is set); the stored byte is the biased
 *    exponent, value 2^(byte-127);
 *  - rows with m_indices outside [0, G), masked rows r >= min(count, cap), and experts whose
 *    K_e is not a multiple of 128 or overflows K_cap are not computed (outputs untouched);
 *  - FP4 weights (named only): OCP e2m1 codes with the weight-scale rule of the FP8 path over
 *    128x128 blocks, the maximum 448 replaced by e2m1's 6 and the scale rounded up to a power of
 *    two (the page's "2^k" weight scales); e2m1 conversion is round-to-nearest-even with
 *    saturation to +-6 (NaN -> +6); two codes per byte along K, the even element in the low
 *    nibble.
 *
 * All dot products accumulate in fp64 over dequantized values decode(q) * sf, with no
 * blocking or reordering beyond the definition.  Compile with -ffp-contract=off.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ----------------------------------------------------------------------------------------
 * e4m3 (OCP FP8 E4M3FN): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no inf,
 * NaN = S.1111.111.  Normal: (1 + m/8) * 2^(e-7); subnormal (e = 0): m/8 * 2^-6.
 * --------------------------------------------------------------------------------------*/
double oracle_e4m3_decode(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);            /* m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);  /* (8+m)/8 * 2^(e-7) */
    return sign ? -v : v;
}

/* Values of the non-negative finite codes 0x00..0x7E, increasing with the code. */
static double g_pos[127];
static double g_dec[256];

__attribute__((constructor)) static void oracle_init(void) {
    for (int c = 0; c < 127; ++c) g_pos[c] = oracle_e4m3_decode((uint8_t)c);
    for (int c = 0; c < 256; ++c) g_dec[c] = oracle_e4m3_decode((uint8_t)c);
}

/* Nearest e4m3 value to y; on a tie the code with the even mantissa (even code) wins;
 * |y| >= 448 saturates to +-448; NaN -> 0x7F; the sign of zero is kept. */
uint8_t oracle_e4m3_encode(float y) {
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    for (int c = 0; c < 126; ++c) {
        double lo = g_pos[c], hi = g_pos[c + 1];
        if (a <= hi) {
            double dlo = a - lo, dhi = hi - a;
            int pick;
            if (dlo < dhi) pick = c;
            else if (dhi < dlo) pick = c + 1;
            else pick = (c % 2 == 0) ? c : c + 1;
            return (uint8_t)(sign | pick);
        }
    }
    return (uint8_t)(sign | 0x7E); /* not reached: a < 448 = g_pos[126] */
}

/* ----------------------------------------------------------------------------------------
 * e2m1 (OCP FP4 E2M1): 1 sign bit (bit 3), 2 exponent bits (bias 1), 1 mantissa bit, no inf or
 * NaN.  Normal (e > 0): (1 + m/2) * 2^(e-1); subnormal (e = 0): m/2.  Non-negative values, by
 * code 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 * --------------------------------------------------------------------------------------*/
double oracle_e2m1_decode(uint8_t code) {
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 0x3;
    int m = code & 0x1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

static double g_pos4[8];
static double g_dec4[16];

__attribute__((constructor)) static void oracle_init_fp4(void) {
    for (int c = 0; c < 8; ++c) g_pos4[c] = oracle_e2m1_decode((uint8_t)c);
    for (int c = 0; c < 16; ++c) g_dec4[c] = oracle_e2m1_decode((uint8_t)c);
}

/* Nearest e2m1 value to y; on a tie the code with the even mantissa (even code) wins;
 * |y| >= 6 saturates to +-6; NaN -> +6 (0x7); the sign of zero is kept. */
uint8_t oracle_e2m1_encode(float y) {
    if (isnan(y)) return 0x7;
    uint8_t sign = signbit(y) ? 0x8 : 0x0;
    double a = fabs((double)y);
    if (a >= 6.0) return (uint8_t)(sign | 0x7);
    for (int c = 0; c < 7; ++c) {
        double lo = g_pos4[c], hi = g_pos4[c + 1];
        if (a <= hi) {
            double dlo = a - lo, dhi = hi - a;
            int pick;
            if (dlo < dhi) pick = c;
            else if (dhi < dlo) pick = c + 1;
            else pick = (c % 2 == 0) ? c : c + 1;
            return (uint8_t)(sign | pick);
        }
    }
    return (uint8_t)(sign | 0x7); /* not reached: a < 6 = g_pos4[7] */
}

void oracle_e2m1_encode_array(const float* y, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_encode(y[i]);
}

void oracle_e2m1_decode_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_decode(c[i]);
}

/* bf16 bits -> fp32 (exact) */
static float bf16_to_float(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ----------------------------------------------------------------------------------------
 * Scale rule of the per-channel cast in the #365 repro, shared by the three casts:
 *   sf = amax / 448 (fp32); if sf == 0: sf = sf_zero; sf = max(sf, 1e-30)
 * then optionally rounded up to a power of two (UE8M0).  Returns the scale; *ue_byte gets
 * the UE8M0 byte (biased exponent) when ue8m0 != 0.
 * --------------------------------------------------------------------------------------*/
static float scale_rule_max(float amax, float qmax, float sf_zero, int ue8m0, uint8_t* ue_byte) {
    const float floor_sf = 1e-30f;
    float sf = amax / qmax;
    if (sf == 0.0f) sf = sf_zero;
    if (sf < floor_sf) sf = floor_sf;
    if (ue8m0) {
        uint32_t bits;
        memcpy(&bits, &sf, 4);
        int e = (int)((bits >> 23) & 0xFF);
        if ((bits & 0x7FFFFFu) != 0) e += 1;  /* round up to the next power of two */
        sf = ldexpf(1.0f, e - 127);
        if (ue_byte) *ue_byte = (uint8_t)e;
    }
    return sf;
}

static float scale_rule(float amax, float sf_zero, int ue8m0, uint8_t* ue_byte) {
    return scale_rule_max(amax, 448.0f, sf_zero, ue8m0, ue_byte);
}

/* q = e4m3(fl32(x * fl32(1/sf))) */
static uint8_t quantize_one(float x, float sf) {
    float r = 1.0f / sf;
    float p = x * r;
    return oracle_e4m3_encode(p);
}

void oracle_scale_from_amax(const float* amax, int64_t n, float sf_zero, int ue8m0,
                            float* sf, uint8_t* ue_bytes) {
    for (int64_t i = 0; i < n; ++i)
        sf[i] = scale_rule(amax[i], sf_zero, ue8m0, ue_bytes ? &ue_bytes[i] : NULL);
}

void oracle_e4m3_encode_array(const float* y, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(y[i]);
}

void oracle_e4m3_decode_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/* ----------------------------------------------------------------------------------------
 * 1x128 per-token cast.  x: bf16 [M, K] with row stride ldx (elements).  K % 128 == 0.
 * Outputs (natural layouts): q [M][K], sf [M][K/128] (fp32 value of the scale), and, when
 * ue8m0, ue [M][K/128] bytes.  If row_counts != NULL the M rows form G equal groups of
 * M/G rows and only rows r < clamp(row_counts[g], 0, M/G) of group g are cast; other rows
 * are left untouched.
 * --------------------------------------------------------------------------------------*/
void oracle_quant_per_token_1x128(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                                  const int32_t* row_counts, int G, float sf_zero, int ue8m0,
                                  uint8_t* q, float* sf, uint8_t* ue) {
    int64_t KB = K / 128;
    int64_t rpg = (row_counts && G > 0) ? M / G : M;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        if (row_counts) {
            int64_t g = m / rpg, r = m % rpg;
            int64_t lim = row_counts[g];
            if (lim < 0) lim = 0;
            if (lim > rpg) lim = rpg;
            if (r >= lim) continue;
        }
        for (int64_t kb = 0; kb < KB; ++kb) {
            const uint16_t* xb = x + m * ldx + kb * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(bf16_to_float(xb[i]));
                if (v > amax) amax = v;
            }
            uint8_t byte = 0;
            float s = scale_rule(amax, sf_zero, ue8m0, &byte);
            sf[m * KB + kb] = s;
            if (ue8m0 && ue) ue[m * KB + kb] = byte;
            for (int i = 0; i < 128; ++i)
                q[m * K + kb * 128 + i] = quantize_one(bf16_to_float(xb[i]), s);
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * 128x128 per-block cast of weights w: bf16 [G][N][K], N % 128 == K % 128 == 0.
 * Outputs: q [G][N][K], sf [G][N/128][K/128], ue bytes likewise when ue8m0.
 * --------------------------------------------------------------------------------------*/
void oracle_quant_block_128x128(const uint16_t* w, int G, int64_t N, int64_t K, float sf_zero,
                                int ue8m0, uint8_t* q, float* sf, uint8_t* ue) {
    int64_t NB = N / 128, KB = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t nb = 0; nb < NB; ++nb) {
            for (int64_t kb = 0; kb < KB; ++kb) {
                const uint16_t* base = w + (g * N + nb * 128) * K + kb * 128;
                float amax = 0.0f;
                for (int r = 0; r < 128; ++r)
                    for (int c = 0; c < 128; ++c) {
                        float v = fabsf(bf16_to_float(base[r * K + c]));
                        if (v > amax) amax = v;
                    }
                uint8_t byte = 0;
                float s = scale_rule(amax, sf_zero, ue8m0, &byte);
                int64_t si = (g * NB + nb) * KB + kb;
                sf[si] = s;
                if (ue8m0 && ue) ue[si] = byte;
                for (int r = 0; r < 128; ++r)
                    for (int c = 0; c < 128; ++c) {
                        int64_t off = (g * N + nb * 128 + r) * K + kb * 128 + c;
                        q[off] = quantize_one(bf16_to_float(w[off]), s);
                    }
            }
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * FP4 weight cast (the FP4 operand of m_grouped_fp8_fp4_gemm_nt_contiguous, #444): per 128x128
 * block of w [G][N][K], amax in fp32; sf = amax / 6, zero -> sf_zero, >= 1e-30, rounded up to a
 * power of two (UE8M0 byte = biased exponent); q = e2m1(fl32(x * fl32(1/sf))).
 * Outputs: q_packed [G][N][K/2] (element k of a row in byte k/2, the low nibble for even k),
 * ue [G][N/128][K/128].
 * --------------------------------------------------------------------------------------*/
void oracle_quant_block_128x128_fp4(const uint16_t* w, int G, int64_t N, int64_t K, float sf_zero,
                                    uint8_t* q_packed, uint8_t* ue) {
    int64_t NB = N / 128, KB = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t nb = 0; nb < NB; ++nb) {
            for (int64_t kb = 0; kb < KB; ++kb) {
                const uint16_t* base = w + (g * N + nb * 128) * K + kb * 128;
                float amax = 0.0f;
                for (int r = 0; r < 128; ++r)
                    for (int c = 0; c < 128; ++c) {
                        float v = fabsf(bf16_to_float(base[r * K + c]));
                        if (v > amax) amax = v;
                    }
                uint8_t byte = 0;
                float s = scale_rule_max(amax, 6.0f, sf_zero, 1, &byte);
                ue[(g * NB + nb) * KB + kb] = byte;
                float rcp = 1.0f / s;
                for (int r = 0; r < 128; ++r)
                    for (int c = 0; c < 128; c += 2) {
                        int64_t off = (g * N + nb * 128 + r) * K + kb * 128 + c;
                        uint8_t lo = oracle_e2m1_encode(bf16_to_float(w[off]) * rcp);
                        uint8_t hi = oracle_e2m1_encode(bf16_to_float(w[off + 1]) * rcp);
                        q_packed[off / 2] = (uint8_t)(lo | (hi << 4));
                    }
            }
        }
    }
}

/* Value of weight element (e, n, k) of packed FP4 codes [G][N][K/2]. */
static double fp4_at(const uint8_t* qb_packed, int64_t e, int64_t n, int64_t k, int64_t N, int64_t K) {
    uint8_t byte = qb_packed[(e * N + n) * (K / 2) + k / 2];
    return g_dec4[(k & 1) ? (byte >> 4) : (byte & 0xF)];
}

/* ----------------------------------------------------------------------------------------
 * Per-channel cast over 128-token blocks (#365 repro, `_per_channel_cast_to_fp8`).
 * x: bf16 [T][C] token-major, T % 128 == 0.  Outputs q [T][C] and sf [T/128][C].
 * --------------------------------------------------------------------------------------*/
void oracle_quant_per_channel_128(const uint16_t* x, int64_t T, int64_t C, float sf_zero,
                                  uint8_t* q, float* sf) {
    int64_t TB = T / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t tb = 0; tb < TB; ++tb) {
        for (int64_t c = 0; c < C; ++c) {
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(bf16_to_float(x[(tb * 128 + i) * C + c]));
                if (v > amax) amax = v;
            }
            float s = scale_rule(amax, sf_zero, 0, NULL);
            sf[tb * C + c] = s;
            for (int i = 0; i < 128; ++i) {
                int64_t off = (tb * 128 + i) * C + c;
                q[off] = quantize_one(bf16_to_float(x[off]), s);
            }
        }
    }
}

/* Per-expert K-major pack (#365 repro, `_pack_kmajor`): expert e, with token span
 * [o_e, o_e + ks[e]), gets its codes transposed into a [C][ks[e]] row-major block at
 * element offset o_e * C.  q: [T][C] token-major. */
void oracle_pack_kmajor(const uint8_t* q, const int32_t* ks, int G, int64_t C, uint8_t* packed) {
    int64_t o = 0;
    for (int e = 0; e < G; ++e) {
        int64_t k = ks[e];
        for (int64_t c = 0; c < C; ++c)
            for (int64_t t = 0; t < k; ++t)
                packed[o * C + c * k + t] = q[(o + t) * C + c];
        o += k;
    }
}

/* ----------------------------------------------------------------------------------------
 * m-grouped contiguous GEMM (#444 description): for each row m with e = m_indices[m] in
 * [0, G):  D[m][n] = sum_k decode(qa[m][k]) sfa[m][k/128] * decode(qb[e][n][k]) sfb[e][n/128][k/128]
 * in fp64.  Other rows of d are not written.  sfa: [M][K/128], sfb: [G][N/128][K/128].
 * --------------------------------------------------------------------------------------*/
void oracle_gemm_contiguous(const uint8_t* qa, const float* sfa, const uint8_t* qb,
                            const float* sfb, const int32_t* m_indices, int64_t M, int G,
                            int64_t N, int64_t K, double* d) {
    int64_t KB = K / 128, NB = N / 128;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        int64_t e = m_indices[m];
        if (e < 0 || e >= G) continue;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double xa = g_dec[qa[m * K + k]] * (double)sfa[m * KB + k / 128];
                double xb = g_dec[qb[(e * N + n) * K + k]] *
                            (double)sfb[(e * NB + n / 128) * KB + k / 128];
                acc += xa * xb;
            }
            d[m * N + n] = acc;
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * m-grouped masked GEMM (#469 reproduction): for r < min(max(counts[g], 0), cap):
 *   D[g][r][n] = sum_k decode(qa[g][r][k]) sfa[g][r][k/128] * decode(qb[g][n][k]) sfb[g][n/128][k/128]
 * qa [G][cap][K], sfa [G][cap][K/128], qb [G][N][K], sfb [G][N/128][K/128], d [G][cap][N].
 * Rows at or beyond the count are not written.
 * --------------------------------------------------------------------------------------*/
void oracle_gemm_masked(const uint8_t* qa, const float* sfa, const uint8_t* qb, const float* sfb,
                        const int32_t* counts, int G, int64_t cap, int64_t N, int64_t K,
                        double* d) {
    int64_t KB = K / 128, NB = N / 128;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t r = 0; r < cap; ++r) {
            int64_t v = counts[g];
            if (v < 0) v = 0;
            if (v > cap) v = cap;
            if (r >= v) continue;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double xa = g_dec[qa[(g * cap + r) * K + k]] *
                                (double)sfa[(g * cap + r) * KB + k / 128];
                    double xb = g_dec[qb[(g * N + n) * K + k]] *
                                (double)sfb[(g * NB + n / 128) * KB + k / 128];
                    acc += xa * xb;
                }
                d[(g * cap + r) * N + n] = acc;
            }
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * The contiguous and masked GEMMs above with FP4 weights (#444: FP8 activations, FP4 weights):
 * the same sums with decode(qb) the e2m1 value of the packed code.  qb_packed [G][N][K/2].
 * --------------------------------------------------------------------------------------*/
void oracle_gemm_contiguous_fp4(const uint8_t* qa, const float* sfa, const uint8_t* qb_packed,
                                const float* sfb, const int32_t* m_indices, int64_t M, int G,
                                int64_t N, int64_t K, double* d) {
    int64_t KB = K / 128, NB = N / 128;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        int64_t e = m_indices[m];
        if (e < 0 || e >= G) continue;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double xa = g_dec[qa[m * K + k]] * (double)sfa[m * KB + k / 128];
                double xb = fp4_at(qb_packed, e, n, k, N, K) * (double)sfb[(e * NB + n / 128) * KB + k / 128];
                acc += xa * xb;
            }
            d[m * N + n] = acc;
        }
    }
}

void oracle_gemm_masked_fp4(const uint8_t* qa, const float* sfa, const uint8_t* qb_packed,
                            const float* sfb, const int32_t* counts, int G, int64_t cap, int64_t N,
                            int64_t K, double* d) {
    int64_t KB = K / 128, NB = N / 128;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t r = 0; r < cap; ++r) {
            int64_t v = counts[g];
            if (v < 0) v = 0;
            if (v > cap) v = cap;
            if (r >= v) continue;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double xa = g_dec[qa[(g * cap + r) * K + k]] * (double)sfa[(g * cap + r) * KB + k / 128];
                    double xb = fp4_at(qb_packed, g, n, k, N, K) * (double)sfb[(g * NB + n / 128) * KB + k / 128];
                    acc += xa * xb;
                }
                d[(g * cap + r) * N + n] = acc;
            }
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * Plain and batched FP8 GEMM with accumulation (#469 validation: the adjacent-path checks of
 * ordinary GEMM layouts, output dtypes and accumulation, and batched GEMM): for every batch
 * entry b < B, row m < M and column n < N,
 *   D[b][m][n] = C[b][m][n] + sum_k decode(qa[b][m][k]) sfa[b][m][k/128]
 *                                  * decode(qb[b][n][k]) sfb[b][n/128][k/128]
 * with C taken as 0 when c is NULL.  A plain GEMM is B = 1.
 * qa [B][M][K], sfa [B][M][K/128], qb [B][N][K], sfb [B][N/128][K/128], c and d [B][M][N].
 * --------------------------------------------------------------------------------------*/
void oracle_gemm_batched(const uint8_t* qa, const float* sfa, const uint8_t* qb, const float* sfb,
                         const double* c, int64_t B, int64_t M, int64_t N, int64_t K, double* d) {
    int64_t KB = K / 128, NB = N / 128;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b) {
        for (int64_t m = 0; m < M; ++m) {
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double xa = g_dec[qa[(b * M + m) * K + k]] * (double)sfa[(b * M + m) * KB + k / 128];
                    double xb = g_dec[qb[(b * N + n) * K + k]] *
                                (double)sfb[(b * NB + n / 128) * KB + k / 128];
                    acc += xa * xb;
                }
                d[(b * M + m) * N + n] = (c != NULL ? c[(b * M + m) * N + n] : 0.0) + acc;
            }
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * k-grouped wgrad GEMM (#365 repro): for each expert e with span [o_e, o_e + K_e) along K,
 *   D_e[n][h] = C_e[n][h] + sum_{t < K_e} decode(a_e[n][t]) sfa[(o_e+t)/128][n]
 *                                      * decode(b_e[h][t]) sfb[(o_e+t)/128][h]
 * where a_e / b_e are the K-major packed blocks of `oracle_pack_kmajor` (a: [C=N], b: [C=H]).
 * c may be NULL (zero).  K_e = 0 gives D_e = C_e.  An expert with K_e % 128 != 0, K_e < 0,
 * or a span past K_cap is skipped (d_e untouched), as is every later expert.  d is fp64;
 * the GPU output is fp32.
 * --------------------------------------------------------------------------------------*/
void oracle_gemm_kgrouped(const uint8_t* a_packed, const float* sfa, const uint8_t* b_packed,
                          const float* sfb, const float* c, const int32_t* ks, int G,
                          int64_t K_cap, int64_t N, int64_t H, double* d) {
    int64_t o = 0;
    for (int e = 0; e < G; ++e) {
        int64_t k = ks[e];
        if (k < 0 || k % 128 != 0 || o + k > K_cap) break;
        const uint8_t* ae = a_packed + o * N;
        const uint8_t* be = b_packed + o * H;
#pragma omp parallel for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            for (int64_t h = 0; h < H; ++h) {
                double acc = 0.0;
                for (int64_t t = 0; t < k; ++t) {
                    int64_t kb = (o + t) / 128;
                    double xa = g_dec[ae[n * k + t]] * (double)sfa[kb * N + n];
                    double xb = g_dec[be[h * k + t]] * (double)sfb[kb * H + h];
                    acc += xa * xb;
                }
                int64_t off = ((int64_t)e * N + n) * H + h;
                d[off] = (c ? (double)c[off] : 0.0) + acc;
            }
        }
        o += k;
    }
}

/* ----------------------------------------------------------------------------------------
 * Output rounding and comparison.
 * --------------------------------------------------------------------------------------*/

/* ----------------------------------------------------------------------------------------
 * BF16 m-grouped GEMMs (#469 reproduction: `m_grouped_bf16_gemm_nt_masked`, checked against
 * torch.bmm(a.double(), b.double().mT) rounded to bf16).  No scales: the bf16 inputs are
 * exact in fp64 and the products accumulate in fp64.
 *   masked:     D[g][r][n] = sum_k a[g][r][k] b[g][n][k] for r < min(max(counts[g], 0), cap)
 *   contiguous: D[m][n]    = sum_k a[m][k] b[e][n][k]    for e = m_indices[m] in [0, G)
 * Rows that are not valid are not written.
 * --------------------------------------------------------------------------------------*/
void oracle_gemm_masked_bf16(const uint16_t* a, const uint16_t* b, const int32_t* counts, int G,
                             int64_t cap, int64_t N, int64_t K, double* d) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t r = 0; r < cap; ++r) {
            int64_t v = counts[g];
            if (v < 0) v = 0;
            if (v > cap) v = cap;
            if (r >= v) continue;
            for (int64_t n = 0; n < N; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (double)bf16_to_float(a[(g * cap + r) * K + k]) *
                           (double)bf16_to_float(b[(g * N + n) * K + k]);
                d[(g * cap + r) * N + n] = acc;
            }
        }
    }
}

void oracle_gemm_contiguous_bf16(const uint16_t* a, const uint16_t* b, const int32_t* m_indices,
                                 int64_t M, int G, int64_t N, int64_t K, double* d) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t m = 0; m < M; ++m) {
        int64_t e = m_indices[m];
        if (e < 0 || e >= G) continue;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += (double)bf16_to_float(a[m * K + k]) * (double)bf16_to_float(b[(e * N + n) * K + k]);
            d[m * N + n] = acc;
        }
    }
}

/* ----------------------------------------------------------------------------------------
 * Prefix-sum ("psum") grouped layouts: `use_psum_layout` of the k-grouped call in #365's
 * repro listing, and the m_indices / psum / masked modes of #444's graph-mutation test.
 * Readings (the pages name the option but not its encoding):
 *  - k-grouped: psum[e] = K_0 + ... + K_e, so K_e = psum[e] - psum[e-1] (psum[-1] = 0); a
 *    decreasing entry gives a negative K_e, which stops the walk of oracle_gemm_kgrouped;
 *  - m-grouped contiguous: psum[e] is the exclusive end row of expert e, whose rows start at
 *    the previous end rounded up to 128 (the 128-aligned segments of the m_indices layout).
 *    An entry below its predecessor, past M, or ending inside the rounding gap stops the walk:
 *    that expert and every later one stay unrouted (-1).
 * --------------------------------------------------------------------------------------*/
void oracle_sizes_from_psum(const int32_t* psum, int G, int32_t* ks) {
    for (int e = 0; e < G; ++e) ks[e] = psum[e] - (e > 0 ? psum[e - 1] : 0);
}

void oracle_m_indices_from_psum(const int32_t* psum, int G, int64_t M, int32_t* m_indices) {
    for (int64_t m = 0; m < M; ++m) m_indices[m] = -1;
    for (int e = 0; e < G; ++e) {
        int64_t prev = e > 0 ? psum[e - 1] : 0, end = psum[e];
        int64_t start = (prev + 127) / 128 * 128;
        if (prev < 0 || end < prev || end > M || (end > prev && end < start)) break;
        for (int64_t m = start; m < end; ++m) m_indices[m] = e;
    }
}

/* fp64 -> bf16 bits, a single round-to-nearest-even (no intermediate fp32 rounding).
 * bf16: 8 exponent bits (bias 127), 7 mantissa bits; min normal 2^-126, subnormal step
 * 2^-133; overflow past the largest finite value plus half an ulp gives inf. */
uint16_t oracle_round_bf16(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
    int ulp_exp = (e - 1) - 7;    /* 8 significant bits for normals */
    if (ulp_exp < -133) ulp_exp = -133; /* subnormal range: fixed step 2^-133 */
    double steps = ldexp(a, -ulp_exp);  /* exact */
    double r = nearbyint(steps);        /* default rounding mode: nearest, ties to even */
    double rv = ldexp(r, ulp_exp);
    const double maxbf = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
    if (rv > maxbf) return (uint16_t)(sign | 0x7F80);
    float f = (float)rv;                    /* exact: rv is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

void oracle_round_bf16_array(const double* v, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(v[i]);
}

/* Similarity difference of two vectors: 1 - 2 sum(x y) / sum(x^2 + y^2), in fp64. */
double oracle_calc_diff(const double* x, const double* y, int64_t n) {
    double sxy = 0.0, sxx = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        sxy += x[i] * y[i];
        sxx += x[i] * x[i] + y[i] * y[i];
    }
    if (sxx == 0.0) return 0.0;
    return 1.0 - 2.0 * sxy / sxx;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
