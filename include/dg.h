/*
 * dg.h - C ABI of the GB300 (sm_103a) blockwise-scaled FP8 grouped-GEMM library (libdg.so).
 *
 * The library computes the data-parallel hot path of FP8 Mixture-of-Experts layers as they
 * are described on three DeepGEMM issue/PR pages:
 *   [P1] "Non-deterministic numerical problem of k_grouped_fp8_gemm_nt_contiguous" (#365):
 *        the per-channel cast listing, the K-major per-expert pack, the k-grouped wgrad call
 *        k_grouped_fp8_gemm_nt_contiguous(a, b, d, ks, ks_tensor, c, recipe=(1,1,128)).
 *   [P2] "Fix cross-expert output overwrites in SM90 masked GEMM" (#469): the masked call
 *        m_grouped_*_gemm_nt_masked(a, b, d, masked_m, expected_m) and its output boundary.
 *   [P3] "SM120 m_grouped_fp8 contiguous kernel: illegal memory access at CUDA graph replay"
 *        (#444): the m-grouped contiguous call routed by m_indices, UE8M0 scale factors, and
 *        graph replay with a changed expert distribution.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless stated.  The
 *     library allocates nothing, never copies device data to the host and never
 *     synchronises: each call only enqueues kernels on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  The one exception is the debug aid dg_debug_word (end of file).  Calls are therefore capturable into CUDA graphs, and a
 *     captured call re-reads m_indices / counts / ks from device memory on every replay.
 *   - Return value: DG_OK, or an error code with nothing enqueued.  dg_last_error() gives a
 *     message for the calling thread's most recent failure.
 *   - `status` (optional, may be NULL): a caller-owned device int32.  Kernels OR DG_STATUS_*
 *     bits into it when they meet bad device-side data (an m_indices value outside [-1, G),
 *     count > cap, K_e not a multiple of 128, ks overflowing K_cap, a wait that timed out);
 *     the offending work is skipped.  Kernels never trap.  The caller clears it.
 *   - Every wait inside a kernel is bounded: after DG_WAIT_LIMIT_MS milliseconds (environment,
 *     read once per process; default 2000) the kernel sets DG_STATUS_TIMEOUT, drains the copies
 *     and MMAs it issued, frees its tensor memory and returns.
 *   - Alignment: buffers read or written by TMA (fp8 operands, outputs, C) must be 16-byte
 *     aligned; N, K (and H) must be multiples of 128.
 *   - e4m3 = OCP FP8 E4M3FN (max 448).  bf16 buffers are passed as `const void*`.
 *   - Scale factors: DG_SF_FP32 = fp32 values; DG_SF_UE8M0 = one byte per scale, value
 *     2^(byte-127).
 *
 * Scale-factor layouts (all row-major in the order written)
 *   sfa, per-token 1x128 (MN-major, "column-major TMA-aligned"): [K/128][Mp] where
 *        Mp = round_up(M, 4) for fp32, round_up(M, 16) for UE8M0 bytes; element (kb, m).
 *   sfb, per-128x128 block: [G][N/128][K/128].
 *   sf, per-channel over 128 tokens ([P1] `sf.T` is a view of this): [K_cap/128][C].
 */
#ifndef DG_H
#define DG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum dg_result { DG_OK = 0, DG_ERR_INVALID_ARG = 1, DG_ERR_UNSUPPORTED = 2, DG_ERR_CUDA = 3 };
enum dg_sf_format { DG_SF_FP32 = 0, DG_SF_UE8M0 = 1 };
enum dg_out_dtype { DG_OUT_BF16 = 0, DG_OUT_FP32 = 1 };
enum dg_status_bits {
    DG_STATUS_BAD_INDEX = 1,     /* m_indices outside [-1, G), or a row of another expert in a block */
    DG_STATUS_COUNT_GT_CAP = 2,  /* masked count > cap (clamped to cap) or < 0 (taken as 0) */
    DG_STATUS_K_NOT_ALIGNED = 4, /* some K_e < 0 or not a multiple of 128 */
    DG_STATUS_K_OVERFLOW = 8,    /* prefix of ks runs past K_cap */
    DG_STATUS_TIMEOUT = 16,      /* a bounded wait inside a kernel gave up */
    DG_STATUS_TOO_MANY_RUNS = 32 /* contiguous layout has more expert segments than supported */
};
enum dg_op { DG_OP_M_GROUPED_CONTIGUOUS = 0, DG_OP_M_GROUPED_MASKED = 1, DG_OP_K_GROUPED_WGRAD = 2 };

/* Largest supported values (DG_ERR_UNSUPPORTED beyond them). */
#define DG_MAX_GROUPS 1024          /* G for every grouped call */
#define DG_MAX_M_BLOCKS 4096        /* ceil(M/128) for the contiguous call: M <= 524288 */

/* Message describing the calling thread's most recent error ("" if none). */
const char* dg_last_error(void);

/* Bytes of device workspace `op` needs (0 if none).  The workspace must be 128-byte aligned
 * and must not be used by two calls that may run at the same time. */
size_t dg_workspace_size(int op, int G, int64_t M, int64_t N, int64_t K);

/*
 * 1x128 per-token cast ([P2] "1d" activation scales of sm90_fp8_gemm_1d2d; [P3] "activations
 * quantized with column-major TMA-aligned packed scales").  For every row m < M and K block
 * kb: amax = max |x[m, kb*128 : kb*128+128]| (fp32), sf = amax / 448, sf == 0 -> sf_zero,
 * sf = max(sf, 1e-30) ([P1] per-channel listing, same rules taken along K); for UE8M0 sf is
 * rounded up to a power of two.  q = e4m3_rne_satfinite(x * (1/sf)) with an fp32 reciprocal
 * and an fp32 product.
 *   x:  bf16 [M, K], row stride ldx elements (ldx >= K, ldx*2 a multiple of 16).
 *   q:  e4m3 [M, K], row stride K.   sfa: see "Scale-factor layouts" (per sf_format).
 *   row_counts: optional int32 [G]; when given, the M rows form G groups of M/G rows (the
 *     masked [G, cap, K] activation) and only rows r < clamp(row_counts[g], 0, M/G) are read
 *     and written, so padding rows cost no traffic.  G is ignored when row_counts is NULL.
 */
int dg_quant_per_token_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                             void* sfa, int sf_format, float sf_zero, const int32_t* row_counts,
                             int G, void* stream);

/*
 * The same 1x128 per-token cast over the rows of a contiguous m-grouped activation that are
 * routed to an expert ([P3] m_grouped_fp8_fp4_gemm_nt_contiguous: rows whose m_indices entry is
 * -1 are padding that the GEMM never writes).  Rows m < M with m_indices[m] >= 0 are cast
 * exactly as by dg_quant_per_token_1x128; rows with m_indices[m] < 0 are neither read nor
 * written (their codes and scales keep whatever the buffers held).
 *   x, ldx, q, sfa, sf_format, sf_zero: as for dg_quant_per_token_1x128.
 *   m_indices: int32 [M] device array, the contiguous GEMM's routing (only its sign is used).
 */
int dg_quant_per_token_1x128_routed(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                                    void* sfa, int sf_format, float sf_zero,
                                    const int32_t* m_indices, void* stream);

/*
 * The masked per-token cast reading its rows packed: the tokens routed to each expert arrive
 * one expert after another ([P2] masked call: group g holds masked_m[g] valid rows of its
 * [cap, K] slice), and are cast straight into the masked [G, cap, K] layout the masked GEMM
 * reads, with no scatter in between.  Group g's valid rows r < v_g = clamp(row_counts[g], 0, cap)
 * are rows P_g + r of x, P_g = v_0 + ... + v_(g-1); each is cast exactly as by
 * dg_quant_per_token_1x128 into row g*cap + r of q and sfa.  Rows of q and sfa at or past a
 * group's count are not written.
 *   x:  bf16, the packed rows at its front; its capacity is G*cap rows (row stride ldx).
 *   q, sfa: as for dg_quant_per_token_1x128 with M = G*cap.   row_counts: int32 [G].
 *   1 <= G <= DG_MAX_GROUPS.
 */
int dg_quant_per_token_1x128_packed(const void* x, int64_t K, int64_t ldx, uint8_t* q, void* sfa,
                                    int sf_format, float sf_zero, const int32_t* row_counts, int G,
                                    int64_t cap, void* stream);

/*
 * The inverse movement for an output: the valid rows of a masked [G, cap] array of rows (the
 * masked GEMM's [G, cap, N] output, [P2] 3-D store) packed one group after another, so that
 * they leave the device in one copy.  Row r < v_g of group g (v_g as above) is copied byte for
 * byte to row P_g + r of dst.
 *   src: [G, cap] rows of row_bytes bytes (a multiple of 16); dst: capacity G*cap rows of
 *   row_bytes; both 16-byte aligned.   counts: int32 [G].   1 <= G <= DG_MAX_GROUPS.
 */
int dg_pack_masked_rows(const void* src, int G, int64_t cap, int64_t row_bytes, const int32_t* counts,
                        void* dst, void* stream);

/*
 * Per-channel cast over 128-token blocks with the per-expert K-major pack ([P1] repro:
 * `_per_channel_cast_to_fp8(x, gran_k=128, sf_val)` then `_pack_kmajor`).  For every
 * 128-token block tb inside sum(ks) and every column c: amax over the 128 tokens, then the
 * scale and code rules of dg_quant_per_token_1x128 (fp32 scales only).
 *   x:  bf16 [K_cap, C] token-major (row stride C); rows at or past sum(ks) are not read.
 *   ks: int32 [G] device token counts per expert, each a multiple of 128, sum <= K_cap.
 *   q_packed: e4m3, expert e's codes transposed into a [C, K_e] row-major block at element
 *     offset prefix_e * C (prefix_e = ks[0] + ... + ks[e-1]).
 *   sf: fp32 [K_cap/128][C].
 * Bad ks set DG_STATUS_K_NOT_ALIGNED / DG_STATUS_K_OVERFLOW and stop the walk over experts at
 * the first bad one (later experts are not written).
 */
int dg_quant_per_channel_128(const void* x, int64_t K_cap, int64_t C, const int32_t* ks, int G,
                             uint8_t* q_packed, float* sf, float sf_zero, int32_t* status,
                             void* stream);

/*
 * Both operands of a k-grouped wgrad cast in one launch: the same results as
 * dg_quant_per_channel_128(x_a, K_cap, C_a, ks, ...) followed by
 * dg_quant_per_channel_128(x_b, K_cap, C_b, ks, ...) with the same ks, sf_zero and status
 * ([P1] repro: `_make_operand` applied to grad_y and to the activation).  The two calls are
 * independent, so one launch covers both and saves a kernel boundary on the wgrad path.
 *   x_a / x_b: bf16 [K_cap, C_a] / [K_cap, C_b].  q_a / q_b, sf_a / sf_b: as in
 *   dg_quant_per_channel_128.
 */
int dg_quant_per_channel_128_pair(const void* x_a, int64_t C_a, uint8_t* q_a, float* sf_a,
                                  const void* x_b, int64_t C_b, uint8_t* q_b, float* sf_b,
                                  int64_t K_cap, const int32_t* ks, int G, float sf_zero,
                                  int32_t* status, void* stream);

/*
 * 128x128 per-block cast of expert weights ([P2] "2d" weight scales of sm90_fp8_gemm_1d2d;
 * [P3] "weights requantized to 2^k scales" for UE8M0).  amax over each 128x128 block, then
 * the rules of dg_quant_per_token_1x128.
 *   w: bf16 [G, N, K].  q: e4m3 [G, N, K].  sfb: [G][N/128][K/128] fp32 or UE8M0 bytes.
 */
int dg_quant_block_128x128(const void* w, int G, int64_t N, int64_t K, uint8_t* q, void* sfb,
                           int sf_format, float sf_zero, void* stream);

/*
 * m-grouped contiguous FP8 GEMM ([P3] m_grouped_fp8_fp4_gemm_nt_contiguous, FP8 operands):
 *   D[m, n] = sum_k A[m, k] sfa[k/128, m] * B[e, n, k] sfb[e, n/128, k/128],  e = m_indices[m]
 * for rows with e >= 0; rows with m_indices = -1 are never written.  Expert segments are
 * aligned to 128 rows: the expert of 128-row block b is m_indices[128 b]; a block whose first
 * row is -1 is padding and skipped; inside a block, rows whose index differs from the block's
 * expert are not written (DG_STATUS_BAD_INDEX if it is another valid expert).
 *   a: e4m3 [M, K].  b: e4m3 [G, N, K].  d: [M, N] bf16 or fp32 (out_dtype).
 *   sfa: [K/128][Mp] (per sf_format), sfb: [G][N/128][K/128] (same sf_format).
 *   m_indices: int32 [M] device.  Accumulation is fp32 in tensor memory, promoted per 128-K
 *   block; results are bitwise reproducible run to run.
 */
int dg_m_grouped_fp8_contiguous(const uint8_t* a, const void* sfa, const uint8_t* b,
                                const void* sfb, void* d, int out_dtype, const int32_t* m_indices,
                                int64_t M, int G, int64_t N, int64_t K, int sf_format,
                                void* workspace, size_t workspace_bytes, int32_t* status,
                                void* stream);

/*
 * dg_m_grouped_fp8_contiguous with the grouped layout given as prefix sums ([P1] and [P3]:
 * the `use_psum_layout` option of the grouped GEMMs, and the graph-mutation test "across
 * m_indices/psum/masked modes").  Reading taken: psum[e] is the exclusive end row of expert
 * e's rows, which start at the previous expert's end rounded up to a multiple of 128
 * (psum[-1] = 0) - the 128-aligned segments of the m_indices layout, described by G integers.
 *   psum: int32 [G] device, non-decreasing, psum[G-1] <= M.  An entry below its predecessor,
 *   past M, or ending inside the rounding gap sets DG_STATUS_BAD_INDEX; that expert and every
 *   later one are skipped.  Everything else is as dg_m_grouped_fp8_contiguous; the result is
 *   bitwise that of the equivalent m_indices call.
 */
int dg_m_grouped_fp8_contiguous_psum(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb, void* d,
                                     int out_dtype, const int32_t* psum, int64_t M, int G, int64_t N, int64_t K,
                                     int sf_format, void* workspace, size_t workspace_bytes, int32_t* status,
                                     void* stream);

/*
 * m-grouped masked FP8 GEMM ([P2] m_grouped_*_gemm_nt_masked(a, b, d, masked_m, expected_m)):
 *   D[g, r, n] = sum_k A[g, r, k] sfa[k/128, g*cap + r] * B[g, n, k] sfb[g, n/128, k/128]
 * for r < min(counts[g], cap).  Rows at or past the count are never written: the output is
 * kept per expert as a 3-D [G, cap, N] tensor (the fix of [P2]), so no tile can reach the
 * next expert's rows, and rows in [count, cap) inside a tile are not stored either.
 *   a: e4m3 [G, cap, K].  b: e4m3 [G, N, K].  d: [G, cap, N] bf16 or fp32.
 *   sfa: [K/128][Mp] with M = G*cap.  counts: int32 [G] device.
 *   expected_m: a hint only; it never changes the result.
 */
int dg_m_grouped_fp8_masked(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb,
                            void* d, int out_dtype, const int32_t* counts, int G, int64_t cap,
                            int64_t N, int64_t K, int expected_m, int sf_format, void* workspace,
                            size_t workspace_bytes, int32_t* status, void* stream);

/*
 * Plain FP8 GEMM with the same scaling ([P2] validation: the adjacent-path checks of ordinary
 * GEMM layouts, output dtypes and accumulation, and batched GEMM):
 *   D[m, n] = C[m, n] + sum_k A[m, k] sfa[k/128, m] * B[n, k] sfb[n/128, k/128]
 * for m < M (C omitted when c is NULL).
 *   a: e4m3 [M, K] row-major.  sfa: [K/128][Mp] per-token scales ("Scale-factor layouts").
 *   b: e4m3 [N, K] row-major.  sfb: [N/128][K/128] (the [G][N/128][K/128] layout with G = 1).
 *   c: optional fp32 [M, N]; needs out_dtype DG_OUT_FP32; may equal d (in-place accumulate).
 *   d: [M, N] bf16 or fp32 (out_dtype).  M >= 0 (0: nothing enqueued), M <= 524288.
 * Runs the contiguous m-grouped kernel with one expert owning every row; no routing tensor.
 */
int dg_fp8_gemm_nt(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb,
                   const float* c, void* d, int out_dtype, int64_t M, int64_t N, int64_t K,
                   int sf_format, int32_t* status, void* stream);

/*
 * Batched FP8 GEMM ([P2] validation, batched GEMM; also the masked layout with every count
 * equal to the capacity):  D[i] = C[i] + A[i] . B[i]^T for i < batch.
 *   a: e4m3 [batch, M, K].  sfa: [K/128][Mp] over the batch*M rows.  b: e4m3 [batch, N, K].
 *   sfb: [batch][N/128][K/128].  c: optional fp32 [batch, M, N] (fp32 output only; may equal d).
 *   d: [batch, M, N] bf16 or fp32.  1 <= batch <= DG_MAX_GROUPS.
 */
int dg_fp8_gemm_nt_batched(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb,
                           const float* c, void* d, int out_dtype, int batch, int64_t M,
                           int64_t N, int64_t K, int sf_format, int32_t* status, void* stream);

/*
 * m-grouped masked BF16 GEMM ([P2] m_grouped_bf16_gemm_nt_masked(a, b, d, masked_m, expected_m),
 * the GEMM of the pages' reproduction, checked there against bmm(a.double(), b.double().mT)
 * rounded to bf16):
 *   D[g, r, n] = sum_k A[g, r, k] * B[g, n, k]   (fp32 accumulation)   for r < min(counts[g], cap)
 * with the same per-expert output boundary as the FP8 masked GEMM: rows at or past the count
 * are never written.
 *   a: bf16 [G, cap, K].  b: bf16 [G, N, K].  d: [G, cap, N] bf16 or fp32 (out_dtype).
 *   counts: int32 [G] device (clamped to [0, cap]; out-of-range counts set
 *   DG_STATUS_COUNT_GT_CAP).  N % 128 == 0, K % 64 == 0; a, b, d 16-byte aligned.
 *   expected_m: a hint only (with the capacity it picks the tile width); it never changes the
 *   result.
 */
int dg_m_grouped_bf16_masked(const void* a, const void* b, void* d, int out_dtype, const int32_t* counts,
                             int G, int64_t cap, int64_t N, int64_t K, int expected_m, int32_t* status,
                             void* stream);

/*
 * m-grouped contiguous BF16 GEMM: the BF16 GEMM of [P2] on the contiguous layout of [P3]
 * (rows routed by m_indices, -1 = padding, segments aligned to 128 rows):
 *   D[m, n] = sum_k A[m, k] * B[m_indices[m], n, k]   for rows with m_indices[m] in [0, G).
 *   a: bf16 [M, K].  b: bf16 [G, N, K].  d: [M, N] bf16 or fp32.  m_indices: int32 [M] device.
 *   Row validity, the skipping of all-padding blocks and the status bits are those of
 *   dg_m_grouped_fp8_contiguous.  N % 128 == 0, K % 64 == 0.
 */
int dg_m_grouped_bf16_contiguous(const void* a, const void* b, void* d, int out_dtype, const int32_t* m_indices,
                                 int64_t M, int G, int64_t N, int64_t K, int32_t* status, void* stream);

/*
 * k-grouped FP8 weight-gradient GEMM ([P1] k_grouped_fp8_gemm_nt_contiguous with
 * recipe (1, 1, 128)): for each expert e with token span [o_e, o_e + K_e) along K,
 *   D_e[n, h] = C_e[n, h] + sum_{t < K_e} A_e[n, t] sfa[(o_e+t)/128, n] * B_e[h, t] sfb[(o_e+t)/128, h]
 * where A_e / B_e are the K-major packed blocks written by dg_quant_per_channel_128.
 *   a_packed: e4m3, [N, K_e] blocks at offset o_e*N.  b_packed: e4m3, [H, K_e] at o_e*H.
 *   sfa: fp32 [K_cap/128][N].  sfb: fp32 [K_cap/128][H].
 *   c: fp32 [G, N, H] or NULL (zero); may alias d (the pages pass the same tensor).
 *   d: fp32 [G, N, H].  ks: int32 [G] device.
 *   K_e = 0 gives D_e = C_e.  Bad ks stop the walk as in dg_quant_per_channel_128.
 *   workspace: dg_workspace_size(DG_OP_K_GROUPED_WGRAD, G, 0, N, H) bytes; it receives the
 *   per-expert TMA descriptors, rebuilt from ks by a separate launch on every call (so a
 *   replayed graph never uses descriptors derived from stale counts).
 */
int dg_k_grouped_fp8_wgrad(const uint8_t* a_packed, const float* sfa, const uint8_t* b_packed,
                           const float* sfb, const float* c, float* d, const int32_t* ks, int G,
                           int64_t K_cap, int64_t N, int64_t H, void* workspace,
                           size_t workspace_bytes, int32_t* status, void* stream);

/*
 * The whole wgrad of [P1]'s listing from bf16 inputs in two launches: the per-channel casts
 * with the per-expert K-major packs of grad_y [K_cap, N] (A) and act [K_cap, H] (B), exactly as
 * dg_quant_per_channel_128_pair fills a_packed/sfa and b_packed/sfb, and in the same launch the
 * per-expert descriptors; then the GEMM of dg_k_grouped_fp8_wgrad.  The casts and the
 * descriptors are independent and run side by side, which saves the separate descriptor launch.
 *   grad_y, act: bf16, row-major, 16-byte aligned.  sf_zero as for the per-channel cast.
 *   a_packed, sfa, b_packed, sfb: caller buffers of dg_k_grouped_fp8_wgrad's layouts (written).
 *   ks, G, K_cap, N, H, c, d, workspace, status: as for dg_k_grouped_fp8_wgrad.
 * The _psum form takes the expert spans as inclusive prefix sums (see dg_k_grouped_fp8_wgrad_psum).
 */
int dg_k_grouped_fp8_wgrad_from_bf16(const void* grad_y, const void* act, const int32_t* ks, int G,
                                     int64_t K_cap, int64_t N, int64_t H, uint8_t* a_packed,
                                     float* sfa, uint8_t* b_packed, float* sfb, const float* c,
                                     float* d, float sf_zero, void* workspace,
                                     size_t workspace_bytes, int32_t* status, void* stream);
int dg_k_grouped_fp8_wgrad_from_bf16_psum(const void* grad_y, const void* act, const int32_t* psum,
                                          int G, int64_t K_cap, int64_t N, int64_t H,
                                          uint8_t* a_packed, float* sfa, uint8_t* b_packed,
                                          float* sfb, const float* c, float* d, float sf_zero,
                                          void* workspace, size_t workspace_bytes, int32_t* status,
                                          void* stream);

/*
 * dg_k_grouped_fp8_wgrad, dg_quant_per_channel_128 and dg_quant_per_channel_128_pair with the
 * expert spans given as inclusive prefix sums ([P1] k_grouped_fp8_gemm_nt_contiguous(...,
 * use_psum_layout=True)): psum[e] = K_0 + ... + K_e, so K_e = psum[e] - psum[e-1] (psum[-1] = 0).
 * A decreasing entry gives a negative K_e and stops the walk like any bad K_e.  Results are
 * bitwise those of the equivalent ks calls.
 */
int dg_k_grouped_fp8_wgrad_psum(const uint8_t* a_packed, const float* sfa, const uint8_t* b_packed,
                                const float* sfb, const float* c, float* d, const int32_t* psum, int G,
                                int64_t K_cap, int64_t N, int64_t H, void* workspace, size_t workspace_bytes,
                                int32_t* status, void* stream);
int dg_quant_per_channel_128_psum(const void* x, int64_t K_cap, int64_t C, const int32_t* psum, int G,
                                  uint8_t* q_packed, float* sf, float sf_zero, int32_t* status, void* stream);
int dg_quant_per_channel_128_pair_psum(const void* x_a, int64_t C_a, uint8_t* q_a, float* sf_a, const void* x_b,
                                       int64_t C_b, uint8_t* q_b, float* sf_b, int64_t K_cap, const int32_t* psum,
                                       int G, float sf_zero, int32_t* status, void* stream);

/*
 * FP4 weights ([P3]: the kernel is named m_grouped_fp8_fp4_gemm_nt_contiguous, FP8 activations
 * with FP8 or FP4 weights, "weights requantized to 2^k scales").  The pages name the FP4 form
 * only; reading taken: OCP e2m1 codes (values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives)
 * with one power-of-two (UE8M0) scale per 128x128 block, the rule of the FP8 weight cast with
 * e2m1's maximum 6 in place of 448.
 *
 * dg_quant_block_128x128_fp4: per 128x128 block of w, amax (fp32), sf = amax / 6, sf == 0 ->
 * sf_zero, sf = max(sf, 1e-30), rounded up to a power of two; q = e2m1_rne_satfinite(x * (1/sf)).
 *   w: bf16 [G, N, K] (16-byte aligned).  q_packed: [G, N, K/2] bytes, two codes per byte along K,
 *   element 2i in the low nibble and 2i+1 in the high nibble (4-byte aligned).
 *   sfb: UE8M0 bytes [G][N/128][K/128].  N, K multiples of 128.
 */
int dg_quant_block_128x128_fp4(const void* w, int G, int64_t N, int64_t K, uint8_t* q_packed,
                               uint8_t* sfb, float sf_zero, void* stream);

/*
 * m-grouped contiguous and masked GEMMs with FP4 weights ([P3]
 * m_grouped_fp8_fp4_gemm_nt_contiguous): the results of dg_m_grouped_fp8_contiguous /
 * dg_m_grouped_fp8_masked with sf_format DG_SF_UE8M0, with each weight element the e2m1 value
 * of its code times its block's scale.
 *   a: e4m3 [M, K] / [G, cap, K].  sfa: UE8M0 bytes [K/128][round_up(M or G*cap, 16)].
 *   b_packed: FP4 codes [G, N, K/2] as written by dg_quant_block_128x128_fp4 (16-byte aligned).
 *   sfb: UE8M0 bytes [G][N/128][K/128].  d: bf16 or fp32 (out_dtype).
 *   m_indices / counts, G, cap, expected_m, status, stream: as for the FP8 calls.
 *   N must be a multiple of 256 (DG_ERR_UNSUPPORTED otherwise): these calls run on the
 *   block-scaled MMA kernel's 128 x 256 tiles.  Rows that are not valid are never written.
 */
int dg_m_grouped_fp8_fp4_contiguous(const uint8_t* a, const uint8_t* sfa, const uint8_t* b_packed,
                                    const uint8_t* sfb, void* d, int out_dtype,
                                    const int32_t* m_indices, int64_t M, int G, int64_t N, int64_t K,
                                    int32_t* status, void* stream);
int dg_m_grouped_fp8_fp4_masked(const uint8_t* a, const uint8_t* sfa, const uint8_t* b_packed,
                                const uint8_t* sfb, void* d, int out_dtype, const int32_t* counts,
                                int G, int64_t cap, int64_t N, int64_t K, int expected_m,
                                int32_t* status, void* stream);

/* Largest G accepted by dg_k_grouped_fp8_wgrad_noalloc. */
#define DG_NOALLOC_MAX_GROUPS 256

/*
 * dg_k_grouped_fp8_wgrad without a workspace.  This entry point has no counterpart on the
 * source pages; it exists for callers that cannot allocate device memory when they make the
 * call: runtimes that carve all device memory into a fixed arena at start-up and forbid later
 * allocation, serving loops that must not pay cudaMalloc's implicit device-wide
 * synchronisation, and plain C callers that have no device allocator of their own to provide
 * the workspace.  The caller still owns and passes every input and output.
 *   Arguments, layouts, results and status bits are those of dg_k_grouped_fp8_wgrad.
 *   The per-expert descriptors go to a 64 KiB array compiled into the library
 *   (2 * DG_NOALLOC_MAX_GROUPS descriptors of 128 bytes), held by every device that loads the
 *   library until the process exits.  G > DG_NOALLOC_MAX_GROUPS returns DG_ERR_UNSUPPORTED.
 *   The first call in each CUDA context (normally once per device: its primary context, with
 *   that device current) looks up the array's device address and caches it for that context;
 *   a context created later (after cudaDeviceReset, or a caller's own driver context) gets its
 *   own lookup on its first call.  Make the first call in a context before any stream capture.
 *   All calls share the one array: calls that may overlap on the GPU (other streams, other
 *   host threads) race on it and must be serialised by the caller.  Every descriptor a call
 *   reads is rewritten by that same call, so nothing is carried over from the previous call.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
int dg_k_grouped_fp8_wgrad_noalloc(const uint8_t* a_packed, const float* sfa, const uint8_t* b_packed,
                                   const float* sfb, const float* c, float* d, const int32_t* ks, int G,
                                   int64_t K_cap, int64_t N, int64_t H, int32_t* status, void* stream);

/*
 * Debug aids ([P3], "What fails" and "Evidence / repro kit": the arguments of the failing
 * call were dumped inside the serving process and replayed offline).  Here the same search uses
 * a host-side argument log, and a debug build whose kernels check the indices they compute
 * (the kernels never trap, so a bad index shows as a bit, not as a fault).
 *
 * Argument log.  dg_set_arg_log(path) makes every entry point above append one text line to
 * the file `path` before it checks its arguments: a sequence number, the entry point's name
 * and name=value for every argument (pointers in hex, sizes in decimal, floats with 9
 * significant digits).  NULL or "" stops the log.  The environment variable DG_ARG_LOG, read
 * when the library is loaded, sets the first path.  The log reads nothing from the device, so
 * it is safe inside stream capture; it records calls, not graph replays.  Returns DG_OK.
 *
 * Debug build.  Built with -DDG_DEBUG=1 (libdg_debug.so), every kernel checks each index it
 * computes for a scale read, an owner-thread store, a C read or a cast's element access against
 * the extent the layouts above give that buffer; an index outside it ORs a DG_DEBUG_* bit into
 * the library's debug word and the access is skipped.  Its kernels' bounded waits give up after
 * 250 ms instead of 2000 ms (DG_WAIT_LIMIT_MS overrides both).  In the release build nothing is
 * checked.
 *   dg_debug_build(): 1 for the debug build, 0 for the release build.
 *   dg_debug_word(out, clear): waits for the current device (cudaDeviceSynchronize), then
 *   stores in *out (a HOST pointer) the OR of the bits raised on it since the last clear, and
 *   clears them if `clear` != 0.  The release build stores 0.  Returns DG_OK or DG_ERR_CUDA.
 */
enum dg_debug_bits {
    DG_DEBUG_A_SCALE = 1,  /* an activation-scale (sfa) index outside [K/128][Mp] */
    DG_DEBUG_B_SCALE = 2,  /* a weight-scale (sfb) index outside [G][N/128][K/128] */
    DG_DEBUG_OUT = 4,      /* an output (or C) row or column outside D */
    DG_DEBUG_CAST_IN = 8,  /* a cast's input element outside x / w */
    DG_DEBUG_CAST_OUT = 16 /* a cast's code or scale outside q / sf */
};
int dg_set_arg_log(const char* path);
int dg_debug_build(void);
int dg_debug_word(uint32_t* out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* DG_H */
