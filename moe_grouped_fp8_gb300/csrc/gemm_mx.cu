// gemm_mx.cu - m-grouped FP8 (e4m3) GEMM for UE8M0 scale factors, scaled by the tensor core.
//
// With UE8M0 scales ("SM120 m_grouped_fp8 contiguous kernel: illegal memory access at CUDA graph
// replay", #444, environment: weights requantized to 2^k scales, activations with packed
// power-of-two scales) every scale is a power of two, which is what the block-scaled MMA of
// sm_103a (tcgen05.mma.kind::mxf8f6f4.block_scale.scale_vec::1X) applies itself: one UE8M0 scale
// per row of A and per row of B for each 32-element K block of an instruction.  A 1x128 activation
// scale and a 128x128 weight scale are constant over a 128-K block, so the four 32-K MMAs of the
// block take the same scales (the scale replicated per 32-K), and the weight scale is the same for
// all 128 rows of a weight tile.  The tensor core then accumulates the scaled products over the
// whole K of a tile in tensor memory: no per-block promotion, one hand-off per tile.
//
// Roles (352 threads): warps 0-7 drain the finished accumulator (TMEM lane quarter = warp % 4,
// column half = warp / 4) and write each valid row from registers; warp 8 issues the TMA loads of
// the A / B tiles; warp 9 writes the scale bytes of each group of four 128-K blocks into the
// tensor-memory scale layout in shared memory; warp 10 copies a group's scales into tensor memory
// (tcgen05.cp) and issues the MMAs (it owns the tensor memory).  Tiles are 128 x 256: a
// 256-column accumulator leaves room for the scale columns but not for a second accumulator, so
// the MMAs of the next tile wait for the drain of the last (the drain warps hand it back as soon as
// it is in registers) - a few per cent of a tile of 16 or more blocks, which is why the library
// takes this kernel for K >= 2048 only.  Against 128 x 128 tiles the wide tile halves the A-operand
// traffic and shared-memory reads per FLOP: with 128 x 128 tiles (three accumulators) this kernel
// measured 0.44 of the FP8 peak on a compute-bound shape, with 128 x 256 tiles 0.72.
//
// Scale layout in tensor memory (scale_vec::1X, M = 128 or N = 128 rows): the scale of row
// 32 j + i sits in lane i, column c0 + j of each 32-lane quarter (tcgen05.cp.32x128b.warpx4 copies
// 32 rows of four 32-bit words and replicates them into the four quarters).  Byte u of a word is
// the row's scale for 128-K block u of the group, which the MMAs of that block select with
// scale-factor id u: one copy of 1 KB serves four blocks.
//
// FP4 weights (the FP8 x FP4 form of the same kernel name, m_grouped_fp8_fp4_gemm_nt_contiguous):
// B holds e2m1 codes, two per byte in global memory; the TMA unpacks each 16-code group of 8 bytes
// into 16 bytes of shared memory (CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B), the form kind::mxf8f6f4
// reads for 4-bit operands, so a 128-K block of B takes the same 128 bytes per row of shared memory
// as FP8 and every descriptor and swizzle is unchanged; the instruction's B format changes, and the
// stage's transaction count, which counts the packed bytes the load reads (a count of the unpacked
// footprint never completed: every wait ran out).
//
// The schedule comes from the device-side routing tensor in every CTA on every launch (as in
// gemm.cu), so graph replays with changed routing never use stale state.  The K order of the
// accumulation is fixed, with no split-K and no atomics, so every call is bitwise reproducible.
// Rows that are not valid (masked rows at or past the count, m_indices = -1, rows of another
// expert) are never written.
#include <cuda_bf16.h>

#include <atomic>

#include "host_common.hpp"
#include "kernel_common.cuh"
#include "mgrouped.cuh"
#include "ptx.cuh"

namespace dg {
namespace mx {

constexpr int EPI_WARPS = 8;
constexpr int PRODUCER_WARP = 8, SF_WARP = 9, MMA_WARP = 10;
constexpr int NT = 11 * 32;
constexpr int SFG = 4;              // 128-K blocks per scale group (the four bytes of a word)
constexpr int SF_SLOTS = 4;         // scale groups in shared / tensor memory at once
constexpr int KG = 4;               // scale groups whose bytes the scale warp has in flight
constexpr int SF_ROWS_BYTES = 512;  // 32 rows x 16 bytes: the scales of 128 rows
constexpr uint32_t TMEM_COLS = 512;

// The tile plan: 128 x 256 tiles, four 48 KB ring stages, one accumulator.
struct Plan {
    static constexpr int BN = 256;                               // tile columns
    static constexpr int STAGES = 4;
    static constexpr int ACC = 1;
    static constexpr int A_BYTES = BM * BK;                      // 16 KB
    static constexpr int B_BYTES = BN * BK;                      // 32 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int NB128 = BN / 128;                       // 128-row weight blocks of a tile
    static constexpr int SFB_BYTES = NB128 * SF_ROWS_BYTES;      // B scales of BN rows
    static constexpr int SF_SLOT = SF_ROWS_BYTES + SFB_BYTES;    // A scales, then B scales
    static constexpr uint32_t SF_COLS = 16;                      // tensor-memory columns of a group (4 + 8, padded)
    static constexpr int CPT = BN / 2;                           // accumulator columns per drain thread
    static constexpr int RING_OFF = 0;
    static constexpr int SF_OFF = STAGES * STAGE_BYTES;
    static constexpr int SCHED_OFF = SF_OFF + SF_SLOTS * SF_SLOT;
    static constexpr int BAR_OFF = (SCHED_OFF + SCHED_BYTES + 127) / 128 * 128;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * SF_SLOTS + 2 * ACC;  // full, empty; sfull, sempty; tfull, tempty
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int TOTAL = MISC_OFF + 256 + 1024;          // + alignment slack
    static constexpr uint32_t SF_COL0 = ACC * BN;                // group slot q: A scales at SF_COL0 + SF_COLS q
    static_assert(SF_COL0 + SF_COLS * SF_SLOTS <= TMEM_COLS, "scale columns inside the allocation");
    static_assert(SF_COL0 % 8 == 0 && SF_COLS % 8 == 0 && SF_COLS >= 4 + BN / 32, "scale columns 8-aligned");
    static_assert(A_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0 && SF_OFF % 1024 == 0, "swizzle atoms aligned");
    static_assert(SF_SLOT % 128 == 0 && SCHED_OFF % 16 == 0, "scale slots 16-byte aligned");
    static_assert(BAR_OFF % 8 == 0 && MISC_OFF % 8 == 0, "mbarriers 8-byte aligned");
    static_assert(TOTAL <= 232448, "shared memory");
    static_assert(CPT % 32 == 0, "drain loads of 32 columns");
};
static_assert(BM == 128, "the scale layout covers 128 rows of A");

// The scale warp's walk over this CTA's (tile, scale group) items: group kb0 covers the 128-K
// blocks kb0 .. kb0 + SFG - 1 of the tile (fewer at the tile's end).
template <Layout L>
struct Walk {
    int t, kb0;
    TileInfo ti;
    bool valid;
    __device__ void start(int num_tiles, const RunTable& rt, int R, const GemmArgs& a) {
        t = blockIdx.x;
        kb0 = 0;
        valid = t < num_tiles;
        if (valid) ti = decode_tile<L>(t, rt, R, a);
    }
    __device__ void next(int num_tiles, const RunTable& rt, int R, const GemmArgs& a) {
        kb0 += SFG;
        if (kb0 < ti.kbt) return;
        kb0 = 0;
        t += gridDim.x;
        valid = t < num_tiles;
        if (valid) ti = decode_tile<L>(t, rt, R, a);
    }
};

// The UE8M0 bytes of one group: ba[j][u] = block kb0 + u of row 32 j + lane of the tile's A rows,
// bb[n][u] = block kb0 + u of the tile's n-th 128-row weight block.  Rows outside the layout and blocks past the
// tile's K read 127 (scale 1): they are never used for a stored result.
template <Layout L, int NB128>
__device__ __forceinline__ void load_group(const Walk<L>& w, const GemmArgs& a, int lane, uint8_t (&ba)[4][SFG],
                                           uint8_t (&bb)[NB128][SFG]) {
    const uint8_t* sfa = static_cast<const uint8_t*>(a.sfa);
    const uint8_t* sfb =
        static_cast<const uint8_t*>(a.sfb) + (static_cast<int64_t>(w.ti.e) * a.n128 + w.ti.nb * NB128) * a.KB;
#pragma unroll
    for (int u = 0; u < SFG; ++u) {
        const bool kin = w.kb0 + u < w.ti.kbt;
        const int64_t kbase = static_cast<int64_t>(w.kb0 + u) * a.sfa_ld;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t r = static_cast<int64_t>(w.ti.row0) + j * 32 + lane;
            const bool in = kin && r < a.M;  // Masked: a.M = cap; Contiguous: rows
            const int64_t m = L == Layout::Masked ? static_cast<int64_t>(w.ti.e) * a.M + r : r;
            ba[j][u] = in && DG_CHECKED(sfa_in<L>(a, w.kb0 + u, m), DG_DEBUG_A_SCALE) ? __ldg(sfa + kbase + m)
                                                                                      : static_cast<uint8_t>(127);
        }
#pragma unroll
        for (int n = 0; n < NB128; ++n)
            bb[n][u] = kin && DG_CHECKED(sfb_in(a, w.ti.e, w.ti.nb * NB128 + n, w.kb0 + u), DG_DEBUG_B_SCALE)
                           ? __ldg(sfb + n * a.KB + w.kb0 + u)
                           : static_cast<uint8_t>(127);
    }
}

__device__ __forceinline__ uint32_t pack4(const uint8_t (&b)[SFG]) {
    return static_cast<uint32_t>(b[0]) | (static_cast<uint32_t>(b[1]) << 8) | (static_cast<uint32_t>(b[2]) << 16) |
           (static_cast<uint32_t>(b[3]) << 24);
}

template <Layout L, bool OUT_FP32, bool B_FP4>
__global__ void __launch_bounds__(NT, 1)
    k_grouped_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const GemmArgs a) {
    using P = Plan;
    constexpr int BN = P::BN, STAGES = P::STAGES, ACC = P::ACC, A_BYTES = P::A_BYTES, STAGE_BYTES = P::STAGE_BYTES;
    constexpr int SF_SLOT = P::SF_SLOT, NB128 = P::NB128;
    // Bytes a stage's TMA loads complete: an unpacking FP4 load counts the packed bytes it reads
    // (half a B tile), though it fills the same shared-memory footprint as FP8.
    constexpr uint32_t STAGE_TX = A_BYTES + (B_FP4 ? P::B_BYTES / 2 : P::B_BYTES);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

    uint8_t* ring = smem + P::RING_OFF;
    uint8_t* sfbuf = smem + P::SF_OFF;
    const RunTable rt = RunTable::at(smem + P::SCHED_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::BAR_OFF);
    uint64_t* full = bars;                 // A / B tiles landed (TMA bytes)
    uint64_t* empty = bars + STAGES;       // the stage's MMAs are done
    uint64_t* sfull = bars + 2 * STAGES;   // a scale group is in shared memory
    uint64_t* sempty = sfull + SF_SLOTS;   // the group's copies and MMAs are done
    uint64_t* tfull = sempty + SF_SLOTS;   // an accumulator holds a finished tile
    uint64_t* tempty = tfull + ACC;        // the drain warps have read it
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + P::MISC_OFF);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + P::MISC_OFF + 4);
    int* s_ntiles = reinterpret_cast<int*>(smem + P::MISC_OFF + 12);
    int* s_scan = reinterpret_cast<int*>(smem + P::MISC_OFF + 64);  // [NT / 32 + 1]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const WaitCtx wc{a.status, s_abort, a.wait_limit_ns};

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int q = 0; q < SF_SLOTS; ++q) {
            mbar_init(&sfull[q], 1);
            mbar_init(&sempty[q], 1);
        }
        for (int b = 0; b < ACC; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], EPI_WARPS);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(s_tmem, TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    pdl_trigger();
    pdl_wait();  // every earlier kernel of the stream has finished: inputs are visible
    __syncthreads();

    // ---------------------------------------------------------------- tile schedule
    const int R = build_runs<L, NT>(a, rt, s_scan, ring);  // the ring is free during set-up
    const int num_tiles = tile_prefix<NT, 1>(R, a.num_nb, rt, s_scan, s_ntiles);
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    if (warp == PRODUCER_WARP) {
        // ------------------------------------------------------------ A / B tiles
        if (lane == 0 && R > 0) {
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile<L>(t, rt, R, a);
                for (int kb = 0; kb < ti.kbt; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
                    uint8_t* sa = ring + stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], STAGE_TX);
                    if constexpr (L == Layout::Masked)
                        tma_load_3d(sa, &tmA, &full[stage], kb * BK, ti.row0, ti.e);
                    else
                        tma_load_2d(sa, &tmA, &full[stage], kb * BK, ti.row0);
                    tma_load_3d(sa + A_BYTES, &tmB, &full[stage], kb * BK, ti.nb * BN, ti.e);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // drain: every load this thread issued has landed before the CTA may exit
            const int n_drain = issued < STAGES ? issued : STAGES;
            for (int i = 0; i < n_drain; ++i) {
                int s = stage - 1 - i;
                uint32_t ph = phase;
                while (s < 0) { s += STAGES; ph ^= 1u; }
                drain_wait(&full[s], ph, a.drain_limit_ns);
            }
        }
        __syncwarp();
    } else if (warp == SF_WARP) {
        // ------------------------------------------------------------ scale groups -> shared memory
        // KG register slots: slot g is written to shared memory, then reloaded with the group KG
        // places further on, so KG groups' global loads are in flight while the slots fill.
        if (R > 0) {
            Walk<L> st, ld;
            st.start(num_tiles, rt, R, a);
            ld.start(num_tiles, rt, R, a);
            uint8_t ba[KG][4][SFG], bb[KG][NB128][SFG];
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                if (ld.valid) {
                    load_group<L, NB128>(ld, a, lane, ba[g], bb[g]);
                    ld.next(num_tiles, rt, R, a);
                }
            }
            int slot = 0;
            uint32_t phase = 0;
            bool ok = true;
            while (st.valid && ok) {
#pragma unroll
                for (int g = 0; g < KG; ++g) {
                    if (!st.valid) break;
                    bool w = true;
                    if (lane == 0) w = mbar_wait(&sempty[slot], phase ^ 1u, wc);
                    if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) { ok = false; break; }
                    __syncwarp();  // orders every lane's writes below after lane 0's wait
                    uint8_t* sl = sfbuf + slot * SF_SLOT;
                    *reinterpret_cast<uint4*>(sl + 16 * lane) =
                        make_uint4(pack4(ba[g][0]), pack4(ba[g][1]), pack4(ba[g][2]), pack4(ba[g][3]));
#pragma unroll
                    for (int n = 0; n < NB128; ++n) {
                        const uint32_t wb = pack4(bb[g][n]);  // one scale for the 128 rows of weight block n
                        *reinterpret_cast<uint4*>(sl + SF_ROWS_BYTES * (1 + n) + 16 * lane) = make_uint4(wb, wb, wb, wb);
                    }
                    fence_async_smem();  // generic-proxy writes -> visible to tcgen05.cp
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sfull[slot]);
                    if (++slot == SF_SLOTS) { slot = 0; phase ^= 1u; }
                    st.next(num_tiles, rt, R, a);
                    if (ld.valid) {
                        load_group<L, NB128>(ld, a, lane, ba[g], bb[g]);
                        ld.next(num_tiles, rt, R, a);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ scale copies + MMAs
        if (lane == 0 && R > 0) {
            int stage = 0, j = 0, slot = 0;
            uint32_t phase = 0, sphase = 0;
            bool ok = true;
            uint64_t* last = nullptr;  // the barrier of this thread's last commit, and its phase
            uint32_t last_ph = 0;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++j) {
                const TileInfo ti = decode_tile<L>(t, rt, R, a);
                const int tb = j % ACC;
                const uint32_t tv = static_cast<uint32_t>(j / ACC) & 1u;
                if (!mbar_wait(&tempty[tb], tv ^ 1u, wc)) { ok = false; break; }
                tc_fence_after();
                const uint32_t dt = tmem_base + static_cast<uint32_t>(tb * BN);
                uint32_t sfa_t = 0, sfb_t = 0;
                for (int kb = 0; kb < ti.kbt; ++kb) {
                    const uint32_t u = static_cast<uint32_t>(kb % SFG);
                    if (u == 0) {
                        // a new scale group: its bytes into tensor memory (ordered before the MMAs)
                        if (!mbar_wait(&sfull[slot], sphase, wc)) { ok = false; break; }
                        tc_fence_after();
                        sfa_t = tmem_base + P::SF_COL0 + P::SF_COLS * static_cast<uint32_t>(slot);
                        sfb_t = sfa_t + 4u;
                        const uint32_t sf_s = smem_u32(sfbuf + slot * SF_SLOT);
                        tmem_cp_32x128b_x4(sfa_t, sdesc_rows16(sf_s));
#pragma unroll
                        for (int n = 0; n < NB128; ++n)  // B rows 128 n .. 128 n + 127: columns 4 n ..
                            tmem_cp_32x128b_x4(sfb_t + 4u * n, sdesc_rows16(sf_s + SF_ROWS_BYTES * (1 + n)));
                    }
                    if (!mbar_wait(&full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t idesc = idesc_mxf8_e4m3_ue8m0(BM, BN, u, u, B_FP4 ? MXF_E2M1 : MXF_E4M3);
                    const uint32_t sa = smem_u32(ring + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_mxf8_1x(dt, sdesc_k_sw128(sa + 32 * k), sdesc_k_sw128(sb + 32 * k), idesc, sfa_t, sfb_t,
                                     (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);  // frees the stage's tiles
                    last = &empty[stage];
                    last_ph = phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    if (u == SFG - 1 || kb == ti.kbt - 1) {
                        umma_commit(&sempty[slot]);  // frees the group's scale slot
                        last = &sempty[slot];
                        last_ph = sphase;
                        if (++slot == SF_SLOTS) { slot = 0; sphase ^= 1u; }
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[tb]);
                last = &tfull[tb];
                last_ph = tv;
            }
            // the tensor core is done with every copy and MMA this thread issued
            if (last != nullptr) drain_wait(last, last_ph, a.drain_limit_ns);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ drain accumulators, store rows
        const int q = warp & 3;   // TMEM lane quarter
        const int h = warp >> 2;  // column half
        const int row = q * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        constexpr int ESIZE = OUT_FP32 ? 4 : 2;
        int j = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++j) {
            const TileInfo ti = decode_tile<L>(t, rt, R, a);
            const int tb = j % ACC;
            const uint32_t tv = static_cast<uint32_t>(j / ACC) & 1u;
            bool row_ok;
            int64_t grow;
            if constexpr (L == Layout::Masked) {
                row_ok = row < ti.valid;
                grow = static_cast<int64_t>(ti.e) * a.M + ti.row0 + row;
            } else {
                grow = static_cast<int64_t>(ti.row0) + row;
                if (a.psum) {
                    row_ok = row < ti.valid;
                } else {
                    const int mi = grow < a.M ? a.routing[grow] : -1;
                    row_ok = mi == ti.e;
                    if (mi >= 0 && mi != ti.e) status_or(a.status, DG_STATUS_BAD_INDEX);
                }
            }
            if (!mbar_wait(&tfull[tb], tv, wc)) break;
            tc_fence_after();
            constexpr int CPT = P::CPT;
            uint32_t v[CPT / 32][32];
            const uint32_t col = tmem_base + t_lane + static_cast<uint32_t>(tb * BN + h * CPT);
#pragma unroll
            for (int c = 0; c < CPT / 32; ++c) tmem_ld_x32(col + 32 * c, v[c]);
#pragma unroll
            for (int c = 0; c < CPT / 32; ++c) tmem_wait_ld(v[c]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[tb]);  // the accumulator is in registers
            const int64_t c0 = static_cast<int64_t>(ti.nb) * BN + h * CPT;
            if (!row_ok || !DG_CHECKED(out_in<L>(a, grow, c0, CPT), DG_DEBUG_OUT)) continue;
            uint8_t* dst = static_cast<uint8_t*>(a.d) + (grow * a.ldd + c0) * ESIZE;
            if constexpr (OUT_FP32) {
                const float* crow = a.c != nullptr ? a.c + grow * a.ldd + c0 : nullptr;
#pragma unroll
                for (int p = 0; p < CPT / 4; ++p) {
                    const int i = 4 * p;
                    float4 o = make_float4(__uint_as_float(v[i / 32][i % 32]), __uint_as_float(v[i / 32][i % 32 + 1]),
                                           __uint_as_float(v[i / 32][i % 32 + 2]),
                                           __uint_as_float(v[i / 32][i % 32 + 3]));
                    if (crow != nullptr) {
                        // C may alias D: this thread reads each element before it writes it
                        const float4 cv = *reinterpret_cast<const float4*>(crow + i);
                        o.x = cv.x + o.x;
                        o.y = cv.y + o.y;
                        o.z = cv.z + o.z;
                        o.w = cv.w + o.w;
                    }
                    *reinterpret_cast<float4*>(dst + 16 * p) = o;
                }
            } else {
#pragma unroll
                for (int p = 0; p < CPT / 8; ++p) {
                    uint32_t w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = 8 * p + 2 * u;
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[i / 32][i % 32]),
                                                                        __uint_as_float(v[i / 32][i % 32 + 1]));
                        w[u] = *reinterpret_cast<const uint32_t*>(&b2);
                    }
                    *reinterpret_cast<uint4*>(dst + 16 * p) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
        __syncwarp();
    }

    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <Layout L, bool OUT_FP32, bool B_FP4>
int launch(const CUtensorMap& tA, const CUtensorMap& tB, GemmArgs args, cudaStream_t stream) {
    auto kern = k_grouped_gemm_mx<L, OUT_FP32, B_FP4>;
    DG_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Plan::TOTAL));
    int sms = 0;
    if (int rc = device_sm_count(&sms)) return rc;
    args.num_nb = static_cast<int>(args.N / Plan::BN);
    return launch_pdl(kern, dim3(sms), dim3(NT), Plan::TOTAL, stream, tA, tB, args);
}

template <Layout L>
int launch_l(bool out_fp32, bool b_fp4, const CUtensorMap& tA, const CUtensorMap& tB, const GemmArgs& args,
             cudaStream_t stream) {
    if (b_fp4)
        return out_fp32 ? launch<L, true, true>(tA, tB, args, stream) : launch<L, false, true>(tA, tB, args, stream);
    return out_fp32 ? launch<L, true, false>(tA, tB, args, stream) : launch<L, false, false>(tA, tB, args, stream);
}

}  // namespace mx

int launch_mgrouped_mx(Layout L, bool out_fp32, bool b_fp4, const CUtensorMap& tA, const CUtensorMap& tB,
                       const GemmArgs& args, cudaStream_t stream) {
    if (L == Layout::Masked) return mx::launch_l<Layout::Masked>(out_fp32, b_fp4, tA, tB, args, stream);
    return mx::launch_l<Layout::Contiguous>(out_fp32, b_fp4, tA, tB, args, stream);
}

}  // namespace dg

namespace dg {
int debug_word_gemm_mx(uint32_t* out, bool clear) { return debug_word_local(out, clear); }
}  // namespace dg
