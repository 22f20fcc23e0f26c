// gemm_pair.cu - the m-grouped FP8 (e4m3) GEMM on CTA pairs (tcgen05 cta_group::2), sm_103a.
//
// A cluster of two CTAs on two SMs computes a 256 x 192 output tile of one expert: CTA r of
// the pair holds m-block 2j + r of the expert's run (128 rows of A) and B rows [96 r, 96 r + 96)
// of the tile's 192 columns.  One thread of the even CTA issues tcgen05.mma.cta_group::2
// (M = 256, N = 192, K = 32), which reads both CTAs' shared memory and leaves each CTA's
// 128 x 192 fp32 partial in its own tensor memory.  Against a 128 x 128 tile per SM this cuts
// the operand bytes each SM fetches per FLOP by 42%, and with them the bytes that must be in
// flight to keep the tensor core busy.  (N = 192 rather than 256 keeps each promotion thread at
// 64 accumulators within the 128 registers that 14 warps per SM leave.)
//
// Roles (480 threads per CTA): warps 0-11 promote and store (lane quarter = warp % 4, 64-column
// group = warp / 4), warp 12 loads A and B with TMA, warp 13 owns tensor memory; in the even
// CTA lane 0 of warps 13 and 14 issue the MMAs of the pair, on alternate 128-K blocks.  Per 128-K block the partial P goes to one of two
// TMEM buffers; the promotion warps read it and accumulate
// acc += sfa * sfb * P in fp32 registers - the per-128-K-block promotion of the 1x128 / 128x128
// scaling ("FP8 GEMM with fine-grained scaling": per-token activation scales, per-block weight
// scales).  K order, accumulation and rounding are fixed: every call is bitwise reproducible.
//
// Barriers: full[s] of the even CTA counts the bytes of both CTAs' loads of stage s; empty[s]
// and tfull[b] are completed in both CTAs by one multicast tcgen05.commit; tempty[b] of the
// even CTA collects the 24 promotion warps of the pair.  Every wait is bounded; a CTA leaves
// only after a cluster barrier, so no signal ever reaches a CTA that has exited.
//
// A run with an odd number of m-blocks pairs its last block with a block the odd CTA computes
// but never stores (rows of another expert, padding, or out of range, which TMA fills with
// zeros).  Row validity, the owner-thread tail stores and the 3-D masked stores follow the
// single-CTA kernel of gemm.cu: rows that are not valid are never written.
#include <cuda_bf16.h>

#include <atomic>

#include "host_common.hpp"
#include "kernel_common.cuh"
#include "mgrouped.cuh"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int P_EPI_WARPS = 12;
constexpr int P_PRODUCER_WARP = 12;
constexpr int P_MMA_WARP = 13;         // and P_MMA_WARP + 1: two issuers taking alternate 128-K blocks
constexpr int P_MMA_WARPS = 2;
constexpr int P_THREADS = 480;
constexpr int P_EPI_BAR = 1;             // named barrier of the 384 promotion/store threads
constexpr int P_BN = PAIR_BN;            // output columns of a pair tile
constexpr int P_BHALF = PAIR_B_ROWS;     // B rows held by each CTA
constexpr int P_TBUFS = 2;               // TMEM partial buffers
constexpr int P_TSTRIDE = 256;           // TMEM columns between buffers
constexpr int P_CPT = 64;                // output columns per promotion thread
constexpr int P_SF_GROUP = 4;            // 128-K blocks whose scales a promotion thread loads together
constexpr int P_STAGES = 5;

struct PairPlan {
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = P_BHALF * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int CHUNKS = P_BN * 2 / 128;  // 128-byte column chunks of a bf16 tile row
    static constexpr int CHUNK_BYTES = BM * 128;
    static constexpr int STG_BYTES = CHUNKS * CHUNK_BYTES;
    static constexpr int RING_OFF = 0;
    static constexpr int STG_OFF = P_STAGES * STAGE_BYTES;
    static constexpr int SCHED_OFF = STG_OFF + STG_BYTES;
    static constexpr int BAR_OFF = (SCHED_OFF + SCHED_BYTES + 127) / 128 * 128;
    static constexpr int NUM_BARS = 2 * P_STAGES + 2 * P_TBUFS;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int MISC_BYTES = 256;
    static constexpr int TOTAL = MISC_OFF + MISC_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = 512;
    static_assert(P_EPI_WARPS * 32 + 32 + 32 * P_MMA_WARPS == P_THREADS, "roles");
    static_assert(P_CPT * (P_EPI_WARPS / 4) == P_BN && P_CPT % 32 == 0, "column groups");
    static_assert(P_CPT * 2 == 128, "a promotion thread's bf16 columns fill one 128-byte chunk row");
    static_assert(STG_OFF % 1024 == 0 && SCHED_OFF % 1024 == 0, "TMA / swizzle buffers are 1024-byte aligned");
    static_assert(BAR_OFF % 8 == 0 && MISC_OFF % 8 == 0, "mbarrier objects are 8-byte aligned");
    static_assert(P_TBUFS * P_TSTRIDE <= TMEM_COLS && P_BN <= P_TSTRIDE, "TMEM allocation");
    static_assert(B_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(P_BN == 2 * P_BHALF && P_BN % 64 == 0, "B halves; 64-column groups never straddle a 128-column scale block");
    static_assert(STG_BYTES >= 2 * DG_MAX_M_BLOCKS, "run scratch fits in the staging buffer");
    static_assert(64 + 4 * (P_THREADS / 32) <= MISC_BYTES, "scan scratch");
    static_assert(TOTAL <= 232448, "shared memory");
};

struct PairTile {
    int e;       // expert / group
    int nb;      // output column tile (P_BN columns)
    int row0;    // this CTA's first row: Contiguous global row, Masked row within the group
    int valid;   // Masked: valid rows of this CTA's block
    bool blk_ok; // this CTA's m-block belongs to the run
};

// Tiles of a run: ceil(L / 2) m-pairs (fastest) x num_nb column tiles.
template <Layout L>
__device__ __forceinline__ PairTile decode_pair(int t, const RunTable& rt, int R, uint32_t rank, const GemmArgs& a) {
    const int r = find_run(rt.prefix, R, t);
    const int local = t - rt.prefix[r];
    const int Lr = rt.L[r];
    const int pairs = (Lr + 1) >> 1;
    const int nb = local / pairs, j = local - nb * pairs;
    const int blk = 2 * j + static_cast<int>(rank);
    PairTile ti;
    ti.e = rt.e[r];
    ti.nb = nb;
    ti.blk_ok = blk < Lr;
    ti.valid = 0;
    if constexpr (L == Layout::Contiguous) {
        ti.row0 = (rt.first[r] + blk) * BM;
        if (a.psum) {
            const int v = rt.x[r] - ti.row0;
            ti.valid = (!ti.blk_ok || v < 0) ? 0 : (v < BM ? v : BM);
        }
    } else {
        ti.row0 = blk * BM;
        const int v = rt.x[r] - ti.row0;
        ti.valid = v < 0 ? 0 : (v < BM ? v : BM);
    }
    return ti;
}

template <Layout L, bool SF_UE8M0>
__global__ void __launch_bounds__(P_THREADS, 1)
    k_grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD8,
                        const GemmArgs a) {
    using P = PairPlan;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);  // same offsets in both CTAs

    uint8_t* ring = smem + P::RING_OFF;
    uint8_t* stg = smem + P::STG_OFF;
    const RunTable rt = RunTable::at(smem + P::SCHED_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::BAR_OFF);
    uint64_t* full = bars;
    uint64_t* empty = bars + P_STAGES;
    uint64_t* tfull = bars + 2 * P_STAGES;
    uint64_t* tempty = tfull + P_TBUFS;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + P::MISC_OFF);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + P::MISC_OFF + 4);
    int* s_ntiles = reinterpret_cast<int*>(smem + P::MISC_OFF + 12);
    uint32_t* s_ballot = reinterpret_cast<uint32_t*>(smem + P::MISC_OFF + 32);  // [2][4]
    int* s_scan = reinterpret_cast<int*>(smem + P::MISC_OFF + 64);              // [P_THREADS / 32]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const WaitCtx wc{a.status, s_abort, a.wait_limit_ns};

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < P_TBUFS; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 2 * P_EPI_WARPS);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == P_MMA_WARP) {
        tmem_alloc_pair(s_tmem, P::TMEM_COLS);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    if (warp == P_PRODUCER_WARP && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmD);
        prefetch_tmap(&tmD8);
    }
    pdl_trigger();
    pdl_wait();  // every earlier kernel of the stream has finished: inputs are visible
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any signal crosses the pair

    // ---------------------------------------------------------------- tile schedule
    const int R = build_runs<L, P_THREADS>(a, rt, s_scan, stg);  // staging is free during set-up
    const int num_tiles = tile_prefix<P_THREADS, 2>(R, a.num_nb, rt, s_scan, s_ntiles);
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(cluster_count_x());

    // ---------------------------------------------------------------- roles
    if (warp == P_PRODUCER_WARP) {
        if (lane == 0 && num_tiles > 0) {
            const uint32_t full0 = mapa_shared(smem_u32(full), 0);  // the even CTA's full[0]
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int t = cid; t < num_tiles && ok; t += ncl) {
                const PairTile ti = decode_pair<L>(t, rt, R, rank, a);
                const int brow = ti.nb * P_BN + static_cast<int>(rank) * P_BHALF;
                for (int kb = 0; kb < a.KB; ++kb) {
                    if (!mbar_wait_cl(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
                    uint8_t* sa = ring + stage * P::STAGE_BYTES;
                    uint8_t* sb = sa + P::A_BYTES;
                    const uint32_t fb = full0 + static_cast<uint32_t>(stage) * 8u;
                    if (leader) mbar_arrive_expect_tx(&full[stage], 2 * P::STAGE_BYTES);
                    if constexpr (L == Layout::Masked)
                        tma_load_3d_pair(sa, &tmA, fb, kb * BK, ti.row0, ti.e);
                    else
                        tma_load_2d_pair(sa, &tmA, fb, kb * BK, ti.row0);
                    tma_load_3d_pair(sb, &tmB, fb, kb * BK, brow, ti.e);
                    ++issued;
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            // drain: the MMA has consumed every stage this thread filled, so all its loads landed
            const int n_drain = issued < P_STAGES ? issued : P_STAGES;
            for (int i = 0; i < n_drain; ++i) {
                int s = stage - 1 - i;
                uint32_t ph = phase;
                while (s < 0) { s += P_STAGES; ph ^= 1u; }
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait_cl(&empty[s], ph)) {
                    if (globaltimer_ns() - t0 > a.wait_limit_ns) break;
                }
            }
        }
        __syncwarp();
    } else if (warp >= P_MMA_WARP && warp < P_MMA_WARP + P_MMA_WARPS) {
        // Two issuers in the even CTA take alternate 128-K blocks (block number n of the pair), as
        // in the single-CTA kernel: while one is blocked issuing, the other has passed its waits.
        // Each waits for its TMEM buffer before its stage: with an odd stage count a stage's uses
        // alternate between the issuers, and the buffer wait (after the in-order promotion of block
        // n - TBUFS) orders the stage's previous use first.
        static_assert(P_STAGES % P_MMA_WARPS == 0 || P_TBUFS <= P_STAGES - 1, "stage phase order");
        static_assert(P_TBUFS % P_MMA_WARPS == 0, "one issuer per TMEM buffer");
        const uint32_t me = static_cast<uint32_t>(warp - P_MMA_WARP);
        if (leader && lane == 0 && num_tiles > 0) {
            bool ok = true, any = false;
            int last_tb = 0;
            uint32_t last_tphase = 0;
            uint32_t n = 0;
            constexpr uint32_t IDESC = idesc_e4m3_f32(2 * BM, P_BN);
            for (int t = cid; t < num_tiles && ok; t += ncl) {
                for (int kb = 0; kb < a.KB; ++kb, ++n) {
                    if (n % P_MMA_WARPS != me) continue;
                    const int stage = static_cast<int>(n % P_STAGES);
                    const uint32_t phase = (n / P_STAGES) & 1u;
                    const int tb = static_cast<int>(n % P_TBUFS);
                    const uint32_t tphase = (n / P_TBUFS) & 1u;
                    if (!mbar_wait_cl(&tempty[tb], tphase ^ 1u, wc)) { ok = false; break; }
                    if (!mbar_wait_cl(&full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(ring + stage * P::STAGE_BYTES);
                    const uint32_t sb = sa + P::A_BYTES;
                    const uint32_t dt = tmem_base + static_cast<uint32_t>(tb * P_TSTRIDE);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_e4m3_pair(dt, sdesc_k_sw128(sa + 32 * k), sdesc_k_sw128(sb + 32 * k), IDESC,
                                       k > 0 ? 1u : 0u);
                    umma_commit_pair(&empty[stage], 3);
                    umma_commit_pair(&tfull[tb], 3);
                    any = true;
                    last_tb = tb;
                    last_tphase = tphase;
                }
            }
            if (any) {
                // this issuer's last commit: every MMA it issued has completed
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait_cl(&tfull[last_tb], last_tphase)) {
                    if (globaltimer_ns() - t0 > a.wait_limit_ns) break;
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ promotion + store
        const int q = warp & 3;    // TMEM lane quarter
        const int cg = warp >> 2;  // 64-column group
        const int row = q * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);  // the even CTA's tempty[0]
        int tb = 0;
        uint32_t tphase = 0;
        bool have_store = false;
        int parity_slot = 0;
        for (int t = cid; t < num_tiles; t += ncl) {
            const PairTile ti = decode_pair<L>(t, rt, R, rank, a);
            bool failed = false;
            bool row_ok = false;
            int64_t grow = 0;
            if constexpr (L == Layout::Masked) {
                row_ok = row < ti.valid;
                grow = static_cast<int64_t>(ti.e) * a.M + ti.row0 + row;
            } else if (a.psum) {
                grow = static_cast<int64_t>(ti.row0) + row;
                row_ok = row < ti.valid;
            } else {
                grow = static_cast<int64_t>(ti.row0) + row;
                const int mi = (ti.blk_ok && grow < a.M) ? a.routing[grow] : -1;
                row_ok = (mi == ti.e);
                if (mi >= 0 && mi != ti.e) status_or(a.status, DG_STATUS_BAD_INDEX);
                const uint32_t bal = __ballot_sync(0xffffffffu, row_ok);
                if (cg == 0 && lane == 0) s_ballot[parity_slot * 4 + q] = bal;
            }
            const int64_t col0 = static_cast<int64_t>(ti.nb) * P_BN + cg * P_CPT;
            const bool col_ok = col0 < a.N;
            const bool use = row_ok && col_ok;

            float acc[P_CPT];
#pragma unroll
            for (int i = 0; i < P_CPT; ++i) acc[i] = 0.0f;

            // scales in registers, P_SF_GROUP blocks at a time, the next group in flight
            const int64_t sbi0 = (static_cast<int64_t>(ti.e) * a.n128 + col0 / 128) * a.KB;
            // raw scale bits (fp32, or the UE8M0 byte): converted where used, so that no
            // instruction waits on the loads until the group's first block is promoted
            auto load_group = [&](int g, uint32_t (&sa)[P_SF_GROUP], uint32_t (&sb)[P_SF_GROUP]) {
#pragma unroll
                for (int u = 0; u < P_SF_GROUP; ++u) {
                    const int kbi = g * P_SF_GROUP + u;
                    sa[u] = 0u;
                    sb[u] = 0u;
                    if (use && kbi < a.KB) {
                        const int64_t idx = static_cast<int64_t>(kbi) * a.sfa_ld + grow;
                        if constexpr (SF_UE8M0) {
                            sa[u] = __ldg(static_cast<const uint8_t*>(a.sfa) + idx);
                            sb[u] = __ldg(static_cast<const uint8_t*>(a.sfb) + sbi0 + kbi);
                        } else {
                            sa[u] = __float_as_uint(__ldg(static_cast<const float*>(a.sfa) + idx));
                            sb[u] = __float_as_uint(__ldg(static_cast<const float*>(a.sfb) + sbi0 + kbi));
                        }
                    }
                }
            };
            auto scale_of = [&](uint32_t sa, uint32_t sb) -> float {
                if constexpr (SF_UE8M0)
                    return ue8m0_to_float(static_cast<uint8_t>(sa)) * ue8m0_to_float(static_cast<uint8_t>(sb));
                else
                    return __uint_as_float(sa) * __uint_as_float(sb);
            };
            uint32_t sa_c[P_SF_GROUP], sb_c[P_SF_GROUP], sa_n[P_SF_GROUP], sb_n[P_SF_GROUP];
            load_group(0, sa_c, sb_c);
            load_group(1, sa_n, sb_n);
            for (int kb0 = 0; kb0 < a.KB && !failed; kb0 += P_SF_GROUP) {
#pragma unroll
                for (int u = 0; u < P_SF_GROUP; ++u) {
                    if (kb0 + u >= a.KB) break;
                    const float s = scale_of(sa_c[u], sb_c[u]);
                    if (!mbar_wait_cl(&tfull[tb], tphase, wc)) { failed = true; break; }
                    tc_fence_after();
                    const uint32_t tcol = tmem_base + t_lane + static_cast<uint32_t>(tb * P_TSTRIDE + cg * P_CPT);
                    uint32_t v[32];
                    tmem_ld_x32(tcol, v);
                    tmem_wait_ld(v);
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        ffma2(acc[i], acc[i + 1], s, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                    tmem_ld_x32(tcol + 32, v);
                    tmem_wait_ld(v);
                    // both halves are in registers: hand the TMEM buffer back before the FMAs
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(tb) * 8u);
                    if (++tb == P_TBUFS) { tb = 0; tphase ^= 1u; }
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        ffma2(acc[32 + i], acc[32 + i + 1], s, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                }
#pragma unroll
                for (int u = 0; u < P_SF_GROUP; ++u) {
                    sa_c[u] = sa_n[u];
                    sb_c[u] = sb_n[u];
                }
                load_group(kb0 / P_SF_GROUP + 2, sa_n, sb_n);
            }

            // ---- stage the tile in shared memory (chunk cg, row `row`: this thread's 64 columns)
            if (tid == 0 && have_store) bulk_wait_read_all();  // the previous store has read the staging
            named_bar_sync(P_EPI_BAR, P_EPI_WARPS * 32);
            if (!failed) {
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    uint8_t* dst = stg + cg * P::CHUNK_BYTES + row * 128 + ((p ^ (row & 7)) << 4);
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[8 * p + 2 * i], acc[8 * p + 2 * i + 1]);
                        w[i] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            fence_async_smem();
            if (bar_or(P_EPI_BAR, P_EPI_WARPS * 32, failed || *s_abort != 0)) break;

            // ---- store: TMA for the leading 8-row-aligned valid rows, owner threads for the rest
            int v = 0;
            if (L == Layout::Masked || a.psum) {
                v = ti.valid;
            } else {
                for (int qq = 0; qq < 4; ++qq) {
                    const uint32_t bal = s_ballot[parity_slot * 4 + qq];
                    if (bal == 0xffffffffu) { v += 32; continue; }
                    v += __ffs(~bal) - 1;
                    break;
                }
            }
            const int v8 = v & ~7;
            if (tid == 0 && v8 > 0) {
                for (int c = 0; c < P::CHUNKS; ++c) {
                    const int x = ti.nb * P_BN + c * 64;
                    if (x >= a.N) break;
                    const uint8_t* src = stg + c * P::CHUNK_BYTES;
                    if (v8 == BM) {
                        if constexpr (L == Layout::Contiguous) tma_store_2d(&tmD, src, x, ti.row0);
                        else tma_store_3d(&tmD, src, x, ti.row0, ti.e);
                    } else {
                        for (int r8 = 0; r8 < v8; r8 += 8) {
                            if constexpr (L == Layout::Contiguous)
                                tma_store_2d(&tmD8, src + r8 * 128, x, ti.row0 + r8);
                            else
                                tma_store_3d(&tmD8, src + r8 * 128, x, ti.row0 + r8, ti.e);
                        }
                    }
                }
                bulk_commit();
                have_store = true;
            }
            if (use && row >= v8) {
                uint8_t* dst = static_cast<uint8_t*>(a.d) + (grow * a.ldd + col0) * 2;
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[8 * p + 2 * i], acc[8 * p + 2 * i + 1]);
                        w[i] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                    *reinterpret_cast<uint4*>(dst + 16 * p) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            parity_slot ^= 1;
        }
        if (tid == 0 && have_store) bulk_wait_all();
        __syncwarp();
    }

    __syncthreads();
    cluster_sync();  // neither CTA leaves while its partner may still signal its barriers
    if (warp == P_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, P::TMEM_COLS);
    }
}

// Co-resident clusters of one instantiation on the current device (cached per device).
template <Layout L, bool UE8M0>
int pair_clusters(int* out) {
    static std::atomic<int> cache[64];
    int dev = 0;
    DG_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) { *out = c; return DG_OK; }
    }
    int sms = 0;
    if (int rc = device_sm_count(&sms)) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms / 2 * 2));
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = PairPlan::TOTAL;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    DG_CHECK_CUDA(cudaOccupancyMaxActiveClusters(&n, k_grouped_gemm_pair<L, UE8M0>, &cfg));
    if (n < 1) return set_error(DG_ERR_UNSUPPORTED, "no CTA pair of the m-grouped kernel fits on this device");
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return DG_OK;
}

template <Layout L, bool UE8M0>
int launch_pair_t(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tD, const CUtensorMap& tD8,
                  const GemmArgs& args, cudaStream_t stream) {
    auto kern = k_grouped_gemm_pair<L, UE8M0>;
    // The attribute is per device: set it on every call (cheap, host-only, capture-safe).
    DG_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PairPlan::TOTAL));
    int ncl = 0;
    if (int rc = pair_clusters<L, UE8M0>(&ncl)) return rc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * ncl));
    cfg.blockDim = dim3(P_THREADS);
    cfg.dynamicSmemBytes = PairPlan::TOTAL;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tA, tB, tD, tD8, args);
    if (e != cudaSuccess) return set_error(DG_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return DG_OK;
}

}  // namespace

int launch_mgrouped_pair(Layout L, bool sf_ue8m0, const CUtensorMap& tA, const CUtensorMap& tB,
                         const CUtensorMap& tD, const CUtensorMap& tD8, GemmArgs args, void* stream) {
    args.num_nb = static_cast<int>((args.N + P_BN - 1) / P_BN);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (L == Layout::Masked) {
        if (sf_ue8m0) return launch_pair_t<Layout::Masked, true>(tA, tB, tD, tD8, args, s);
        return launch_pair_t<Layout::Masked, false>(tA, tB, tD, tD8, args, s);
    }
    if (sf_ue8m0) return launch_pair_t<Layout::Contiguous, true>(tA, tB, tD, tD8, args, s);
    return launch_pair_t<Layout::Contiguous, false>(tA, tB, tD, tD8, args, s);
}

}  // namespace dg
