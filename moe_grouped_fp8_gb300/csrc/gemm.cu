// gemm.cu - persistent, warp-specialised FP8 (e4m3) m-grouped GEMM for sm_103a.
//
// One kernel template serves the two m-grouped layouts of the source pages:
//   Contiguous - rows stacked per expert, routed by m_indices (-1 = padding row), segments
//                aligned to 128 rows ("SM120 m_grouped_fp8 contiguous kernel: illegal memory
//                access at CUDA graph replay", #444);
//   Masked     - [G, cap, K] activations with a valid-row count per expert ("Fix cross-expert
//                output overwrites in SM90 masked GEMM", #469).
// (The k-grouped weight-gradient GEMM lives in kgrouped.cu.)
//
// Roles (EW promotion warps + 3): warps 0..EW-1 promote and store (TMEM lane quarter = warp % 4,
// column group = warp / 4; EW = 8 for 128-column tiles, 16 for 256-column tiles, so that a thread
// always holds 64 accumulators), warp EW issues TMA loads, warps EW+1 and EW+2 issue tcgen05.mma on
// alternate 128-K blocks (warp EW+1 owns tensor memory).
// Per 128-K block the MMA writes a fresh fp32 partial P into one of the TMEM buffers; the
// promotion warps read it (tcgen05.ld) and accumulate acc += sfa * sfb * P in fp32 registers
// while the tensor core fills the next buffer.  The K order is fixed, there is no split-K
// and no atomic on outputs, so every call is bitwise reproducible.
//
// The tile schedule is rebuilt in shared memory by every CTA from the device-side routing
// tensor (m_indices / counts) at the start of every launch, and the TMA descriptors are static
// kernel parameters, so a CUDA graph replayed after the routing tensor changed in place never
// uses stale schedule or descriptor state.
//
// Outputs: with long K the epilogue stages the tile in shared memory (128-byte swizzle) and
// stores rows [0, 8*floor(v/8)) of the tile's v valid leading rows with TMA boxes of 128 or 8
// rows through a descriptor that keeps the expert dimension (3-D [G, cap, N] for the masked
// layout), so a store can never cross into the next expert; the remaining valid rows are written
// by their owner threads.  With short K every valid row is written by its owner thread from
// registers.  Rows that are not valid are never written.
#include <cuda_bf16.h>

#include <atomic>

#include "host_common.hpp"
#include "kernel_common.cuh"
#include "mgrouped.cuh"
#include "ptx.cuh"

namespace dg {

constexpr int NUM_MMA_WARPS = 2;
// How a tile reaches the output: staged in shared memory and stored with TMA by thread 0 of the
// promotion warps (ST_THREAD0), or written from registers by each row's owner thread (ST_DIRECT:
// no staging buffer).
constexpr int ST_THREAD0 = 0, ST_DIRECT = 1;
// Threads of a CTA: EW promotion warps, the producer and two MMA issuers; with 16 promotion warps
// one idle warp completes the fifth warpgroup of the register split below.
template <int EW>
__host__ __device__ constexpr int num_threads() { return (EW + (EW == 16 ? 4 : 1 + NUM_MMA_WARPS)) * 32; }

// Register split of the 16-warp CTA (640 threads, 96 registers each at launch: an SM sub-partition
// holds 16384 registers and runs 5 of the 20 warps).  The control warpgroup (producer, MMA issuers,
// idle warp) gives registers back, the promotion warpgroups take them: per sub-partition
// 4 x 32 x (RS_PROMO - RS_LAUNCH) <= 32 x (RS_LAUNCH - RS_CONTROL), so every increase is covered by
// the decreases (an increase that the pool cannot cover would wait forever).  The host checks the
// compiled register count equals RS_LAUNCH before it launches.
constexpr int RS_LAUNCH = 96, RS_CONTROL = 40, RS_PROMO = 104;
static_assert(4 * (RS_PROMO - RS_LAUNCH) <= RS_LAUNCH - RS_CONTROL, "register split exceeds the pool");
static_assert(RS_LAUNCH * 640 <= 65536 && RS_LAUNCH * 5 * 32 <= 16384, "launch registers");
constexpr int EPI_BAR = 1;  // named barrier of the promotion/store threads


template <Layout L, int BN, int STAGES, bool OUT_FP32, bool STAGED, int EW>
struct Plan {
    // TMEM partial buffers (the tensor core runs up to TB - 1 blocks ahead of the promotion; 512
    // columns hold two 256-column or four 128-column buffers) and the 128-K blocks whose scales
    // a promotion thread prefetches together.
    static constexpr int TB = BN == 256 ? 2 : 4;
    static constexpr int SFG = BN == 256 ? 2 : 4;
    static constexpr int CGROUPS = EW / 4;             // column groups (warps per TMEM lane quarter)
    // Columns of the partial loaded per tcgen05.ld round: all 64 at once when the registers allow
    // (8 warps with 64 accumulators: 352 threads, 168 registers each), 16 beside 128 accumulators
    // (8 warps of a 128 x 256 tile), 16 with 16 warps (104 registers each after the split).
    static constexpr int RC = EW == 16 ? 16 : (BN / CGROUPS == 64 ? 64 : 16);
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int ESIZE = OUT_FP32 ? 4 : 2;
    static constexpr int CPT = BN / CGROUPS;           // output columns per promotion thread
    static constexpr int CHUNKS = BN * ESIZE / 128;    // 128-byte column chunks of a tile row
    static constexpr int CHUNK_BYTES = BM * 128;
    static constexpr int STG_BYTES = STAGED ? CHUNKS * CHUNK_BYTES : 0;
    static constexpr int RING_OFF = 0;
    static constexpr int STG_OFF = STAGES * STAGE_BYTES;
    static constexpr int SCHED_OFF = STG_OFF + STG_BYTES;
    static constexpr int BAR_OFF = (SCHED_OFF + SCHED_BYTES + 127) / 128 * 128;  // mbarriers: 8-byte aligned
    static constexpr int NUM_BARS = 2 * STAGES + 2 * TB;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int MISC_BYTES = 256;
    static constexpr int TOTAL = MISC_OFF + MISC_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = TB * BN;
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
    static_assert(CPT % 32 == 0, "promotion threads read 32-column groups");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(STG_OFF % 1024 == 0 && SCHED_OFF % 1024 == 0, "TMA / swizzle buffers are 1024-byte aligned");
    static_assert(BAR_OFF % 8 == 0 && MISC_OFF % 8 == 0, "mbarrier objects are 8-byte aligned");
    static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation: power of two <= 512");
    static_assert(CPT % RC == 0 && (RC == 16 || RC % 32 == 0), "promotion rounds of whole loads");
    static_assert(EW == 8 || EW == 16, "promotion warps");
    static_assert(BN == 128 || (BN == 256 && !OUT_FP32), "256-column tiles stage bf16 output only");
    static_assert(TOTAL <= 232448, "shared memory");
};

// ------------------------------------------------------------------------- the kernel

template <Layout L, int BN, int STAGES, bool OUT_FP32, bool SF_UE8M0, int SM, int EW>
__global__ void __launch_bounds__(num_threads<EW>(), 1)
    k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD8,
                   const GemmArgs a) {
    constexpr bool DIRECT = SM == ST_DIRECT;
    using P = Plan<L, BN, STAGES, OUT_FP32, !DIRECT, EW>;
    constexpr int NUM_THREADS = num_threads<EW>();
    constexpr int NUM_EPI_WARPS = EW;
    constexpr int PRODUCER_WARP = EW;
    constexpr int MMA_WARP = EW + 1;  // and MMA_WARP + 1: the two MMA issuers
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

    uint8_t* ring = smem + P::RING_OFF;
    uint8_t* stg = smem + P::STG_OFF;
    const RunTable rt = RunTable::at(smem + P::SCHED_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P::BAR_OFF);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + P::TB;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + P::MISC_OFF);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + P::MISC_OFF + 4);
    int* s_ntiles = reinterpret_cast<int*>(smem + P::MISC_OFF + 12);
    uint32_t* s_ballot = reinterpret_cast<uint32_t*>(smem + P::MISC_OFF + 32);  // [2][4]
    int* s_scan = reinterpret_cast<int*>(smem + P::MISC_OFF + 64);              // [NUM_THREADS / 32]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const WaitCtx wc{a.status, s_abort, a.wait_limit_ns};

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < P::TB; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], NUM_EPI_WARPS);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(s_tmem, P::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == PRODUCER_WARP && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmD);
        prefetch_tmap(&tmD8);
    }
    pdl_trigger();
    pdl_wait();  // every earlier kernel of the stream has finished: inputs are visible
    __syncthreads();

    // ---------------------------------------------------------------- tile schedule
    // scratch: the staging buffer (or, without one, the ring) is free during set-up
    const int R = build_runs<L, NUM_THREADS>(a, rt, s_scan, DIRECT ? ring : stg);
    const int num_tiles = tile_prefix<NUM_THREADS, 1>(R, a.num_nb, rt, s_scan, s_ntiles);
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    // TMA stores of a staged tile: the leading v8 valid rows (a multiple of 8)
    auto issue_stores = [&](const TileInfo& ti, int v8) {
        for (int c = 0; c < P::CHUNKS; ++c) {
            const uint8_t* src = stg + c * P::CHUNK_BYTES;
            const int x = ti.nb * BN + c * (128 / P::ESIZE);
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
    };

    // ---------------------------------------------------------------- roles
    // (each warpgroup changes its register limit before its roles' code, which it dominates)
    if (warp >= EW) {
    if constexpr (EW == 16) setmaxnreg_dec<RS_CONTROL>();
    if (warp == PRODUCER_WARP) {
        if (lane == 0 && R > 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile<L>(t, rt, R, a);
                for (int kb = 0; kb < ti.kbt; ++kb) {
                    if (!mbar_wait_inl(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
#if DG_DEBUG
                    // debug build, test hook: the producer stops as if stalled, so the MMA issuers'
                    // bounded waits for this stage run out and the CTA takes its abort path
                    if (blockIdx.x == 0 && a.dbg_stop_at > 0 && issued + 1 == a.dbg_stop_at) { ok = false; break; }
#endif
                    uint8_t* sa = ring + stage * P::STAGE_BYTES;
                    uint8_t* sb = sa + P::A_BYTES;
                    mbar_arrive_expect_tx(&full[stage], P::STAGE_BYTES);
                    if constexpr (L == Layout::Masked)
                        tma_load_3d(sa, &tmA, &full[stage], kb * BK, ti.row0, ti.e);
                    else
                        tma_load_2d(sa, &tmA, &full[stage], kb * BK, ti.row0);
                    tma_load_3d(sb, &tmB, &full[stage], kb * BK, ti.nb * BN, ti.e);
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
    } else if (warp >= MMA_WARP && warp < MMA_WARP + NUM_MMA_WARPS) {
        // Two issuers take alternate 128-K blocks (global block number n of this CTA): an issue
        // blocks until the tensor core has taken the MMAs, so while one issuer is blocked the
        // other has already passed its barrier waits and queues its block at once.  A commit
        // tracks only its own thread's MMAs, so each issuer signals its own blocks' barriers.
        const uint32_t me = static_cast<uint32_t>(warp - MMA_WARP);
        if (lane == 0 && R > 0) {
            bool ok = true, any = false;
            int last_tb = 0;
            uint32_t last_tphase = 0;
            uint32_t n = 0;
            constexpr uint32_t IDESC = idesc_e4m3_f32(BM, BN);
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const TileInfo ti = decode_tile<L>(t, rt, R, a);
                for (int kb = 0; kb < ti.kbt; ++kb, ++n) {
                    if (n % NUM_MMA_WARPS != me) continue;
                    const int stage = static_cast<int>(n % STAGES);
                    const uint32_t phase = (n / STAGES) & 1u;
                    const int tb = static_cast<int>(n % P::TB);
                    const uint32_t tphase = (n / P::TB) & 1u;
                    // Order matters.  With an odd stage count a stage's consecutive uses alternate
                    // between the issuers, and a parity wait cannot tell phase k from k + 2, so
                    // the full wait of block n is sound only once block n - STAGES has taken its
                    // phase.  Waiting for the TMEM buffer first ensures that: it comes back after
                    // the promotion of block n - TB, which runs after block n - TB - 1 >= n - STAGES
                    // (TB <= STAGES - 1) was promoted, hence after its MMA consumed the stage.
                    // (Each TMEM buffer belongs to one issuer, which consumes its phases in order.)
                    static_assert(STAGES % NUM_MMA_WARPS == 0 || P::TB <= STAGES - 1, "stage phase order");
                    static_assert(P::TB % NUM_MMA_WARPS == 0, "one issuer per TMEM buffer");
                    if (!mbar_wait_inl(&tempty[tb], tphase ^ 1u, wc)) { ok = false; break; }
                    if (!mbar_wait_inl(&full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(ring + stage * P::STAGE_BYTES);
                    const uint32_t sb = sa + P::A_BYTES;
                    const uint32_t dt = tmem_base + static_cast<uint32_t>(tb * BN);
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_e4m3(dt, sdesc_k_sw128(sa + 32 * k), sdesc_k_sw128(sb + 32 * k), IDESC, k > 0 ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    umma_commit(&tfull[tb]);
                    any = true;
                    last_tb = tb;
                    last_tphase = tphase;
                }
            }
            // this issuer's last commit: the tensor core is done with every MMA it issued
            if (any) drain_wait(&tfull[last_tb], last_tphase, a.drain_limit_ns);
        }
        __syncwarp();
    }
    } else {
        // ------------------------------------------------------------ promotion + staging
        if constexpr (EW == 16) setmaxnreg_inc<RS_PROMO>();
        const int q = warp & 3;       // TMEM lane quarter
        const int h2 = warp >> 2;     // column group
        const int row = q * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        int tb = 0;
        uint32_t tphase = 0;
        int parity_slot = 0;
        int tix = 0;  // this CTA's tile count so far
        bool have_store = false;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const TileInfo ti = decode_tile<L>(t, rt, R, a);
            bool failed = false;
            // With m_indices routing and short K (owner-thread stores) a row's scales are loaded
            // whether or not the row is valid (an invalid row's result is never stored), so that
            // they do not wait for the row's routing entry: tiles of a few valid rows spend most
            // of their time in such hand-offs (many-expert w2 at 1 token per expert: -11%).  With
            // long K the waiting is hidden and the extra live registers cost more (+1-4%).
            constexpr bool EARLY_SCALES = L == Layout::Contiguous && DIRECT;
            bool row_ok = false, row_in = false;
            int64_t grow = 0;
            int mi = -1;
            if constexpr (L == Layout::Masked) {
                row_ok = row < ti.valid;
                grow = static_cast<int64_t>(ti.e) * a.M + ti.row0 + row;
            } else if (a.psum) {
                grow = static_cast<int64_t>(ti.row0) + row;
                row_ok = row < ti.valid;
            } else {
                grow = static_cast<int64_t>(ti.row0) + row;
                row_in = grow < a.M;
                mi = row_in ? a.routing[grow] : -1;
                if constexpr (!EARLY_SCALES) {
                    row_ok = (mi == ti.e);
                    if (mi >= 0 && mi != ti.e) status_or(a.status, DG_STATUS_BAD_INDEX);
                    const uint32_t bal = __ballot_sync(0xffffffffu, row_ok);
                    if (h2 == 0 && lane == 0) s_ballot[parity_slot * 4 + q] = bal;
                }
            }
            // the rows whose scales are loaded
            const bool row_sc = (EARLY_SCALES && !a.psum) ? row_in : row_ok;

            float acc[P::CPT];
#pragma unroll
            for (int i = 0; i < P::CPT; ++i) acc[i] = 0.0f;

            // Scales travel in registers, P::SFG 128-K blocks at a time (2 for 256-column tiles, 4
            // for 128): while the blocks of group g are promoted, the loads of group g + 1 are in
            // flight (issued one group earlier).
            const int sbi0 = (ti.e * a.n128 + (ti.nb * BN + h2 * P::CPT) / 128) * a.KB;
            // raw scale bits (fp32, or the UE8M0 byte): converted where used, so that no
            // instruction waits on the loads until the group's first block is promoted
            auto load_group = [&](int g, uint32_t (&sa)[P::SFG], uint32_t (&sb)[P::SFG]) {
#pragma unroll
                for (int u = 0; u < P::SFG; ++u) {
                    const int kbi = g * P::SFG + u;
                    sa[u] = 0u;
                    sb[u] = 0u;
                    if (row_sc && kbi < ti.kbt && DG_CHECKED(sfa_in<L>(a, kbi, grow), DG_DEBUG_A_SCALE) &&
                        DG_CHECKED(sfb_in(a, ti.e, (ti.nb * BN + h2 * P::CPT) / 128, kbi), DG_DEBUG_B_SCALE)) {
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
            uint32_t sa_c[P::SFG], sb_c[P::SFG], sa_n[P::SFG], sb_n[P::SFG];
            load_group(0, sa_c, sb_c);
            load_group(1, sa_n, sb_n);
            if constexpr (EARLY_SCALES) {
                if (!a.psum) {
                    row_ok = (mi == ti.e);
                    if (mi >= 0 && mi != ti.e) status_or(a.status, DG_STATUS_BAD_INDEX);
                    const uint32_t bal = __ballot_sync(0xffffffffu, row_ok);
                    if (h2 == 0 && lane == 0) s_ballot[parity_slot * 4 + q] = bal;
                }
            }
            for (int kb0 = 0; kb0 < ti.kbt && !failed; kb0 += P::SFG) {
#pragma unroll
                for (int u = 0; u < P::SFG; ++u) {
                    if (kb0 + u >= ti.kbt) break;
                    const float s = scale_of(sa_c[u], sb_c[u]);
                    if (!mbar_wait_inl(&tfull[tb], tphase, wc)) { failed = true; break; }
                    tc_fence_after();
                    // P::RC columns per round: the round's loads, one wait, then (after the last
                    // round) the TMEM buffer goes back to the MMA issuers before the round's FMAs
#pragma unroll
                    for (int c0 = 0; c0 < P::CPT; c0 += P::RC) {
                        constexpr int W = P::RC < 32 ? P::RC : 32;  // columns per tcgen05.ld
                        uint32_t v[P::RC / W][W];
                        const uint32_t col = tmem_base + t_lane + static_cast<uint32_t>(tb * BN + h2 * P::CPT + c0);
#pragma unroll
                        for (int c2 = 0; c2 < P::RC / W; ++c2) tmem_ld(col + c2 * W, v[c2]);
#pragma unroll
                        for (int c2 = 0; c2 < P::RC / W; ++c2) tmem_wait_ld(v[c2]);
                        if (c0 + P::RC == P::CPT) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&tempty[tb]);
                            if (++tb == P::TB) { tb = 0; tphase ^= 1u; }
                        }
#pragma unroll
                        for (int c2 = 0; c2 < P::RC / W; ++c2)
#pragma unroll
                            for (int i = 0; i < W; i += 2)
                                ffma2(acc[c0 + c2 * W + i], acc[c0 + c2 * W + i + 1], s, __uint_as_float(v[c2][i]),
                                      __uint_as_float(v[c2][i + 1]));
                    }
                }
#pragma unroll
                for (int u = 0; u < P::SFG; ++u) {
                    sa_c[u] = sa_n[u];
                    sb_c[u] = sb_n[u];
                }
                load_group(kb0 / P::SFG + 2, sa_n, sb_n);
            }

            // ---- accumulate: D = C + result (fp32 output; C may alias D: each element is read by
            // the thread that later writes it, before any store of this tile)
            if constexpr (OUT_FP32) {
                if (a.c != nullptr && row_ok && !failed &&
                    DG_CHECKED(out_in<L>(a, grow, static_cast<int64_t>(ti.nb) * BN + h2 * P::CPT, P::CPT),
                               DG_DEBUG_OUT)) {
                    const float* crow = a.c + grow * a.ldd + static_cast<int64_t>(ti.nb) * BN + h2 * P::CPT;
#pragma unroll
                    for (int i = 0; i < P::CPT; i += 4) {
                        const float4 v = *reinterpret_cast<const float4*>(crow + i);
                        acc[i] += v.x;
                        acc[i + 1] += v.y;
                        acc[i + 2] += v.z;
                        acc[i + 3] += v.w;
                    }
                }
            }

            // this thread's row of the tile (CPT columns), written from registers
            auto store_own_row = [&]() {
                if (!DG_CHECKED(out_in<L>(a, grow, static_cast<int64_t>(ti.nb) * BN + h2 * P::CPT, P::CPT),
                                DG_DEBUG_OUT))
                    return;
                uint8_t* dst = static_cast<uint8_t*>(a.d) +
                               ((grow * a.ldd) + ti.nb * BN + h2 * P::CPT) * static_cast<int64_t>(P::ESIZE);
                constexpr int PIECES = P::CPT * P::ESIZE / 16;
#pragma unroll
                for (int p = 0; p < PIECES; ++p) {
                    if constexpr (OUT_FP32) {
                        *reinterpret_cast<float4*>(dst + 16 * p) =
                            make_float4(acc[4 * p], acc[4 * p + 1], acc[4 * p + 2], acc[4 * p + 3]);
                    } else {
                        uint32_t w[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const __nv_bfloat162 h = __floats2bfloat162_rn(acc[8 * p + 2 * i], acc[8 * p + 2 * i + 1]);
                            w[i] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                        *reinterpret_cast<uint4*>(dst + 16 * p) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            };

            if constexpr (DIRECT) {
                // ---- every valid row by its owner thread; no barrier: a failed wait ends this
                // warp's loop, and the abort flag ends the others' waits
                if (failed || *s_abort != 0) break;
                if (row_ok) store_own_row();
            } else {
                // ---- stage the tile in shared memory once the previous tile's stores have read it
                if (tid == 0 && tix > 0) bulk_wait_read_all();
                named_bar_sync(EPI_BAR, NUM_EPI_WARPS * 32);
                if (!failed) {
                    constexpr int PIECES = P::CPT * P::ESIZE / 16;
#pragma unroll
                    for (int p = 0; p < PIECES; ++p) {
                        const int off = h2 * P::CPT * P::ESIZE + 16 * p;  // byte offset in the tile row
                        const int chunk = off >> 7, j = (off & 127) >> 4;
                        uint8_t* dst = stg + chunk * P::CHUNK_BYTES + row * 128 + ((j ^ (row & 7)) << 4);
                        if constexpr (OUT_FP32) {
                            *reinterpret_cast<float4*>(dst) =
                                make_float4(acc[4 * p], acc[4 * p + 1], acc[4 * p + 2], acc[4 * p + 3]);
                        } else {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const __nv_bfloat162 h = __floats2bfloat162_rn(acc[8 * p + 2 * i], acc[8 * p + 2 * i + 1]);
                                w[i] = *reinterpret_cast<const uint32_t*>(&h);
                            }
                            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                fence_async_smem();
                if (bar_or(EPI_BAR, NUM_EPI_WARPS * 32, failed || *s_abort != 0)) break;

                // ---- stores: TMA for the leading 8-row-aligned valid rows (issued by thread 0), owner
                // threads for the rest
                const int v8 = stored_rows<L>(ti, a, s_ballot + parity_slot * 4) & ~7;
                if (tid == 0 && v8 > 0) {
                    issue_stores(ti, v8);
                    have_store = true;
                }
                if (row_ok && row >= v8) store_own_row();
            }
            parity_slot ^= 1;
            ++tix;
        }
        if (SM == ST_THREAD0 && tid == 0 && have_store) bulk_wait_all();
        __syncwarp();
    }

    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, P::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------- host launchers

namespace {

// Tile stores.  With few 128-K blocks per tile the tile transitions dominate: staging the tile and
// the TMA store's shared-memory reads sit between one tile's last partial and the next tile's
// first.  Up to 32 blocks each row's owner thread writes it from registers (no staging, no wait
// on a store): the many-expert w2 shape (K = 256) 0.140 -> 0.124 ms at 113 tokens per expert,
// 0.067 -> 0.052 ms at 1, and even at K = 4096.  With long K the TMA stores issued by thread 0
// measured faster (decode, K = 7168).  Both write the same bits.
constexpr int DIRECT_MAX_KB = 32;
// testing: 0 automatic, 1 TMA stores issued by thread 0 of the promotion warps, 3 owner-thread stores
std::atomic<int> g_force_store{0};
// testing (debug build): the output rows the index checks let the stores reach; 0 = the layout's
std::atomic<int64_t> g_debug_out_rows{0};
// testing (debug build): CTA 0's producer stops before its n-th stage load; 0 = never
std::atomic<int> g_debug_stop_at{0};

int store_mode(int KB) {
    switch (g_force_store.load(std::memory_order_relaxed)) {
        case 1: return ST_THREAD0;
        case 3: return ST_DIRECT;
        default: return KB <= DIRECT_MAX_KB ? ST_DIRECT : ST_THREAD0;
    }
}

template <Layout L, int BN, int STAGES, bool OUT_FP32, bool SF_UE8M0, int SM, int EW>
int launch_gemm_sm(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tD, const CUtensorMap& tD8,
                   const GemmArgs& args, cudaStream_t stream) {
    using P = Plan<L, BN, STAGES, OUT_FP32, SM != ST_DIRECT, EW>;
    auto kern = k_grouped_gemm<L, BN, STAGES, OUT_FP32, SF_UE8M0, SM, EW>;
    // The attribute is per device: set it on every call (cheap, host-only, capture-safe).
    DG_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::TOTAL));
    if constexpr (EW == 16) {
        // the register split assumes the launch gives every thread RS_LAUNCH registers
        static int regs = 0;
        if (regs == 0) {
            cudaFuncAttributes fa{};
            DG_CHECK_CUDA(cudaFuncGetAttributes(&fa, kern));
            regs = fa.numRegs;
        }
        DG_CHECK_SUPPORTED(regs == RS_LAUNCH, "m-grouped kernel compiled for %d registers, its register split needs %d",
                           regs, RS_LAUNCH);
    }
    int sms = 0;
    if (int rc = device_sm_count(&sms)) return rc;
    return launch_pdl(kern, dim3(sms), dim3(num_threads<EW>()), P::TOTAL, stream, tA, tB, tD, tD8, args);
}

// Promotion warps of a 128 x 256 tile: 16 (64 accumulators per thread, the partial read in two
// 32-column rounds) or 8 (128 accumulators, eight 16-column rounds).  testing: 0 automatic.
std::atomic<int> g_force_warps{0};

template <Layout L, int BN, int STAGES, bool OUT_FP32, bool SF_UE8M0, int EW>
int launch_gemm_ew(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tD, const CUtensorMap& tD8,
                   const GemmArgs& args, cudaStream_t stream) {
    if (store_mode(args.KB) == ST_DIRECT)
        return launch_gemm_sm<L, BN, STAGES, OUT_FP32, SF_UE8M0, ST_DIRECT, EW>(tA, tB, tD, tD8, args, stream);
    return launch_gemm_sm<L, BN, STAGES, OUT_FP32, SF_UE8M0, ST_THREAD0, EW>(tA, tB, tD, tD8, args, stream);
}

template <Layout L, int BN, int STAGES, bool OUT_FP32, bool SF_UE8M0>
int launch_gemm(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tD, const CUtensorMap& tD8,
                const GemmArgs& args, cudaStream_t stream) {
    if constexpr (BN == 256) {
        if (g_force_warps.load(std::memory_order_relaxed) != 8)
            return launch_gemm_ew<L, BN, STAGES, OUT_FP32, SF_UE8M0, 16>(tA, tB, tD, tD8, args, stream);
    }
    return launch_gemm_ew<L, BN, STAGES, OUT_FP32, SF_UE8M0, 8>(tA, tB, tD, tD8, args, stream);
}

constexpr int MG_BN = 128;
constexpr int MG_STAGES = 4;
constexpr int MG_STAGES_BF16 = 5;
constexpr int MG_BN_WIDE = 256;      // bf16 output with N % 256 == 0: 128 x 256 tiles
constexpr int MG_STAGES_WIDE = 3;    // 48 KB stages

// Columns of a single-CTA tile: 256 when the output is bf16 and N is a multiple of 256 of at
// least 1024 (half the MMA instructions and TMEM handshakes per FLOP, 25% fewer operand bytes
// through shared memory; measured 0.408 -> 0.329 ms on the prefill shape, 0.478 -> 0.419 ms on
// decode), else 128 (narrow N: twice the tiles for the same weights, measured faster at N = 512).
// Both tile widths give bitwise the same results.
std::atomic<int> g_force_bn{0};  // testing: 0 automatic, else the tile width (128, or 256 when allowed)

int single_bn(int out, int64_t N) {
    const bool wide_ok = out == DG_OUT_BF16 && N % MG_BN_WIDE == 0;
    const int f = g_force_bn.load(std::memory_order_relaxed);
    if (f == MG_BN) return MG_BN;
    if (f == MG_BN_WIDE && wide_ok) return MG_BN_WIDE;
    return (wide_ok && N >= 4 * MG_BN_WIDE) ? MG_BN_WIDE : MG_BN;
}

CUtensorMapDataType out_tmap_type(int out) {
    return out == DG_OUT_FP32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// Kernel choice for UE8M0 scales: the block-scaled MMA kernel (gemm_mx.cu: the tensor core applies
// the power-of-two scales and accumulates the whole K of a 128 x 256 tile, no per-block promotion)
// when N % 256 == 0 and K has at least MX_MIN_KB blocks, else the promotion kernel above (fp32
// promotion per 128-K block; the only choice for fp32 scales).  Measured: the block-scaled kernel
// 0.704 ms against 0.812 ms on a compute-bound shape (8 x 4096 rows, N = 4096, K = 7168), equal or
// up to 4% faster on the many-expert w13 shapes (K = 4096); with K = 256 (w2) its single
// accumulator leaves the tensor core idle during each tile's drain and the promotion kernel wins.
// The two round differently (the tensor core's accumulation order against fp32 promotion), each
// within the oracle's tolerance.  testing: 0 automatic, 1 promotion, 2 block-scaled MMA wherever
// N % 256 == 0.
std::atomic<int> g_force_kernel{0};
constexpr int MX_MIN_KB = 16;

bool use_mx(int fmt, int64_t N, int64_t K) {
    if (fmt != DG_SF_UE8M0 || N % MX_BN != 0) return false;
    const int f = g_force_kernel.load(std::memory_order_relaxed);
    if (f == 1 || g_force_bn.load(std::memory_order_relaxed) == MG_BN) return false;
    return f == 2 || K / BK >= MX_MIN_KB;
}

// The element type of the weight operand (a distinct type, so that it cannot be passed for an
// int argument).
enum class Weights { Fp8, Fp4 };

template <Layout L>
int dispatch_mgrouped(int out, int fmt, Weights wt, const CUtensorMap& tA, const CUtensorMap& tB,
                      const CUtensorMap& tD, const CUtensorMap& tD8, GemmArgs args, cudaStream_t s) {
    if (wt == Weights::Fp4) return launch_mgrouped_mx(L, out == DG_OUT_FP32, true, tA, tB, args, s);
    if (use_mx(fmt, args.N, args.K)) return launch_mgrouped_mx(L, out == DG_OUT_FP32, false, tA, tB, args, s);
    const int bn = single_bn(out, args.N);
    args.num_nb = static_cast<int>(args.N / bn);
    // bf16 output stages half as much as fp32, which leaves room for a fifth ring stage
    if (out == DG_OUT_FP32) {
        if (fmt == DG_SF_UE8M0) return launch_gemm<L, MG_BN, MG_STAGES, true, true>(tA, tB, tD, tD8, args, s);
        return launch_gemm<L, MG_BN, MG_STAGES, true, false>(tA, tB, tD, tD8, args, s);
    }
    if (bn == MG_BN_WIDE) {
        if (fmt == DG_SF_UE8M0) return launch_gemm<L, MG_BN_WIDE, MG_STAGES_WIDE, false, true>(tA, tB, tD, tD8, args, s);
        return launch_gemm<L, MG_BN_WIDE, MG_STAGES_WIDE, false, false>(tA, tB, tD, tD8, args, s);
    }
    if (fmt == DG_SF_UE8M0) return launch_gemm<L, MG_BN, MG_STAGES_BF16, false, true>(tA, tB, tD, tD8, args, s);
    return launch_gemm<L, MG_BN, MG_STAGES_BF16, false, false>(tA, tB, tD, tD8, args, s);
}

// Shapes and codes; then (for a non-empty call) the pointers.
int check_shape_mg(int out, int G, int64_t N, int64_t K, int fmt) {
    DG_CHECK_ARG(G >= 1 && G <= DG_MAX_GROUPS, "G must be in [1, %d] (%d)", DG_MAX_GROUPS, G);
    DG_CHECK_ARG(N > 0 && K > 0 && N % 128 == 0 && K % 128 == 0, "N and K must be positive multiples of 128");
    DG_CHECK_ARG(out == DG_OUT_BF16 || out == DG_OUT_FP32, "bad out_dtype %d", out);
    DG_CHECK_ARG(fmt == DG_SF_FP32 || fmt == DG_SF_UE8M0, "bad sf_format %d", fmt);
    DG_CHECK_SUPPORTED(K <= (1 << 30) && N <= (1 << 24), "N or K too large");
    return DG_OK;
}

int check_ptrs_mg(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb, void* d) {
    DG_CHECK_ARG(a && sfa && b && sfb && d, "null pointer argument");
    DG_CHECK_ARG(aligned16(a) && aligned16(b) && aligned16(d), "a, b and d must be 16-byte aligned");
    return DG_OK;
}

// The weight tensor map: FP8 codes [G, N, K], or (b_fp4) FP4 codes packed two per byte
// [G, N, K/2] that the TMA unpacks to 16-byte groups of 16 codes in shared memory; boxes of 128 (K)
// x brows rows.
int encode_weights(CUtensorMap* tB, const uint8_t* b, bool b_fp4, int G, int64_t N, int64_t K, uint32_t brows) {
    uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(G)};
    const uint64_t row = b_fp4 ? static_cast<uint64_t>(K / 2) : static_cast<uint64_t>(K);
    uint64_t str[2] = {row, row * static_cast<uint64_t>(N)};
    uint32_t box[3] = {BK, brows, 1};
    return encode_tmap(tB, b_fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, b, dims,
                       str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// FP4 weights run only on the block-scaled kernel: UE8M0 scales and N % 256 == 0.
int check_fp4(bool b_fp4, int fmt, int64_t N) {
    if (!b_fp4) return DG_OK;
    DG_CHECK_ARG(fmt == DG_SF_UE8M0, "FP4 weights need UE8M0 scales");
    DG_CHECK_SUPPORTED(N % MX_BN == 0, "FP4 weights need N %% %d == 0 (N=%lld)", MX_BN, (long long)N);
    return DG_OK;
}

}  // namespace
}  // namespace dg

using namespace dg;

namespace dg {
namespace {

int check_accumulator(const float* c, int out_dtype) {
    if (c == nullptr) return DG_OK;
    DG_CHECK_ARG(out_dtype == DG_OUT_FP32, "accumulation (c != NULL) needs fp32 output");
    DG_CHECK_ARG(aligned16(c), "c must be 16-byte aligned");
    return DG_OK;
}

// The masked layout [G, cap, K]; dense: every group has cap rows (a batched GEMM), no counts.
int m_grouped_masked(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb, const float* c, void* d,
                     int out_dtype, const int32_t* counts, bool dense, int G, int64_t cap, int64_t N, int64_t K,
                     int expected_m, int sf_format, int32_t* status, void* stream, bool b_fp4 = false) {
    DG_CHECK_ARG(cap >= 0, "cap must be >= 0");
    if (int rc = check_shape_mg(out_dtype, G, N, K, sf_format)) return rc;
    if (int rc = check_fp4(b_fp4, sf_format, N)) return rc;
    DG_CHECK_ARG(c == nullptr || out_dtype == DG_OUT_FP32, "accumulation (c != NULL) needs fp32 output");
    if (cap == 0) return DG_OK;
    if (int rc = check_ptrs_mg(a, sfa, b, sfb, d)) return rc;
    if (int rc = check_accumulator(c, out_dtype)) return rc;
    DG_CHECK_ARG(dense || counts != nullptr, "counts is null");
    DG_CHECK_SUPPORTED(cap <= (1 << 24) && static_cast<int64_t>(G) * cap < (1ll << 31), "cap too large");
    const int esize = out_dtype == DG_OUT_FP32 ? 4 : 2;
    const int64_t M = static_cast<int64_t>(G) * cap;
    const int64_t Mp = sf_format == DG_SF_FP32 ? (M + 3) / 4 * 4 : (M + 15) / 16 * 16;
    (void)expected_m;  // a hint only: the schedule comes from the device-side counts
    CUtensorMap tA, tB, tD, tD8;
    {
        uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(cap), static_cast<uint64_t>(G)};
        uint64_t str[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(cap * K)};
        uint32_t box[3] = {BK, BM, 1};
        if (int rc = encode_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, a, dims, str, box,
                                 CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }
    {
        const bool mx = b_fp4 || use_mx(sf_format, N, K);
        const uint32_t brows = static_cast<uint32_t>(mx ? MX_BN : single_bn(out_dtype, N));
        if (int rc = encode_weights(&tB, b, b_fp4, G, N, K, brows)) return rc;
    }
    {
        uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(cap), static_cast<uint64_t>(G)};
        uint64_t str[2] = {static_cast<uint64_t>(N * esize), static_cast<uint64_t>(cap * N * esize)};
        uint32_t box[3] = {static_cast<uint32_t>(128 / esize), BM, 1};
        if (int rc = encode_tmap(&tD, out_tmap_type(out_dtype), 3, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
        box[1] = 8;
        if (int rc = encode_tmap(&tD8, out_tmap_type(out_dtype), 3, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }
    GemmArgs args{};
#if DG_DEBUG
    args.dbg_rows = g_debug_out_rows.load(std::memory_order_relaxed);
    args.dbg_stop_at = g_debug_stop_at.load(std::memory_order_relaxed);
#endif
    args.routing = counts;
    args.dense = dense ? 1 : 0;
    args.c = c;
    args.sfa = sfa;
    args.sfb = sfb;
    args.d = d;
    args.status = status;
    args.wait_limit_ns = wait_limit_ns();
    args.drain_limit_ns = drain_limit_ns();
    args.M = cap;
    args.sfa_ld = Mp;
    args.ldd = N;
    args.G = G;
    args.K = static_cast<int>(K);
    args.KB = static_cast<int>(K / BK);
    args.n128 = static_cast<int>(N / 128);
    args.N = N;
    return dispatch_mgrouped<Layout::Masked>(out_dtype, sf_format, b_fp4 ? Weights::Fp4 : Weights::Fp8, tA, tB, tD,
                                             tD8, args,
                                             static_cast<cudaStream_t>(stream));
}

// The contiguous layout, routed by m_indices [M] or (psum) by per-expert end rows [G]; dense:
// one expert owning all M rows (a plain GEMM), no routing tensor.
int m_grouped_contiguous(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb, const float* c,
                         void* d, int out_dtype, const int32_t* routing, bool psum, bool dense, int64_t M, int G,
                         int64_t N, int64_t K, int sf_format, int32_t* status, void* stream, bool b_fp4 = false) {
    DG_CHECK_ARG(M >= 0, "M must be >= 0");
    if (int rc = check_shape_mg(out_dtype, G, N, K, sf_format)) return rc;
    if (int rc = check_fp4(b_fp4, sf_format, N)) return rc;
    DG_CHECK_ARG(c == nullptr || out_dtype == DG_OUT_FP32, "accumulation (c != NULL) needs fp32 output");
    if (M == 0) return DG_OK;
    if (int rc = check_ptrs_mg(a, sfa, b, sfb, d)) return rc;
    if (int rc = check_accumulator(c, out_dtype)) return rc;
    DG_CHECK_ARG(dense || routing != nullptr, psum ? "psum is null" : "m_indices is null");
    DG_CHECK_SUPPORTED((M + BM - 1) / BM <= DG_MAX_M_BLOCKS, "M too large (at most %d rows)", DG_MAX_M_BLOCKS * BM);
    const int esize = out_dtype == DG_OUT_FP32 ? 4 : 2;
    const int64_t Mp = sf_format == DG_SF_FP32 ? (M + 3) / 4 * 4 : (M + 15) / 16 * 16;
    CUtensorMap tA, tB, tD, tD8;
    {
        uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
        uint64_t str[1] = {static_cast<uint64_t>(K)};
        uint32_t box[2] = {BK, BM};
        if (int rc = encode_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a, dims, str, box,
                                 CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }
    {
        const bool mx = b_fp4 || use_mx(sf_format, N, K);
        const uint32_t brows = static_cast<uint32_t>(mx ? MX_BN : single_bn(out_dtype, N));
        if (int rc = encode_weights(&tB, b, b_fp4, G, N, K, brows)) return rc;
    }
    {
        uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(M)};
        uint64_t str[1] = {static_cast<uint64_t>(N * esize)};
        uint32_t box[2] = {static_cast<uint32_t>(128 / esize), BM};
        if (int rc = encode_tmap(&tD, out_tmap_type(out_dtype), 2, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
        box[1] = 8;
        if (int rc = encode_tmap(&tD8, out_tmap_type(out_dtype), 2, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }
    GemmArgs args{};
#if DG_DEBUG
    args.dbg_rows = g_debug_out_rows.load(std::memory_order_relaxed);
    args.dbg_stop_at = g_debug_stop_at.load(std::memory_order_relaxed);
#endif
    args.routing = routing;
    args.psum = psum ? 1 : 0;
    args.dense = dense ? 1 : 0;
    args.c = c;
    args.sfa = sfa;
    args.sfb = sfb;
    args.d = d;
    args.status = status;
    args.wait_limit_ns = wait_limit_ns();
    args.drain_limit_ns = drain_limit_ns();
    args.M = M;
    args.sfa_ld = Mp;
    args.ldd = N;
    args.G = G;
    args.K = static_cast<int>(K);
    args.KB = static_cast<int>(K / BK);
    args.n128 = static_cast<int>(N / 128);
    args.N = N;
    return dispatch_mgrouped<Layout::Contiguous>(out_dtype, sf_format, b_fp4 ? Weights::Fp4 : Weights::Fp8, tA, tB,
                                                 tD, tD8, args,
                                                 static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace dg

extern "C" int dg_m_grouped_fp8_contiguous(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb,
                                           void* d, int out_dtype, const int32_t* m_indices, int64_t M, int G,
                                           int64_t N, int64_t K, int sf_format, void* workspace,
                                           size_t workspace_bytes, int32_t* status, void* stream) {
    DG_ARG_LOG(a, sfa, b, sfb, d, out_dtype, m_indices, M, G, N, K, sf_format, workspace, workspace_bytes, status,
               stream);
    (void)workspace;
    (void)workspace_bytes;
    return m_grouped_contiguous(a, sfa, b, sfb, nullptr, d, out_dtype, m_indices, false, false, M, G, N, K,
                                sf_format, status, stream);
}

extern "C" int dg_m_grouped_fp8_masked(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb, void* d,
                                       int out_dtype, const int32_t* counts, int G, int64_t cap, int64_t N, int64_t K,
                                       int expected_m, int sf_format, void* workspace, size_t workspace_bytes,
                                       int32_t* status, void* stream) {
    DG_ARG_LOG(a, sfa, b, sfb, d, out_dtype, counts, G, cap, N, K, expected_m, sf_format, workspace, workspace_bytes,
               status, stream);
    (void)workspace;
    (void)workspace_bytes;
    return m_grouped_masked(a, sfa, b, sfb, nullptr, d, out_dtype, counts, false, G, cap, N, K, expected_m,
                            sf_format, status, stream);
}

extern "C" int dg_fp8_gemm_nt(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb, const float* c,
                              void* d, int out_dtype, int64_t M, int64_t N, int64_t K, int sf_format,
                              int32_t* status, void* stream) {
    DG_ARG_LOG(a, sfa, b, sfb, c, d, out_dtype, M, N, K, sf_format, status, stream);
    return m_grouped_contiguous(a, sfa, b, sfb, c, d, out_dtype, nullptr, true, true, M, 1, N, K, sf_format, status,
                                stream);
}

extern "C" int dg_fp8_gemm_nt_batched(const uint8_t* a, const void* sfa, const uint8_t* b, const void* sfb,
                                      const float* c, void* d, int out_dtype, int batch, int64_t M, int64_t N,
                                      int64_t K, int sf_format, int32_t* status, void* stream) {
    DG_ARG_LOG(a, sfa, b, sfb, c, d, out_dtype, batch, M, N, K, sf_format, status, stream);
    return m_grouped_masked(a, sfa, b, sfb, c, d, out_dtype, nullptr, true, batch, M, N, K, static_cast<int>(M),
                            sf_format, status, stream);
}

extern "C" int dg_m_grouped_fp8_contiguous_psum(const uint8_t* a, const void* sfa, const uint8_t* b,
                                                const void* sfb, void* d, int out_dtype, const int32_t* psum,
                                                int64_t M, int G, int64_t N, int64_t K, int sf_format,
                                                void* workspace, size_t workspace_bytes, int32_t* status,
                                                void* stream) {
    DG_ARG_LOG(a, sfa, b, sfb, d, out_dtype, psum, M, G, N, K, sf_format, workspace, workspace_bytes, status, stream);
    (void)workspace;
    (void)workspace_bytes;
    return m_grouped_contiguous(a, sfa, b, sfb, nullptr, d, out_dtype, psum, true, false, M, G, N, K, sf_format,
                                status, stream);
}

extern "C" int dg_m_grouped_fp8_fp4_contiguous(const uint8_t* a, const uint8_t* sfa, const uint8_t* b_packed,
                                               const uint8_t* sfb, void* d, int out_dtype, const int32_t* m_indices,
                                               int64_t M, int G, int64_t N, int64_t K, int32_t* status,
                                               void* stream) {
    DG_ARG_LOG(a, sfa, b_packed, sfb, d, out_dtype, m_indices, M, G, N, K, status, stream);
    return m_grouped_contiguous(a, sfa, b_packed, sfb, nullptr, d, out_dtype, m_indices, false, false, M, G, N, K,
                                DG_SF_UE8M0, status, stream, true);
}

extern "C" int dg_m_grouped_fp8_fp4_masked(const uint8_t* a, const uint8_t* sfa, const uint8_t* b_packed,
                                           const uint8_t* sfb, void* d, int out_dtype, const int32_t* counts, int G,
                                           int64_t cap, int64_t N, int64_t K, int expected_m, int32_t* status,
                                           void* stream) {
    DG_ARG_LOG(a, sfa, b_packed, sfb, d, out_dtype, counts, G, cap, N, K, expected_m, status, stream);
    return m_grouped_masked(a, sfa, b_packed, sfb, nullptr, d, out_dtype, counts, false, G, cap, N, K, expected_m,
                            DG_SF_UE8M0, status, stream, true);
}

// ------------------------------------------------------------------------- test hooks
// Each selects, for later calls in this process, one choice the library otherwise makes
// itself, so that the tests hold every variant to the oracle and to each other.
// Debug build: the index checks of the m-grouped FP8 kernels' owner-thread stores treat the output
// as `rows` rows (0 restores the layout's): rows past it are skipped and raise DG_DEBUG_OUT, which
// exercises the checks without any access out of bounds.  No effect on the release build.
extern "C" int dg_testing_debug_out_rows(int64_t rows) {
    DG_CHECK_ARG(rows >= 0, "rows must be >= 0");
    dg::g_debug_out_rows.store(rows, std::memory_order_relaxed);
    return DG_OK;
}

// Debug build: the first CTA's TMA producer of the m-grouped FP8 promotion kernel stops before its
// n-th stage load (0 restores normal operation), as a stalled producer would: the waits for that
// stage run out after the wait limit, the kernel sets DG_STATUS_TIMEOUT, drains what it issued and
// returns.  No effect on the release build.
extern "C" int dg_testing_debug_stop_producer(int n) {
    DG_CHECK_ARG(n >= 0, "n must be >= 0");
    dg::g_debug_stop_at.store(n, std::memory_order_relaxed);
    return DG_OK;
}

// The single-CTA tile width: 0 automatic, 128, or 256 (where N allows).
extern "C" int dg_testing_mgrouped_bn(int bn) {
    DG_CHECK_ARG(bn == 0 || bn == MG_BN || bn == MG_BN_WIDE, "bn must be 0, %d or %d", MG_BN, MG_BN_WIDE);
    g_force_bn.store(bn, std::memory_order_relaxed);
    return DG_OK;
}

// How the kernel stores tiles: 0 automatic, 1 TMA stores issued by thread 0 of the promotion
// warps, 3 owner-thread stores from registers.
extern "C" int dg_testing_mgrouped_store(int which) {
    DG_CHECK_ARG(which == 0 || which == 1 || which == 3, "which must be 0 (automatic), 1 (thread 0) or 3 (owner threads)");
    g_force_store.store(which, std::memory_order_relaxed);
    return DG_OK;
}

// The m-grouped kernel of UE8M0-scale calls: 0 automatic, 1 the promotion kernel, 2 the
// block-scaled MMA kernel wherever N % 256 == 0 (and no 128-column tile width is forced).
extern "C" int dg_testing_mgrouped_kernel(int which) {
    DG_CHECK_ARG(which >= 0 && which <= 2, "which must be 0 (automatic), 1 (promotion) or 2 (block-scaled MMA)");
    g_force_kernel.store(which, std::memory_order_relaxed);
    return DG_OK;
}

// Promotion warps of 128 x 256 tiles: 0 automatic (16), 8 or 16.
extern "C" int dg_testing_mgrouped_warps(int warps) {
    DG_CHECK_ARG(warps == 0 || warps == 8 || warps == 16, "warps must be 0, 8 or 16");
    g_force_warps.store(warps, std::memory_order_relaxed);
    return DG_OK;
}

namespace dg {
int debug_word_gemm(uint32_t* out, bool clear) { return debug_word_local(out, clear); }
}  // namespace dg
