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
// Roles (352 threads): warps 0-7 drain finished accumulators (TMEM lane quarter = warp % 4, column
// half = warp / 4) and write each valid row from registers; warp 8 issues the TMA loads of the A / B
// tiles; warp 9 turns each 128-K block's scale bytes into the tensor-memory scale layout in shared
// memory; warp 10 copies the scales into tensor memory (tcgen05.cp) and issues the MMAs (it owns the
// tensor memory).  Tiles are 128 x 128; three 128-column accumulators let the MMAs of the next
// tiles run while a finished one is drained.
//
// Scale layout in tensor memory (scale_vec::1X, M = 128 or N = 128 rows): the scale of row
// 32 j + i sits in lane i, column c0 + j of each 32-lane quarter (tcgen05.cp.32x128b.warpx4 copies
// 32 rows of four 32-bit words and replicates them into the four quarters).  Each word holds the
// row's scale byte in all four byte positions, so the byte the instruction's scale-factor id picks
// is the scale whatever the id.
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

constexpr int BN = 128;             // tile columns
constexpr int STAGES = 6;           // shared-memory ring of 128-K blocks
constexpr int ACC = 3;              // tensor-memory accumulators (128 columns each)
constexpr int EPI_WARPS = 8;
constexpr int PRODUCER_WARP = 8, SF_WARP = 9, MMA_WARP = 10;
constexpr int NT = 11 * 32;
constexpr int KG = 8;               // 128-K blocks whose scale bytes the scale warp has in flight
constexpr int A_BYTES = BM * BK;    // 16 KB
constexpr int B_BYTES = BN * BK;    // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SF_ROWS_BYTES = 512;  // 32 rows x 16 bytes: the scales of 128 rows
constexpr int SF_SLOT = 2 * SF_ROWS_BYTES;  // A scales, then B scales
constexpr int RING_OFF = 0;
constexpr int SF_OFF = STAGES * STAGE_BYTES;
constexpr int SCHED_OFF = SF_OFF + STAGES * SF_SLOT;
constexpr int BAR_OFF = (SCHED_OFF + SCHED_BYTES + 127) / 128 * 128;
constexpr int NUM_BARS = 3 * STAGES + 2 * ACC;  // full, sfull, empty; tfull, tempty
constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
constexpr int TOTAL = MISC_OFF + 256 + 1024;    // + alignment slack
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_COL0 = ACC * BN;          // stage s: A scales at SF_COL0 + 8 s, B scales 4 later
static_assert(SF_COL0 + 8 * STAGES <= TMEM_COLS, "scale columns inside the allocation");
static_assert(A_BYTES % 1024 == 0 && STAGE_BYTES % 1024 == 0 && SF_OFF % 1024 == 0, "swizzle atoms aligned");
static_assert(SF_SLOT % 128 == 0 && SCHED_OFF % 16 == 0, "scale slots 16-byte aligned");
static_assert(BAR_OFF % 8 == 0 && MISC_OFF % 8 == 0, "mbarriers 8-byte aligned");
static_assert(TOTAL <= 232448, "shared memory");
static_assert(BM == 128 && BN == 128, "the scale layout covers 128 rows of A and of B");

// The scale warp's walk over this CTA's (tile, 128-K block) items.
template <Layout L>
struct Walk {
    int t, kb;
    TileInfo ti;
    bool valid;
    __device__ void start(int num_tiles, const RunTable& rt, int R, const GemmArgs& a) {
        t = blockIdx.x;
        kb = 0;
        valid = t < num_tiles;
        if (valid) ti = decode_tile<L>(t, rt, R, a);
    }
    __device__ void next(int num_tiles, const RunTable& rt, int R, const GemmArgs& a) {
        if (++kb < ti.kbt) return;
        kb = 0;
        t += gridDim.x;
        valid = t < num_tiles;
        if (valid) ti = decode_tile<L>(t, rt, R, a);
    }
};

// The UE8M0 bytes of one item: rows 32 j + lane of the tile's A rows (sa[j]) and the tile's weight
// block (sb).  Rows outside the layout read 127 (scale 1): they are never stored.
template <Layout L>
__device__ __forceinline__ void load_scales(const Walk<L>& w, const GemmArgs& a, int lane, uint32_t (&sa)[4],
                                            uint32_t& sb) {
    const uint8_t* sfa = static_cast<const uint8_t*>(a.sfa);
    const uint8_t* sfb = static_cast<const uint8_t*>(a.sfb);
    const int64_t kbase = static_cast<int64_t>(w.kb) * a.sfa_ld;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t r = static_cast<int64_t>(w.ti.row0) + j * 32 + lane;
        bool in;
        int64_t m;
        if constexpr (L == Layout::Masked) {
            in = r < a.M;  // a.M = cap
            m = static_cast<int64_t>(w.ti.e) * a.M + r;
        } else {
            in = r < a.M;
            m = r;
        }
        sa[j] = in ? static_cast<uint32_t>(__ldg(sfa + kbase + m)) : 127u;
    }
    sb = __ldg(sfb + (static_cast<int64_t>(w.ti.e) * a.n128 + w.ti.nb) * a.KB + w.kb);
}

template <Layout L, bool OUT_FP32>
__global__ void __launch_bounds__(NT, 1)
    k_grouped_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);

    uint8_t* ring = smem + RING_OFF;
    uint8_t* sfbuf = smem + SF_OFF;
    const RunTable rt = RunTable::at(smem + SCHED_OFF);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + BAR_OFF);
    uint64_t* full = bars;                 // A / B tiles landed (TMA bytes)
    uint64_t* sfull = bars + STAGES;       // the stage's scales are in shared memory
    uint64_t* empty = bars + 2 * STAGES;   // the stage's MMAs (and scale copies) are done
    uint64_t* tfull = bars + 3 * STAGES;   // an accumulator holds a finished tile
    uint64_t* tempty = tfull + ACC;        // the drain warps have read it
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + MISC_OFF);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + MISC_OFF + 4);
    int* s_ntiles = reinterpret_cast<int*>(smem + MISC_OFF + 12);
    int* s_scan = reinterpret_cast<int*>(smem + MISC_OFF + 64);  // [NT / 32 + 1]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const WaitCtx wc{a.status, s_abort, a.wait_limit_ns};

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&sfull[s], 1);
            mbar_init(&empty[s], 1);
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
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
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
        // ------------------------------------------------------------ scales -> shared memory
        // KG register slots: slot g is written to shared memory, then reloaded with the item KG
        // places further on, so KG items' global loads are in flight while the ring fills.
        if (R > 0) {
            Walk<L> st, ld;
            st.start(num_tiles, rt, R, a);
            ld.start(num_tiles, rt, R, a);
            uint32_t sa[KG][4], sb[KG];
#pragma unroll
            for (int g = 0; g < KG; ++g) {
                sa[g][0] = sa[g][1] = sa[g][2] = sa[g][3] = 127u;
                sb[g] = 127u;
                if (ld.valid) {
                    load_scales<L>(ld, a, lane, sa[g], sb[g]);
                    ld.next(num_tiles, rt, R, a);
                }
            }
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            while (st.valid && ok) {
#pragma unroll
                for (int g = 0; g < KG; ++g) {
                    if (!st.valid) break;
                    bool w = true;
                    if (lane == 0) w = mbar_wait(&empty[stage], phase ^ 1u, wc);
                    if (!__shfl_sync(0xffffffffu, w ? 1 : 0, 0)) { ok = false; break; }
                    __syncwarp();  // orders every lane's writes below after lane 0's wait
                    uint8_t* slot = sfbuf + stage * SF_SLOT;
                    const uint4 va = make_uint4(sa[g][0] * 0x01010101u, sa[g][1] * 0x01010101u,
                                                sa[g][2] * 0x01010101u, sa[g][3] * 0x01010101u);
                    const uint32_t wb = sb[g] * 0x01010101u;
                    *reinterpret_cast<uint4*>(slot + 16 * lane) = va;
                    *reinterpret_cast<uint4*>(slot + SF_ROWS_BYTES + 16 * lane) = make_uint4(wb, wb, wb, wb);
                    fence_async_smem();  // generic-proxy writes -> visible to tcgen05.cp
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sfull[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    st.next(num_tiles, rt, R, a);
                    if (ld.valid) {
                        load_scales<L>(ld, a, lane, sa[g], sb[g]);
                        ld.next(num_tiles, rt, R, a);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ scale copies + MMAs
        if (lane == 0 && R > 0) {
            constexpr uint32_t IDESC = idesc_mxf8_e4m3_ue8m0(BM, BN);
            int stage = 0, j = 0;
            uint32_t phase = 0;
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
                for (int kb = 0; kb < ti.kbt; ++kb) {
                    if (!mbar_wait(&full[stage], phase, wc)) { ok = false; break; }
                    if (!mbar_wait(&sfull[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sfa_t = tmem_base + SF_COL0 + 8u * static_cast<uint32_t>(stage);
                    const uint32_t sfb_t = sfa_t + 4u;
                    const uint32_t sf_s = smem_u32(sfbuf + stage * SF_SLOT);
                    tmem_cp_32x128b_x4(sfa_t, sdesc_rows16(sf_s));
                    tmem_cp_32x128b_x4(sfb_t, sdesc_rows16(sf_s + SF_ROWS_BYTES));
                    const uint32_t sa = smem_u32(ring + stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / 32; ++k)
                        umma_mxf8_1x(dt, sdesc_k_sw128(sa + 32 * k), sdesc_k_sw128(sb + 32 * k), IDESC, sfa_t, sfb_t,
                                     (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);  // frees the stage's tiles and scale slot
                    last = &empty[stage];
                    last_ph = phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
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
            uint32_t v[2][32];
            const uint32_t col = tmem_base + t_lane + static_cast<uint32_t>(tb * BN + h * 64);
            tmem_ld_x32(col, v[0]);
            tmem_ld_x32(col + 32, v[1]);
            tmem_wait_ld(v[0]);
            tmem_wait_ld(v[1]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[tb]);  // the accumulator is in registers
            if (!row_ok) continue;
            const int64_t c0 = static_cast<int64_t>(ti.nb) * BN + h * 64;
            uint8_t* dst = static_cast<uint8_t*>(a.d) + (grow * a.ldd + c0) * ESIZE;
            if constexpr (OUT_FP32) {
                const float* crow = a.c != nullptr ? a.c + grow * a.ldd + c0 : nullptr;
#pragma unroll
                for (int p = 0; p < 16; ++p) {
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
                for (int p = 0; p < 8; ++p) {
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

template <Layout L, bool OUT_FP32>
int launch(const CUtensorMap& tA, const CUtensorMap& tB, GemmArgs args, cudaStream_t stream) {
    auto kern = k_grouped_gemm_mx<L, OUT_FP32>;
    DG_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TOTAL));
    int sms = 0;
    if (int rc = device_sm_count(&sms)) return rc;
    args.num_nb = static_cast<int>(args.N / BN);
    return launch_pdl(kern, dim3(sms), dim3(NT), TOTAL, stream, tA, tB, args);
}

}  // namespace mx

int launch_mgrouped_mx(Layout L, bool out_fp32, const CUtensorMap& tA, const CUtensorMap& tB, const GemmArgs& args,
                       cudaStream_t stream) {
    if (L == Layout::Masked)
        return out_fp32 ? mx::launch<Layout::Masked, true>(tA, tB, args, stream)
                        : mx::launch<Layout::Masked, false>(tA, tB, args, stream);
    return out_fp32 ? mx::launch<Layout::Contiguous, true>(tA, tB, args, stream)
                    : mx::launch<Layout::Contiguous, false>(tA, tB, args, stream);
}

}  // namespace dg
