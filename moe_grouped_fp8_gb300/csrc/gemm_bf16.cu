// gemm_bf16.cu - persistent, warp-specialised BF16 m-grouped GEMM for sm_103a: the BF16 masked
// GEMM of the reproduction in "Fix cross-expert output overwrites in SM90 masked GEMM" (#469,
// m_grouped_bf16_gemm_nt_masked(a, b, d, masked_m, expected_m)), and the same GEMM on the
// contiguous layout routed by m_indices.
//
// D[rows of expert e, :] = A[rows, :] . B_e^T with bf16 operands and fp32 accumulation over the
// whole K in tensor memory - no scales, no promotion.  Per tile the MMA thread issues
// tcgen05.mma.kind::f16 (M = 128, N = BN, K = 16, both operands bf16) for every 64-element K
// stage into one of two TMEM tile buffers and commits once; the eight epilogue warps read the
// finished tile, round it to bf16 (or keep fp32) and store it while the tensor core fills the
// other buffer.  Tiles are 128 x 256 (bf16 output, N % 256 == 0: three 48 KB ring stages) or
// 128 x 128 (five 32 KB stages for bf16, four for fp32 output); the wider tile moves 25% fewer
// operand bytes from L2 into shared memory per MMA.  A 64-element bf16 stage row is 128 bytes, so the 128-byte-swizzled stage tiles
// and the 32-byte K advance per MMA are those of the FP8 kernels.
//
// Schedule (rebuilt on device from counts / m_indices at every launch), row validity and the
// row-exact store (3-D [G, cap, N] TMA boxes of 128 or 8 rows, owner-thread tails) follow the FP8
// kernel of gemm.cu: rows that are not valid are never written.
#include <cuda_bf16.h>

#include <atomic>

#include "host_common.hpp"
#include "kernel_common.cuh"
#include "mgrouped.cuh"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int H_EPI_WARPS = 8;
constexpr int H_PRODUCER_WARP = 8;
constexpr int H_MMA_WARP = 9;
constexpr int H_THREADS = 320;
constexpr int H_EPI_BAR = 1;
constexpr int H_BK = 64;     // bf16 elements of K per stage (128-byte rows)
constexpr int H_TBUFS = 2;   // TMEM tile buffers (BN fp32 columns each)

template <int BN, int STAGES, bool OUT_FP32>
struct HPlan {
    static constexpr int A_BYTES = BM * H_BK * 2;
    static constexpr int B_BYTES = BN * H_BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int ESIZE = OUT_FP32 ? 4 : 2;
    static constexpr int CPT = BN / 2;               // output columns per epilogue thread
    static constexpr int CHUNKS = BN * ESIZE / 128;  // 128-byte column chunks of a tile row
    static constexpr int CHUNK_BYTES = BM * 128;
    static constexpr int STG_BYTES = CHUNKS * CHUNK_BYTES;
    static constexpr int RING_OFF = 0;
    static constexpr int STG_OFF = STAGES * STAGE_BYTES;
    static constexpr int SCHED_OFF = STG_OFF + STG_BYTES;
    static constexpr int BAR_OFF = (SCHED_OFF + SCHED_BYTES + 127) / 128 * 128;
    static constexpr int NUM_BARS = 2 * STAGES + 2 * H_TBUFS;
    static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr int MISC_BYTES = 256;
    static constexpr int TOTAL = MISC_OFF + MISC_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = H_TBUFS * BN;
    static_assert(H_BK * 2 == 128, "a stage row is one 128-byte swizzle row");
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms");
    static_assert(STG_OFF % 1024 == 0 && SCHED_OFF % 1024 == 0, "TMA / swizzle buffers are 1024-byte aligned");
    static_assert(BAR_OFF % 8 == 0 && MISC_OFF % 8 == 0, "mbarrier objects are 8-byte aligned");
    static_assert(STG_BYTES >= 2 * DG_MAX_M_BLOCKS, "run scratch fits in the staging buffer");
    static_assert(BN == 128 || (BN == 256 && !OUT_FP32), "256-column tiles stage bf16 output only");
    static_assert(TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation");
    static_assert(CPT % 32 == 0, "32-column TMEM loads per epilogue thread");
    static_assert(TOTAL <= 232448, "shared memory");
};

struct HTile {
    int e, nb, row0, valid;
};

template <Layout L>
__device__ __forceinline__ HTile decode_h(int t, const RunTable& rt, int R, const GemmArgs& a) {
    const int r = find_run(rt.prefix, R, t);
    const int local = t - rt.prefix[r];
    const int Lr = rt.L[r];
    const int nb = local / Lr, j = local - nb * Lr;  // m-blocks fastest: concurrent tiles share B
    HTile ti;
    ti.nb = nb;
    ti.e = rt.e[r];
    ti.valid = 0;
    if constexpr (L == Layout::Contiguous) {
        ti.row0 = (rt.first[r] + j) * BM;
        if (a.psum) {
            const int v = rt.x[r] - ti.row0;
            ti.valid = v < BM ? v : BM;
        }
    } else {
        ti.row0 = j * BM;
        const int v = rt.x[r] - ti.row0;
        ti.valid = v < BM ? v : BM;
    }
    return ti;
}

template <Layout L, int BN, int STAGES, bool OUT_FP32>
__global__ void __launch_bounds__(H_THREADS, 1)
    k_grouped_gemm_bf16(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmD, const __grid_constant__ CUtensorMap tmD8,
                        const GemmArgs a) {
    using P = HPlan<BN, STAGES, OUT_FP32>;
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
    uint64_t* tempty = tfull + H_TBUFS;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + P::MISC_OFF);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + P::MISC_OFF + 4);
    int* s_ntiles = reinterpret_cast<int*>(smem + P::MISC_OFF + 12);
    uint32_t* s_ballot = reinterpret_cast<uint32_t*>(smem + P::MISC_OFF + 32);  // [2][4]
    int* s_scan = reinterpret_cast<int*>(smem + P::MISC_OFF + 64);              // [H_THREADS / 32]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const WaitCtx wc{a.status, s_abort, a.wait_limit_ns};

    // ---------------------------------------------------------------- set-up
    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < H_TBUFS; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], H_EPI_WARPS);
        }
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == H_MMA_WARP) {
        tmem_alloc(s_tmem, P::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == H_PRODUCER_WARP && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmD);
        prefetch_tmap(&tmD8);
    }
    pdl_trigger();
    pdl_wait();  // every earlier kernel of the stream has finished: inputs are visible
    __syncthreads();

    const int R = build_runs<L, H_THREADS>(a, rt, s_scan, stg);  // staging is free during set-up
    const int num_tiles = tile_prefix<H_THREADS, 1>(R, a.num_nb, rt, s_scan, s_ntiles);
    tc_fence_after();
    const uint32_t tmem_base = *s_tmem;

    // ---------------------------------------------------------------- roles
    if (warp == H_PRODUCER_WARP) {
        if (lane == 0 && num_tiles > 0) {
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const HTile ti = decode_h<L>(t, rt, R, a);
                for (int kb = 0; kb < a.KB; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, wc)) { ok = false; break; }
                    uint8_t* sa = ring + stage * P::STAGE_BYTES;
                    uint8_t* sb = sa + P::A_BYTES;
                    mbar_arrive_expect_tx(&full[stage], P::STAGE_BYTES);
                    if constexpr (L == Layout::Masked)
                        tma_load_3d(sa, &tmA, &full[stage], kb * H_BK, ti.row0, ti.e);
                    else
                        tma_load_2d(sa, &tmA, &full[stage], kb * H_BK, ti.row0);
                    tma_load_3d(sb, &tmB, &full[stage], kb * H_BK, ti.nb * BN, ti.e);
                    ++issued;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            const int n_drain = issued < STAGES ? issued : STAGES;
            for (int i = 0; i < n_drain; ++i) {
                int s = stage - 1 - i;
                uint32_t ph = phase;
                while (s < 0) { s += STAGES; ph ^= 1u; }
                drain_wait(&full[s], ph, a.drain_limit_ns);
            }
        }
        __syncwarp();
    } else if (warp == H_MMA_WARP) {
        if (lane == 0 && num_tiles > 0) {
            int stage = 0, tb = 0;
            uint32_t phase = 0, tphase = 0;
            bool ok = true, any = false;
            constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                if (!mbar_wait(&tempty[tb], tphase ^ 1u, wc)) { ok = false; break; }
                const uint32_t dt = tmem_base + static_cast<uint32_t>(tb * BN);
                for (int kb = 0; kb < a.KB; ++kb) {
                    if (!mbar_wait(&full[stage], phase, wc)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(ring + stage * P::STAGE_BYTES);
                    const uint32_t sb = sa + P::A_BYTES;
#pragma unroll
                    for (int k = 0; k < H_BK / 16; ++k)
                        umma_bf16(dt, sdesc_k_sw128(sa + 32 * k), sdesc_k_sw128(sb + 32 * k), IDESC,
                                  (kb > 0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                // the tile's accumulator (committed on the way out too, so the drain covers it)
                umma_commit(&tfull[tb]);
                any = true;
                if (++tb == H_TBUFS) { tb = 0; tphase ^= 1u; }
            }
            if (any) {
                int lt = tb - 1;
                uint32_t lp = tphase;
                if (lt < 0) { lt = H_TBUFS - 1; lp ^= 1u; }
                drain_wait(&tfull[lt], lp, a.drain_limit_ns);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue: TMEM -> D
        const int q = warp & 3;    // TMEM lane quarter
        const int h2 = warp >> 2;  // column half
        const int row = q * 32 + lane;
        const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
        int tb = 0;
        uint32_t tphase = 0;
        bool have_store = false;
        int parity_slot = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const HTile ti = decode_h<L>(t, rt, R, a);
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
                const int mi = grow < a.M ? a.routing[grow] : -1;
                row_ok = (mi == ti.e);
                if (mi >= 0 && mi != ti.e) status_or(a.status, DG_STATUS_BAD_INDEX);
                const uint32_t bal = __ballot_sync(0xffffffffu, row_ok);
                if (h2 == 0 && lane == 0) s_ballot[parity_slot * 4 + q] = bal;
            }
            bool failed = !mbar_wait(&tfull[tb], tphase, wc);
            float acc[P::CPT];
            if (!failed) {
                tc_fence_after();
                constexpr int LOADS = P::CPT / 32;
                uint32_t v[LOADS][32];
#pragma unroll
                for (int c2 = 0; c2 < LOADS; ++c2)
                    tmem_ld_x32(tmem_base + t_lane + static_cast<uint32_t>(tb * BN + h2 * P::CPT + c2 * 32), v[c2]);
#pragma unroll
                for (int c2 = 0; c2 < LOADS; ++c2) tmem_wait_ld(v[c2]);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[tb]);  // the accumulator is in registers
#pragma unroll
                for (int c2 = 0; c2 < LOADS; ++c2)
#pragma unroll
                    for (int i = 0; i < 32; ++i) acc[c2 * 32 + i] = __uint_as_float(v[c2][i]);
            }
            if (++tb == H_TBUFS) { tb = 0; tphase ^= 1u; }

            // ---- stage the tile in shared memory
            if (tid == 0 && have_store) bulk_wait_read_all();  // the previous store has read the staging
            named_bar_sync(H_EPI_BAR, H_EPI_WARPS * 32);
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
            if (bar_or(H_EPI_BAR, H_EPI_WARPS * 32, failed || *s_abort != 0)) break;

            // ---- store: TMA for the leading 8-row-aligned valid rows, owner threads for the rest
            int v = BM;
            if (L == Layout::Masked || a.psum) {
                v = ti.valid;
            } else {
                v = 0;
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
                have_store = true;
            }
            if (row_ok && row >= v8 &&
                DG_CHECKED(out_in<L>(a, grow, static_cast<int64_t>(ti.nb) * BN + h2 * P::CPT, P::CPT),
                           DG_DEBUG_OUT)) {
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
            }
            parity_slot ^= 1;
        }
        if (tid == 0 && have_store) bulk_wait_all();
        __syncwarp();
    }

    __syncthreads();
    if (warp == H_MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, P::TMEM_COLS);
    }
}

// ------------------------------------------------------------------------- host side

template <Layout L, int BN, int STAGES, bool OUT_FP32>
int launch_h(const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tD, const CUtensorMap& tD8,
             const GemmArgs& args, cudaStream_t stream) {
    using P = HPlan<BN, STAGES, OUT_FP32>;
    auto kern = k_grouped_gemm_bf16<L, BN, STAGES, OUT_FP32>;
    DG_CHECK_CUDA(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P::TOTAL));
    int sms = 0;
    if (int rc = device_sm_count(&sms)) return rc;
    return launch_pdl(kern, dim3(sms), dim3(H_THREADS), P::TOTAL, stream, tA, tB, tD, tD8, args);
}

// testing: the tile width of later calls (0 automatic, 128, or 256 where N and the output allow)
std::atomic<int> g_force_bn_h{0};

// 128 x 256 tiles for bf16 output with N % 256 == 0 when they still fill the GPU (at least one
// 256-column tile per SM for the m-blocks the call is expected to have), else 128 x 128: the
// reproduction's shape (8 experts of 32 rows, N = 256) has 8 wide tiles, 5.2 us with 16 narrow
// ones against 6.1 us; decode and prefill take 11% and 21% less time with wide tiles.
int tile_bn(int out, int64_t N, int64_t m_blocks) {
    const int f = g_force_bn_h.load(std::memory_order_relaxed);
    if (f == 128 || out != DG_OUT_BF16 || N % 256 != 0) return 128;
    if (f == 256) return 256;
    int sms = 0;
    if (device_sm_count(&sms) != DG_OK) sms = 1;
    return m_blocks * (N / 256) >= sms ? 256 : 128;
}

template <Layout L>
int dispatch_h(int out, const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tD, const CUtensorMap& tD8,
               const GemmArgs& args, cudaStream_t s) {
    // bf16 output stages half as much as fp32, which leaves room for a fifth ring stage
    if (out == DG_OUT_FP32) return launch_h<L, 128, 4, true>(tA, tB, tD, tD8, args, s);
    if (args.num_nb * 256 == args.N) return launch_h<L, 256, 3, false>(tA, tB, tD, tD8, args, s);
    return launch_h<L, 128, 5, false>(tA, tB, tD, tD8, args, s);
}

CUtensorMapDataType out_type(int out) {
    return out == DG_OUT_FP32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

int check_common_h(const void* a, const void* b, void* d, int out, int G, int64_t N, int64_t K) {
    DG_CHECK_ARG(G >= 1 && G <= DG_MAX_GROUPS, "G must be in [1, %d] (%d)", DG_MAX_GROUPS, G);
    DG_CHECK_ARG(N > 0 && K > 0 && N % 128 == 0 && K % 64 == 0,
                 "N must be a positive multiple of 128 and K of 64 (N=%lld K=%lld)", (long long)N, (long long)K);
    DG_CHECK_ARG(out == DG_OUT_BF16 || out == DG_OUT_FP32, "bad out_dtype %d", out);
    DG_CHECK_ARG(a && b && d, "null pointer argument");
    DG_CHECK_ARG(aligned16(a) && aligned16(b) && aligned16(d), "a, b and d must be 16-byte aligned");
    DG_CHECK_SUPPORTED(K <= (1 << 30) && N <= (1 << 24), "N or K too large");
    return DG_OK;
}

int encode_b_and_d(const void* b, void* d, int out, int G, int64_t rows, int64_t G_out, int64_t N, int64_t K,
                   bool masked, int bn, CUtensorMap* tB, CUtensorMap* tD, CUtensorMap* tD8) {
    {
        uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(N), static_cast<uint64_t>(G)};
        uint64_t str[2] = {static_cast<uint64_t>(K * 2), static_cast<uint64_t>(N * K * 2)};
        uint32_t box[3] = {H_BK, static_cast<uint32_t>(bn), 1};
        if (int rc = encode_tmap(tB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, b, dims, str, box,
                                 CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }
    const int esize = out == DG_OUT_FP32 ? 4 : 2;
    if (masked) {
        uint64_t dims[3] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows), static_cast<uint64_t>(G_out)};
        uint64_t str[2] = {static_cast<uint64_t>(N * esize), static_cast<uint64_t>(rows * N * esize)};
        uint32_t box[3] = {static_cast<uint32_t>(128 / esize), BM, 1};
        if (int rc = encode_tmap(tD, out_type(out), 3, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return rc;
        box[1] = 8;
        return encode_tmap(tD8, out_type(out), 3, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    uint64_t dims[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(rows)};
    uint64_t str[1] = {static_cast<uint64_t>(N * esize)};
    uint32_t box[2] = {static_cast<uint32_t>(128 / esize), BM};
    if (int rc = encode_tmap(tD, out_type(out), 2, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return rc;
    box[1] = 8;
    return encode_tmap(tD8, out_type(out), 2, d, dims, str, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" int dg_m_grouped_bf16_masked(const void* a, const void* b, void* d, int out_dtype, const int32_t* counts,
                                        int G, int64_t cap, int64_t N, int64_t K, int expected_m, int32_t* status,
                                        void* stream) {
    DG_ARG_LOG(a, b, d, out_dtype, counts, G, cap, N, K, expected_m, status, stream);
    DG_CHECK_ARG(cap >= 0, "cap must be >= 0");
    if (int rc = check_common_h(a, b, d, out_dtype, G, N, K)) return rc;
    DG_CHECK_ARG(counts != nullptr, "counts is null");
    if (cap == 0) return DG_OK;
    DG_CHECK_SUPPORTED(cap <= (1 << 24) && static_cast<int64_t>(G) * cap < (1ll << 31), "cap too large");
    CUtensorMap tA, tB, tD, tD8;
    {
        uint64_t dims[3] = {static_cast<uint64_t>(K), static_cast<uint64_t>(cap), static_cast<uint64_t>(G)};
        uint64_t str[2] = {static_cast<uint64_t>(K * 2), static_cast<uint64_t>(cap * K * 2)};
        uint32_t box[3] = {H_BK, BM, 1};
        if (int rc = encode_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a, dims, str, box,
                                 CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }
    const int64_t rows_hint = expected_m > 0 && expected_m < cap ? expected_m : cap;
    const int bn = tile_bn(out_dtype, N, static_cast<int64_t>(G) * ((rows_hint + BM - 1) / BM));
    if (int rc = encode_b_and_d(b, d, out_dtype, G, cap, G, N, K, true, bn, &tB, &tD, &tD8)) return rc;
    GemmArgs args{};
    args.routing = counts;
    args.d = d;
    args.status = status;
    args.wait_limit_ns = wait_limit_ns();
    args.drain_limit_ns = drain_limit_ns();
    args.M = cap;
    args.ldd = N;
    args.N = N;
    args.G = G;
    args.K = static_cast<int>(K);
    args.KB = static_cast<int>(K / H_BK);
    args.num_nb = static_cast<int>(N / bn);
    args.n128 = static_cast<int>(N / 128);
    return dispatch_h<Layout::Masked>(out_dtype, tA, tB, tD, tD8, args, static_cast<cudaStream_t>(stream));
}

extern "C" int dg_m_grouped_bf16_contiguous(const void* a, const void* b, void* d, int out_dtype,
                                            const int32_t* m_indices, int64_t M, int G, int64_t N, int64_t K,
                                            int32_t* status, void* stream) {
    DG_ARG_LOG(a, b, d, out_dtype, m_indices, M, G, N, K, status, stream);
    DG_CHECK_ARG(M >= 0, "M must be >= 0");
    if (int rc = check_common_h(a, b, d, out_dtype, G, N, K)) return rc;
    DG_CHECK_ARG(m_indices != nullptr, "m_indices is null");
    if (M == 0) return DG_OK;
    DG_CHECK_SUPPORTED((M + BM - 1) / BM <= DG_MAX_M_BLOCKS, "M too large (at most %d rows)", DG_MAX_M_BLOCKS * BM);
    CUtensorMap tA, tB, tD, tD8;
    {
        uint64_t dims[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(M)};
        uint64_t str[1] = {static_cast<uint64_t>(K * 2)};
        uint32_t box[2] = {H_BK, BM};
        if (int rc = encode_tmap(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a, dims, str, box,
                                 CU_TENSOR_MAP_SWIZZLE_128B))
            return rc;
    }
    const int bn = tile_bn(out_dtype, N, (M + BM - 1) / BM);
    if (int rc = encode_b_and_d(b, d, out_dtype, G, M, 1, N, K, false, bn, &tB, &tD, &tD8)) return rc;
    GemmArgs args{};
    args.routing = m_indices;
    args.d = d;
    args.status = status;
    args.wait_limit_ns = wait_limit_ns();
    args.drain_limit_ns = drain_limit_ns();
    args.M = M;
    args.ldd = N;
    args.N = N;
    args.G = G;
    args.K = static_cast<int>(K);
    args.KB = static_cast<int>(K / H_BK);
    args.num_nb = static_cast<int>(N / bn);
    args.n128 = static_cast<int>(N / 128);
    return dispatch_h<Layout::Contiguous>(out_dtype, tA, tB, tD, tD8, args, static_cast<cudaStream_t>(stream));
}

// Test hook: the BF16 GEMM's tile width for later calls (0 automatic, 128, or 256 where the output
// is bf16 and N % 256 == 0).
extern "C" int dg_testing_bf16_bn(int bn) {
    DG_CHECK_ARG(bn == 0 || bn == 128 || bn == 256, "bn must be 0, 128 or 256");
    dg::g_force_bn_h.store(bn, std::memory_order_relaxed);
    return DG_OK;
}

namespace dg {
int debug_word_gemm_bf16(uint32_t* out, bool clear) { return debug_word_local(out, clear); }
}  // namespace dg
