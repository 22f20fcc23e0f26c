// mgrouped.cuh - pieces shared by the m-grouped GEMM kernels (gemm.cu, gemm_bf16.cu): the
// layouts, the kernel arguments, and the on-device tile schedule that every CTA rebuilds at the start of a launch
// from the routing tensor ("SM120 m_grouped_fp8 contiguous kernel: illegal memory access at
// CUDA graph replay", #444 - nothing derived from routing is cached across launches).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dg.h"
#include "kernel_common.cuh"

namespace dg {

enum class Layout : int { Contiguous = 0, Masked = 1 };

constexpr int BM = 128;        // rows of an m-block (TMEM lanes)
constexpr int BK = 128;        // K per pipeline stage = scale-block size
constexpr int MAX_RUNS = 1024;  // runs of consecutive same-expert m-blocks kept in shared memory

struct GemmArgs {
    const int32_t* routing;      // m_indices [M] | psum [G] (psum != 0) | counts [G]
    const void* sfa;             // see the layout notes of each entry point
    const void* sfb;
    void* d;                     // output base (owner-thread stores of tail rows)
    int32_t* status;
    uint64_t wait_limit_ns;      // work waits
    uint64_t drain_limit_ns;     // drains of issued copies / MMAs on the way out
    int64_t M;       // Contiguous: rows; Masked: cap
    int64_t sfa_ld;  // Mp of the [K/128][Mp] activation scales
    int64_t ldd;     // output row length in elements
    int64_t N;       // output columns
    int G;
    int K;           // m-grouped K
    int KB;          // m-grouped K / 128
    int num_nb;      // output column tiles of the launched kernel
    int n128;        // N / 128 (sfb row count)
    int psum;        // Contiguous: routing holds per-expert end rows (prefix sums), not m_indices
    int dense;       // no routing tensor: Masked counts all equal cap; Contiguous (psum) one expert ending at M
    const float* c;  // fp32 accumulator added to the result (fp32 output only), row stride ldd; may alias d
#if DG_DEBUG
    int64_t dbg_rows;  // output rows the store checks allow if below the layout's (test hook); 0 = all
    int dbg_stop_at;   // test hook: CTA 0's producer stops before its n-th stage load (0 = never)
#endif
};

#if DG_DEBUG
// ---- debug-build index predicates (used through DG_CHECKED) against the extents the layouts
// give each buffer.  Rows of A, of the output and of the sfa columns in use: Masked G x cap,
// Contiguous M.
template <Layout L>
__device__ __forceinline__ int64_t layout_rows(const GemmArgs& a) {
    return L == Layout::Masked ? static_cast<int64_t>(a.G) * a.M : a.M;
}
// sfa [K/128][sfa_ld]: element (kb, m)
template <Layout L>
__device__ __forceinline__ bool sfa_in(const GemmArgs& a, int64_t kb, int64_t m) {
    return kb >= 0 && kb < a.KB && m >= 0 && m < layout_rows<L>(a) && layout_rows<L>(a) <= a.sfa_ld;
}
// sfb [G][N/128][K/128]: element (e, n-block, kb)
__device__ __forceinline__ bool sfb_in(const GemmArgs& a, int64_t e, int64_t nblk, int64_t kb) {
    return e >= 0 && e < a.G && nblk >= 0 && nblk < a.n128 && kb >= 0 && kb < a.KB;
}
// output (and C) row `row`, columns [c0, c0 + n) of a [rows][ldd] buffer with N columns in use
template <Layout L>
__device__ __forceinline__ bool out_in(const GemmArgs& a, int64_t row, int64_t c0, int n) {
    const int64_t rows = a.dbg_rows > 0 && a.dbg_rows < layout_rows<L>(a) ? a.dbg_rows : layout_rows<L>(a);
    return row >= 0 && row < rows && c0 >= 0 && c0 + n <= a.N && a.N <= a.ldd;
}
#endif

// Shared-memory bytes of the run table used by build_runs / tile_prefix: int32 prefix and x,
// int16 first / L / e (m-blocks < DG_MAX_M_BLOCKS, experts < DG_MAX_GROUPS).
constexpr int SCHED_BYTES = (MAX_RUNS + 1) * 4 + MAX_RUNS * 4 + 3 * MAX_RUNS * 2;
static_assert(DG_MAX_M_BLOCKS <= 32767 && DG_MAX_GROUPS <= 32767, "int16 run-table fields");

struct RunTable {
    int* prefix;     // [MAX_RUNS + 1] first tile of each run
    int* x;          // [MAX_RUNS] Masked: valid rows of the group (count clamped to [0, cap]);
                     //            Contiguous with prefix sums: end row of the expert
    int16_t* first;  // [MAX_RUNS] Contiguous: first m-block of the run; Masked: group
    int16_t* L;      // [MAX_RUNS] m-blocks of the run
    int16_t* e;      // [MAX_RUNS] expert of the run
    __device__ static RunTable at(uint8_t* base) {
        RunTable t;
        t.prefix = reinterpret_cast<int*>(base);
        t.x = t.prefix + (MAX_RUNS + 1);
        t.first = reinterpret_cast<int16_t*>(t.x + MAX_RUNS);
        t.L = t.first + MAX_RUNS;
        t.e = t.L + MAX_RUNS;
        return t;
    }
};

// Builds the runs of the launch from the routing tensor; every thread of the CTA calls it and
// gets the run count.  Masked: one run per group, L = ceil(count / 128).  Contiguous: maximal
// sequences of consecutive 128-row blocks whose first row carries the same expert (blocks
// whose first row is -1 are padding and skipped).  Contiguous with prefix sums (a.psum): one
// run per expert; expert e owns rows [round_up(psum[e-1], 128), psum[e]) (psum[-1] = 0) and
// rt.x holds the end row; an expert whose end is below its predecessor's, past M, or inside the
// rounding gap is flagged DG_STATUS_BAD_INDEX and it and every later expert are skipped.
// `scratch` holds one int16 per m-block.
// End row of expert e of a prefix-sum routed call (the dense form has one expert ending at M).
__device__ __forceinline__ int64_t route_end(const GemmArgs& a, int e) {
    return a.dense ? a.M : static_cast<int64_t>(a.routing[e]);
}

template <Layout L, int NT>
__device__ int build_runs(const GemmArgs& a, const RunTable& rt, int* s_scan, void* scratch) {
    const int tid = threadIdx.x;
    int R = 0;
    if constexpr (L == Layout::Masked) {
        R = a.G;
        int bad = 0;
        for (int g = tid; g < a.G; g += NT) {
            int c = a.dense ? static_cast<int>(a.M) : a.routing[g];
            if (c < 0) { bad |= DG_STATUS_COUNT_GT_CAP; c = 0; }
            if (c > a.M) { bad |= DG_STATUS_COUNT_GT_CAP; c = static_cast<int>(a.M); }
            rt.first[g] = static_cast<int16_t>(g);
            rt.e[g] = static_cast<int16_t>(g);
            rt.x[g] = c;
            rt.L[g] = static_cast<int16_t>((c + BM - 1) / BM);
        }
        if (bad && blockIdx.x == 0) status_or(a.status, bad);
        __syncthreads();
    } else if (a.psum) {
        int* s_first_bad = s_scan + NT / 32;  // scan scratch is free here
        if (tid == 0) *s_first_bad = a.G;
        __syncthreads();
        for (int e = tid; e < a.G; e += NT) {
            const int64_t prev = e > 0 ? route_end(a, e - 1) : 0;
            const int64_t end = route_end(a, e);
            const int64_t start = (prev + BM - 1) / BM * BM;
            const bool bad = prev < 0 || end < prev || end > a.M || (end > prev && end < start);
            if (bad) atomicMin(s_first_bad, e);
        }
        __syncthreads();
        const int first_bad = *s_first_bad;
        if (first_bad < a.G && blockIdx.x == 0 && tid == 0) status_or(a.status, DG_STATUS_BAD_INDEX);
        for (int e = tid; e < a.G; e += NT) {
            const int64_t prev = e > 0 ? route_end(a, e - 1) : 0;
            const int64_t end = route_end(a, e);
            const int64_t start = (prev + BM - 1) / BM * BM;
            const bool live = e < first_bad && end > start;
            rt.first[e] = static_cast<int16_t>(live ? start / BM : 0);
            rt.L[e] = static_cast<int16_t>(live ? (end - start + BM - 1) / BM : 0);
            rt.e[e] = static_cast<int16_t>(e);
            rt.x[e] = live ? static_cast<int>(end) : 0;
        }
        R = a.G;
        __syncthreads();
    } else {
        const int nblk = static_cast<int>((a.M + BM - 1) / BM);
        int16_t* blk_e = static_cast<int16_t*>(scratch);
        int bad = 0;
        for (int b = tid; b < nblk; b += NT) {
            int e = a.routing[static_cast<int64_t>(b) * BM];
            if (e < -1 || e >= a.G) { bad |= DG_STATUS_BAD_INDEX; e = -1; }
            blk_e[b] = static_cast<int16_t>(e);
        }
        if (bad && blockIdx.x == 0) status_or(a.status, bad);
        __syncthreads();
        const int ch = (nblk + NT - 1) / NT;
        const int lo = tid * ch, hi = min(nblk, lo + ch);
        int cnt = 0;
        for (int b = lo; b < hi; ++b) {
            const int e = blk_e[b];
            cnt += (e >= 0 && (b == 0 || blk_e[b - 1] != e)) ? 1 : 0;
        }
        int total = 0;
        int r = cta_excl_scan<NT>(cnt, s_scan, &total);
        for (int b = lo; b < hi; ++b) {
            const int e = blk_e[b];
            if (e >= 0 && (b == 0 || blk_e[b - 1] != e)) {
                if (r < MAX_RUNS) {
                    rt.first[r] = static_cast<int16_t>(b);
                    rt.e[r] = static_cast<int16_t>(e);
                }
                ++r;
            }
        }
        int cnt2 = 0;
        for (int b = lo; b < hi; ++b) {
            const int e = blk_e[b];
            cnt2 += (e >= 0 && (b == nblk - 1 || blk_e[b + 1] != e)) ? 1 : 0;
        }
        int total2 = 0;
        int r2 = cta_excl_scan<NT>(cnt2, s_scan, &total2);  // its barriers order the rt.first writes
        for (int b = lo; b < hi; ++b) {
            const int e = blk_e[b];
            if (e >= 0 && (b == nblk - 1 || blk_e[b + 1] != e)) {
                if (r2 < MAX_RUNS) rt.L[r2] = static_cast<int16_t>(b - rt.first[r2] + 1);
                ++r2;
            }
        }
        R = total;
        if (R > MAX_RUNS) {
            if (blockIdx.x == 0 && tid == 0) status_or(a.status, DG_STATUS_TOO_MANY_RUNS);
            R = MAX_RUNS;
        }
        __syncthreads();
    }
    return R;
}

// Tiles per run -> prefix; returns the tile count of the launch (all threads call).  A run of
// L m-blocks holds ceil(L / MB) m-tiles of MB blocks each, times num_nb column tiles.
template <int NT, int MB>
__device__ int tile_prefix(int R, int num_nb, const RunTable& rt, int* s_scan, int* s_ntiles) {
    const int tid = threadIdx.x;
    const int ch = (R + NT - 1) / NT;
    const int lo = tid * ch, hi = min(R, lo + ch);
    int sum = 0;
    for (int r = lo; r < hi; ++r) sum += (rt.L[r] + MB - 1) / MB * num_nb;
    int total = 0;
    int p = cta_excl_scan<NT>(sum, s_scan, &total);
    for (int r = lo; r < hi; ++r) {
        rt.prefix[r] = p;
        p += (rt.L[r] + MB - 1) / MB * num_nb;
    }
    if (tid == 0) {
        rt.prefix[R] = total;
        *s_ntiles = total;
    }
    __syncthreads();
    return *s_ntiles;
}

// The block-scaled MMA kernel for UE8M0 scales (gemm_mx.cu): 128 x 256 tiles, N % 256 == 0; its
// B tensor map has boxes of 128 (K) x 256 rows (FP8 codes, or FP4 codes unpacked to 16-byte
// groups when b_fp4).  Returns DG_OK or an error.
constexpr int MX_BN = 256;
int launch_mgrouped_mx(Layout L, bool out_fp32, bool b_fp4, const CUtensorMap& tA, const CUtensorMap& tB,
                       const GemmArgs& args, cudaStream_t stream);

// A tile of the launch's schedule (decoded from its index by every role of a CTA).
struct TileInfo {
    int e;        // expert / group
    int nb;       // output column tile
    int row0;     // first row of the tile: Contiguous global row, Masked row within the group
    int valid;    // Masked: valid rows of the tile (<= 128)
    int kbt;      // 128-K blocks of this tile
};

template <Layout L>
__device__ __forceinline__ TileInfo decode_tile(int t, const RunTable& rt, int R, const GemmArgs& a) {
    const int r = find_run(rt.prefix, R, t);
    const int local = t - rt.prefix[r];
    const int Lr = rt.L[r];
    const int nb = local / Lr, j = local - nb * Lr;  // m-blocks fastest: consecutive tiles share B
    TileInfo ti;
    ti.nb = nb;
    ti.e = rt.e[r];
    ti.valid = 0;
    ti.kbt = a.KB;
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

// Valid rows at the start of a tile: the count for masked / psum tiles, else the leading rows
// whose m_indices entry is the tile's expert (ballots of the four 32-row quarters).
template <Layout L>
__device__ __forceinline__ int stored_rows(const TileInfo& ti, const GemmArgs& a, const uint32_t* ballot) {
    if (L == Layout::Masked || a.psum) return ti.valid;
    int v = 0;
    for (int qq = 0; qq < 4; ++qq) {
        const uint32_t bal = ballot[qq];
        if (bal == 0xffffffffu) { v += 32; continue; }
        return v + __ffs(~bal) - 1;
    }
    return v;
}

}  // namespace dg
