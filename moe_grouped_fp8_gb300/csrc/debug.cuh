// debug.cuh - device-side index checks of the debug build (compiled with -DDG_DEBUG=1).
//
// Every global access whose address the kernels compute from call arguments (scale reads,
// owner-thread stores, C reads, the casts' element reads and writes) can be guarded by
// DG_CHECKED(in_bounds, bit): in a debug build a failed check ORs `bit` into this translation
// unit's debug word and yields false, so that the caller skips the access (nothing traps,
// nothing is read or written out of bounds).  In the release build the macro is the literal
// `true` and its condition is not compiled at all, so the release kernels are the same code as
// without the checks.  TMA copies need no such check: the tensor map bounds every box.  The host
// reads and clears the words with dg_debug_word().
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "dg.h"

#ifndef DG_DEBUG
#define DG_DEBUG 0
#endif

namespace dg {
namespace {
__device__ uint32_t g_debug_word;  // one per translation unit

// This translation unit's word: copied to *out (ORed in) and, if `clear`, reset to 0.
[[maybe_unused]] int debug_word_local(uint32_t* out, bool clear) {
    uint32_t w = 0;
    if (cudaMemcpyFromSymbol(&w, g_debug_word, sizeof(w)) != cudaSuccess) return DG_ERR_CUDA;
    *out |= w;
    if (clear) {
        const uint32_t z = 0;
        if (cudaMemcpyToSymbol(g_debug_word, &z, sizeof(z)) != cudaSuccess) return DG_ERR_CUDA;
    }
    return DG_OK;
}
}  // namespace

#if DG_DEBUG
__device__ __forceinline__ bool dbg_check(bool ok, uint32_t bit) {
    if (!ok) atomicOr(&g_debug_word, bit);
    return ok;
}
#define DG_CHECKED(cond, bit) ::dg::dbg_check((cond), (bit))
#else
#define DG_CHECKED(cond, bit) true
#endif

}  // namespace dg
