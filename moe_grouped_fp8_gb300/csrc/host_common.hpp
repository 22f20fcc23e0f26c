// host_common.hpp - host-side helpers of the C ABI: thread-local error messages, argument
// checks, device properties, and TMA descriptor encoding through the driver entry point
// (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <string>
#include <type_traits>
#include <utility>

#include "dg.h"

namespace dg {

int set_error(int code, const char* fmt, ...);
const char* last_error();
void clear_error();

#define DG_CHECK_ARG(cond, ...)                                               \
    do {                                                                      \
        if (!(cond)) return ::dg::set_error(DG_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)
#define DG_CHECK_SUPPORTED(cond, ...)                                         \
    do {                                                                      \
        if (!(cond)) return ::dg::set_error(DG_ERR_UNSUPPORTED, __VA_ARGS__); \
    } while (0)
#define DG_CHECK_CUDA(expr)                                                                     \
    do {                                                                                        \
        cudaError_t e_ = (expr);                                                                \
        if (e_ != cudaSuccess)                                                                  \
            return ::dg::set_error(DG_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
    } while (0)

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- argument log: when a log file is set (env DG_ARG_LOG, or dg_set_arg_log), every entry point
// appends one line with its name and arguments before it checks them.
bool arg_log_on();
void arg_log_write(const char* fn, const std::string& body);

template <typename T>
void arg_log_value(std::string& s, const T& v) {
    char b[48];
    if constexpr (std::is_pointer_v<T>)
        snprintf(b, sizeof(b), "%p", static_cast<const void*>(v));
    else if constexpr (std::is_floating_point_v<T>)
        snprintf(b, sizeof(b), "%.9g", static_cast<double>(v));
    else
        snprintf(b, sizeof(b), "%lld", static_cast<long long>(v));
    s += b;
}

// names: the comma-separated argument expressions as written at the call site
template <typename... T>
void arg_log(const char* fn, const char* names, const T&... v) {
    std::string s;
    const char* n = names;
    auto one = [&](const auto& x) {
        while (*n == ' ' || *n == ',') ++n;
        const char* e = n;
        while (*e != '\0' && *e != ',') ++e;
        if (!s.empty()) s += ' ';
        s.append(n, e);
        s += '=';
        arg_log_value(s, x);
        n = e;
    };
    (one(v), ...);
    arg_log_write(fn, s);
}

#define DG_ARG_LOG(...)                                                                       \
    do {                                                                                      \
        if (::dg::arg_log_on()) ::dg::arg_log(__func__, #__VA_ARGS__, __VA_ARGS__);           \
    } while (0)

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count(int* out);

// Upper bound, in nanoseconds, of the kernels' work waits (env DG_WAIT_LIMIT_MS, default 2000 ms,
// 250 ms in the debug build; a test hook may shorten it).
uint64_t wait_limit_ns();
// Upper bound of the waits that drain a kernel's copies and MMAs on its way out (the default limit,
// never shortened by the test hook).
uint64_t drain_limit_ns();

// The debug words of the kernels' translation units (each ORs its word into *out, then clears it
// if `clear`); dg_debug_word() combines them.
int debug_word_quant(uint32_t* out, bool clear);
int debug_word_gemm(uint32_t* out, bool clear);
int debug_word_gemm_mx(uint32_t* out, bool clear);
int debug_word_gemm_bf16(uint32_t* out, bool clear);
int debug_word_kgrouped(uint32_t* out, bool clear);

// cuTensorMapEncodeTiled through cudaGetDriverEntryPointByVersion; returns DG_OK or an error
// code with a message.
int encode_tmap(CUtensorMap* tm, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                const uint64_t* dims, const uint64_t* strides_bytes /* rank-1 entries */,
                const uint32_t* box, CUtensorMapSwizzle swizzle);

// Launch `kernel` on `stream` with programmatic stream serialization, so that its launch and
// set-up overlap the previous kernel in the stream; the kernel calls pdl_wait() before touching
// global memory.  Returns DG_OK or DG_ERR_CUDA.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) return set_error(DG_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return DG_OK;
}

}  // namespace dg
