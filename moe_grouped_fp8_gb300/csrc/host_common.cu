// host_common.cu - error state, device properties, TMA descriptor encoding, workspace sizes.
#include <atomic>
#include <cstdlib>
#include <mutex>

#include "host_common.hpp"

namespace dg {

namespace {
thread_local std::string g_err;
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
cudaError_t g_encode_err = cudaSuccess;
constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
}  // namespace

int set_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

const char* last_error() { return g_err.c_str(); }
void clear_error() { g_err.clear(); }

int device_sm_count(int* out) {
    int dev = 0;
    DG_CHECK_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return set_error(DG_ERR_UNSUPPORTED, "device index %d", dev);
    if (g_sm_count[dev] == 0) {
        int n = 0;
        DG_CHECK_CUDA(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
        g_sm_count[dev] = n;
    }
    *out = g_sm_count[dev];
    return DG_OK;
}

uint64_t drain_limit_ns() {
    static uint64_t v = [] {
#if DG_DEBUG
        constexpr long long kDefaultMs = 250;  // the debug build gives up sooner
#else
        constexpr long long kDefaultMs = 2000;
#endif
        const char* s = std::getenv("DG_WAIT_LIMIT_MS");
        long long ms = s ? std::atoll(s) : kDefaultMs;
        if (ms <= 0) ms = kDefaultMs;
        return static_cast<uint64_t>(ms) * 1000000ull;
    }();
    return v;
}

namespace {
std::atomic<uint64_t> g_wait_override_ns{0};
}

uint64_t wait_limit_ns() {
    const uint64_t o = g_wait_override_ns.load(std::memory_order_relaxed);
    return o != 0 ? o : drain_limit_ns();
}

namespace {
std::mutex g_log_mu;
std::string g_log_path;
std::atomic<bool> g_log_on{false};
uint64_t g_log_seq = 0;

// the environment's log file, read once when the library is loaded
[[maybe_unused]] const bool g_log_env = [] {
    const char* p = std::getenv("DG_ARG_LOG");
    if (p != nullptr && *p != '\0') {
        g_log_path = p;
        g_log_on.store(true);
    }
    return true;
}();
}  // namespace

bool arg_log_on() { return g_log_on.load(std::memory_order_relaxed); }

// One line per call: a sequence number, the entry point, then name=value for every argument.  It
// reads nothing from the device, so it is safe in stream capture and before any check.
void arg_log_write(const char* fn, const std::string& body) {
    std::lock_guard<std::mutex> lk(g_log_mu);
    if (g_log_path.empty()) return;
    FILE* f = std::fopen(g_log_path.c_str(), "a");
    if (f == nullptr) return;
    std::fprintf(f, "%llu %s %s\n", static_cast<unsigned long long>(g_log_seq++), fn, body.c_str());
    std::fclose(f);
}

int encode_tmap(CUtensorMap* tm, CUtensorMapDataType dtype, uint32_t rank, const void* base,
                const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (g_encode == nullptr)
        return set_error(DG_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorString(g_encode_err));
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(tm, dtype, rank, const_cast<void*>(base), reinterpret_cast<const cuuint64_t*>(dims),
                          reinterpret_cast<const cuuint64_t*>(strides_bytes), reinterpret_cast<const cuuint32_t*>(box),
                          elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(DG_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the layout (CUresult %d)", (int)r);
    return DG_OK;
}

}  // namespace dg

extern "C" const char* dg_last_error(void) { return dg::last_error(); }

extern "C" int dg_debug_build(void) {
#if DG_DEBUG
    return 1;
#else
    return 0;
#endif
}

extern "C" int dg_debug_word(uint32_t* out, int clear) {
    DG_CHECK_ARG(out != nullptr, "out must not be NULL");
    *out = 0;
    DG_CHECK_CUDA(cudaDeviceSynchronize());
    for (auto fn : {dg::debug_word_quant, dg::debug_word_gemm, dg::debug_word_gemm_mx, dg::debug_word_gemm_bf16,
                    dg::debug_word_kgrouped})
        if (int rc = fn(out, clear != 0)) return dg::set_error(rc, "reading a debug word failed");
    return DG_OK;
}

extern "C" int dg_set_arg_log(const char* path) {
    std::lock_guard<std::mutex> lk(dg::g_log_mu);
    dg::g_log_path = path != nullptr ? path : "";
    dg::g_log_on.store(!dg::g_log_path.empty(), std::memory_order_relaxed);
    return DG_OK;
}

extern "C" size_t dg_workspace_size(int op, int G, int64_t M, int64_t N, int64_t K) {
    DG_ARG_LOG(op, G, M, N, K);
    (void)M;
    (void)N;
    (void)K;
    if (op == DG_OP_K_GROUPED_WGRAD && G > 0) return static_cast<size_t>(G) * 2 * 128;  // two tensor maps per expert
    return 0;
}

// Test hook: the limit of the kernels' work waits for later calls in this process (0 restores the
// default).  Drains on the way out keep the default limit, so that a kernel whose work waits gave
// up still waits for the copies and MMAs it issued before it frees tensor memory and exits.
extern "C" int dg_testing_wait_limit_ns(uint64_t ns) {
    dg::g_wait_override_ns.store(ns, std::memory_order_relaxed);
    return DG_OK;
}
