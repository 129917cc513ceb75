// kda_abi.cu -- status strings, size helpers, device selection and the
// device-side error word of libkda.so. The compute entry points live beside
// their kernels (kda_decode.cu, kda_shortconv.cu, kda_prefill*.cu).
#include <cstdio>
#include <string>

#include <atomic>
#include <mutex>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {

static thread_local std::string g_detail;

void set_detail(const std::string &msg) { g_detail = msg; }
void clear_detail() { g_detail.clear(); }

kda_status fail(kda_status s, const std::string &msg) {
    set_detail(msg);
    return s;
}

kda_status invalid(const std::string &msg) { return fail(KDA_ERR_INVALID_ARG, msg); }

kda_status check_ptr(const void *p, const char *name) {
    if (p == nullptr) return invalid(std::string(name) + " is NULL");
    if (!aligned16(p)) return invalid(std::string(name) + " is not 16-byte aligned");
    return KDA_OK;
}

kda_status bind_stream_device(kda_stream_t stream) {
    int dev = -1;
    if (stream != nullptr) {
        // A stream being captured into a CUDA graph does not permit
        // cudaStreamGetDevice; the capturing thread's current device is the
        // stream's device then, so it is kept as it is.
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(reinterpret_cast<cudaStream_t>(stream), &cs) == cudaSuccess &&
            cs != cudaStreamCaptureStatusNone)
            return KDA_OK;
        cudaGetLastError();
        cudaError_t e = cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &dev);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(KDA_ERR_CUDA, std::string("cudaStreamGetDevice: ") + cudaGetErrorString(e));
        }
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != dev) {
            e = cudaSetDevice(dev);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(KDA_ERR_CUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(e));
            }
        }
    }
    return KDA_OK;
}

kda_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(KDA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
    return KDA_OK;
}

__device__ unsigned g_device_error_word;

// The CUDA context current on the calling thread, through the driver entry
// point (the library links only the runtime). NULL when none is current.
static void *current_context() {
    typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
    static std::atomic<CtxGetCurrentFn> fn{nullptr};
    CtxGetCurrentFn f = fn.load(std::memory_order_acquire);
    if (f == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || p == nullptr) {
            cudaGetLastError();
            return nullptr;
        }
        f = reinterpret_cast<CtxGetCurrentFn>(p);
        fn.store(f, std::memory_order_release);
    }
    CUcontext c = nullptr;
    return f(&c) == CUDA_SUCCESS ? static_cast<void *>(c) : nullptr;
}

kda_status symbol_address(const void *symbol, SymbolCache &cache, void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(KDA_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    }
    if (dev < 0 || dev >= SymbolCache::MAX_DEV) return fail(KDA_ERR_UNSUPPORTED, "device index above 63");
    std::lock_guard<std::mutex> lock(cache.mu);
    void *ctx = current_context();
    if (cache.addr[dev] != nullptr && ctx != nullptr && ctx == cache.ctx[dev]) {
        *out = cache.addr[dev];
        return KDA_OK;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, symbol);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return fail(KDA_ERR_CUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    }
    // the lookup makes the device's primary context current if none was
    cache.addr[dev] = p;
    cache.ctx[dev] = ctx != nullptr ? ctx : current_context();
    *out = p;
    return KDA_OK;
}

unsigned *device_error_word() {
    static SymbolCache cache;
    void *p = nullptr;
    if (symbol_address(&g_device_error_word, cache, &p) != KDA_OK) return nullptr;
    return static_cast<unsigned *>(p);
}

}  // namespace kda

using namespace kda;

extern "C" const char *kda_status_string(kda_status s) {
    switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: not supported by this build";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA: CUDA runtime error";
    case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: device-side wait timed out";
    case KDA_ERR_DEVICE_CHECK: return "KDA_ERR_DEVICE_CHECK: kernel found invalid input data";
    }
    return "unknown kda_status";
}

extern "C" const char *kda_last_error_detail(void) { return g_detail.c_str(); }

extern "C" int kda_abi_version(void) { return 1; }

extern "C" size_t kda_state_bytes(int layers, int heads, int dk, int dv) {
    if (layers < 0 || heads < 0 || dk < 0 || dv < 0) return 0;
    return (size_t)layers * (size_t)heads * (size_t)dk * (size_t)dv * sizeof(float);
}

extern "C" size_t kda_shortconv_ring_bytes(int layers, int batch, int heads, int d, int elem_bytes) {
    if (layers < 0 || batch < 0 || heads < 0 || d < 0 || elem_bytes < 0) return 0;
    return (size_t)layers * (size_t)batch * (size_t)heads * 3u * 3u * (size_t)d * (size_t)elem_bytes;
}

namespace kda {
// One mbarrier that nothing completes; thread 0 waits on it with the bounded wait.
__global__ void selftest_wait_kernel(long long limit, unsigned *err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
        if (!tc::mbar_wait(&bar, 0, limit)) atomicOr(err, DEVERR_TIMEOUT);
    }
}
}  // namespace kda

extern "C" kda_status kda_selftest_bounded_wait(long long limit_cycles, kda_stream_t stream) {
    clear_detail();
    if (limit_cycles < 1 || limit_cycles > 2000000000LL) return invalid("limit_cycles must be in 1 .. 2e9");
    kda_status st = bind_stream_device(stream);
    if (st != KDA_OK) return st;
    unsigned *err = device_error_word();
    if (!err) return fail(KDA_ERR_CUDA, "device error word unavailable");
    selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_cycles, err);
    return check_launch("selftest_wait_kernel");
}

extern "C" kda_status kda_sync_status(kda_stream_t stream) {
    clear_detail();
    kda_status st = bind_stream_device(stream);
    if (st != KDA_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaStreamSynchronize: ") + cudaGetErrorString(e));
    unsigned word = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("error word: ") + cudaGetErrorString(e));
    if (word & DEVERR_TIMEOUT) return fail(KDA_ERR_TIMEOUT, "a bounded device-side wait gave up");
    if (word & DEVERR_SEQLENS)
        return fail(KDA_ERR_DEVICE_CHECK, "cu_seqlens is not non-decreasing from 0 to T; affected sequences skipped");
    return KDA_OK;
}
