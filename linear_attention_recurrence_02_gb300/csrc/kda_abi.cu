// kda_abi.cu -- status strings, size helpers, device selection and the
// device-side error word of libkda.so. The compute entry points live beside
// their kernels (kda_decode.cu, kda_shortconv.cu, kda_prefill*.cu).
#include <cstdio>
#include <string>

#include <atomic>

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

unsigned *device_error_word() {
    // looked up once per device (the calling thread's current device)
    static std::atomic<unsigned *> cache[64];
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        unsigned *c = cache[dev].load(std::memory_order_acquire);
        if (c) return c;
    } else {
        cudaGetLastError();
        dev = -1;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (dev >= 0) cache[dev].store(static_cast<unsigned *>(p), std::memory_order_release);
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
