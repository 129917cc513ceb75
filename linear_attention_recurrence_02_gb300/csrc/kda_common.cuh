// kda_common.cuh -- internal helpers shared by the libkda.so sources.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>
#include <string>

#include "kda.h"

namespace kda {

// ---------------------------------------------------------------- host side
void set_detail(const std::string &msg);
void clear_detail();
kda_status fail(kda_status s, const std::string &msg);
kda_status invalid(const std::string &msg);

// Make the stream's device current for this library's runtime instance.
kda_status bind_stream_device(kda_stream_t stream);

// Map the last launch error to a status (does not synchronise).
kda_status check_launch(const char *what);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool valid_head_dim(int D) { return D == 16 || D == 32 || D == 64 || D == 128; }

kda_status check_ptr(const void *p, const char *name);

// Device-side error word (one per device): bit 0 = bad cu_seqlens,
// bit 1 = bounded wait timed out.
enum : unsigned { DEVERR_SEQLENS = 1u, DEVERR_TIMEOUT = 2u };
unsigned *device_error_word();  // device address of the word on the current device

// Device address of a file-scope __device__ variable on the current device.
// The lookup is cached per device and keyed on the CUDA context that was
// current when it was made: after a cudaDeviceReset the primary context, and
// with it the variable's address, is new, and the next call looks it up again.
struct SymbolCache {
    static constexpr int MAX_DEV = 64;
    std::mutex mu;
    void *addr[MAX_DEV] = {};
    void *ctx[MAX_DEV] = {};
};
kda_status symbol_address(const void *symbol, SymbolCache &cache, void **out);

// Opt a kernel into more than 48 KiB of dynamic shared memory, once per device.
template <auto Kern>
inline cudaError_t smem_attr_once(int bytes) {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// ---------------------------------------------------------------- device side
template <typename T> struct Elem;
template <> struct Elem<float> {
    __device__ __forceinline__ static float load(const float *p) { return *p; }
    __device__ __forceinline__ static void store(float *p, float x) { *p = x; }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ __forceinline__ static float load(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }
};

// 1 / sqrt(ss + eps), or 0 when ss + eps == 0 (zero vector stays zero).
__device__ __forceinline__ float inv_norm(float ss, float eps) {
    float den = ss + eps;
    return den > 0.f ? 1.0f / sqrtf(den) : 0.f;
}

}  // namespace kda
