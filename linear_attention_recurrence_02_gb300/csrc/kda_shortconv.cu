// kda_shortconv.cu -- decode step of the width-4 causal depthwise short
// convolution + SiLU in front of q, k, v, with its 3-token ring
// ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析",
// sections "KDA 递推公式先衰减再差分" and "414MB 的 KDA 状态从哪来").
//
// Memory-bound elementwise work: each thread owns 16 bytes of channels of one
// (b, projection, h) row: it reads x and the three ring slots with 128-bit
// loads, the 4 taps per channel as float4, writes y and the shifted ring.
// y is written projection-major, [3,B,H,D], so that y[0], y[1], y[2] are the
// contiguous q, k, v operands of the decode step.
#include "kda_common.cuh"

namespace kda {

template <typename T> struct Vec16;  // 16 bytes of T
template <> struct Vec16<float> { static constexpr int N = 4; };
template <> struct Vec16<__nv_bfloat16> { static constexpr int N = 8; };

template <typename T>
__device__ __forceinline__ void load16(const T *p, float (&out)[Vec16<T>::N]) {
    uint4 raw = __ldcs(reinterpret_cast<const uint4 *>(p));
    const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
    for (int i = 0; i < Vec16<T>::N; ++i) out[i] = Elem<T>::load(e + i);
}

template <typename T>
__device__ __forceinline__ void store16(T *p, const float (&in)[Vec16<T>::N]) {
    uint4 raw;
    T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
    for (int i = 0; i < Vec16<T>::N; ++i) Elem<T>::store(e + i, in[i]);
    __stcs(reinterpret_cast<uint4 *>(p), raw);
}

template <typename T>
__global__ void __launch_bounds__(256) shortconv_step_kernel(const T *__restrict__ x, T *__restrict__ ring,
                                                             const float *__restrict__ w, T *__restrict__ y,
                                                             int B, int H, int D) {
    constexpr int V = Vec16<T>::N;
    const int nvec = D / V;
    const size_t total = (size_t)B * 3 * H * nvec;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int cv = (int)(idx % nvec);
    const size_t row = idx / nvec;  // (b*3 + p)*H + h
    const int h = (int)(row % H);
    const int p = (int)((row / H) % 3);
    const size_t b = row / ((size_t)3 * H);
    const size_t xoff = row * D + (size_t)cv * V;
    const size_t yoff = (((size_t)p * B + b) * H + h) * D + (size_t)cv * V;
    const size_t roff = row * 3 * D + (size_t)cv * V;
    const float *wt = w + (((size_t)p * H + h) * D + (size_t)cv * V) * 4;

    float xv[V], r0[V], r1[V], r2[V], yv[V];
    load16(x + xoff, xv);
    load16(ring + roff, r0);
    load16(ring + roff + D, r1);
    load16(ring + roff + 2 * (size_t)D, r2);
#pragma unroll
    for (int i = 0; i < V; ++i) {
        float4 tap = __ldg(reinterpret_cast<const float4 *>(wt) + i);
        float z = tap.x * r0[i] + tap.y * r1[i] + tap.z * r2[i] + tap.w * xv[i];
        yv[i] = z / (1.0f + expf(-z));
    }
    store16(y + yoff, yv);
    store16(ring + roff, r1);
    store16(ring + roff + D, r2);
    store16(ring + roff + 2 * (size_t)D, xv);
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_shortconv_step(const void *x, void *ring, const float *w, void *y, int B, int H,
                                         int D, kda_dtype dtype, kda_stream_t stream) {
    clear_detail();
    if (B < 0) return invalid("B must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (B == 0) return KDA_OK;
    kda_status st;
    if ((st = check_ptr(x, "x")) || (st = check_ptr(ring, "ring")) || (st = check_ptr(w, "w")) ||
        (st = check_ptr(y, "y")))
        return st;
    if (y == x || y == ring) return invalid("y must not alias x or ring");
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int V = dtype == KDA_BF16 ? 8 : 4;
    const size_t total = (size_t)B * 3 * H * (D / V);
    const unsigned blocks = (unsigned)((total + 255) / 256);
    if (dtype == KDA_BF16)
        shortconv_step_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(ring), w,
            static_cast<__nv_bfloat16 *>(y), B, H, D);
    else
        shortconv_step_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float *>(x),
                                                            static_cast<float *>(ring), w,
                                                            static_cast<float *>(y), B, H, D);
    return check_launch("shortconv_step_kernel");
}
