// kda_shortconv.cu -- decode step of the width-4 causal depthwise short
// convolution + SiLU in front of q, k, v, with its 3-token ring
// ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析",
// sections "KDA 递推公式先衰减再差分" and "414MB 的 KDA 状态从哪来").
//
// Memory-bound elementwise work: each thread owns 16 bytes of channels of one
// (projection, h) pair for two sequences: it loads the 4 taps per channel
// once (float4), issues the 128-bit loads of x and the three ring slots of
// both sequences before using any, and writes y and the shifted ring (the
// ring's stored vectors move unchanged).
// y is written projection-major, [3,B,H,D], so that y[0], y[1], y[2] are the
// contiguous q, k, v operands of the decode step.
//
// The prefill form runs the same convolution over packed sequences: each
// thread owns four channels of one (projection, head) and walks
// a tile of 64 tokens with the 3-token window in registers. A tile's history
// comes from the tokens before it, or from the sequence's ring where the
// sequence starts, so tiles are independent; the thread that processes a
// sequence's last token writes its ring for the decode hand-off.
#include <string>

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

// One thread per 16 bytes of channels of one (projection, head) and a group
// of STEP_BPT sequences: the taps of its channels are loaded once and kept in
// registers for every sequence of the group, and the group's loads are all
// issued before any is used (one 16-byte x vector and three ring slots each).
// Measured at 64 sequences x 96 heads (bf16): 1 sequence per thread 14.4 us,
// 2 sequences 12.4 us, 4 sequences 14.4 us (133 registers: 1.3 waves); the
// first form, one thread per (sequence, projection, head) vector re-reading
// the taps for every sequence in 256-thread blocks, 16.4 us.
constexpr int STEP_BPT = 2;
constexpr int STEP_NT = 128;
template <typename T>
__global__ void __launch_bounds__(STEP_NT) shortconv_step_kernel(const T *__restrict__ x, T *__restrict__ ring,
                                                             const float *__restrict__ w, T *__restrict__ y,
                                                             int B, int H, int D) {
    constexpr int V = Vec16<T>::N;
    const int nvec = D / V;
    const int ngroups = (B + STEP_BPT - 1) / STEP_BPT;
    const size_t total = (size_t)ngroups * 3 * H * nvec;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int cv = (int)(idx % nvec);
    const size_t r = idx / nvec;
    const int h = (int)(r % H);
    const int p = (int)((r / H) % 3);
    const int b0 = (int)(r / ((size_t)3 * H)) * STEP_BPT;
    const float4 *wt = reinterpret_cast<const float4 *>(w + (((size_t)p * H + h) * D + (size_t)cv * V) * 4);
    float4 tap[V];
#pragma unroll
    for (int i = 0; i < V; ++i) tap[i] = __ldg(wt + i);

    // raw 16-byte vectors in flight: x and the three slots of every sequence of the group
    uint4 xr[STEP_BPT], rr[STEP_BPT][3];
#pragma unroll
    for (int bb = 0; bb < STEP_BPT; ++bb) {
        if (b0 + bb >= B) break;
        const size_t row = ((size_t)(b0 + bb) * 3 + p) * H + h;  // (b*3 + p)*H + h
        const size_t xoff = row * D + (size_t)cv * V, roff = row * 3 * D + (size_t)cv * V;
        xr[bb] = __ldcs(reinterpret_cast<const uint4 *>(x + xoff));
#pragma unroll
        for (int k = 0; k < 3; ++k) rr[bb][k] = __ldcs(reinterpret_cast<const uint4 *>(ring + roff + (size_t)k * D));
    }
#pragma unroll
    for (int bb = 0; bb < STEP_BPT; ++bb) {
        const int b = b0 + bb;
        if (b >= B) break;
        const size_t row = ((size_t)b * 3 + p) * H + h;
        const size_t roff = row * 3 * D + (size_t)cv * V;
        const size_t yoff = (((size_t)p * B + b) * H + h) * D + (size_t)cv * V;
        const T *xe = reinterpret_cast<const T *>(&xr[bb]);
        const T *e0 = reinterpret_cast<const T *>(&rr[bb][0]);
        const T *e1 = reinterpret_cast<const T *>(&rr[bb][1]);
        const T *e2 = reinterpret_cast<const T *>(&rr[bb][2]);
        float yv[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const float z = tap[i].x * Elem<T>::load(e0 + i) + tap[i].y * Elem<T>::load(e1 + i) +
                            tap[i].z * Elem<T>::load(e2 + i) + tap[i].w * Elem<T>::load(xe + i);
            yv[i] = z / (1.0f + expf(-z));
        }
        store16(y + yoff, yv);
        // the ring shifts: its stored values move unchanged
        __stcs(reinterpret_cast<uint4 *>(ring + roff), rr[bb][1]);
        __stcs(reinterpret_cast<uint4 *>(ring + roff + D), rr[bb][2]);
        __stcs(reinterpret_cast<uint4 *>(ring + roff + 2 * (size_t)D), xr[bb]);
    }
}

constexpr int CONV_TILE = 64;  // tokens per prefill tile

template <typename T>
__device__ __forceinline__ void zero16(float (&out)[Vec16<T>::N]) {
#pragma unroll
    for (int i = 0; i < Vec16<T>::N; ++i) out[i] = 0.f;
}

// 4 channels per thread in the prefill form: 8-byte bf16 or 16-byte fp32 vectors
template <typename T> struct Vec4;
template <> struct Vec4<float> { using Raw = uint4; };
template <> struct Vec4<__nv_bfloat16> { using Raw = uint2; };

template <typename T>
__device__ __forceinline__ void unpack4(typename Vec4<T>::Raw raw, float (&out)[4]) {
    const T *e = reinterpret_cast<const T *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = Elem<T>::load(e + i);
}
template <typename T>
__device__ __forceinline__ void load4(const T *p, float (&out)[4]) {
    unpack4<T>(__ldcs(reinterpret_cast<const typename Vec4<T>::Raw *>(p)), out);
}
template <typename T>
__device__ __forceinline__ void store4(T *p, const float (&in)[4]) {
    typename Vec4<T>::Raw raw;
    T *e = reinterpret_cast<T *>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) Elem<T>::store(e + i, in[i]);
    __stcs(reinterpret_cast<typename Vec4<T>::Raw *>(p), raw);
}

// One work item = (token tile, group of 256 four-channel vectors of a token
// row); a persistent grid walks the items, tile-major.
template <typename T>
__global__ void __launch_bounds__(256, 3) shortconv_prefill_kernel(
    const T *__restrict__ x, const T *__restrict__ ring_in, const float *__restrict__ w, T *__restrict__ y,
    T *__restrict__ ring_out, const int64_t *__restrict__ cu, int N, int64_t Ttot, int H, int D, unsigned *err,
    long long ntiles, int ngroups) {
    constexpr int V = 4;
    using Raw = typename Vec4<T>::Raw;
    constexpr int BATCH = sizeof(Raw) == 8 ? 16 : 4;  // token loads in flight per thread
    const int nvec = D / V;
    const size_t row = (size_t)3 * H * D;      // x elements per token
    const size_t rsz = (size_t)9 * H * D;      // ring elements per sequence
    const size_t ystride = (size_t)H * D;
    for (long long item = blockIdx.x; item < ntiles * ngroups; item += gridDim.x) {
        const long long tile = item / ngroups;
        const int vi = (int)(item % ngroups) * blockDim.x + threadIdx.x;
        if (vi >= 3 * H * nvec) continue;
        const int cv = vi % nvec, ph = vi / nvec;  // ph = p * H + h
        const int h = ph % H, p = ph / H;
        const size_t xo = (size_t)ph * D + (size_t)cv * V;
        const size_t ro = (size_t)ph * 3 * D + (size_t)cv * V;
        T *yb = y + (size_t)p * Ttot * H * D + (size_t)h * D + (size_t)cv * V;  // + t * ystride

        // Sequences with no tokens pass their ring through (first tile only).
        if (tile == 0 && ring_out) {
            for (int n = 0; n < N; ++n) {
                if ((cu ? cu[n + 1] - cu[n] : Ttot) != 0) continue;
                float r[V];
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    if (ring_in) load4(ring_in + n * rsz + ro + (size_t)m * D, r);
                    else r[0] = r[1] = r[2] = r[3] = 0.f;
                    store4(ring_out + n * rsz + ro + (size_t)m * D, r);
                }
            }
        }
        const int64_t t0 = tile * CONV_TILE;
        const int64_t t1 = t0 + CONV_TILE < Ttot ? t0 + CONV_TILE : Ttot;
        if (t0 >= t1) continue;

        // the sequence holding t0: the last n with cu[n] <= t0
        int n = 0;
        int64_t sn = 0, en = Ttot;
        if (cu) {
            if (cu[0] != 0 || cu[N] != Ttot) {
                if (err) atomicOr(err, DEVERR_SEQLENS);
                continue;
            }
            int lo = 0, hi = N - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (cu[mid] <= t0) lo = mid;
                else hi = mid - 1;
            }
            n = lo;
            sn = cu[n];
            en = cu[n + 1];
            if (!(0 <= sn && sn <= t0 && t0 < en && en <= Ttot)) {
                if (err) atomicOr(err, DEVERR_SEQLENS);
                continue;
            }
        }
        float4 tap[V];
#pragma unroll
        for (int i = 0; i < V; ++i)
            tap[i] = __ldg(reinterpret_cast<const float4 *>(w + ((size_t)ph * D + (size_t)cv * V) * 4) + i);

        // window x_{t-3}, x_{t-2}, x_{t-1}: a token of this sequence, else a ring slot
        float r0[V], r1[V], r2[V];
        auto hist = [&](int64_t j, float (&out)[V]) {
            if (j >= sn) load4(x + (size_t)j * row + xo, out);
            else if (ring_in) load4(ring_in + (size_t)n * rsz + ro + (size_t)(j - sn + 3) * D, out);
            else out[0] = out[1] = out[2] = out[3] = 0.f;
        };
        auto step = [&](const float (&xv)[V], int64_t t) {
            float yv[V];
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const float z = tap[i].x * r0[i] + tap[i].y * r1[i] + tap[i].z * r2[i] + tap[i].w * xv[i];
                yv[i] = __fdividef(z, 1.0f + __expf(-z));
                r0[i] = r1[i];
                r1[i] = r2[i];
                r2[i] = xv[i];
            }
            store4(yb + (size_t)t * ystride, yv);
        };
        hist(t0 - 3, r0);
        hist(t0 - 2, r1);
        hist(t0 - 1, r2);
        int64_t t = t0;
        bool bad = false;
        while (t < t1) {
            const int64_t te = en < t1 ? en : t1;
            for (; t + BATCH <= te; t += BATCH) {
                Raw raw[BATCH];
#pragma unroll
                for (int u = 0; u < BATCH; ++u) raw[u] = __ldcs(reinterpret_cast<const Raw *>(x + (size_t)(t + u) * row + xo));
#pragma unroll
                for (int u = 0; u < BATCH; ++u) {
                    float xv[V];
                    unpack4<T>(raw[u], xv);
                    step(xv, t + u);
                }
            }
            for (; t < te; ++t) {
                float xv[V];
                load4(x + (size_t)t * row + xo, xv);
                step(xv, t);
            }
            if (t < en) break;  // tile ends inside the sequence
            if (ring_out) {
                store4(ring_out + (size_t)n * rsz + ro, r0);
                store4(ring_out + (size_t)n * rsz + ro + D, r1);
                store4(ring_out + (size_t)n * rsz + ro + 2 * (size_t)D, r2);
            }
            if (t >= t1) break;
            // next sequence with tokens; it must start here
            do {
                if (n + 1 >= N) {
                    bad = true;
                    break;
                }
                ++n;
                sn = cu[n];
                en = cu[n + 1];
            } while (en == sn && sn == t);
            if (bad || sn != t || en < sn || en > Ttot) {
                bad = true;
                break;
            }
            hist(t - 3, r0);
            hist(t - 2, r1);
            hist(t - 1, r2);
        }
        if (bad && err) atomicOr(err, DEVERR_SEQLENS);
    }
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
    const size_t total = (size_t)((B + STEP_BPT - 1) / STEP_BPT) * 3 * H * (D / V);
    const unsigned blocks = (unsigned)((total + STEP_NT - 1) / STEP_NT);
    if (dtype == KDA_BF16)
        shortconv_step_kernel<__nv_bfloat16><<<blocks, STEP_NT, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<__nv_bfloat16 *>(ring), w,
            static_cast<__nv_bfloat16 *>(y), B, H, D);
    else
        shortconv_step_kernel<float><<<blocks, STEP_NT, 0, s>>>(static_cast<const float *>(x),
                                                            static_cast<float *>(ring), w,
                                                            static_cast<float *>(y), B, H, D);
    return check_launch("shortconv_step_kernel");
}

extern "C" kda_status kda_shortconv_prefill(const void *x, const void *ring_in, const float *w, void *y,
                                            void *ring_out, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                            int D, kda_dtype dtype, kda_stream_t stream) {
    clear_detail();
    if (N < 1) return invalid("N must be >= 1");
    if (T < 0) return invalid("T must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (!cu_seqlens && N != 1) return invalid("cu_seqlens may be NULL only for N = 1");
    kda_status st;
    if ((st = check_ptr(w, "w"))) return st;
    if (T > 0 && ((st = check_ptr(x, "x")) || (st = check_ptr(y, "y")))) return st;
    if (ring_in && (st = check_ptr(ring_in, "ring_in"))) return st;
    if (ring_out && (st = check_ptr(ring_out, "ring_out"))) return st;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 7))
        return invalid("cu_seqlens must be 8-byte aligned");
    if (y && (y == x || y == ring_in || y == ring_out)) return invalid("y must not alias x or a ring");
    if (ring_out && (ring_out == ring_in || ring_out == x)) return invalid("ring_out must not alias ring_in or x");
    if (T == 0 && !ring_out) return KDA_OK;
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const long long vecs = 3LL * H * (D / 4);
    const long long groups = (vecs + 255) / 256;
    const long long tiles = T > 0 ? (T + CONV_TILE - 1) / CONV_TILE : 1;
    if (groups > 0x7fffffffLL || tiles > (1LL << 40)) return fail(KDA_ERR_UNSUPPORTED, "shape too large");
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = dtype == KDA_BF16
                ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, shortconv_prefill_kernel<__nv_bfloat16>, 256, 0)
                : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, shortconv_prefill_kernel<float>, 256, 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(KDA_ERR_CUDA, std::string("occupancy query: ") + cudaGetErrorString(e));
    }
    const long long items = tiles * groups;
    const long long resident = (long long)sms * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(items < resident ? items : resident);
    unsigned *err = device_error_word();
    if (dtype == KDA_BF16)
        shortconv_prefill_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(x), static_cast<const __nv_bfloat16 *>(ring_in), w,
            static_cast<__nv_bfloat16 *>(y), static_cast<__nv_bfloat16 *>(ring_out), cu_seqlens, N, T, H, D, err,
            tiles, (int)groups);
    else
        shortconv_prefill_kernel<float><<<grid, 256, 0, s>>>(
            static_cast<const float *>(x), static_cast<const float *>(ring_in), w, static_cast<float *>(y),
            static_cast<float *>(ring_out), cu_seqlens, N, T, H, D, err, tiles, (int)groups);
    return check_launch("shortconv_prefill_kernel");
}
