// kda_shortconv.cu -- decode step of the width-4 causal depthwise short
// convolution + SiLU in front of q, k, v, with its 3-token ring
// ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析",
// sections "KDA 递推公式先衰减再差分" and "414MB 的 KDA 状态从哪来").
//
// Memory-bound elementwise work. A CTA owns one (projection, head) and a
// block of sequences: one thread copies their x rows and 3-slot ring rows
// into shared memory with two TMA tensor copies, the CTA reads the
// (projection, head)'s taps once, and each thread then convolves 16-byte
// vectors of channels and writes y and the shifted ring (the ring's stored
// vectors move unchanged).
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
#include "kda_tc.cuh"

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

// Decode step: one CTA per (projection, head) and sc_bc(D) consecutive
// sequences (a tile of SC_TILE_BYTES of x and ring). One thread issues the two
// tensor copies (the x rows and the 3-slot ring rows of those sequences) as
// soon as the CTA starts, so the whole launch's input is in flight at once;
// the (projection, head)'s taps are read once per CTA. Threads then own one
// 16-byte vector of channels for a stride of sequences and write y and the
// shifted ring with plain 16-byte stores. A tile reaching past B reads zeros
// there and stores nothing.
// The SiLU takes the fast exponential and division intrinsics (a few ulp, as
// the prefill form does): the CTA's compute sits between its tile landing and
// its stores, on the launch's critical path.
// Measured at 64 sequences x 96 heads (bf16, inputs rotating through six sets
// so every call misses in L2, launches replayed from a CUDA graph): 7.0 us,
// 8.1 us with the exact expf and division. Tiles of 16 KB / 64 threads ran
// about the same, 64 KB or 256 threads 8.7-9.6 us (exact forms).
// Launched as a programmatic dependent launch that prefetches its tiles into
// L2 before griddepcontrol.wait: 7.33 -> 7.11 us replayed from a graph, 10.1 ->
// 8.4 us issued one by one (same outputs).
// The earlier form, one thread per 16-byte vector and two sequences with all
// loads in registers, ran 10.2 us: 1.9 waves with 64 KB of loads in flight
// per SM, and its per-lane tap loads touched a different 128-byte line in
// every lane (two thirds of its L1 sectors).
constexpr int SC_NT = 128;
constexpr int SC_TILE_BYTES = 32768;
constexpr long long WAIT_LIMIT_CONV = 2000000000LL;  // clock cycles (about 1 s)
__host__ __device__ constexpr int sc_bc(int D, int esize) {
    return SC_TILE_BYTES / (4 * D * esize) > 256 ? 256 : SC_TILE_BYTES / (4 * D * esize);
}
template <typename T, int D>
__global__ void __launch_bounds__(SC_NT) shortconv_step_kernel(const __grid_constant__ CUtensorMap tm_x,
                                                               const __grid_constant__ CUtensorMap tm_r,
                                                               T *__restrict__ ring, const float *__restrict__ w,
                                                               T *__restrict__ y, int B, int H, unsigned *err) {
    constexpr int V = Vec16<T>::N, NV = D / V, BC = sc_bc(D, (int)sizeof(T));
    constexpr int BSTEP = SC_NT / NV;  // sequences handled per pass of the CTA
    extern __shared__ __align__(128) unsigned char sc_smem[];
    T *sx = reinterpret_cast<T *>(sc_smem);  // [BC][D]
    T *sr = sx + BC * D;                     // [BC][3][D]
    uint64_t *bar = reinterpret_cast<uint64_t *>(sr + 3 * BC * D);
    const int H3 = 3 * H;
    const int ph = (int)(blockIdx.x % (unsigned)H3);  // p * H + h
    const int b0 = (int)(blockIdx.x / (unsigned)H3) * BC;
    // A programmatic dependent launch: the CTA may start while the kernel before
    // it on the stream drains. Before griddepcontrol.wait it only prefetches its
    // x and ring tiles and its taps into L2, where that kernel's writes land;
    // every load of them comes after the wait, so none can see a stale value.
    // Dependents are released after the wait, so a kernel two launches back has
    // always completed before the next one starts.
    if (threadIdx.x == 0) {
        tc::mbar_init(bar, 1);
        tc::fence_mbar_init();
        tc::tma_prefetch_l2_3d(&tm_x, 0, ph, b0);
        tc::tma_prefetch_l2_4d(&tm_r, 0, 0, ph, b0);
    } else if (threadIdx.x == 32) {
        tc::prefetch_l2_bulk(w + (size_t)ph * D * 4, D * 16);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) {
        tc::mbar_arrive_expect_tx(bar, (uint32_t)(BC * 4 * D * sizeof(T)));
        tc::tma_load_3d(sx, &tm_x, bar, 0, ph, b0);
        tc::tma_load_4d(sr, &tm_r, bar, 0, 0, ph, b0);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int cv = threadIdx.x % NV, bs = threadIdx.x / NV;
    float4 tap[V];
    const float4 *wt = reinterpret_cast<const float4 *>(w + ((size_t)ph * D + (size_t)cv * V) * 4);
#pragma unroll
    for (int i = 0; i < V; ++i) tap[i] = wt[i];
    __syncthreads();  // the barrier's initialisation is visible to every waiting thread
    const bool got = tc::mbar_wait(bar, 0, WAIT_LIMIT_CONV);
    if (__syncthreads_or(!got)) {
        if (threadIdx.x == 0) {
            atomicOr(err, DEVERR_TIMEOUT);
            tc::mbar_wait(bar, 0, WAIT_LIMIT_CONV);  // let the copies land before shared memory goes away
        }
        return;
    }
    const int p = ph / H, h = ph - p * H;
#pragma unroll 4
    for (int bb = bs; bb < BC; bb += BSTEP) {
        const int b = b0 + bb;
        if (b >= B) break;
        const uint4 xr = *reinterpret_cast<const uint4 *>(sx + bb * D + cv * V);
        const uint4 r0 = *reinterpret_cast<const uint4 *>(sr + (bb * 3 + 0) * D + cv * V);
        const uint4 r1 = *reinterpret_cast<const uint4 *>(sr + (bb * 3 + 1) * D + cv * V);
        const uint4 r2 = *reinterpret_cast<const uint4 *>(sr + (bb * 3 + 2) * D + cv * V);
        const T *xe = reinterpret_cast<const T *>(&xr);
        const T *e0 = reinterpret_cast<const T *>(&r0);
        const T *e1 = reinterpret_cast<const T *>(&r1);
        const T *e2 = reinterpret_cast<const T *>(&r2);
        float yv[V];
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const float z = tap[i].x * Elem<T>::load(e0 + i) + tap[i].y * Elem<T>::load(e1 + i) +
                            tap[i].z * Elem<T>::load(e2 + i) + tap[i].w * Elem<T>::load(xe + i);
            yv[i] = __fdividef(z, 1.0f + __expf(-z));
        }
        store16(y + (((size_t)p * B + b) * H + h) * D + (size_t)cv * V, yv);
        // the ring shifts: its stored values move unchanged
        T *rp = ring + ((size_t)b * H3 + ph) * 3 * D + (size_t)cv * V;
        __stcs(reinterpret_cast<uint4 *>(rp), r1);
        __stcs(reinterpret_cast<uint4 *>(rp + D), r2);
        __stcs(reinterpret_cast<uint4 *>(rp + 2 * D), xr);
    }
}

template <typename T, int D>
static kda_status launch_conv_step(const T *x, T *ring, const float *w, T *y, int B, int H, cudaStream_t s) {
    constexpr int BC = sc_bc(D, (int)sizeof(T));
    const CUtensorMapDataType dt = sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const uint64_t e = sizeof(T), H3 = 3 * (uint64_t)H;
    CUtensorMap mx, mr;
    // x [B][3H][D] and ring [B][3H][3][D], dimensions innermost first
    const uint64_t dx[3] = {(uint64_t)D, H3, (uint64_t)B}, sxs[2] = {D * e, H3 * D * e};
    const uint32_t bx[3] = {(uint32_t)D, 1u, (uint32_t)BC};
    const uint64_t dr[4] = {(uint64_t)D, 3u, H3, (uint64_t)B}, srs[3] = {D * e, 3 * D * e, 3 * H3 * D * e};
    const uint32_t br[4] = {(uint32_t)D, 3u, 1u, (uint32_t)BC};
    if (!tc::make_map_nd(&mx, x, dt, 3, dx, sxs, bx) || !tc::make_map_nd(&mr, ring, dt, 4, dr, srs, br))
        return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled failed for the conv step");
    const size_t smem = (size_t)BC * 4 * D * sizeof(T) + 16;
    if (smem_attr_once<shortconv_step_kernel<T, D>>((int)smem) != cudaSuccess)
        return check_launch("shortconv_step_kernel (shared memory attribute)");
    const uint64_t blocks = (((uint64_t)B + BC - 1) / BC) * H3;
    if (blocks > 0x7fffffffULL) return invalid("B * H too large for the conv step grid");
    // a programmatic dependent launch: it may start while the previous kernel drains
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(SC_NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, shortconv_step_kernel<T, D>, mx, mr, ring, w, y, B, H,
                       device_error_word());  // an error is left for check_launch
    return check_launch("shortconv_step_kernel");
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
    if (dtype == KDA_BF16) {
        const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
        __nv_bfloat16 *rb = static_cast<__nv_bfloat16 *>(ring), *yb = static_cast<__nv_bfloat16 *>(y);
        switch (D) {
        case 16: return launch_conv_step<__nv_bfloat16, 16>(xb, rb, w, yb, B, H, s);
        case 32: return launch_conv_step<__nv_bfloat16, 32>(xb, rb, w, yb, B, H, s);
        case 64: return launch_conv_step<__nv_bfloat16, 64>(xb, rb, w, yb, B, H, s);
        default: return launch_conv_step<__nv_bfloat16, 128>(xb, rb, w, yb, B, H, s);
        }
    }
    const float *xf = static_cast<const float *>(x);
    float *rf = static_cast<float *>(ring), *yf = static_cast<float *>(y);
    switch (D) {
    case 16: return launch_conv_step<float, 16>(xf, rf, w, yf, B, H, s);
    case 32: return launch_conv_step<float, 32>(xf, rf, w, yf, B, H, s);
    case 64: return launch_conv_step<float, 64>(xf, rf, w, yf, B, H, s);
    default: return launch_conv_step<float, 128>(xf, rf, w, yf, B, H, s);
    }
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
