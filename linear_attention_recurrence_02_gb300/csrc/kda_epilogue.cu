// kda_epilogue.cu -- output epilogue of a KDA layer: gated RMSNorm.
//
// "KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析",
// section "相关源码与文档导航", lists a gated RMSNorm among the parts of the KDA
// kernel; "为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化",
// section 6 (the Gated DeltaNet architecture figure), says the output passes a
// gate that scales its features. Neither prints the formula; the reading taken
// is the plainest one, per (token, head) row of D value channels:
//   y_j = o_j / sqrt(mean_j' o_j'^2 + eps) * weight_j * act(gate_j)
// with act the logistic sigmoid or SiLU (z * sigmoid(z)); a row whose mean
// square plus eps is exactly zero maps to zero.
//
// Bandwidth-bound: every element of o and gate is read once and y written
// once. A warp covers whole rows: min(32, D) lanes per row, D / 32 channels
// per lane (one 8-byte bf16 or 16-byte fp32 vector at D = 128), and issues
// the loads of its U = 2 row passes before reducing either; the mean square is
// a shuffle reduction over the row's lanes. The issue slots, not HBM alone,
// bound the kernel, so the per-element work is kept short: the row's 1/RMS is
// one reciprocal square root on the special-function unit (within 2 ulp; the
// exact square root and division took about a fifth of the kernel's
// instructions) and is folded into the weight, and for bf16 outputs the
// sigmoid is taken through
// the identity sigmoid(z) = 1/2 + tanh(z/2)/2 with the hardware tanh
// approximation (relative error about 2^-11, far below bf16 rounding; one
// special-function op instead of an exponential and a reciprocal). fp32
// outputs use the fast exponential and division intrinsics (a few ulp).
// Measured at 4096 tokens x 96 heads: 2 rows per warp and 128-thread blocks
// beat 1, 4 or 8 rows, 16-byte bf16 vectors and 256 threads; with the
// reciprocal square root, 47.9 us against 53.4 us (4 rows: 52.5, 1 row: 67.7).
#include "kda_common.cuh"

namespace kda {

template <typename T, int V> struct alignas(sizeof(T) * V) VecN {
    T e[V];
};
// the streaming load/store intrinsics take built-in types: move V elements
// as one integer vector of the same size
template <int BYTES> struct RawOf;
template <> struct RawOf<2> { using type = unsigned short; };
template <> struct RawOf<4> { using type = unsigned int; };
template <> struct RawOf<8> { using type = uint2; };
template <> struct RawOf<16> { using type = uint4; };
template <typename Vec> __device__ __forceinline__ Vec ld_stream(const Vec *p) {
    using Raw = typename RawOf<sizeof(Vec)>::type;
    const Raw r = __ldcs(reinterpret_cast<const Raw *>(p));
    Vec v;
    memcpy(&v, &r, sizeof(Vec));
    return v;
}
template <typename Vec> __device__ __forceinline__ void st_stream(Vec *p, const Vec &v) {
    using Raw = typename RawOf<sizeof(Vec)>::type;
    Raw r;
    memcpy(&r, &v, sizeof(Vec));
    __stcs(reinterpret_cast<Raw *>(p), r);
}

template <int D, typename T, int ACT>
__global__ void __launch_bounds__(128) gated_rmsnorm_kernel(const T *o, const T *gate,
                                                            const float *__restrict__ weight, T *y,
                                                            long long R, float eps) {
    // y may alias o or gate (the in-place epilogue of a prefill output), so
    // none of the three is declared restrict; each thread loads every element
    // it stores before storing it.
    constexpr int LPR = D < 32 ? D : 32;  // lanes per row
    constexpr int V = D / LPR;            // channels per lane
    constexpr int RPW = 32 / LPR;         // rows per warp pass
    constexpr int U = 2;                  // passes whose loads are issued together
    using Vec = VecN<T, V>;
    const int lane = threadIdx.x & 31, sub = lane / LPR, ln = lane % LPR;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long row0 = warp * (RPW * U);

    float w[V];
#pragma unroll
    for (int i = 0; i < V; ++i) w[i] = __ldg(weight + ln * V + i);
    Vec ov[U], gv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const long long r = row0 + u * RPW + sub;
        if (r < R) {
            ov[u] = ld_stream(reinterpret_cast<const Vec *>(o + r * D) + ln);
            gv[u] = ld_stream(reinterpret_cast<const Vec *>(gate + r * D) + ln);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const long long r = row0 + u * RPW + sub;
        float of[V], ss = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i) {
            of[i] = r < R ? Elem<T>::load(&ov[u].e[i]) : 0.f;
            ss = fmaf(of[i], of[i], ss);
        }
#pragma unroll
        for (int m = LPR / 2; m > 0; m >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float den = ss / (float)D + eps;
        const float inv = den > 0.f ? rsqrtf(den) : 0.f;
        if (r < R) {
            Vec out;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const float z = Elem<T>::load(&gv[u].e[i]);
                float sg;
                if constexpr (sizeof(T) == 2) {  // bf16 output: one tanh instead of exp and reciprocal
                    float th;
                    asm("tanh.approx.f32 %0, %1;" : "=f"(th) : "f"(0.5f * z));
                    sg = fmaf(0.5f, th, 0.5f);
                } else {
                    sg = __fdividef(1.0f, 1.0f + __expf(-z));
                }
                Elem<T>::store(&out.e[i], (of[i] * (w[i] * inv)) * (ACT == KDA_ACT_SILU ? z * sg : sg));
            }
            st_stream(reinterpret_cast<Vec *>(y + r * D) + ln, out);
        }
    }
}

template <int D, typename T, int ACT>
static void launch_epi(const void *o, const void *gate, const float *weight, void *y, long long R, float eps,
                       cudaStream_t s) {
    constexpr int LPR = D < 32 ? D : 32, RPW = 32 / LPR, U = 2;
    const long long warps = (R + RPW * U - 1) / (RPW * U);
    const long long blocks = (warps + 3) / 4;
    gated_rmsnorm_kernel<D, T, ACT><<<(unsigned)blocks, 128, 0, s>>>(
        static_cast<const T *>(o), static_cast<const T *>(gate), weight, static_cast<T *>(y), R, eps);
}

template <typename T, int ACT>
static void dispatch_epi(int D, const void *o, const void *gate, const float *weight, void *y, long long R,
                         float eps, cudaStream_t s) {
    switch (D) {
    case 16: launch_epi<16, T, ACT>(o, gate, weight, y, R, eps, s); break;
    case 32: launch_epi<32, T, ACT>(o, gate, weight, y, R, eps, s); break;
    case 64: launch_epi<64, T, ACT>(o, gate, weight, y, R, eps, s); break;
    default: launch_epi<128, T, ACT>(o, gate, weight, y, R, eps, s); break;
    }
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_gated_rmsnorm(const void *o, const void *gate, const float *weight, void *y, int64_t T,
                                        int H, int D, kda_dtype dtype, kda_gate_act act, float eps,
                                        kda_stream_t stream) {
    clear_detail();
    if (T < 0) return invalid("T must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (act != KDA_ACT_SIGMOID && act != KDA_ACT_SILU) return invalid("act must be KDA_ACT_SIGMOID or KDA_ACT_SILU");
    if (!(eps >= 0.f)) return invalid("eps must be >= 0");
    if (T == 0) return KDA_OK;
    const long long R = (long long)T * H;
    if (R > (1LL << 35)) return invalid("T*H too large for one launch");
    kda_status st;
    if ((st = check_ptr(o, "o")) || (st = check_ptr(gate, "gate")) || (st = check_ptr(weight, "weight")) ||
        (st = check_ptr(y, "y")))
        return st;
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16) {
        if (act == KDA_ACT_SILU) dispatch_epi<__nv_bfloat16, KDA_ACT_SILU>(D, o, gate, weight, y, R, eps, s);
        else dispatch_epi<__nv_bfloat16, KDA_ACT_SIGMOID>(D, o, gate, weight, y, R, eps, s);
    } else {
        if (act == KDA_ACT_SILU) dispatch_epi<float, KDA_ACT_SILU>(D, o, gate, weight, y, R, eps, s);
        else dispatch_epi<float, KDA_ACT_SIGMOID>(D, o, gate, weight, y, R, eps, s);
    }
    return check_launch("gated_rmsnorm_kernel");
}
