// kda_decode.cu -- one KDA decode step, the state streamed once.
//
// Recurrence ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析",
// section "KDA 递推公式先衰减再差分"; per-channel gate as in "为什么 Kimi K3 敢把
// KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化", section 7):
//   S' = Diag(exp g) S ; delta = beta (v - S'^T k^) ; S <- S' + k^ delta^T ; o = S^T q^
// Because o = S'^T q^ + (k^.q^) delta, both column reductions S'^T k^ and
// S'^T q^ come from the same sweep over S, so every state element is loaded
// from HBM once and stored once.
//
// Work split: one CTA per (sequence, head, slice of JS value columns). The
// CTA keeps its D x JS fp32 slice of S in registers (RPT rows x one float4
// per thread), issued as 128-bit streaming loads before anything else so the
// HBM requests are in flight while q/k/g are normalised. Rows of a slice are
// JS*4 = 128 contiguous bytes, so every warp load touches whole 128 B lines.
// Column sums are reduced with warp shuffles over the row groups of a warp
// and through shared memory across warps.
//
// The gate form is a template parameter: one log-gate per key channel (KDA),
// one per head (Gated DeltaNet, the same factor on every row of S), or none
// (the plain delta rule: no decay multiply at all).
#include "kda_common.cuh"

namespace kda {

template <int D> struct DecodeShape;
// JS: value columns per CTA, NT: threads per CTA.
template <> struct DecodeShape<16> { static constexpr int JS = 16, NT = 32; };
template <> struct DecodeShape<32> { static constexpr int JS = 32, NT = 64; };
template <> struct DecodeShape<64> { static constexpr int JS = 32, NT = 128; };
template <> struct DecodeShape<128> { static constexpr int JS = 32, NT = 256; };

template <int D, typename T, int GM>
__global__ void __launch_bounds__(DecodeShape<D>::NT)
    decode_step_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       const float *__restrict__ g, const float *__restrict__ beta,
                       float *__restrict__ state, T *__restrict__ out, float eps) {
    constexpr int JS = DecodeShape<D>::JS, NT = DecodeShape<D>::NT;
    constexpr int C4 = JS / 4;       // float4 columns per slice row
    constexpr int RG = NT / C4;      // row groups
    constexpr int RPT = D / RG;      // rows per thread
    constexpr int NW = NT / 32;      // warps
    constexpr int NSLICE = D / JS;
    static_assert(NT % 32 == 0 && NT >= D && NT >= JS && RPT * RG == D, "bad decode shape");

    const int unit = blockIdx.x / NSLICE;  // b*H + h
    const int slice = blockIdx.x % NSLICE;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int c4 = t % C4, rg = t / C4;

    float *Sp = state + (size_t)unit * D * D + slice * JS + c4 * 4;

    // 1. stream this thread's part of the state slice (rows rg, rg+RG, ...)
    float4 s[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) s[m] = __ldcs(reinterpret_cast<const float4 *>(Sp + (size_t)(rg + m * RG) * D));

    __shared__ float s_qa[D], s_ka[D], s_kh[D], s_a[D];
    __shared__ float s_red[NW][3];
    __shared__ float s_part[NW][JS][2];
    __shared__ float s_delta[JS];

    // 2. L2 norms of q, k and their dot, decay a = exp(g)
    const size_t vo = (size_t)unit * D;
    float qv = 0.f, kv = 0.f, av = 0.f;
    if (t < D) {
        qv = Elem<T>::load(q + vo + t);
        kv = Elem<T>::load(k + vo + t);
        if constexpr (GM == KDA_GATE_CHANNEL) av = expf(__ldg(g + vo + t));
        else if constexpr (GM == KDA_GATE_HEAD) av = expf(__ldg(g + unit));
        else av = 1.f;
    }
    float sqq = qv * qv, skk = kv * kv, sqk = qv * kv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sqq += __shfl_xor_sync(0xffffffffu, sqq, o);
        skk += __shfl_xor_sync(0xffffffffu, skk, o);
        sqk += __shfl_xor_sync(0xffffffffu, sqk, o);
    }
    if (lane == 0) {
        s_red[warp][0] = sqq;
        s_red[warp][1] = skk;
        s_red[warp][2] = sqk;
    }
    __syncthreads();
    sqq = skk = sqk = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        sqq += s_red[w][0];
        skk += s_red[w][1];
        sqk += s_red[w][2];
    }
    const float rq = inv_norm(sqq, eps), rk = inv_norm(skk, eps);
    const float kq = sqk * rq * rk;  // k^ . q^
    if (t < D) {
        s_qa[t] = qv * rq * av;
        s_ka[t] = kv * rk * av;
        s_kh[t] = kv * rk;
        s_a[t] = av;
    }
    __syncthreads();

    // 3. partial column sums of S'^T k^ and S'^T q^ over this thread's rows
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rg + m * RG;
        const float ka = s_ka[i], qa = s_qa[i];
        pk[0] += ka * s[m].x; pk[1] += ka * s[m].y; pk[2] += ka * s[m].z; pk[3] += ka * s[m].w;
        pq[0] += qa * s[m].x; pq[1] += qa * s[m].y; pq[2] += qa * s[m].z; pq[3] += qa * s[m].w;
    }
    // 4. reduce over the row groups inside the warp, then across warps
#pragma unroll
    for (int o = C4; o < 32; o <<= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            pk[c] += __shfl_xor_sync(0xffffffffu, pk[c], o);
            pq[c] += __shfl_xor_sync(0xffffffffu, pq[c], o);
        }
    }
    if (lane < C4) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            s_part[warp][c4 * 4 + c][0] = pk[c];
            s_part[warp][c4 * 4 + c][1] = pq[c];
        }
    }
    __syncthreads();
    if (t < JS) {
        float ks = 0.f, qs = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            ks += s_part[w][t][0];
            qs += s_part[w][t][1];
        }
        const int j = slice * JS + t;
        const float d = __ldg(beta + unit) * (Elem<T>::load(v + vo + j) - ks);
        s_delta[t] = d;
        Elem<T>::store(out + vo + j, qs + kq * d);
    }
    __syncthreads();

    // 5. S <- Diag(a) S + k^ delta^T, written back once
    const float d0 = s_delta[c4 * 4 + 0], d1 = s_delta[c4 * 4 + 1], d2 = s_delta[c4 * 4 + 2],
                d3 = s_delta[c4 * 4 + 3];
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rg + m * RG;
        const float a = s_a[i], kh = s_kh[i];
        float4 r;
        r.x = a * s[m].x + kh * d0;
        r.y = a * s[m].y + kh * d1;
        r.z = a * s[m].z + kh * d2;
        r.w = a * s[m].w + kh * d3;
        __stcs(reinterpret_cast<float4 *>(Sp + (size_t)i * D), r);
    }
}

template <int D, typename T, int GM>
static void launch_decode(const void *q, const void *k, const void *v, const float *g, const float *beta,
                          float *state, void *out, int BH, float eps, cudaStream_t s) {
    constexpr int NSLICE = D / DecodeShape<D>::JS;
    decode_step_kernel<D, T, GM><<<(unsigned)BH * NSLICE, DecodeShape<D>::NT, 0, s>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v), g, beta, state,
        static_cast<T *>(out), eps);
}

template <typename T, int GM>
static void dispatch_decode(int D, const void *q, const void *k, const void *v, const float *g,
                            const float *beta, float *state, void *out, int BH, float eps, cudaStream_t s) {
    switch (D) {
    case 16: launch_decode<16, T, GM>(q, k, v, g, beta, state, out, BH, eps, s); break;
    case 32: launch_decode<32, T, GM>(q, k, v, g, beta, state, out, BH, eps, s); break;
    case 64: launch_decode<64, T, GM>(q, k, v, g, beta, state, out, BH, eps, s); break;
    default: launch_decode<128, T, GM>(q, k, v, g, beta, state, out, BH, eps, s); break;
    }
}

template <typename T>
static void dispatch_gate(kda_gate gate, int D, const void *q, const void *k, const void *v, const float *g,
                          const float *beta, float *state, void *out, int BH, float eps, cudaStream_t s) {
    if (gate == KDA_GATE_HEAD) dispatch_decode<T, KDA_GATE_HEAD>(D, q, k, v, g, beta, state, out, BH, eps, s);
    else if (gate == KDA_GATE_NONE) dispatch_decode<T, KDA_GATE_NONE>(D, q, k, v, g, beta, state, out, BH, eps, s);
    else dispatch_decode<T, KDA_GATE_CHANNEL>(D, q, k, v, g, beta, state, out, BH, eps, s);
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_decode_step_gated(const void *q, const void *k, const void *v, const float *g,
                                            const float *beta, float *state, void *out, int B, int H, int D,
                                            kda_dtype dtype, kda_gate gate, float l2_eps, kda_stream_t stream) {
    clear_detail();
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE)
        return invalid("gate must be KDA_GATE_CHANNEL, KDA_GATE_HEAD or KDA_GATE_NONE");
    if (B < 0) return invalid("B must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (!(l2_eps >= 0.f)) return invalid("l2_eps must be >= 0");
    if (B == 0) return KDA_OK;
    if ((long long)B * H * (D / 16) > 0x7fffffffLL) return invalid("B*H too large for one launch");
    kda_status st;
    if ((st = check_ptr(q, "q")) || (st = check_ptr(k, "k")) || (st = check_ptr(v, "v")) ||
        (gate != KDA_GATE_NONE && (st = check_ptr(g, "g"))) || (st = check_ptr(beta, "beta")) ||
        (st = check_ptr(state, "state")) ||
        (st = check_ptr(out, "out")))
        return st;
    if (out == q || out == k || out == v || (const void *)out == (const void *)state)
        return invalid("out must not alias q, k, v or state");
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dtype == KDA_BF16)
        dispatch_gate<__nv_bfloat16>(gate, D, q, k, v, g, beta, state, out, B * H, l2_eps, s);
    else
        dispatch_gate<float>(gate, D, q, k, v, g, beta, state, out, B * H, l2_eps, s);
    return check_launch("decode_step_kernel");
}

extern "C" kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                                      const float *beta, float *state, void *out, int B, int H, int D,
                                      kda_dtype dtype, float l2_eps, kda_stream_t stream) {
    return kda_decode_step_gated(q, k, v, g, beta, state, out, B, H, D, dtype, KDA_GATE_CHANNEL, l2_eps, stream);
}
