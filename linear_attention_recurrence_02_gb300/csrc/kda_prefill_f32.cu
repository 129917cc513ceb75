// kda_prefill_f32.cu -- chunked prefill for d = 128 on CUDA cores in fp32
// arithmetic: the d = 128 path for the shapes neither tensor-core kernel
// takes (fp32 q/k/v with a chunk below 16, bf16 with a chunk other than 16,
// 32 or 64, and an empty token range).
//
// Chunk algebra ("为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化",
// section 5: attention-like work inside a chunk, the state handed from chunk
// to chunk; section 6: the decay between two positions is the product of the
// gates in between). With G_r = sum_{s<=r} g_s per key channel, L2-normalised
// q^, k^, and the chunk entered with state S:
//   Kt_r = e^{G_r} k^_r,  Qt_r = e^{G_r} q^_r,  R_s = e^{-G_s} k^_s
//   [A_raw; P_raw] = [Kt; Qt] R^T      A = beta_r A_raw (s < r),  P = P_raw (s <= r)
//   [X; O_int]     = [Kt; Qt] S
//   (I + A) U = Diag(beta) (V - X)     (blocked forward substitution)
//   O = O_int + P U
//   S <- Diag(e^{G_L}) (S + R^T U)
// e^{G_r - G_s} = e^{G_r} e^{-G_s} needs no anchor in fp32 as long as every
// G_L >= -80 (e^80 is far inside fp32's range); a chunk beyond that computes
// A and P by exact pairwise exponentials and R_s = e^{G_L - G_s} k^_s (Kb),
// with the state update S <- Diag(e^{G_L}) S + Kb^T U.
//
// One CTA (256 threads) per (sequence, head) keeps the 128 x 128 fp32 state in
// shared memory for the whole sequence. The products are register-tiled (8 x 8
// or 4 x 8 outputs per thread): the row operand is read as broadcast scalars
// from rows padded to 129 floats, the column operand as two 16-byte loads.
#include <string>

#include "kda_common.cuh"
#include "kda_prefill.cuh"

namespace kda {
namespace f32p {

constexpr int D = 128, CM = 64, NT = 256;
constexpr int LQ = D + 1;   // row stride of [Kt; Qt] (128 rows) and R (64 rows)
constexpr int LA = CM + 1;  // row stride of A (then the diagonal blocks' inverses) and P
constexpr float SPAN_MAX = 80.f;

// shared memory, in floats
constexpr int O_KQ = 0;                    // [Kt; Qt] [128][LQ]; O_int in rows 64.. after the product
constexpr int O_R = O_KQ + 2 * CM * LQ;    // R [64][LQ]; G (per-channel gate) while the operands are built
constexpr int O_S = O_R + CM * LQ;         // S [128][128]
constexpr int O_V = O_S + D * D;           // V [64][128] -> rhs -> U
constexpr int O_A = O_V + CM * D;          // A [64][LA]; the row norms while the operands are built
constexpr int O_P = O_A + CM * LA;         // P [64][LA]; G (per-head gate) while the operands are built
constexpr int O_F = O_P + CM * LA;         // G_L, e^{G_L}, scale of R^T U in the state update [3][128]
constexpr int SMEM_FLOATS = O_F + 3 * D;
constexpr size_t SMEM = (size_t)SMEM_FLOATS * sizeof(float);
static_assert(SMEM <= 232448, "shared memory of the fp32 prefill");

template <typename T> __device__ __forceinline__ void load4(const T *p, float (&f)[4]);
template <> __device__ __forceinline__ void load4<float>(const float *p, float (&f)[4]) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w;
}
template <> __device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float (&f)[4]) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
    f[0] = __bfloat162float(a.x); f[1] = __bfloat162float(a.y);
    f[2] = __bfloat162float(b.x); f[3] = __bfloat162float(b.y);
}
template <typename T> __device__ __forceinline__ void store8(T *p, const float (&f)[8]);
template <> __device__ __forceinline__ void store8<float>(float *p, const float (&f)[8]) {
    *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
    *reinterpret_cast<float4 *>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}
template <> __device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16 *p, const float (&f)[8]) {
    uint4 u;
    uint32_t *w = reinterpret_cast<uint32_t *>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 t = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
        w[e] = *reinterpret_cast<const uint32_t *>(&t);
    }
    *reinterpret_cast<uint4 *>(p) = u;
}
__device__ __forceinline__ void ld8(const float *p, float (&b)[8]) {
    const float4 x = *reinterpret_cast<const float4 *>(p), y = *reinterpret_cast<const float4 *>(p + 4);
    b[0] = x.x; b[1] = x.y; b[2] = x.z; b[3] = x.w; b[4] = y.x; b[5] = y.y; b[6] = y.z; b[7] = y.w;
}

}  // namespace f32p

template <typename T, int GM>
__global__ void __launch_bounds__(f32p::NT, 1)
    prefill_f32_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                       const float *__restrict__ g, const float *__restrict__ beta, const float *s_init,
                       float *s_final, T *__restrict__ out, const int64_t *__restrict__ cu_seqlens, int N,
                       int64_t Ttot, int H, int C, float eps, unsigned *err, const int *__restrict__ order,
                       int v_zero) {
    using namespace f32p;
    constexpr bool GCH = GM == KDA_GATE_CHANNEL, GHD = GM == KDA_GATE_HEAD;
    extern __shared__ __align__(16) float fsm[];
    float *sKQ = fsm + O_KQ, *sR = fsm + O_R, *sS = fsm + O_S, *sV = fsm + O_V, *sA = fsm + O_A, *sP = fsm + O_P;
    float *sGL = fsm + O_F, *sEA = sGL + D, *sEB = sEA + D;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const int h = blockIdx.x % H, n = order ? order[blockIdx.x / H] : (int)(blockIdx.x / H);
    int64_t start, end;
    if (!seq_range(cu_seqlens, n, N, Ttot, err, start, end)) return;
    const size_t sbase = ((size_t)n * H + h) * D * D;
    for (int p = tid; p < D * D / 4; p += NT) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s_init) x = *reinterpret_cast<const float4 *>(s_init + sbase + 4 * (size_t)p);
        *reinterpret_cast<float4 *>(sS + 4 * p) = x;
    }

    for (int64_t c0 = start; c0 < end; c0 += C) {
        const int L = (int)((end - c0) < (int64_t)C ? (end - c0) : (int64_t)C);
        __syncthreads();  // the previous chunk is done with every buffer
        // 1. L2 norms of the q and k rows (two threads per row, 64 channels each), into the A area
        {
            const int rr = tid >> 1, half = tid & 1, r = rr & 63;
            const bool isq = rr >= 64;
            float ss = 0.f;
            if (r < L) {
                const T *src = (isq ? q : k) + ((size_t)(c0 + r) * H + h) * D + 64 * half;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    float f[4];
                    load4<T>(src + 4 * c, f);
                    ss += f[0] * f[0] + f[1] * f[1] + f[2] * f[2] + f[3] * f[3];
                }
            }
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (half == 0) sA[(isq ? 64 : 0) + r] = r < L ? inv_norm(ss, eps) : 0.f;
        }
        // 2. cumulative log decay G: per channel into the R area, per head into the P area
        bool bad = false;
        if constexpr (GCH) {
            if (tid < D) {
                float acc = 0.f;
                const float *gp = g + ((size_t)c0 * H + h) * D + tid;
                float gv[16];
#pragma unroll 1
                for (int r0 = 0; r0 < CM; r0 += 16) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) gv[r] = r0 + r < L ? gp[(size_t)(r0 + r) * H * D] : 0.f;
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        acc += gv[r];
                        sR[(r0 + r) * LQ + tid] = acc;
                    }
                }
                sGL[tid] = acc;
                bad = !(acc >= -SPAN_MAX);
            }
        } else if constexpr (GHD) {
            if (warp == 0) {  // an inclusive scan over the 64 rows, two per lane
                const float g0 = 2 * lane < L ? g[(size_t)(c0 + 2 * lane) * H + h] : 0.f;
                const float g1 = 2 * lane + 1 < L ? g[(size_t)(c0 + 2 * lane + 1) * H + h] : 0.f;
                float incl = g0 + g1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                sP[2 * lane] = incl - g1;
                sP[2 * lane + 1] = incl;
                const float GL = __shfl_sync(0xffffffffu, incl, 31);
                if (lane == 0) sGL[0] = GL;
                bad = lane == 0 && !(GL >= -SPAN_MAX);
            }
        }
        const bool exact = __syncthreads_or(bad);
        // G of (row r, channel i), wherever step 2 left it
        auto gval = [&](const float *src, int r, int i) -> float {
            if constexpr (GCH) return src[r * LQ + i];
            else if constexpr (GHD) return src[r];
            else return 0.f;
        };
        // 3. operands, rows past L zero. Normal path: Kt and Qt rows, R over G, V.
        //    Exact path: k^ and q^ rows unscaled and Kb over G, with G kept in the V area
        //    until A and P are formed (step 4), then Kt, Qt and V.
        if (exact) {
            for (int p = tid; p < CM * D; p += NT) {  // G into the V area
                const int r = p / D, i = p % D;
                sV[p] = GCH ? sR[r * LQ + i] : (GHD && i == 0 ? sP[r] : 0.f);
            }
            __syncthreads();
        }
        const float *gsrc = exact ? sV : (GCH ? sR : sP);
        const int gld = exact ? D : LQ;
        for (int p = tid; p < CM * (D / 4); p += NT) {
            const int r = p >> 5, i0 = (p & 31) * 4;
            float kf[4] = {0.f, 0.f, 0.f, 0.f}, qf[4] = {0.f, 0.f, 0.f, 0.f}, vf[4] = {0.f, 0.f, 0.f, 0.f};
            if (r < L) {
                const size_t o = ((size_t)(c0 + r) * H + h) * D + i0;
                load4<T>(k + o, kf);
                load4<T>(q + o, qf);
                if (!v_zero && !exact) load4<T>(v + o, vf);
            }
            const float rk = sA[r], rq = sA[64 + r];
            float kt[4], qt[4], rr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int i = i0 + e;
                float G = 0.f, GL = 0.f;
                if constexpr (GCH) {
                    G = gsrc[r * gld + i];
                    GL = sGL[i];
                } else if constexpr (GHD) {
                    G = exact ? gsrc[r * gld] : gsrc[r];
                    GL = sGL[0];
                }
                const float kh = kf[e] * rk, qh = qf[e] * rq;
                const float eg = exact ? 1.f : __expf(G);
                kt[e] = eg * kh;
                qt[e] = eg * qh;
                rr[e] = (exact ? __expf(GL - G) : __expf(-G)) * kh;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sKQ[r * LQ + i0 + e] = kt[e];
                sKQ[(64 + r) * LQ + i0 + e] = qt[e];
                sR[r * LQ + i0 + e] = rr[e];
            }
            if (!exact) *reinterpret_cast<float4 *>(sV + r * D + i0) = make_float4(vf[0], vf[1], vf[2], vf[3]);
        }
        if (tid < D) {
            const float GL = GCH ? sGL[tid] : GHD ? sGL[0] : 0.f;
            const float eg = __expf(GL);
            sEA[tid] = eg;
            sEB[tid] = exact ? 1.f : eg;
        }
        __syncthreads();

        // 4. A and P
        if (!exact) {
            // [A_raw; P_raw] = [Kt; Qt] R^T, each thread 8 rows x 4 columns
            const int r0 = 8 * ty, s0 = 4 * tx;  // r0 over the 128 rows of [Kt; Qt]
            const int rl = r0 & 63;               // row within A or P
            const bool isp = r0 >= 64;
            float *dst = isp ? sP : sA;
            if (s0 <= rl + 7) {  // a tile wholly past the diagonal is zero
                float acc[8][4];
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[m][c] = 0.f;
#pragma unroll 4
                for (int i = 0; i < D; ++i) {
                    float a[8], b[4];
#pragma unroll
                    for (int m = 0; m < 8; ++m) a[m] = sKQ[(r0 + m) * LQ + i];
#pragma unroll
                    for (int c = 0; c < 4; ++c) b[c] = sR[(s0 + c) * LQ + i];
#pragma unroll
                    for (int m = 0; m < 8; ++m)
#pragma unroll
                        for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(a[m], b[c], acc[m][c]);
                }
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int r = rl + m;
                    const float br = !isp && r < L ? beta[(size_t)(c0 + r) * H + h] : 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int s = s0 + c;
                        dst[r * LA + s] = isp ? ((s <= r && r < L) ? acc[m][c] : 0.f)
                                              : ((s < r && r < L) ? br * acc[m][c] : 0.f);
                    }
                }
            } else {
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int c = 0; c < 4; ++c) dst[(rl + m) * LA + s0 + c] = 0.f;
            }
            __syncthreads();
        } else {
            // exact pairwise decays: A_rs = beta_r sum_i k^_ri k^_si e^{G_ri - G_si}, P likewise with q^
            for (int pidx = tid; pidx < CM * CM; pidx += NT) {
                const int r = pidx >> 6, s = pidx & 63;
                float a = 0.f, pq = 0.f;
                if (s <= r && r < L) {
                    for (int i = 0; i < D; ++i) {
                        const float dG = GCH ? sV[r * D + i] - sV[s * D + i] : GHD ? sV[r * D] - sV[s * D] : 0.f;
                        const float ks = sKQ[s * LQ + i] * __expf(dG);
                        a = fmaf(sKQ[r * LQ + i], ks, a);
                        pq = fmaf(sKQ[(64 + r) * LQ + i], ks, pq);
                    }
                }
                sA[r * LA + s] = (s < r && r < L) ? beta[(size_t)(c0 + r) * H + h] * a : 0.f;
                sP[r * LA + s] = pq;
            }
            __syncthreads();
            // then Kt = e^{G} k^, Qt = e^{G} q^ in place, and V over G
            for (int p = tid; p < CM * D; p += NT) {
                const int r = p / D, i = p % D;
                const float eg = __expf(GCH ? sV[r * D + i] : GHD ? sV[r * D] : 0.f);
                sKQ[r * LQ + i] *= eg;
                sKQ[(64 + r) * LQ + i] *= eg;
            }
            __syncthreads();
            for (int p = tid; p < CM * D; p += NT) {
                const int r = p / D, i = p % D;
                sV[p] = (r < L && !v_zero) ? Elem<T>::load(v + ((size_t)(c0 + r) * H + h) * D + i) : 0.f;
            }
            __syncthreads();
        }

        // 5. [X; O_int] = [Kt; Qt] S, each thread 8 x 8. X rows give rhs = beta (V - X) over V;
        //    O_int rows go over the Qt rows (dead once every thread has finished the product).
        {
            const int r0 = 8 * ty, j0 = 8 * tx;
            float acc[8][8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[m][c] = 0.f;
#pragma unroll 2
            for (int i = 0; i < D; ++i) {
                float a[8], b[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) a[m] = sKQ[(r0 + m) * LQ + i];
                ld8(sS + i * D + j0, b);
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[m][c] = fmaf(a[m], b[c], acc[m][c]);
            }
            __syncthreads();
            if (r0 < 64) {
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const int r = r0 + m;
                    const float br = r < L ? beta[(size_t)(c0 + r) * H + h] : 0.f;
                    float vv[8];
                    ld8(sV + r * D + j0, vv);
#pragma unroll
                    for (int c = 0; c < 8; ++c) vv[c] = br * (vv[c] - acc[m][c]);
                    *reinterpret_cast<float4 *>(sV + r * D + j0) = make_float4(vv[0], vv[1], vv[2], vv[3]);
                    *reinterpret_cast<float4 *>(sV + r * D + j0 + 4) = make_float4(vv[4], vv[5], vv[6], vv[7]);
                }
            } else {
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int c = 0; c < 8; ++c) sKQ[(r0 + m) * LQ + j0 + c] = acc[m][c];
            }
        }
        __syncthreads();

        // 6. (I + A) U = rhs by 16-row blocks. Each warp b < 4 inverts its diagonal block
        //    D_b = (I + A_bb)^-1 in place (lane = column; forward substitution), then the blocks
        //    of U follow in order: U_b = D_b (rhs_b - sum_{k<b} A_bk U_k).
        if (warp < 4) {
            const int b0 = 16 * warp, c = lane & 15;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = r == c ? 1.f : 0.f;
#pragma unroll
                for (int t = 0; t < r; ++t) acc = fmaf(-sA[(b0 + r) * LA + b0 + t], x[t], acc);
                x[r] = acc;
            }
            __syncwarp();
            if (lane < 16)
#pragma unroll
                for (int r = 0; r < 16; ++r) sA[(b0 + r) * LA + b0 + c] = x[r];
        }
        __syncthreads();
        {
            const int rr = tid >> 4, j0 = 8 * tx;  // row rr of the block, 8 columns
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
                const int r = 16 * blk + rr;
                float y[8];
                ld8(sV + r * D + j0, y);
                for (int t = 0; t < 16 * blk; ++t) {  // rhs_b - sum_{k<b} A_bk U_k
                    const float a = sA[r * LA + t];
                    float u[8];
                    ld8(sV + t * D + j0, u);
#pragma unroll
                    for (int c = 0; c < 8; ++c) y[c] = fmaf(-a, u[c], y[c]);
                }
                __syncthreads();
                *reinterpret_cast<float4 *>(sV + r * D + j0) = make_float4(y[0], y[1], y[2], y[3]);
                *reinterpret_cast<float4 *>(sV + r * D + j0 + 4) = make_float4(y[4], y[5], y[6], y[7]);
                __syncthreads();
                float u[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int t = 0; t < 16; ++t) {  // U_b = D_b Y_b
                    const float dv = sA[r * LA + 16 * blk + t];
                    float yy[8];
                    ld8(sV + (16 * blk + t) * D + j0, yy);
#pragma unroll
                    for (int c = 0; c < 8; ++c) u[c] = fmaf(dv, yy[c], u[c]);
                }
                __syncthreads();
                *reinterpret_cast<float4 *>(sV + r * D + j0) = make_float4(u[0], u[1], u[2], u[3]);
                *reinterpret_cast<float4 *>(sV + r * D + j0 + 4) = make_float4(u[4], u[5], u[6], u[7]);
                __syncthreads();
            }
        }

        // 7. O = O_int + P U, each thread 4 rows x 8 columns; stored to out
        {
            const int r0 = 4 * ty, j0 = 8 * tx;
            float acc[4][8];
#pragma unroll
            for (int m = 0; m < 4; ++m)  // rows of stride LQ: scalar loads, not 16-byte aligned
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[m][c] = sKQ[(64 + r0 + m) * LQ + j0 + c];
            const int smax = r0 + 4 < L ? r0 + 4 : L;
            for (int t = 0; t < smax; ++t) {
                float a[4], u[8];
#pragma unroll
                for (int m = 0; m < 4; ++m) a[m] = sP[(r0 + m) * LA + t];
                ld8(sV + t * D + j0, u);
#pragma unroll
                for (int m = 0; m < 4; ++m)
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[m][c] = fmaf(a[m], u[c], acc[m][c]);
            }
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (r0 + m < L) store8<T>(out + ((size_t)(c0 + r0 + m) * H + h) * D + j0, acc[m]);
        }

        // 8. S <- Diag(e^{G_L}) S + Diag(eb) R^T U, each thread 8 x 8
        {
            const int i0 = 8 * ty, j0 = 8 * tx;
            float acc[8][8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[m][c] = 0.f;
            for (int t = 0; t < L; ++t) {
                float a[8], u[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) a[m] = sR[t * LQ + i0 + m];
                ld8(sV + t * D + j0, u);
#pragma unroll
                for (int m = 0; m < 8; ++m)
#pragma unroll
                    for (int c = 0; c < 8; ++c) acc[m][c] = fmaf(a[m], u[c], acc[m][c]);
            }
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int i = i0 + m;
                const float ea = sEA[i], eb = sEB[i];
                float sv[8];
                ld8(sS + i * D + j0, sv);
#pragma unroll
                for (int c = 0; c < 8; ++c) sv[c] = fmaf(eb, acc[m][c], ea * sv[c]);
                *reinterpret_cast<float4 *>(sS + i * D + j0) = make_float4(sv[0], sv[1], sv[2], sv[3]);
                *reinterpret_cast<float4 *>(sS + i * D + j0 + 4) = make_float4(sv[4], sv[5], sv[6], sv[7]);
            }
        }
    }
    __syncthreads();
    if (s_final)
        for (int p = tid; p < D * D / 4; p += NT)
            *reinterpret_cast<float4 *>(s_final + sbase + 4 * (size_t)p) = *reinterpret_cast<const float4 *>(sS + 4 * p);
    (void)lane;
}

bool prefill_f32_applicable(const PrefillArgs &a) { return a.D == 128 && a.C >= 1 && a.C <= 64; }

template <typename T, int GM>
static kda_status launch_f32(const PrefillArgs &a, cudaStream_t s) {
    auto kern = prefill_f32_kernel<T, GM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)f32p::SMEM);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    kern<<<launch_seqs(a) * a.H, f32p::NT, f32p::SMEM, s>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v), a.g, a.beta,
        a.s_init, a.s_final, static_cast<T *>(a.out), a.cu_seqlens, a.N, a.T, a.H, a.C, a.eps, a.err, a.order,
        a.v_zero ? 1 : 0);
    return check_launch("prefill_f32_kernel");
}

template <typename T>
static kda_status dispatch_f32(const PrefillArgs &a, cudaStream_t s) {
    if (a.gate == KDA_GATE_HEAD) return launch_f32<T, KDA_GATE_HEAD>(a, s);
    if (a.gate == KDA_GATE_NONE) return launch_f32<T, KDA_GATE_NONE>(a, s);
    return launch_f32<T, KDA_GATE_CHANNEL>(a, s);
}

kda_status prefill_f32(const PrefillArgs &a, cudaStream_t s) {
    return a.bf16 ? dispatch_f32<__nv_bfloat16>(a, s) : dispatch_f32<float>(a, s);
}

}  // namespace kda
