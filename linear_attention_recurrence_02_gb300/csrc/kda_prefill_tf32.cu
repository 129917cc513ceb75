// kda_prefill_tf32.cu -- chunked prefill for fp32 q/k/v, d_k = d_v = 128, on
// the 5th-generation tensor cores (tcgen05 kind::tf32, accumulators in TMEM).
//
// Chunk algebra ("为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化",
// section 5: attention-like work inside a chunk, the state handed from chunk
// to chunk; section 6: the decay between two positions is the product of the
// gates in between). With G the cumulative log decay inside the chunk per key
// channel, a per-channel anchor c = min(0, G_L + 40), L2-normalised q^, k^ and
// the chunk entered with state S:
//   Lk = e^{G-c} k^,  Lq = e^{G-c} q^,  Rk = e^{c-G} k^,  S~ = Diag(e^c) S
//   [A_raw; P_raw] = [Lk; Lq] Rk^T            (G1)  A = mask_<(beta_r A_raw), P = mask_<=(P_raw)
//   [X; O_int]     = [Lk; Lq] S~              (G0)  (= [e^G k^; e^G q^] S)
//   T = (I + A)^-1 Diag(beta)                       (CUDA cores, fp32, 16-row blocks)
//   U = T (V - X)                             (G2)
//   O = O_int + P U                           (G3)
//   S~ + Rk^T U                               (G4)  = Diag(e^{c-G_L}) S_next
// The factor e^{G_L-c} S_next needs is kept per channel and applied, with the
// next chunk's e^{c'}, when the state is read back at the start of that chunk.
// Every factor stays within e^[-40, 40] while the chunk's decay span is at
// most 80; a chunk beyond that uses c = 0, forms A and P with exact pairwise
// exponentials on the CUDA cores, applies Diag(e^{G_L}) to the state before
// G4 and takes Kb = e^{G_L-G} k^ in place of Rk.
//
// fp32 accuracy from tf32 operands: every product X Y is taken as
// X_hi Y_hi + X_hi Y_lo + X_lo Y_hi, X_hi being X with the low 13 mantissa
// bits cleared and X_lo = X - X_hi (exact in fp32); the dropped X_lo Y_lo and
// the rounding of X_lo leave a relative error near 2^-21 per product. The
// state accumulator serves as its own hi part: the tensor core reads a 32-bit
// operand through its top 19 bits.
//
// Layout: TMEM lane = value channel j for G0, G2, G3, G4 (the state lives in
// TMEM as S~^T, lane j, column i, for the whole sequence and is G0's A
// operand; W^T = (V - X)^T and U^T are written back to TMEM as hi / lo A
// operands). G1 puts the 128 rows of [Lk; Lq] on the lanes. The B operands
// ([Lk; Lq], Rk, T, P, Rk^T) are fp32 hi / lo tiles in 128-byte-swizzled
// K-major shared memory written by the CUDA cores.
//
// One CTA (256 threads) per (sequence, head); its phases run in order with
// block barriers between them, the MMAs issued by one elected lane of warp 0.
// Every wait is bounded.
#include <string>

#include "kda_common.cuh"
#include "kda_prefill.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace tfp {

using namespace tc;

constexpr int C = 64, D = 128, NT = 256;
constexpr long long WAIT_LIMIT = 4000000000LL;  // clock cycles (about 2 s)
constexpr float ANCHOR = 40.f, SPAN_MAX = 2.f * ANCHOR;

// shared memory, bytes from a 1024-byte aligned base
constexpr uint32_t KQH = 0, KQL = 65536;        // [Lk; Lq] hi / lo: 128 rows x 128, four 16 KB blocks each
constexpr uint32_t RKH = 131072, RKL = 163840;  // Rk hi / lo: 64 rows x 128 (four 8 KB blocks);
                                                // then Rk^T (Kb^T) hi / lo: 128 rows x 64 (two 16 KB blocks)
// reused once G0 and G1 are done with [Lk; Lq]
constexpr uint32_t TH = 0, TL = 16384, PH = 32768, PL = 49152;  // T, P hi / lo: 64 rows x 64 (two 8 KB blocks)
constexpr uint32_t AF = 65536;                  // A fp32 [64][65]
constexpr uint32_t NI = AF + 64 * 65 * 4;       // (I + A)^-1 fp32 [64][65]
constexpr uint32_t AT = NI + 64 * 65 * 4;       // D_i A_ik below the diagonal blocks, fp32 [64][65]
constexpr uint32_t RTH = 65536, RTL = 98304;
constexpr uint32_t OSTG = RKH;                  // once Rk^T is formed: a whole chunk of O, row-major [64][128] fp32    // once T is formed: Rk^T (Kb^T) hi / lo, 128 rows x 64 (two 16 KB blocks)
// exact chunks: k^, q^, G fp32 [64][129] in the [Lk; Lq] area before it is built
constexpr int XLD = 129;
constexpr uint32_t XK = 0, XQ = 64 * XLD * 4, XG = 2 * 64 * XLD * 4;
constexpr uint32_t SMALL = 196608;
constexpr uint32_t SMEM = SMALL + 3344 + 16 + 4096 + 1024;  // vectors, barrier, norm partials, alignment
static_assert(AT + 64 * 65 * 4 <= RKH && XG + 64 * XLD * 4 <= RKH && PL + 16384 <= RTH, "tile overlap");
static_assert(SMEM <= 232448, "shared memory of the tf32 prefill");
// TMEM columns
constexpr uint32_t T_S = 0;    // S~^T (fp32 accumulator; also the hi part of G0's A operand)
constexpr uint32_t T_W = 128;  // S~ lo | W^T hi, lo | U^T hi, lo (A operands)
constexpr uint32_t T_XO = 256; // X^T (64 columns), O^T (64)
constexpr uint32_t T_AP = 384; // [A_raw; P_raw] (lanes = rows of [Lk; Lq])
constexpr uint32_t T_U = 448;  // U^T

constexpr uint32_t ID_N64 = idesc_tf32(128, 64), ID_N128 = idesc_tf32(128, 128);

__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xffffe000u); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// byte offset of element (row, k) in a K-major fp32 tile of `rows` rows, 128-byte swizzle
__device__ __forceinline__ uint32_t kmaj(int row, int k, int rows) {
    return (uint32_t)((k >> 5) * rows * 128 + row * 128 + ((((k & 31) >> 2) ^ (row & 7)) << 4) + ((k & 3) << 2));
}
__device__ __forceinline__ void put_hilo(uint8_t *sm, uint32_t hi, uint32_t lo, uint32_t off, float x) {
    const float h = tf32_hi(x);
    *reinterpret_cast<float *>(sm + hi + off) = h;
    *reinterpret_cast<float *>(sm + lo + off) = x - h;
}
__device__ __forceinline__ void put_hilo4(uint8_t *sm, uint32_t hi, uint32_t lo, uint32_t off, const float (&x)[4]) {
    float4 h, l;
    h.x = tf32_hi(x[0]); h.y = tf32_hi(x[1]); h.z = tf32_hi(x[2]); h.w = tf32_hi(x[3]);
    l.x = x[0] - h.x; l.y = x[1] - h.y; l.z = x[2] - h.z; l.w = x[3] - h.w;
    *reinterpret_cast<float4 *>(sm + hi + off) = h;
    *reinterpret_cast<float4 *>(sm + lo + off) = l;
}

__device__ __forceinline__ bool elect_one() {
    uint32_t p;
    asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(p));
    return p != 0;
}

// D (+)= A B^T in 3xTF32 over NK steps of K = 8. A and B K-major in shared
// memory (hi / lo descriptors), K blocks of 32 elements ABLK / BBLK bytes
// apart; the first step overwrites D unless `acc`.
template <int NK, uint32_t ABLK, uint32_t BBLK>
__device__ __forceinline__ void prod_ss(uint32_t d, uint64_t ah, uint64_t al, uint64_t bh, uint64_t bl,
                                        uint32_t idesc, bool acc) {
#pragma unroll 1
    for (int kb = 0; kb < NK / 4; ++kb) {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const uint64_t oa = (uint64_t)((kb * ABLK + k4 * 32) >> 4), ob = (uint64_t)((kb * BBLK + k4 * 32) >> 4);
            mma_tf32(d, ah + oa, bh + ob, idesc, (acc || kb > 0 || k4 > 0) ? 1u : 0u);
            mma_tf32(d, ah + oa, bl + ob, idesc, 1u);
            mma_tf32(d, al + oa, bh + ob, idesc, 1u);
        }
    }
}
// The same with A in TMEM (hi / lo columns ah / al, one element per column).
template <int NK, uint32_t BBLK>
__device__ __forceinline__ void prod_ts(uint32_t d, uint32_t ah, uint32_t al, uint64_t bh, uint64_t bl,
                                        uint32_t idesc, bool acc) {
#pragma unroll 1
    for (int kb = 0; kb < NK / 4; ++kb) {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
            const uint64_t ob = (uint64_t)((kb * BBLK + k4 * 32) >> 4);
            const uint32_t ka = 32 * kb + 8 * k4;
            mma_tf32_ts(d, ah + ka, bh + ob, idesc, (acc || kb > 0 || k4 > 0) ? 1u : 0u);
            mma_tf32_ts(d, ah + ka, bl + ob, idesc, 1u);
            mma_tf32_ts(d, al + ka, bh + ob, idesc, 1u);
        }
    }
}

}  // namespace tfp

template <int GM>
__global__ void __launch_bounds__(tfp::NT, 1)
    prefill_tf32_kernel(const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ q,
                        const float *__restrict__ k, const float *__restrict__ v,
                        const float *__restrict__ g, const float *__restrict__ beta, const float *s_init,
                        float *s_final, float *__restrict__ out, const int64_t *__restrict__ cu_seqlens, int N,
                        int64_t Ttot, int H, int Cc, float eps, unsigned *err, const int *__restrict__ order,
                        int v_zero) {
    using namespace tfp;
    constexpr bool GCH = GM == KDA_GATE_CHANNEL, GHD = GM == KDA_GATE_HEAD;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base derived from the shared array itself (accesses compile to shared-memory instructions)
    uint8_t *sm = smem_raw + ((1024u - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023u)) & 1023u);
    float *vec = reinterpret_cast<float *>(sm + SMALL);
    float *s_rk = vec, *s_rq = vec + 64, *s_beta = vec + 128;
    float *s_fac = vec + 448, *s_fpend = vec + 576, *s_egl = vec + 704;
    float *s_part = reinterpret_cast<float *>(sm + SMALL + 3344 + 16);  // [8 row groups][128] decay totals
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + SMALL + 3328);
    uint32_t *s_taddr = reinterpret_cast<uint32_t *>(sm + SMALL + 3336);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, q4 = warp & 3, half = warp >> 2;
    // front (loads, norms, decay, operand build): warp = 8-row group, lane = 4-channel group
    const int h = blockIdx.x % H, n = order ? order[blockIdx.x / H] : (int)(blockIdx.x / H);
    int64_t start, end;
    if (!seq_range(cu_seqlens, n, N, Ttot, err, start, end)) return;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(s_taddr, 512);
        tmem_relinquish();
    }
    if (tid < 128) s_fpend[tid] = 1.f;
    sync_tc();
    const uint32_t tbase = *s_taddr;
    const uint32_t lq = (uint32_t)(32 * q4) << 16;  // this warp's TMEM lane quarter
    const int jl = 32 * q4 + lane;                    // this thread's TMEM lane (value channel)
    const uint32_t sb = smem_u32(sm);
    const size_t soff = ((size_t)n * H + h) * D * D;
    // the entry state, S^T: lane j, column i
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {
        const int i0 = 64 * half + 32 * part;
        uint32_t r[32];
#pragma unroll
        for (int m = 0; m < 32; ++m) r[m] = s_init ? f2u(s_init[soff + (size_t)(i0 + m) * D + jl]) : 0u;
        tmem_st32(tbase + lq + T_S + i0, r);
    }
    tmem_st_wait();

    uint32_t phase = 0;
    bool ok = true;
    auto issue = [&](auto &&body) {
        if (warp == 0) {
            if (elect_one()) body();
            __syncwarp();
        }
    };
    auto wait_mma = [&]() {
        const bool w = mbar_wait(bar, phase, WAIT_LIMIT);
        ok = __syncthreads_and(w) != 0;
        if (ok) phase ^= 1u;
        tc_fence_after();
    };

    // this thread's g, k, q (rows 8 warp.., channels 4 lane..) and beta of the chunk at c0 into registers,
    // 16-byte loads in one round trip; the loads of the next chunk are issued once G3/G4 of this one run
    float4 gr[8], kr[8], qr[8];
    float br = 0.f;
    auto load_chunk = [&](int64_t c0, int L) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const int r = 8 * warp + m;
            gr[m] = kr[m] = qr[m] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < L) {
                const size_t o = ((size_t)(c0 + r) * H + h) * D + 4 * lane;
                kr[m] = *reinterpret_cast<const float4 *>(k + o);
                qr[m] = *reinterpret_cast<const float4 *>(q + o);
                if constexpr (GCH) {
                    gr[m] = *reinterpret_cast<const float4 *>(g + o);
                } else if constexpr (GHD) {
                    const float gv = g[(size_t)(c0 + r) * H + h];
                    gr[m] = make_float4(gv, gv, gv, gv);
                }
            }
        }
        if (tid < 64) br = tid < L ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
    };
    auto f4 = [](const float4 &x, int e) -> float { return e == 0 ? x.x : e == 1 ? x.y : e == 2 ? x.z : x.w; };
    if (start < end) load_chunk(start, (int)((end - start) < (int64_t)Cc ? (end - start) : (int64_t)Cc));
    for (int64_t c0 = start; c0 < end; c0 += Cc) {
        const int L = (int)((end - c0) < (int64_t)Cc ? (end - c0) : (int64_t)Cc);
        // ---- the next chunk's rows of q, k, v (and g) into L2 while this one is processed
        if (c0 + Cc < end) {
            const int64_t n0 = c0 + Cc;
            const int Ln = (int)((end - n0) < (int64_t)Cc ? (end - n0) : (int64_t)Cc);
            const int which = tid >> 6, r = tid & 63;
            const float *src = which == 0 ? q : which == 1 ? k : which == 2 ? (v_zero ? nullptr : v)
                                                                            : (GCH ? g : nullptr);
            if (r < Ln && src != nullptr) prefetch_l2_bulk(src + ((size_t)(n0 + r) * H + h) * D, D * 4);
        }
        // the previous chunk's output copy has read its staging (the Rk area this chunk's build writes)
        if (tid == 0) bulk_wait_read();
        if (tid < 64) s_beta[tid] = br;
        // row norms: the warp holds all 128 channels of its 8 rows; a halving butterfly over lane bits 2..0
        // leaves row (lane & 7)'s partial on the lane, and lane bits 3, 4 finish the sum
        {
            float a[8], b[8];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                a[m] = kr[m].x * kr[m].x + kr[m].y * kr[m].y + kr[m].z * kr[m].z + kr[m].w * kr[m].w;
                b[m] = qr[m].x * qr[m].x + qr[m].y * qr[m].y + qr[m].z * qr[m].z + qr[m].w * qr[m].w;
            }
#pragma unroll
            for (int w = 4; w > 0; w >>= 1) {
                const bool up = (lane & w) != 0;
#pragma unroll
                for (int m = 0; m < w; ++m) {
                    const float sa = up ? a[m] : a[m + w], sb = up ? b[m] : b[m + w];
                    const float ra = __shfl_xor_sync(0xffffffffu, sa, w), rb = __shfl_xor_sync(0xffffffffu, sb, w);
                    a[m] = (up ? a[m + w] : a[m]) + ra;
                    b[m] = (up ? b[m + w] : b[m]) + rb;
                }
            }
            a[0] += __shfl_xor_sync(0xffffffffu, a[0], 8);
            b[0] += __shfl_xor_sync(0xffffffffu, b[0], 8);
            a[0] += __shfl_xor_sync(0xffffffffu, a[0], 16);
            b[0] += __shfl_xor_sync(0xffffffffu, b[0], 16);
            if (lane < 8) {
                const int r = 8 * warp + lane;
                s_rk[r] = r < L ? inv_norm(a[0], eps) : 0.f;
                s_rq[r] = r < L ? inv_norm(b[0], eps) : 0.f;
            }
        }
        {  // decay totals of this row group per channel
            float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                t.x += gr[m].x; t.y += gr[m].y; t.z += gr[m].z; t.w += gr[m].w;
            }
            *reinterpret_cast<float4 *>(s_part + warp * 128 + 4 * lane) = t;
        }
        __syncthreads();
        // G of row r runs as (G of the row groups before) + its g, in row order; G_L and the anchors per channel
        float off[4] = {0.f, 0.f, 0.f, 0.f}, GL[4] = {0.f, 0.f, 0.f, 0.f}, cI[4];
#pragma unroll
        for (int w2 = 0; w2 < 8; ++w2) {
            const float4 t = *reinterpret_cast<const float4 *>(s_part + w2 * 128 + 4 * lane);
            const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (w2 < warp) off[e] += tv[e];
                GL[e] += tv[e];
            }
        }
        const bool exact = __syncthreads_or(!(GL[0] >= -SPAN_MAX && GL[1] >= -SPAN_MAX && GL[2] >= -SPAN_MAX &&
                                              GL[3] >= -SPAN_MAX)) != 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) cI[e] = exact ? 0.f : fminf(0.f, GL[e] + ANCHOR);
        if (warp == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s_fac[4 * lane + e] = s_fpend[4 * lane + e] * expf(cI[e]);
                s_egl[4 * lane + e] = expf(GL[e]);
            }
        }

        // ---- operand tiles: [Lk; Lq] and, row-major, the state-update operand Rk (Kb on exact chunks)
        if (!exact) {
            float acc[4] = {off[0], off[1], off[2], off[3]};
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = 8 * warp + m;
                const float rk = s_rk[r], rq = s_rq[r];
                float lk[4], lq[4], rkv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[e] += f4(gr[m], e);
                    const float kh = f4(kr[m], e) * rk, qh = f4(qr[m], e) * rq;
                    const float e1 = expf(acc[e] - cI[e]), e2 = expf(cI[e] - acc[e]);
                    lk[e] = e1 * kh;
                    lq[e] = e1 * qh;
                    rkv[e] = e2 * kh;
                }
                put_hilo4(sm, KQH, KQL, kmaj(r, 4 * lane, 128), lk);
                put_hilo4(sm, KQH, KQL, kmaj(64 + r, 4 * lane, 128), lq);
                put_hilo4(sm, RKH, RKL, kmaj(r, 4 * lane, 64), rkv);
            }
        } else {
            // exact pairwise decays: stage k^, q^, G; A_raw and P_raw straight into TMEM; then [Lk; Lq], c = 0
            float *xk = reinterpret_cast<float *>(sm + XK), *xq = reinterpret_cast<float *>(sm + XQ);
            float *xg = reinterpret_cast<float *>(sm + XG);
            float acc[4] = {off[0], off[1], off[2], off[3]};
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = 8 * warp + m;
                const float rk = s_rk[r], rq = s_rq[r];
                float kb[4], gg[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[e] += f4(gr[m], e);
                    gg[e] = acc[e];
                    const float kh = f4(kr[m], e) * rk;
                    xk[r * XLD + 4 * lane + e] = kh;
                    xq[r * XLD + 4 * lane + e] = f4(qr[m], e) * rq;
                    xg[r * XLD + 4 * lane + e] = acc[e];
                    kb[e] = expf(GL[e] - acc[e]) * kh;
                }
                gr[m] = make_float4(gg[0], gg[1], gg[2], gg[3]);  // G from here on
                put_hilo4(sm, RKH, RKL, kmaj(r, 4 * lane, 64), kb);
            }
            __syncthreads();
            {
                // lane = row of [A_raw; P_raw] (key row r for A, query row r for P), 32 columns s
                const int rr = jl & 63;
                const float *xa = jl < 64 ? xk : xq;
                uint32_t o[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const int s = 32 * half + m;
                    float a = 0.f;
                    if (s <= rr) {
#pragma unroll 4
                        for (int i = 0; i < D; ++i)
                            a = fmaf(xa[rr * XLD + i], xk[s * XLD + i] * expf(xg[rr * XLD + i] - xg[s * XLD + i]), a);
                    }
                    o[m] = f2u(a);
                }
                tmem_st32(tbase + lq + T_AP + 32 * half, o);
                tmem_st_wait();
            }
            __syncthreads();
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const int r = 8 * warp + m;
                const float rk = s_rk[r], rq = s_rq[r];
                float lk[4], lq[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float e1 = expf(f4(gr[m], e));
                    lk[e] = e1 * f4(kr[m], e) * rk;
                    lq[e] = e1 * f4(qr[m], e) * rq;
                }
                put_hilo4(sm, KQH, KQL, kmaj(r, 4 * lane, 128), lk);
                put_hilo4(sm, KQH, KQL, kmaj(64 + r, 4 * lane, 128), lq);
            }
        }
        fence_async_smem();
        __syncthreads();
        // G1 runs while the state is read back
        if (!exact)
            issue([&] {
                prod_ss<16, 16384, 8192>(tbase + T_AP, sdesc_sw128(sb + KQH, 16, 1024), sdesc_sw128(sb + KQL, 16, 1024),
                                         sdesc_sw128(sb + RKH, 16, 1024), sdesc_sw128(sb + RKL, 16, 1024), ID_N64,
                                         false);
            });
        // ---- state read-back: S~ = Diag(pending factor x e^c) Acc, written back with its lo part
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
            uint32_t r[32], lo[32];
            tmem_ld32(tbase + lq + T_S + i0, r);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                const float x = u2f(r[m]) * s_fac[i0 + m];
                r[m] = f2u(x);
                lo[m] = f2u(x - tf32_hi(x));
            }
            tmem_st32(tbase + lq + T_S + i0, r);
            tmem_st32(tbase + lq + T_W + i0, lo);
        }
        tmem_st_wait();
        sync_tc();
        issue([&] {
            prod_ts<16, 16384>(tbase + T_XO, tbase + T_S, tbase + T_W, sdesc_sw128(sb + KQH, 16, 1024),
                               sdesc_sw128(sb + KQL, 16, 1024), ID_N128, false);
            mma_commit(bar);
        });
        // v^T of this thread's value channel (warps 4-7), loaded while G0 runs
        float vv[64];
        if (half == 1) {
#pragma unroll
            for (int s = 0; s < 64; ++s) vv[s] = (s < L && !v_zero) ? v[((size_t)(c0 + s) * H + h) * D + jl] : 0.f;
        }
        wait_mma();
        if (!ok) break;

        // ---- A and P rows (warps 0-3: lane = row of [A; P]); W^T = V^T - X^T (warps 4-7: lane = j)
        if (half == 0) {
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
                float a[32];
                {
                    uint32_t r0[32];
                    tmem_ld32(tbase + lq + T_AP + 32 * part, r0);
                    tmem_ld_wait();
#pragma unroll
                    for (int m = 0; m < 32; ++m) a[m] = u2f(r0[m]);
                }
                if (jl < 64) {
                    float *af = reinterpret_cast<float *>(sm + AF);
                    const float br = s_beta[jl];
#pragma unroll
                    for (int m = 0; m < 32; ++m) {
                        const int s = 32 * part + m;
                        af[jl * 65 + s] = s < jl ? br * a[m] : 0.f;
                    }
                } else {
                    const int r = jl - 64;
#pragma unroll
                    for (int s4 = 0; s4 < 8; ++s4) {
                        float p[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int s = 32 * part + 4 * s4 + u;
                            p[u] = (s <= r && r < L) ? a[4 * s4 + u] : 0.f;
                        }
                        put_hilo4(sm, PH, PL, kmaj(r, 32 * part + 4 * s4, 64), p);
                    }
                }
            }
        } else {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                uint32_t x[32], hi[32];
                tmem_ld32(tbase + lq + T_XO + 32 * part, x);
                tmem_ld_wait();
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const float w = vv[32 * part + m] - u2f(x[m]);
                    const float wh = tf32_hi(w);
                    hi[m] = f2u(wh);
                    x[m] = f2u(w - wh);
                }
                tmem_st32(tbase + lq + T_W + 32 * part, hi);
                tmem_st32(tbase + lq + T_W + 64 + 32 * part, x);
            }
            tmem_st_wait();
        }
        __syncthreads();

        // ---- T = (I + A)^-1 Diag(beta): diagonal 16 x 16 blocks by forward substitution
        //      (warp b, lane = column), then block row by block row
        {
            const float *af = reinterpret_cast<const float *>(sm + AF);
            float *ni = reinterpret_cast<float *>(sm + NI), *at = reinterpret_cast<float *>(sm + AT);
            if (warp < 4 && lane < 16) {
                const int b0 = 16 * warp, c = lane;  // column c of D_b, rows in order
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = r == c ? 1.f : 0.f;
#pragma unroll
                    for (int t = 0; t < r; ++t) acc = fmaf(-af[(b0 + r) * 65 + b0 + t], x[t], acc);
                    x[r] = acc;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) ni[(b0 + r) * 65 + b0 + c] = x[r];
            }
            __syncthreads();
            // At_ik = D_i A_ik for the six blocks below the diagonal (i > k)
            // every thread one element (row rr, column cc) of each of the six blocks: six independent chains
            const int rr = tid >> 4, cc = tid & 15;
#pragma unroll
            for (int pb = 0; pb < 6; ++pb) {
                const int i = pb < 1 ? 1 : pb < 3 ? 2 : 3, kb = pb - (i * (i - 1)) / 2;
                float y = 0.f;
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    if (t <= rr) y = fmaf(ni[(16 * i + rr) * 65 + 16 * i + t], af[(16 * i + t) * 65 + 16 * kb + cc], y);
                at[(16 * i + rr) * 65 + 16 * kb + cc] = y;
            }
            __syncthreads();
            // block row i: Ninv_ij = -sum_{j <= kb < i} At_i,kb Ninv_kb,j for j < i
#pragma unroll
            for (int i = 1; i < 4; ++i) {
                float y[3];
#pragma unroll
                for (int j = 0; j < i; ++j) {  // element (rr, cc) of block (i, j): i independent chains
                    float acc = 0.f;
#pragma unroll
                    for (int kb = j; kb < i; ++kb)
#pragma unroll
                        for (int t = 0; t < 16; ++t)
                            acc = fmaf(at[(16 * i + rr) * 65 + 16 * kb + t], ni[(16 * kb + t) * 65 + 16 * j + cc], acc);
                    y[j] = acc;
                }
#pragma unroll
                for (int j = 0; j < i; ++j) ni[(16 * i + rr) * 65 + 16 * j + cc] = -y[j];
                __syncthreads();
            }
            for (int e = tid; e < C * 16; e += NT) {
                const int r = e >> 4, s4 = e & 15;
                float t[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int s = 4 * s4 + u;
                    t[u] = s <= r ? ni[r * 65 + s] * s_beta[s] : 0.f;
                }
                put_hilo4(sm, TH, TL, kmaj(r, 4 * s4, 64), t);
            }
        }
        fence_async_smem();
        sync_tc();
        issue([&] {
            prod_ts<8, 8192>(tbase + T_U, tbase + T_W, tbase + T_W + 64, sdesc_sw128(sb + TH, 16, 1024),
                             sdesc_sw128(sb + TL, 16, 1024), ID_N64, false);
            mma_commit(bar);
        });
        wait_mma();
        if (!ok) break;

        // ---- U^T hi / lo into TMEM; Rk^T (Kb^T) tile; on exact chunks the state decays now
        {
            uint32_t u[32], hi[32];
            tmem_ld32(tbase + lq + T_U + 32 * half, u);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                const float x = u2f(u[m]), xh = tf32_hi(x);
                hi[m] = f2u(xh);
                u[m] = f2u(x - xh);
            }
            tmem_st32(tbase + lq + T_W + 32 * half, hi);
            tmem_st32(tbase + lq + T_W + 64 + 32 * half, u);
        }
        // Rk^T (Kb^T) from the row-major tile: thread (channel ci, rows 32 ch..), 16-byte groups of 4 rows
        const int ci = tid & 127, ch = tid >> 7;
#pragma unroll 2
        for (int g4 = 0; g4 < 8; ++g4) {
            const int r0 = 32 * ch + 4 * g4;
            float4 hv, lv;
            hv.x = *reinterpret_cast<const float *>(sm + RKH + kmaj(r0, ci, 64));
            hv.y = *reinterpret_cast<const float *>(sm + RKH + kmaj(r0 + 1, ci, 64));
            hv.z = *reinterpret_cast<const float *>(sm + RKH + kmaj(r0 + 2, ci, 64));
            hv.w = *reinterpret_cast<const float *>(sm + RKH + kmaj(r0 + 3, ci, 64));
            lv.x = *reinterpret_cast<const float *>(sm + RKL + kmaj(r0, ci, 64));
            lv.y = *reinterpret_cast<const float *>(sm + RKL + kmaj(r0 + 1, ci, 64));
            lv.z = *reinterpret_cast<const float *>(sm + RKL + kmaj(r0 + 2, ci, 64));
            lv.w = *reinterpret_cast<const float *>(sm + RKL + kmaj(r0 + 3, ci, 64));
            const uint32_t off = kmaj(ci, r0, 128);
            *reinterpret_cast<float4 *>(sm + RTH + off) = hv;
            *reinterpret_cast<float4 *>(sm + RTL + off) = lv;
        }
        if (exact) {
#pragma unroll 1
            for (int part = 0; part < 2; ++part) {
                const int i0 = 64 * half + 32 * part;
                uint32_t r[32];
                tmem_ld32(tbase + lq + T_S + i0, r);
                tmem_ld_wait();
#pragma unroll
                for (int m = 0; m < 32; ++m) r[m] = f2u(u2f(r[m]) * s_egl[i0 + m]);
                tmem_st32(tbase + lq + T_S + i0, r);
            }
        }
        tmem_st_wait();
        fence_async_smem();
        sync_tc();
        if (warp == 0)
#pragma unroll
            for (int e = 0; e < 4; ++e) s_fpend[4 * lane + e] = exact ? 1.f : expf(GL[e] - cI[e]);
        issue([&] {
            prod_ts<8, 8192>(tbase + T_XO + 64, tbase + T_W, tbase + T_W + 64, sdesc_sw128(sb + PH, 16, 1024),
                             sdesc_sw128(sb + PL, 16, 1024), ID_N64, true);
            prod_ts<8, 16384>(tbase + T_S, tbase + T_W, tbase + T_W + 64, sdesc_sw128(sb + RTH, 16, 1024),
                              sdesc_sw128(sb + RTL, 16, 1024), ID_N128, true);
            mma_commit(bar);
        });
        if (c0 + Cc < end) load_chunk(c0 + Cc, (int)((end - c0 - Cc) < (int64_t)Cc ? (end - c0 - Cc) : (int64_t)Cc));
        wait_mma();
        if (!ok) break;

        // ---- O^T -> out (warp half: 32 rows). A whole chunk is staged row-major in the dead Rk area and
        //      leaves by one tensor copy; a sequence's short last chunk by plain stores of its own rows
        //      (the rows after it belong to the next sequence)
        {
            uint32_t o[32];
            tmem_ld32(tbase + lq + T_XO + 64 + 32 * half, o);
            tmem_ld_wait();
            if (L == C) {
                float *ost = reinterpret_cast<float *>(sm + OSTG);
#pragma unroll
                for (int m = 0; m < 32; ++m) ost[(32 * half + m) * D + jl] = u2f(o[m]);
                fence_async_smem();
                __syncthreads();
                if (tid == 0) {
                    tma_store_2d(&tm_o, ost, h * D, (int)c0);
                    bulk_commit();
                }
            } else {
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const int r = 32 * half + m;
                    if (r < L) out[((size_t)(c0 + r) * H + h) * D + jl] = u2f(o[m]);
                }
            }
        }
        __syncthreads();
    }
    sync_tc();
    if (ok && s_final) {
#pragma unroll 1
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * half + 32 * part;
            uint32_t r[32];
            tmem_ld32(tbase + lq + T_S + i0, r);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < 32; ++m) s_final[soff + (size_t)(i0 + m) * D + jl] = u2f(r[m]) * s_fpend[i0 + m];
        }
    }
    if (tid == 0) bulk_wait_all();  // output copies complete before the CTA's shared memory goes away
    if (!ok) {
        if (tid == 0) {
            atomicOr(err, DEVERR_TIMEOUT);
            mbar_wait(bar, phase, WAIT_LIMIT);  // the MMAs still in flight finish before TMEM is freed
        }
    }
    sync_tc();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// fp32, d = 128, C >= 16; the output copy's row coordinate is 32-bit
bool prefill_tf32_applicable(const PrefillArgs &a) {
    return !a.bf16 && a.D == 128 && a.C >= 16 && a.C <= 64 && a.T > 0 && a.T <= 0x7fffffffLL;
}

template <int GM>
static kda_status launch_tf32(const PrefillArgs &a, cudaStream_t s) {
    auto kern = prefill_tf32_kernel<GM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tfp::SMEM);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    // whole output chunks leave through this map: 64 rows x one head's 128 channels
    CUtensorMap mo;
    if (!tcp::make_map(&mo, a.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)a.H * tfp::D, (uint64_t)a.T, tfp::D,
                       tfp::C, CU_TENSOR_MAP_SWIZZLE_NONE))
        return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    kern<<<launch_seqs(a) * a.H, tfp::NT, tfp::SMEM, s>>>(
        mo, static_cast<const float *>(a.q), static_cast<const float *>(a.k), static_cast<const float *>(a.v), a.g,
        a.beta, a.s_init, a.s_final, static_cast<float *>(a.out), a.cu_seqlens, a.N, a.T, a.H, a.C, a.eps, a.err,
        a.order, a.v_zero ? 1 : 0);
    return check_launch("prefill_tf32_kernel");
}

kda_status prefill_tf32(const PrefillArgs &a, cudaStream_t s) {
    if (a.gate == KDA_GATE_HEAD) return launch_tf32<KDA_GATE_HEAD>(a, s);
    if (a.gate == KDA_GATE_NONE) return launch_tf32<KDA_GATE_NONE>(a, s);
    return launch_tf32<KDA_GATE_CHANNEL>(a, s);
}

}  // namespace kda
