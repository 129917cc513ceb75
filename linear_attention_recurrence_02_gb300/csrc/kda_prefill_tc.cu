// kda_prefill_tc.cu -- chunked KDA prefill on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA) for bf16 q/k/v, d_k = d_v = 128, chunk 64.
//
// Method: the chunk algebra of the general kernel (kda_prefill.cu; "为什么 Kimi
// K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化", section 5: attention-
// like work inside a chunk, state hand-off between chunks; section 6:
// cumulative decay as a product of gates; the WY/UT reparameterisation it
// names is realised here as T = (I + A)^-1 Diag(beta)). With G the
// cumulative log decay inside the chunk and a per-channel anchor c:
//   Lk = e^{G-c} k^,  Lq = e^{G-c} q^,  Rk = e^{c-G} k^,  Kb = e^{G_L-G} k^,
//   S~ = Diag(e^c) S
//   [A_raw; P_raw] = [Lk; Lq] Rk^T            (G1)   A = mask_<(beta A_raw)
//   T = (I + A)^-1 Diag(beta)                  (CUDA cores, fp32)
//   W' = T Lk,  U0 = T V                       (G2, G3)
//   U = U0 - W' S~                             (G4)
//   O = Lq S~ + P U                            (G5, G6)
//   S <- Diag(e^{G_L}) S + Kb^T U              (G7)
// Lk S~ = Diag-folded e^G k^ S, so W' S~ = T Kt S and Lq S~ = Qt S exactly.
// c = min(0, G_L + 80) keeps every factor inside e^[-80, 80] whenever the
// chunk's decay span G_0 - G_L is at most 160; a chunk beyond that computes
// A and P with exact pairwise exponentials on CUDA cores and uses c = 0.
//
// Layout: every MMA has M = 128 on a channel axis, so TMEM lane = channel
// (key channel i or value channel j) throughout, and the fp32 master state
// S^T (lane j, column i) never leaves TMEM between chunks. Operands are bf16
// in 128-byte-swizzled shared memory tiles, loaded by TMA (q, k, v, g) or
// written by the CUDA cores from TMEM read-backs.
//
// One CTA (256 threads, 2 warpgroups) per (sequence, head) walks the chunks
// of its sequence; thread 0 issues TMA and MMAs, every wait is bounded.
#include <cuda.h>

#include <string>

#include "kda_common.cuh"
#include "kda_prefill.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace tcp {

using namespace tc;

constexpr int C = 64, D = 128, NT = 256;
// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_QRAW = 0;        // q tile (TMA) -> W' tile (MN-major, rows i)
constexpr uint32_t OFF_KRAW = 16384;    // k tile (TMA) -> U^T tile (K-major, rows j)
constexpr uint32_t OFF_V = 32768;       // v tile (TMA)
constexpr uint32_t OFF_G = 49152;       // g fp32 [64][128] (TMA) -> G -> M^-1 (fp32, column-major) + scratch
constexpr uint32_t OFF_LKQ = 81920;     // [Lk; Lq] 128 rows
constexpr uint32_t OFF_RK = 114688;     // Rk 64 rows -> A^T fp32 [64][64]
constexpr uint32_t OFF_KB = 131072;     // Kb 64 rows
constexpr uint32_t OFF_SOP = 147456;    // S~^T 128 rows (j) x 128 (i)
constexpr uint32_t OFF_T = 180224;      // T 64 rows (r) x 64 (s)
constexpr uint32_t OFF_P = 188416;      // P 64 rows (r) x 64 (s)
constexpr uint32_t OFF_SMALL = 196608;  // per-row / per-channel vectors, barriers
constexpr uint32_t SMEM_BYTES = OFF_SMALL + 4096 + 1024;
constexpr uint32_t LOAD_BYTES = 3 * 16384 + 32768;
// TMEM columns (512 allocated)
constexpr uint32_t TM_S = 0, TM_AP = 128, TM_W = 192, TM_U0 = 256, TM_X = 320, TM_O = 384;
constexpr long long WAIT_LIMIT = 4000000000LL;  // clock cycles (about 2 s)
constexpr float SPAN_MAX = 160.f, ANCHOR = 80.f;

constexpr uint32_t ID_KK64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_MK64 = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_KM64 = idesc_bf16(128, 64, 0, 1);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, 0, 1);

// byte offset of 16-byte chunk cc (channels 8cc..8cc+7) of `row` in a
// 128-byte-swizzled tile whose 64-channel blocks hold `rows` rows each
__device__ __forceinline__ uint32_t swz(int row, int cc, int rows) {
    return (uint32_t)((cc >> 3) * rows * 128 + row * 128 + (((cc & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    __nv_bfloat162 t;
    t = __floats2bfloat162_rn(f[0], f[1]);
    u.x = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2bfloat162_rn(f[2], f[3]);
    u.y = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2bfloat162_rn(f[4], f[5]);
    u.z = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2bfloat162_rn(f[6], f[7]);
    u.w = *reinterpret_cast<uint32_t *>(&t);
    return u;
}

__device__ __forceinline__ void unpack8(uint4 u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 t = *reinterpret_cast<const __nv_bfloat162 *>(&w[e]);
        f[2 * e] = __bfloat162float(t.x);
        f[2 * e + 1] = __bfloat162float(t.y);
    }
}

__device__ __forceinline__ void sync_tc() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__device__ __forceinline__ void sync_for_mma() {
    fence_async_smem();
    sync_tc();
}

__global__ void __launch_bounds__(NT, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                      const float *__restrict__ beta, const float *s_init, float *s_final,
                      __nv_bfloat16 *__restrict__ out, const int64_t *__restrict__ cu_seqlens, int N,
                      int64_t Ttot, int H, float eps, unsigned *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float *s_rq = reinterpret_cast<float *>(sm + OFF_SMALL);
    float *s_rk = s_rq + 64;
    float *s_beta = s_rk + 64;
    float *s_gl = s_beta + 64;
    float *s_c = s_gl + 128;
    float *s_expc = s_c + 128;
    float *s_expgl = s_expc + 128;
    uint64_t *bar_load = reinterpret_cast<uint64_t *>(s_expgl + 128);
    uint64_t *bar_mma = bar_load + 1;
    uint32_t *s_taddr = reinterpret_cast<uint32_t *>(bar_mma + 1);
    float *gt = reinterpret_cast<float *>(sm + OFF_G);
    float *AT = reinterpret_cast<float *>(sm + OFF_RK);  // A^T: AT[s*64 + r] = A[r][s]
    float *MT = gt;                                      // M^-1 column-major: MT[s*64 + r]
    float *Yb = gt + 4096;                               // scratch for the blocked inverse

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3, hh = warp >> 2;
    const int h = blockIdx.x % H, n = blockIdx.x / H;
    int64_t start, end;
    if (!seq_range(cu_seqlens, n, N, Ttot, err, start, end)) return;

    if (tid == 0) {
        mbar_init(bar_load, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_g);
    }
    if (warp == 0) {
        tmem_alloc(s_taddr, 512);
        tmem_relinquish();
    }
    sync_tc();
    const uint32_t tbase = *s_taddr;
    const uint32_t lrow = (uint32_t)(32 * q4) << 16;  // this warp's TMEM lane quarter
    const uint32_t sbase = smem_u32(sm);
    const int jl = 32 * q4 + lane;                    // this thread's TMEM lane (channel)
    const size_t soff = ((size_t)n * H + h) * D * D;

    // initial state -> TMEM (S^T: lane j, column i)
#pragma unroll
    for (int part = 0; part < 2; ++part) {
        uint32_t r[32];
        const int i0 = 64 * hh + 32 * part;
#pragma unroll
        for (int m = 0; m < 32; ++m)
            r[m] = s_init ? __float_as_uint(s_init[soff + (size_t)(i0 + m) * D + jl]) : 0u;
        tmem_st32(tbase + lrow + TM_S + i0, r);
    }
    tmem_st_wait();

    uint32_t ph_load = 0, ph_mma = 0;
    bool ok = true;
    for (int64_t c0 = start; c0 < end; c0 += C) {
        const int L = (int)((end - c0) < (int64_t)C ? (end - c0) : (int64_t)C);
        sync_for_mma();  // previous chunk fully consumed before its buffers are refilled
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_load, LOAD_BYTES);
            const int x0 = h * D, y0 = (int)c0;
            tma_load_2d(sm + OFF_QRAW, &tm_q, bar_load, x0, y0);
            tma_load_2d(sm + OFF_QRAW + 8192, &tm_q, bar_load, x0 + 64, y0);
            tma_load_2d(sm + OFF_KRAW, &tm_k, bar_load, x0, y0);
            tma_load_2d(sm + OFF_KRAW + 8192, &tm_k, bar_load, x0 + 64, y0);
            tma_load_2d(sm + OFF_V, &tm_v, bar_load, x0, y0);
            tma_load_2d(sm + OFF_V + 8192, &tm_v, bar_load, x0 + 64, y0);
            tma_load_2d(sm + OFF_G, &tm_g, bar_load, x0, y0);
        }
        if (tid < C) s_beta[tid] = tid < L ? beta[(size_t)(c0 + tid) * H + h] : 0.f;
        bool got = mbar_wait(bar_load, ph_load, WAIT_LIMIT);
        if (__syncthreads_or(!got)) {
            mbar_wait(bar_load, ph_load, WAIT_LIMIT);
            ok = false;
            break;
        }
        ph_load ^= 1;

        // rows past the end of the sequence: zero q, k, v, g (so beta = 0,
        // k = 0 and G stays at G_{L-1}); they then contribute nothing
        if (L < C) {
            const uint4 z4 = make_uint4(0, 0, 0, 0);
            for (int p = tid; p < (C - L) * 16; p += NT) {
                const int r = L + (p >> 4), cc = p & 15;
                const uint32_t o = swz(r, cc, 64);
                *reinterpret_cast<uint4 *>(sm + OFF_QRAW + o) = z4;
                *reinterpret_cast<uint4 *>(sm + OFF_KRAW + o) = z4;
                *reinterpret_cast<uint4 *>(sm + OFF_V + o) = z4;
            }
            for (int p = tid; p < (C - L) * 32; p += NT)
                *reinterpret_cast<uint4 *>(sm + OFF_G + (L + (p >> 5)) * 512 + (p & 31) * 16) = z4;
            __syncthreads();
        }

        // L2 norms of the q and k rows (one warp per row, 8 bytes per lane)
        for (int rr = warp; rr < 2 * C; rr += NT / 32) {
            const int r = rr & 63;
            const uint8_t *tile = sm + (rr < C ? OFF_QRAW : OFF_KRAW);
            const int kb = lane >> 4, ch = (lane & 15) >> 1, half = lane & 1;
            const uint2 u = *reinterpret_cast<const uint2 *>(tile + kb * 8192 + r * 128 + ((ch ^ (r & 7)) << 4) +
                                                             half * 8);
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
            const float f0 = __bfloat162float(a.x), f1 = __bfloat162float(a.y), f2 = __bfloat162float(b.x),
                        f3 = __bfloat162float(b.y);
            float ss = f0 * f0 + f1 * f1 + f2 * f2 + f3 * f3;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            if (lane == 0) (rr < C ? s_rq : s_rk)[r] = inv_norm(ss, eps);
        }
        // cumulative log decay G along the chunk (two halves, then fix-up)
        {
            const int i = tid & 127, r0 = (tid >> 7) * 32;
            float acc = 0.f;
            for (int r = r0; r < r0 + 32; ++r) {
                acc += gt[r * 128 + i];
                gt[r * 128 + i] = acc;
            }
        }
        __syncthreads();
        if (tid >= 128) {
            const int i = tid - 128;
            const float base = gt[31 * 128 + i];
            for (int r = 32; r < 64; ++r) gt[r * 128 + i] += base;
        }
        __syncthreads();
        // per-channel anchor; a chunk whose decay span exceeds SPAN_MAX takes the exact path
        int bad = 0;
        if (tid < 128) bad = !(gt[tid] - gt[63 * 128 + tid] <= SPAN_MAX);
        const int exact = __syncthreads_or(bad);
        if (tid < 128) {
            const float GL = gt[63 * 128 + tid];
            const float c = exact ? 0.f : fminf(0.f, GL + ANCHOR);
            s_gl[tid] = GL;
            s_c[tid] = c;
            s_expc[tid] = expf(c);
            s_expgl[tid] = expf(GL);
        }
        __syncthreads();

        // operand tiles Lk, Lq, Rk, Kb (bf16, swizzled) from q^, k^ and G
        for (int p = tid; p < C * 16; p += NT) {
            const int r = p >> 4, cc = p & 15;
            const uint32_t o64 = swz(r, cc, 64);
            float qf[8], kf[8];
            unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_QRAW + o64), qf);
            unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_KRAW + o64), kf);
            const float rq = s_rq[r], rk = s_rk[r];
            const float4 ga = *reinterpret_cast<const float4 *>(gt + r * 128 + cc * 8);
            const float4 gb = *reinterpret_cast<const float4 *>(gt + r * 128 + cc * 8 + 4);
            const float G[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
            float lk[8], lq[8], rkv[8], kbv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = cc * 8 + e;
                const float kh = kf[e] * rk, qh = qf[e] * rq;
                const float e1 = __expf(G[e] - s_c[i]);
                lk[e] = e1 * kh;
                lq[e] = e1 * qh;
                rkv[e] = __expf(s_c[i] - G[e]) * kh;
                kbv[e] = __expf(s_gl[i] - G[e]) * kh;
            }
            *reinterpret_cast<uint4 *>(sm + OFF_LKQ + swz(r, cc, 128)) = pack8(lk);
            *reinterpret_cast<uint4 *>(sm + OFF_LKQ + swz(r + 64, cc, 128)) = pack8(lq);
            if (!exact) *reinterpret_cast<uint4 *>(sm + OFF_RK + o64) = pack8(rkv);
            *reinterpret_cast<uint4 *>(sm + OFF_KB + o64) = pack8(kbv);
        }

        // S~^T = S^T Diag(e^c) as a bf16 operand; S^T <- S^T Diag(e^{G_L}) in TMEM
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * hh + 32 * part;
            uint32_t r[32];
            tmem_ld32(tbase + lrow + TM_S + i0, r);
            tmem_ld_wait();
            float so[32];
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                const float s = __uint_as_float(r[m]);
                so[m] = s * s_expc[i0 + m];
                r[m] = __float_as_uint(s * s_expgl[i0 + m]);
            }
            tmem_st32(tbase + lrow + TM_S + i0, r);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const int cc = part * 4 + qd;
                *reinterpret_cast<uint4 *>(sm + OFF_SOP + hh * 16384 + jl * 128 + ((cc ^ (jl & 7)) << 4)) =
                    pack8(so + 8 * qd);
            }
        }
        tmem_st_wait();

        if (exact) {
            // A^T and P with exact pairwise decays (rare: decay span > e^160)
            for (int p = tid; p < C * C; p += NT) {
                const int r = p & 63, s = p >> 6;
                float a = 0.f, pq = 0.f;
                if (s <= r) {
                    const float rkr = s_rk[r], rks = s_rk[s], rqr = s_rq[r];
                    for (int cc = 0; cc < 16; ++cc) {
                        float kr[8], ks[8], qr[8];
                        unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_KRAW + swz(r, cc, 64)), kr);
                        unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_KRAW + swz(s, cc, 64)), ks);
                        unpack8(*reinterpret_cast<const uint4 *>(sm + OFF_QRAW + swz(r, cc, 64)), qr);
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int i = cc * 8 + e;
                            const float x = ks[e] * rks * __expf(gt[r * 128 + i] - gt[s * 128 + i]);
                            a += kr[e] * rkr * x;
                            pq += qr[e] * rqr * x;
                        }
                    }
                }
                AT[s * 64 + r] = (s < r) ? s_beta[r] * a : 0.f;
                *reinterpret_cast<__nv_bfloat16 *>(sm + OFF_P + r * 128 + ((((s >> 3) ^ (r & 7))) << 4) +
                                                   (s & 7) * 2) = __float2bfloat16_rn(pq);
            }
        }
        sync_for_mma();

        // G1: [A_raw; P_raw] = [Lk; Lq] Rk^T   and   G5: O = Lq S~ (as O^T = S~^T Lq^T)
        if (tid == 0) {
            if (!exact) {
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
                    mma_bf16(tbase + TM_AP, sdesc_sw128(sbase + OFF_LKQ + kb * 16384 + ko, 16, 1024),
                             sdesc_sw128(sbase + OFF_RK + kb * 8192 + ko, 16, 1024), ID_KK64, ks > 0);
                }
            }
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
                mma_bf16(tbase + TM_O, sdesc_sw128(sbase + OFF_SOP + kb * 16384 + ko, 16, 1024),
                         sdesc_sw128(sbase + OFF_LKQ + 8192 + kb * 16384 + ko, 16, 1024), ID_KK64, ks > 0);
            }
            mma_commit(bar_mma);
        }
        got = mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
        if (__syncthreads_or(!got)) {
            mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
            ok = false;
            break;
        }
        ph_mma ^= 1;
        tc_fence_after();

        // read back A (lanes 0-63, masked, times beta) and P (lanes 64-127, masked)
        if (!exact) {
            uint32_t r32[32];
            tmem_ld32(tbase + lrow + TM_AP + 32 * hh, r32);
            tmem_ld_wait();
            const int s0 = 32 * hh;
            if (q4 < 2) {
                const int r = 32 * q4 + lane;
                const float br = s_beta[r];
#pragma unroll
                for (int m = 0; m < 32; ++m) AT[(s0 + m) * 64 + r] = (s0 + m < r) ? br * __uint_as_float(r32[m]) : 0.f;
            } else {
                const int r = 32 * (q4 - 2) + lane;
                float pv[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) pv[m] = (s0 + m <= r) ? __uint_as_float(r32[m]) : 0.f;
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                    const int cc = 4 * hh + qd;
                    *reinterpret_cast<uint4 *>(sm + OFF_P + r * 128 + ((cc ^ (r & 7)) << 4)) = pack8(pv + 8 * qd);
                }
            }
        }
        __syncthreads();

        // T = (I + A)^-1 Diag(beta): diagonal 16x16 blocks by forward substitution ...
        if (tid < 64) {
            const int s0 = tid, b0 = (tid >> 4) * 16;
            float x[16];
#pragma unroll
            for (int rl = 0; rl < 16; ++rl) {
                const int r = b0 + rl;
                float v = (r == s0) ? 1.f : 0.f;
#pragma unroll
                for (int kl = 0; kl < 16; ++kl) {
                    const int k = b0 + kl;
                    if (kl < rl && k >= s0) v -= AT[k * 64 + r] * x[kl];
                }
                x[rl] = v;
            }
#pragma unroll
            for (int rl = 0; rl < 16; ++rl) MT[s0 * 64 + b0 + rl] = x[rl];
            for (int r = 0; r < b0; ++r) MT[s0 * 64 + r] = 0.f;
        }
        __syncthreads();
        // ... then the blocks below the diagonal, one block-diagonal at a time
        for (int dl = 1; dl < 4; ++dl) {
            const int nblk = 4 - dl;
            for (int e = tid; e < nblk * 256; e += NT) {
                const int b = e >> 8, w = e & 255;
                const int r = 16 * (b + dl) + (w & 15), s = 16 * b + (w >> 4);
                float acc = 0.f;
                for (int k = 16 * b; k < 16 * (b + dl); ++k) acc += AT[k * 64 + r] * MT[s * 64 + k];
                Yb[e] = acc;
            }
            __syncthreads();
            for (int e = tid; e < nblk * 256; e += NT) {
                const int b = e >> 8, w = e & 255;
                const int rl = w & 15, sl = w >> 4, Rb = 16 * (b + dl);
                float acc = 0.f;
                for (int kl = 0; kl <= rl; ++kl) acc += MT[(Rb + kl) * 64 + Rb + rl] * Yb[b * 256 + sl * 16 + kl];
                MT[(16 * b + sl) * 64 + Rb + rl] = -acc;
            }
            __syncthreads();
        }
        for (int p = tid; p < C * 8; p += NT) {
            const int r = p & 63, cc = p >> 6;
            float tv[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) tv[e] = MT[(cc * 8 + e) * 64 + r] * s_beta[cc * 8 + e];
            *reinterpret_cast<uint4 *>(sm + OFF_T + r * 128 + ((cc ^ (r & 7)) << 4)) = pack8(tv);
        }
        sync_for_mma();

        // G2: W'^T = Lk^T T^T   and   G3: U0^T = V^T T^T
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t b = sdesc_sw128(sbase + OFF_T + ks * 32, 16, 1024);
                mma_bf16(tbase + TM_W, sdesc_sw128(sbase + OFF_LKQ + ks * 2048, 16384, 1024), b, ID_MK64, ks > 0);
                mma_bf16(tbase + TM_U0, sdesc_sw128(sbase + OFF_V + ks * 2048, 8192, 1024), b, ID_MK64, ks > 0);
            }
            mma_commit(bar_mma);
        }
        got = mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
        if (__syncthreads_or(!got)) {
            mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
            ok = false;
            break;
        }
        ph_mma ^= 1;
        tc_fence_after();

        // W'^T (lane i, column r) -> bf16 tile rows i (MN-major operand)
        {
            uint32_t r32[32];
            tmem_ld32(tbase + lrow + TM_W + 32 * hh, r32);
            tmem_ld_wait();
            float wv[32];
#pragma unroll
            for (int m = 0; m < 32; ++m) wv[m] = __uint_as_float(r32[m]);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const int cc = 4 * hh + qd;
                *reinterpret_cast<uint4 *>(sm + OFF_QRAW + jl * 128 + ((cc ^ (jl & 7)) << 4)) = pack8(wv + 8 * qd);
            }
        }
        sync_for_mma();

        // G4: X^T = S~^T W'^T
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, ko = (ks & 3) * 32;
                mma_bf16(tbase + TM_X, sdesc_sw128(sbase + OFF_SOP + kb * 16384 + ko, 16, 1024),
                         sdesc_sw128(sbase + OFF_QRAW + ks * 2048, 8192, 1024), ID_KM64, ks > 0);
            }
            mma_commit(bar_mma);
        }
        got = mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
        if (__syncthreads_or(!got)) {
            mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
            ok = false;
            break;
        }
        ph_mma ^= 1;
        tc_fence_after();

        // U^T = U0^T - X^T -> bf16 tile rows j (K-major operand)
        {
            uint32_t u0[32], x[32];
            tmem_ld32(tbase + lrow + TM_U0 + 32 * hh, u0);
            tmem_ld32(tbase + lrow + TM_X + 32 * hh, x);
            tmem_ld_wait();
            float uv[32];
#pragma unroll
            for (int m = 0; m < 32; ++m) uv[m] = __uint_as_float(u0[m]) - __uint_as_float(x[m]);
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
                const int cc = 4 * hh + qd;
                *reinterpret_cast<uint4 *>(sm + OFF_KRAW + jl * 128 + ((cc ^ (jl & 7)) << 4)) = pack8(uv + 8 * qd);
            }
        }
        sync_for_mma();

        // G6: O^T += U^T P^T   and   G7: S^T += U^T Kb
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = sdesc_sw128(sbase + OFF_KRAW + ks * 32, 16, 1024);
                mma_bf16(tbase + TM_O, a, sdesc_sw128(sbase + OFF_P + ks * 32, 16, 1024), ID_KK64, 1);
                mma_bf16(tbase + TM_S, a, sdesc_sw128(sbase + OFF_KB + ks * 2048, 8192, 1024), ID_KM128, 1);
            }
            mma_commit(bar_mma);
        }
        got = mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
        if (__syncthreads_or(!got)) {
            mbar_wait(bar_mma, ph_mma, WAIT_LIMIT);
            ok = false;
            break;
        }
        ph_mma ^= 1;
        tc_fence_after();

        // O^T (lane j, column r) -> out[t, h, j]
        {
            uint32_t o32[32];
            tmem_ld32(tbase + lrow + TM_O + 32 * hh, o32);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < 32; ++m) {
                const int r = 32 * hh + m;
                if (r < L) out[((size_t)(c0 + r) * H + h) * D + jl] = __float2bfloat16_rn(__uint_as_float(o32[m]));
            }
        }
    }

    sync_tc();
    if (ok && s_final) {
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            const int i0 = 64 * hh + 32 * part;
            uint32_t r[32];
            tmem_ld32(tbase + lrow + TM_S + i0, r);
            tmem_ld_wait();
#pragma unroll
            for (int m = 0; m < 32; ++m) s_final[soff + (size_t)(i0 + m) * D + jl] = __uint_as_float(r[m]);
        }
    }
    if (!ok && tid == 0) atomicOr(err, DEVERR_TIMEOUT);
    sync_tc();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

static bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t elem, uint64_t inner,
                     uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * elem};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcp

bool prefill_tc_applicable(const PrefillArgs &a) {
    return a.bf16 && a.D == 128 && a.C == 64 && a.T > 0 && a.T <= 0x7fffffffLL;
}

kda_status prefill_tc(const PrefillArgs &a, cudaStream_t s) {
    using namespace tcp;
    CUtensorMap mq, mk, mv, mg;
    const uint64_t inner = (uint64_t)a.H * D, rows = (uint64_t)a.T;
    if (!make_map(&mq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, inner, rows, 128, 64, CU_TENSOR_MAP_SWIZZLE_NONE))
        return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    prefill_tc_kernel<<<(unsigned)a.N * a.H, NT, SMEM_BYTES, s>>>(
        mq, mk, mv, mg, a.beta, a.s_init, a.s_final, static_cast<__nv_bfloat16 *>(a.out), a.cu_seqlens, a.N, a.T,
        a.H, a.eps, a.err);
    return check_launch("prefill_tc_kernel");
}

}  // namespace kda
