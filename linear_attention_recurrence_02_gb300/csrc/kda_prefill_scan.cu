// kda_prefill_scan.cu -- chunked prefill of one long sequence split into
// segments that run in parallel.
//
// The chunked form ("为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构
// 进化", section 5) hands the state from chunk to chunk, so one sequence is a
// serial chain per head. Every step of that chain is affine in the state and
// acts on the key axis only: S <- A_c S + B_c, with A_c a D x D matrix
// (decay, then the delta correction) and B_c collecting the new writes. Over a
// segment of chunks the same holds, S_t = A_t S_start + B_t after any token t
// of it, and so does the readout: o_t = S_t^T q_t = S_start^T (A_t^T q_t) +
// B_t^T q_t. So, with the segments run side by side as one packed batch:
//   1. from zero states: B of every segment (final states) and the outputs
//      B_t^T q_t (written to `out`);
//   2. from identity states with v read as zero: A of every segment (final
//      states) and the outputs A_t^T q_t (to the workspace);
//   3. the true state at every segment start, and the final state:
//      S_{p+1} = A_p S_p + B_p (a short serial scan of D x D products);
//   4. the outputs' missing term: out[t] += (A_t^T q_t)^T S_p for every token
//      t of segment p, one [tokens x D] x [D x D] product per segment and head
//      (tensor cores for bf16 at D = 128, with S_p split into two bf16 terms).
// Two prefill passes for a P-fold wider launch: it pays when a long sequence
// has few heads, so the serial chain leaves most SMs idle.
#include <string>

#include "kda_common.cuh"
#include "kda_prefill.cuh"
#include "kda_tc.cuh"

namespace kda {

// segment p covers tokens [p * seg_tokens, min(T, (p + 1) * seg_tokens))
__global__ void scan_bounds_kernel(int64_t *cu, int P, int64_t seg_tokens, int64_t T) {
    const int p = threadIdx.x + blockIdx.x * blockDim.x;
    if (p <= P) cu[p] = p == P ? T : (int64_t)p * seg_tokens;
}

// [P*H] identity D x D matrices
__global__ void identity_states_kernel(float *S, long long n, int D) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int r = (int)((i / D) % D), c = (int)(i % D);
    S[i] = r == c ? 1.f : 0.f;
}

// One CTA per (head, 32 value columns): Sp[0] = S0 (or zeros), then
// Sp[p] = A[p-1] Sp[p-1] + B[p-1] for p = 1..P (Sp[P] is the final state). The 32-column slice of the
// state stays in shared memory; A streams from L2 a 32-wide k tile at a time.
constexpr int SCAN_JS = 32, SCAN_NT = 256;
template <int D>
__global__ void __launch_bounds__(SCAN_NT) segment_scan_kernel(const float *__restrict__ A, const float *__restrict__ B,
                                                               const float *__restrict__ S0, float *__restrict__ Sp,
                                                               int P, int H) {
    constexpr int NS = D / SCAN_JS < 1 ? 1 : D / SCAN_JS;
    constexpr int JS = D < SCAN_JS ? D : SCAN_JS;
    __shared__ float sS[D][JS];
    __shared__ float sA[D][33];
    const int h = blockIdx.x / NS, j0 = (blockIdx.x % NS) * JS, tid = threadIdx.x;
    const size_t DD = (size_t)D * D;
    for (int e = tid; e < D * JS; e += SCAN_NT) {
        const int i = e / JS, j = e % JS;
        const float v = S0 ? S0[(size_t)h * DD + (size_t)i * D + j0 + j] : 0.f;
        sS[i][j] = v;
        Sp[(size_t)h * DD + (size_t)i * D + j0 + j] = v;
    }
    __syncthreads();
    constexpr int OUT = D * JS / SCAN_NT;  // outputs per thread (16 at D = 128)
    for (int p = 1; p <= P; ++p) {
        const float *Ap = A + ((size_t)(p - 1) * H + h) * DD;
        const float *Bp = B + ((size_t)(p - 1) * H + h) * DD;
        float acc[OUT > 0 ? OUT : 1];
#pragma unroll
        for (int o = 0; o < (OUT > 0 ? OUT : 1); ++o) acc[o] = 0.f;
        for (int k0 = 0; k0 < D; k0 += 32) {
            __syncthreads();
            for (int e = tid; e < D * 32; e += SCAN_NT) {
                const int i = e / 32, kk = e % 32;
                sA[i][kk] = k0 + kk < D ? Ap[(size_t)i * D + k0 + kk] : 0.f;
            }
            __syncthreads();
            const int kmax = D - k0 < 32 ? D - k0 : 32;
#pragma unroll
            for (int o = 0; o < (OUT > 0 ? OUT : 1); ++o) {
                const int e = tid + o * SCAN_NT;
                if (e >= D * JS) break;
                const int i = e / JS, j = e % JS;
                float sum = acc[o];
                for (int kk = 0; kk < kmax; ++kk) sum = fmaf(sA[i][kk], sS[k0 + kk][j], sum);
                acc[o] = sum;
            }
        }
        __syncthreads();
#pragma unroll
        for (int o = 0; o < (OUT > 0 ? OUT : 1); ++o) {
            const int e = tid + o * SCAN_NT;
            if (e >= D * JS) break;
            const int i = e / JS, j = e % JS;
            const float v = acc[o] + Bp[(size_t)i * D + j0 + j];
            sS[i][j] = v;
            Sp[((size_t)p * H + h) * DD + (size_t)i * D + j0 + j] = v;
        }
        __syncthreads();
    }
}

// D = 128: one CTA per (head, 16 value columns), 256 threads, each a 2 x 4
// register tile of the output. A_p sits in shared memory transposed (so that
// a k step is one 8-byte load of A and one 16-byte load of S for 8 FMAs)
// for the whole step, while the next A_{p+1} and B_p are loaded into
// registers: a step pays the L2 latency once, hidden behind its products.
// With `tiles` non-null, every Sp[p] also leaves as the two bf16 terms of the
// correction's operand (hi = bf16(S), lo = bf16(S - hi)), each [i][j] with j in
// two 64-column halves of 128-byte rows, 128-byte swizzled: the layout the
// correction kernel copies straight into shared memory.
constexpr int SCAN128_JS = 16, SCAN128_LDA = 130;
constexpr int SCAN128_SMEM = (128 * SCAN128_LDA + 128 * SCAN128_JS) * 4;
__global__ void __launch_bounds__(SCAN_NT) segment_scan128_kernel(const float *__restrict__ A,
                                                                   const float *__restrict__ B,
                                                                   const float *__restrict__ S0,
                                                                   float *__restrict__ Sp, uint8_t *__restrict__ tiles,
                                                                   int P, int H) {
    constexpr int D = 128, JS = SCAN128_JS, NS = D / JS, LDA = SCAN128_LDA, PER = D * D / SCAN_NT;
    extern __shared__ __align__(16) float scan_sm[];
    float (*sAT)[LDA] = reinterpret_cast<float (*)[LDA]>(scan_sm);               // [k][i]
    float (*sS)[JS] = reinterpret_cast<float (*)[JS]>(scan_sm + D * LDA);         // [i][j]
    const int h = blockIdx.x / NS, j0 = (blockIdx.x % NS) * JS, tid = threadIdx.x;
    const int i0 = (tid >> 2) * 2, c0 = (tid & 3) * 4;  // rows i0, i0+1; columns c0..c0+3 of the slice
    const size_t DD = (size_t)D * D;
    auto put_tiles = [&](int p, int i, int j, const float (&v)[4]) {  // 4 consecutive j of row i
        uint8_t *t = tiles + ((size_t)p * H + h) * (2 * D * 128 * 2);
        const uint32_t off = (uint32_t)((j >> 6) * (D * 128) + i * 128 + ((((j & 63) >> 3) ^ (i & 7)) << 4) + (j & 7) * 2);
        __nv_bfloat162 h0 = __floats2bfloat162_rn(v[0], v[1]), h1 = __floats2bfloat162_rn(v[2], v[3]);
        __nv_bfloat162 l0 = __floats2bfloat162_rn(v[0] - __bfloat162float(h0.x), v[1] - __bfloat162float(h0.y));
        __nv_bfloat162 l1 = __floats2bfloat162_rn(v[2] - __bfloat162float(h1.x), v[3] - __bfloat162float(h1.y));
        *reinterpret_cast<uint2 *>(t + off) =
            make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
        *reinterpret_cast<uint2 *>(t + D * 128 * 2 + off) =
            make_uint2(*reinterpret_cast<uint32_t *>(&l0), *reinterpret_cast<uint32_t *>(&l1));
    };
    for (int e = tid; e < D * JS; e += SCAN_NT) {
        const int i = e / JS, j = e % JS;
        const float v = S0 ? S0[(size_t)h * DD + (size_t)i * D + j0 + j] : 0.f;
        sS[i][j] = v;
        Sp[(size_t)h * DD + (size_t)i * D + j0 + j] = v;
    }
    if (tiles && S0) {  // the initial state is the correction operand of the first segment
        for (int e = tid; e < D * JS / 4; e += SCAN_NT) {
            const int i = e / (JS / 4), jj = (e % (JS / 4)) * 4;
            const float4 x = *reinterpret_cast<const float4 *>(S0 + (size_t)h * DD + (size_t)i * D + j0 + jj);
            const float v[4] = {x.x, x.y, x.z, x.w};
            put_tiles(0, i, j0 + jj, v);
        }
    }
    // A_p into registers: element (i, k) for e = tid + n * SCAN_NT, i = e / D, k = e % D (coalesced rows)
    float pre[PER];
    auto load_a = [&](const float *Ap) {
#pragma unroll
        for (int n = 0; n < PER; ++n) pre[n] = Ap[(size_t)tid + (size_t)n * SCAN_NT];
    };
    if (P >= 1) load_a(A + (size_t)h * DD);
    for (int p = 1; p <= P; ++p) {
        const float *Bp = B + ((size_t)(p - 1) * H + h) * DD;
        __syncthreads();  // every thread is done with the previous step's A
#pragma unroll
        for (int n = 0; n < PER; ++n) {
            const int e = tid + n * SCAN_NT;
            sAT[e % D][e / D] = pre[n];
        }
        __syncthreads();
        float bv[2][4];
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) bv[r][c] = Bp[(size_t)(i0 + r) * D + j0 + c0 + c];
        if (p < P) load_a(A + ((size_t)p * H + h) * DD);  // the next step's A, while this one computes
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 8
        for (int k = 0; k < D; ++k) {
            const float2 a = *reinterpret_cast<const float2 *>(&sAT[k][i0]);
            const float4 sv = *reinterpret_cast<const float4 *>(&sS[k][c0]);
            acc[0][0] = fmaf(a.x, sv.x, acc[0][0]); acc[0][1] = fmaf(a.x, sv.y, acc[0][1]);
            acc[0][2] = fmaf(a.x, sv.z, acc[0][2]); acc[0][3] = fmaf(a.x, sv.w, acc[0][3]);
            acc[1][0] = fmaf(a.y, sv.x, acc[1][0]); acc[1][1] = fmaf(a.y, sv.y, acc[1][1]);
            acc[1][2] = fmaf(a.y, sv.z, acc[1][2]); acc[1][3] = fmaf(a.y, sv.w, acc[1][3]);
        }
        __syncthreads();  // every thread is done reading the old state
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float v[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = i0 + r, j = c0 + c;
                v[c] = acc[r][c] + bv[r][c];
                sS[i][j] = v[c];
                Sp[((size_t)p * H + h) * DD + (size_t)i * D + j0 + j] = v[c];
            }
            if (tiles && p < P) put_tiles(p, i0 + r, j0 + c0, v);
        }
    }
}

// ---------------------------------------------------------------- step 4
// out[t] += OA[t] S_p for the tokens t of segment p (OA[t] = A_t^T q_t, the
// identity pass's output row; S_p the state at the segment's start).

// CUDA cores, any D and dtype: one CTA per (32-token block of a segment,
// head); S_p and the block's OA rows in shared memory, fp32 arithmetic.
constexpr int FIX_ROWS = 32, FIX_NT = 256;
template <int D, typename T>
__global__ void __launch_bounds__(FIX_NT) scan_fixup_kernel(const T *__restrict__ oa, const float *__restrict__ Sp,
                                                            T *__restrict__ out, const int64_t *__restrict__ cu,
                                                            int p0, int H, int nblk) {
    extern __shared__ float fsm[];
    float *sS = fsm;              // [D][D]
    float *sO = fsm + D * D;      // [FIX_ROWS][D]
    const int h = blockIdx.x % H, rest = blockIdx.x / H, blk = rest % nblk, p = p0 + rest / nblk;
    const int64_t s0 = cu[p], s1 = cu[p + 1], t0 = s0 + (int64_t)blk * FIX_ROWS;
    if (t0 >= s1) return;
    const int rows = (int)(s1 - t0 < FIX_ROWS ? s1 - t0 : FIX_ROWS);
    const float *S = Sp + ((size_t)p * H + h) * D * D;
    for (int e = threadIdx.x; e < D * D; e += FIX_NT) sS[e] = S[e];
    for (int e = threadIdx.x; e < FIX_ROWS * D; e += FIX_NT) {
        const int r = e / D, i = e % D;
        sO[e] = r < rows ? Elem<T>::load(oa + ((size_t)(t0 + r) * H + h) * D + i) : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < rows * D; e += FIX_NT) {
        const int r = e / D, j = e % D;
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < D; ++i) acc = fmaf(sO[r * D + i], sS[i * D + j], acc);
        T *o = out + ((size_t)(t0 + r) * H + h) * D + j;
        Elem<T>::store(o, Elem<T>::load(o) + acc);
    }
}

// Tensor cores, bf16 at D = 128: one CTA (4 warps) per (128-token block of a
// segment, head). OA's block lands by TMA as the K-major A operand; S_p
// arrives as its two bf16 terms hi = bf16(S_p) and lo = bf16(S_p - hi),
// prepared once per (segment, head) by the scan, in one bulk copy, each an
// MN-major B operand, so the product keeps about 16 bits of S_p.
// D = OA S_hi + OA S_lo accumulates in TMEM (lane = token). Each thread loads
// its token's output row before the product completes and adds the row to it.
namespace fixtc {
constexpr int NT = 128, D = 128, ROWS = 128;
constexpr uint32_t A_ = 0;           // OA block: two 64-channel halves of 128 rows x 128 B (32 KB)
constexpr uint32_t BH = 32768;       // S_p hi: two 64-column halves of 128 rows x 128 B (32 KB)
constexpr uint32_t BL = 65536;       // S_p lo (32 KB), right after hi: one copy fills both
constexpr uint32_t TILE = 65536;     // bytes of one (segment, head)'s hi + lo in global memory
constexpr uint32_t BAR = 98304;      // two mbarriers and the TMEM address
constexpr uint32_t SMEM = BAR + 64 + 1024;
constexpr uint32_t IDESC = tc::idesc_bf16(128, 128, 0, 1);
constexpr long long WAIT_LIMIT = 2000000000LL;  // clock cycles (about 1 s)
}  // namespace fixtc

__global__ void __launch_bounds__(fixtc::NT) scan_fixup_tc_kernel(const __grid_constant__ CUtensorMap tm_oa,
                                                                  const uint8_t *__restrict__ tiles,
                                                                  __nv_bfloat16 *__restrict__ out,
                                                                  const int64_t *__restrict__ cu, int p0, int H,
                                                                  int nblk, unsigned *err) {
    using namespace fixtc;
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base derived from the shared array itself (accesses compile to shared-memory instructions)
    uint8_t *sm = smem_raw + ((1024u - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar_a = reinterpret_cast<uint64_t *>(sm + BAR), *bar_m = bar_a + 1;
    uint32_t *s_taddr = reinterpret_cast<uint32_t *>(bar_a + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x % H, rest = blockIdx.x / H, blk = rest % nblk, p = p0 + rest / nblk;
    const int64_t s0 = cu[p], s1 = cu[p + 1], t0 = s0 + (int64_t)blk * ROWS;
    if (t0 >= s1) return;  // the whole CTA: the block lies past its segment
    const uint32_t sbase = smem_u32(sm);
    if (tid == 0) {
        mbar_init(bar_a, 1);
        mbar_init(bar_m, 1);
        fence_mbar_init();
        tma_prefetch_desc(&tm_oa);
        mbar_arrive_expect_tx(bar_a, 2 * ROWS * 128 + TILE);
        tma_load_2d(sm + A_, &tm_oa, bar_a, h * D, (int)t0);
        tma_load_2d(sm + A_ + ROWS * 128, &tm_oa, bar_a, h * D + 64, (int)t0);
        bulk_load(sm + BH, tiles + ((size_t)p * H + h) * TILE, TILE, bar_a);
    }
    if (warp == 0) {
        tmem_alloc(s_taddr, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *s_taddr;
    bool ok = true;
    if (tid == 0) {
        ok = mbar_wait(bar_a, 0, WAIT_LIMIT);
        if (ok) {
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t ad = sdesc_sw128(sbase + A_ + (ks >> 2) * (ROWS * 128) + (ks & 3) * 32, 16, 1024);
                mma_bf16(tbase, ad, sdesc_sw128(sbase + BH + ks * 2048, D * 128, 1024), IDESC, ks > 0);
                mma_bf16(tbase, ad, sdesc_sw128(sbase + BL + ks * 2048, D * 128, 1024), IDESC, 1);
            }
            mma_commit(bar_m);
        } else {
            mbar_wait(bar_a, 0, WAIT_LIMIT);  // let the copies land before shared memory goes away
        }
    }
    // this thread's output row, loaded while the product runs
    const int r = 32 * warp + lane;
    const int64_t t = t0 + r;
    uint4 orow[16];
    if (t < s1) {
        const uint4 *o = reinterpret_cast<const uint4 *>(out + ((size_t)t * H + h) * D);
#pragma unroll
        for (int w4 = 0; w4 < 16; ++w4) orow[w4] = o[w4];
    }
    if (tid == 0 && ok) ok = mbar_wait(bar_m, 0, WAIT_LIMIT);
    if (tid == 0 && !ok) atomicOr(err, DEVERR_TIMEOUT);
    ok = !__syncthreads_or(!ok);
    tc_fence_after();
    if (ok) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // unrolled: orow is indexed by q
            uint32_t v[32];
            tmem_ld32(tbase + ((uint32_t)(32 * warp) << 16) + 32 * q, v);
            tmem_ld_wait();
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
                uint32_t *uw = reinterpret_cast<uint32_t *>(&orow[4 * q + w4]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&uw[e]);
                    const __nv_bfloat162 n =
                        __floats2bfloat162_rn(__bfloat162float(b.x) + __uint_as_float(v[8 * w4 + 2 * e]),
                                              __bfloat162float(b.y) + __uint_as_float(v[8 * w4 + 2 * e + 1]));
                    uw[e] = *reinterpret_cast<const uint32_t *>(&n);
                }
            }
        }
        if (t < s1) {
            uint4 *o = reinterpret_cast<uint4 *>(out + ((size_t)t * H + h) * D);
#pragma unroll
            for (int w4 = 0; w4 < 16; ++w4) o[w4] = orow[w4];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, 128);
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Streaming multiprocessors of the current device (0 if unknown).
int current_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

// Requested segment count, with 0 meaning: enough segments that one pass of
// the prefill over them fills the GPU's SMs once (at least 2, at most 4096).
static int requested_segments(int segments, int H) {
    if (segments != 0) return segments;
    const int sms = current_sms();
    int p = H > 0 ? sms / H : 0;
    return p < 2 ? 2 : (p > 4096 ? 4096 : p);
}

// The automatic split of one long sequence inside kda_chunk_prefill: with
// P = floor(SMs / H) segments one pass over them fills the GPU once, and the
// split (two passes of 1/P of the chain each, the scan, the correction)
// pays when P >= 4 and every segment keeps at least 8 chunks. 0: no split.
int prefill_auto_segments(int64_t T, int H, int C) {
    if (T <= 0 || H < 1 || C < 1) return 0;
    const int sms = current_sms();
    const int P = H > 0 ? sms / H : 0;
    if (P < 4) return 0;
    const int64_t chunks = (T + C - 1) / C;
    return chunks >= 8LL * P ? (P > 4096 ? 4096 : P) : 0;
}

// segments actually used for P requested over T tokens in chunks of C
static int scan_segments(int64_t T, int C, int P, int64_t *seg_tokens) {
    const int64_t nch = (T + C - 1) / C;
    const int64_t per = (nch + P - 1) / P;  // chunks per segment
    *seg_tokens = per * C;
    return (int)((nch + per - 1) / per);
}


// Workspace layout of the split: segment bounds, then B, A and the identity
// initial states of every segment, the states at the segment starts plus the
// final state, and the identity pass's outputs.
struct ScanWs {
    int64_t *cu;
    float *Bs, *As, *Id, *Sp;
    uint8_t *tiles;  // bf16 hi/lo operand of every segment start (tensor-core correction only)
    void *oa;
};
static size_t scan_ws_layout(int64_t T, int H, int D, int P, size_t elt, uint8_t *base, ScanWs *w) {
    const size_t states = align256((size_t)P * H * D * D * sizeof(float));
    const size_t sp = align256((size_t)(P + 1) * H * D * D * sizeof(float));
    size_t off = 0;
    auto take = [&](size_t n) {
        uint8_t *q = base ? base + off : nullptr;
        off += n;
        return q;
    };
    uint8_t *cu = take(align256((size_t)(P + 1) * sizeof(int64_t)));
    uint8_t *bs = take(states), *as = take(states), *id = take(states), *spp = take(sp);
    uint8_t *tiles = take(D == 128 ? align256((size_t)P * H * fixtc::TILE) : 0);
    uint8_t *oa = take(align256((size_t)T * H * D * elt));
    if (w) {
        w->cu = reinterpret_cast<int64_t *>(cu);
        w->Bs = reinterpret_cast<float *>(bs);
        w->As = reinterpret_cast<float *>(as);
        w->Id = reinterpret_cast<float *>(id);
        w->Sp = reinterpret_cast<float *>(spp);
        w->tiles = tiles;
        w->oa = oa;
    }
    return off;
}

template <int D, typename T>
static kda_status launch_fixup_simt(const void *oa, const float *Sp, void *out, const int64_t *cu, int p0, int np,
                                    int H, int64_t seg_tokens, cudaStream_t s) {
    const int nblk = (int)((seg_tokens + FIX_ROWS - 1) / FIX_ROWS);
    const int smem = (D * D + FIX_ROWS * D) * (int)sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(scan_fixup_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    scan_fixup_kernel<D, T><<<(unsigned)((long long)np * nblk * H), FIX_NT, smem, s>>>(
        static_cast<const T *>(oa), Sp, static_cast<T *>(out), cu, p0, H, nblk);
    return check_launch("scan_fixup_kernel");
}

template <typename T>
static kda_status dispatch_fixup_simt(int D, const void *oa, const float *Sp, void *out, const int64_t *cu, int p0,
                                      int np, int H, int64_t seg_tokens, cudaStream_t s) {
    switch (D) {
    case 16: return launch_fixup_simt<16, T>(oa, Sp, out, cu, p0, np, H, seg_tokens, s);
    case 32: return launch_fixup_simt<32, T>(oa, Sp, out, cu, p0, np, H, seg_tokens, s);
    case 64: return launch_fixup_simt<64, T>(oa, Sp, out, cu, p0, np, H, seg_tokens, s);
    default: return launch_fixup_simt<128, T>(oa, Sp, out, cu, p0, np, H, seg_tokens, s);
    }
}

// the tensor-core correction: bf16 at D = 128
static bool fixup_tc(bool bf16, int D, int64_t T) { return bf16 && D == 128 && T <= 0x7fffffffLL; }

static kda_status launch_fixup(bool bf16, int D, const void *oa, const float *Sp, const uint8_t *tiles, void *out,
                               const int64_t *cu, int p0, int np, int64_t T, int H, int64_t seg_tokens, unsigned *err,
                               cudaStream_t s) {
    if (np <= 0) return KDA_OK;
    if (fixup_tc(bf16, D, T)) {
        CUtensorMap m;
        if (!tcp::make_map(&m, oa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)H * D, (uint64_t)T, 64,
                           fixtc::ROWS, CU_TENSOR_MAP_SWIZZLE_128B))
            return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
        cudaError_t e = cudaFuncSetAttribute(scan_fixup_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)fixtc::SMEM);
        if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
        const int nblk = (int)((seg_tokens + fixtc::ROWS - 1) / fixtc::ROWS);
        scan_fixup_tc_kernel<<<(unsigned)((long long)np * nblk * H), fixtc::NT, fixtc::SMEM, s>>>(
            m, tiles, static_cast<__nv_bfloat16 *>(out), cu, p0, H, nblk, err);
        return check_launch("scan_fixup_tc_kernel");
    }
    if (bf16) return dispatch_fixup_simt<__nv_bfloat16>(D, oa, Sp, out, cu, p0, np, H, seg_tokens, s);
    return dispatch_fixup_simt<float>(D, oa, Sp, out, cu, p0, np, H, seg_tokens, s);
}

}  // namespace kda

using namespace kda;

extern "C" size_t kda_chunk_prefill_scan_workspace_bytes(int64_t T, int H, int D, int C, int segments) {
    if (T <= 0 || H < 1 || D < 1 || C < 1 || segments < 0) return 0;
    segments = requested_segments(segments, H);
    int64_t seg_tokens = 0;
    const int P = scan_segments(T, C, segments, &seg_tokens);
    // sized for the wider element (fp32) so that one size serves both dtypes
    return scan_ws_layout(T, H, D, P, sizeof(float), nullptr, nullptr);
}

extern "C" kda_status kda_chunk_prefill_scan(const void *q, const void *k, const void *v, const float *g,
                                             const float *beta, const float *initial_state, float *final_state,
                                             void *out, int64_t T, int H, int D, int C, kda_dtype dtype,
                                             kda_gate gate, float l2_eps, int segments, void *workspace,
                                             size_t workspace_bytes, kda_stream_t stream) {
    clear_detail();
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE)
        return invalid("gate must be KDA_GATE_CHANNEL, KDA_GATE_HEAD or KDA_GATE_NONE");
    if (segments < 0 || segments > 4096) return invalid("segments must be in 0..4096");
    if (T < 0) return invalid("T must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    segments = requested_segments(segments, H);
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (C < 1 || C > 64) return invalid("C must be in 1..64");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (!(l2_eps >= 0.f)) return invalid("l2_eps must be >= 0");
    if (T == 0 || segments == 1 || T <= C)  // nothing to split: the ordinary prefill
        return kda_chunk_prefill_gated(q, k, v, g, beta, initial_state, final_state, out, nullptr, 1, T, H, D, C,
                                       dtype, gate, l2_eps, nullptr, 0, stream);
    const size_t need = kda_chunk_prefill_scan_workspace_bytes(T, H, D, C, segments);
    if (workspace_bytes < need) return invalid("workspace too small");
    kda_status st;
    if ((st = check_ptr(q, "q")) || (st = check_ptr(k, "k")) || (st = check_ptr(v, "v")) ||
        (gate != KDA_GATE_NONE && (st = check_ptr(g, "g"))) || (st = check_ptr(beta, "beta")) ||
        (st = check_ptr(out, "out")) || (st = check_ptr(workspace, "workspace")))
        return st;
    if (initial_state && (st = check_ptr(initial_state, "initial_state"))) return st;
    if (final_state && (st = check_ptr(final_state, "final_state"))) return st;
    if (out == q || out == k || out == v) return invalid("out must not alias q, k or v");
    if ((long long)segments * H * 2 > 0x7fffffffLL) return invalid("segments*H too large for one launch");
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned *err = device_error_word();
    if (err == nullptr) return fail(KDA_ERR_CUDA, "device error word unavailable");

    int64_t seg_tokens = 0;
    const int P = scan_segments(T, C, segments, &seg_tokens);
    const bool bf16 = dtype == KDA_BF16;
    ScanWs w;
    scan_ws_layout(T, H, D, P, bf16 ? 2 : 4, static_cast<uint8_t *>(workspace), &w);

    scan_bounds_kernel<<<(P + 1 + 255) / 256, 256, 0, s>>>(w.cu, P, seg_tokens, T);
    if ((st = check_launch("scan_bounds_kernel"))) return st;
    const long long nid = (long long)P * H * D * D;
    identity_states_kernel<<<(unsigned)((nid + 255) / 256), 256, 0, s>>>(w.Id, nid, D);
    if ((st = check_launch("identity_states_kernel"))) return st;

    // the segments are equally long except the last, so natural order is longest-first enough
    PrefillArgs a{q, k, v, g, beta, nullptr, w.Bs, out, w.cu, P, T, H, D, C, bf16, l2_eps, nullptr, 0,
                  err, nullptr, (int)gate};
    auto run = [&](const PrefillArgs &x) { return prefill_run(x, s); };
    if ((st = run(a))) return st;  // 1. B of each segment; outputs from zero states into out
    PrefillArgs ai = a;
    ai.s_init = w.Id;
    ai.s_final = w.As;
    ai.out = w.oa;
    ai.v_zero = true;
    if ((st = run(ai))) return st;  // 2. A of each segment; outputs A_t^T q_t
    // 3. the state at every segment start and the final state
    const int ns = D / SCAN_JS < 1 ? 1 : D / SCAN_JS;
    switch (D) {
    case 16: segment_scan_kernel<16><<<H * ns, SCAN_NT, 0, s>>>(w.As, w.Bs, initial_state, w.Sp, P, H); break;
    case 32: segment_scan_kernel<32><<<H * ns, SCAN_NT, 0, s>>>(w.As, w.Bs, initial_state, w.Sp, P, H); break;
    case 64: segment_scan_kernel<64><<<H * ns, SCAN_NT, 0, s>>>(w.As, w.Bs, initial_state, w.Sp, P, H); break;
    default:
    {
        cudaError_t e = cudaFuncSetAttribute(segment_scan128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             SCAN128_SMEM);
        if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
        segment_scan128_kernel<<<H * (128 / SCAN128_JS), SCAN_NT, SCAN128_SMEM, s>>>(
            w.As, w.Bs, initial_state, w.Sp, fixup_tc(bf16, D, T) ? w.tiles : nullptr, P, H);
    }
        break;
    }
    if ((st = check_launch("segment_scan_kernel"))) return st;
    // 4. the carried state's part of every output (segment 0 has one only with an initial state)
    const int p0 = initial_state ? 0 : 1;
    if ((st = launch_fixup(bf16, D, w.oa, w.Sp, w.tiles, out, w.cu, p0, P - p0, T, H, seg_tokens, err, s)))
        return st;
    if (final_state) {
        const size_t one = (size_t)H * D * D * sizeof(float);
        cudaError_t e = cudaMemcpyAsync(final_state, reinterpret_cast<uint8_t *>(w.Sp) + (size_t)P * one, one,
                                        cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("final state copy: ") + cudaGetErrorString(e));
    }
    return KDA_OK;
}
