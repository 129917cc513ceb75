// kda_fused_decode.cu -- short conv + decode step in one launch.
//
// Same arithmetic as kda_shortconv_step followed by kda_decode_step
// ("KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析",
// section "KDA 递推公式先衰减再差分": a width-4 causal conv with SiLU runs in
// front of q/k/v, then decay, delta correction and readout), except that the
// post-conv q, k, v stay in fp32 on chip instead of being stored and read back.
//
// One CTA per (sequence, head) owns the head's whole D x D state and every
// ring channel of that head, so the in-place ring shift cannot race with
// another CTA's read. For D < 128 the state lives in registers; for D = 128
// one bulk copy stages it in shared memory (fused_decode_bulk_kernel, three
// heads per SM). Either way the state's loads are issued first and stay in
// flight while the conv, the norms and the decay run; column sums of S'^T k^
// and S'^T q^ are reduced through shared memory across the row groups; S is
// written once. The gate form (per channel, per head, none) is a template
// parameter as in kda_decode.cu.
//
// With an output epilogue (template parameter EP = the gate activation), the
// head's output vector o never leaves the CTA: it is normalised by its RMS,
// scaled per channel by the norm weight and multiplied by act(gate) before
// the one store ("WARP中Kimi Delta Attention线性注意力原理剖析", section
// "相关源码与文档导航": a gated RMSNorm follows the recurrence; "为什么 Kimi K3
// 敢把 KV Cache 扔掉？", section 6: an output gate scales the features). The
// reading is that of kda_gated_rmsnorm, per (sequence, head) row of D value
// channels: y = o / sqrt(mean(o^2) + eps) * weight * act(gate), a row whose
// mean square plus eps is zero giving zeros. o is taken in fp32, before any
// rounding to the storage type.
#include <string>

#include "kda_common.cuh"
#include "kda_tc.cuh"

namespace kda {

template <int D> struct FusedShape;
template <> struct FusedShape<16> { static constexpr int NT = 32; };
template <> struct FusedShape<32> { static constexpr int NT = 64; };
template <> struct FusedShape<64> { static constexpr int NT = 128; };

// Output epilogue selector: no epilogue (o is stored), or the gate
// activation of the gated RMSNorm (KDA_ACT_SIGMOID, KDA_ACT_SILU).
constexpr int EP_NONE = -1;

// act(z) of the output gate, fp32 (one element per thread: exact forms)
template <int EP> __device__ __forceinline__ float gate_act(float z) {
    const float sg = 1.0f / (1.0f + expf(-z));
    return EP == KDA_ACT_SILU ? z * sg : sg;
}

template <int D, typename T, int GM, int EP>
__global__ void __launch_bounds__(FusedShape<D>::NT)
    fused_decode_kernel(const T *__restrict__ x, T *__restrict__ ring, const float *__restrict__ w,
                        const float *__restrict__ g, const float *__restrict__ beta, float *__restrict__ state,
                        T *__restrict__ out, int H, float eps, const T *__restrict__ gate_in,
                        const float *__restrict__ nweight, float neps) {
    constexpr int NT = FusedShape<D>::NT;
    constexpr int C4 = D / 4;     // float4 columns per state row
    constexpr int RG = NT / C4;   // row groups
    constexpr int RPT = D / RG;   // rows per thread
    constexpr int NW = NT / 32;   // warps
    static_assert(NT % 32 == 0 && RPT * RG == D && C4 <= 32, "bad fused decode shape");

    const int unit = blockIdx.x;  // b*H + h
    const int b = unit / H, h = unit % H;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int c4 = t % C4, rg = t / C4;

    float *Sp = state + (size_t)unit * D * D + c4 * 4;
    float4 s[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) s[m] = __ldcs(reinterpret_cast<const float4 *>(Sp + (size_t)(rg + m * RG) * D));

    __shared__ float s_y[3][D];
    __shared__ float s_qa[D], s_ka[D], s_kh[D], s_a[D], s_delta[D];
    __shared__ float s_red[NW][3];
    __shared__ float s_part[NW][D][2];

    // 1. width-4 causal conv + SiLU for q, k, v; shift the ring
    for (int idx = t; idx < 3 * D; idx += NT) {
        const int p = idx / D, c = idx % D;
        const size_t row = ((size_t)b * 3 + p) * H + h;
        const size_t xo = row * D + c, ro = row * 3 * D + c;
        const float xv = Elem<T>::load(x + xo);
        const float r0 = Elem<T>::load(ring + ro), r1 = Elem<T>::load(ring + ro + D),
                    r2 = Elem<T>::load(ring + ro + 2 * D);
        const float4 tap = __ldg(reinterpret_cast<const float4 *>(w) + (((size_t)p * H + h) * D + c));
        const float z = tap.x * r0 + tap.y * r1 + tap.z * r2 + tap.w * xv;
        s_y[p][c] = z / (1.0f + expf(-z));
        Elem<T>::store(ring + ro, r1);
        Elem<T>::store(ring + ro + D, r2);
        Elem<T>::store(ring + ro + 2 * D, xv);
    }
    const size_t vo = (size_t)unit * D;
    float av = 0.f, gz = 0.f, nw = 0.f;
    if (t < D) {
        if constexpr (GM == KDA_GATE_CHANNEL) av = expf(__ldg(g + vo + t));
        else if constexpr (GM == KDA_GATE_HEAD) av = expf(__ldg(g + unit));
        else av = 1.f;
        if constexpr (EP != EP_NONE) {
            gz = Elem<T>::load(gate_in + vo + t);
            nw = __ldg(nweight + t);
        }
    }
    __syncthreads();

    // 2. L2 norms of q, k and their dot
    float qv = 0.f, kv = 0.f;
    if (t < D) {
        qv = s_y[0][t];
        kv = s_y[1][t];
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
    for (int wi = 0; wi < NW; ++wi) {
        sqq += s_red[wi][0];
        skk += s_red[wi][1];
        sqk += s_red[wi][2];
    }
    const float rq = inv_norm(sqq, eps), rk = inv_norm(skk, eps);
    const float kq = sqk * rq * rk;
    if (t < D) {
        s_qa[t] = qv * rq * av;
        s_ka[t] = kv * rk * av;
        s_kh[t] = kv * rk;
        s_a[t] = av;
    }
    __syncthreads();  // also: every thread has read s_red, which the epilogue reuses

    // 3. partial column sums over this thread's rows, then across row groups
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int i = rg + m * RG;
        const float ka = s_ka[i], qa = s_qa[i];
        pk[0] += ka * s[m].x; pk[1] += ka * s[m].y; pk[2] += ka * s[m].z; pk[3] += ka * s[m].w;
        pq[0] += qa * s[m].x; pq[1] += qa * s[m].y; pq[2] += qa * s[m].z; pq[3] += qa * s[m].w;
    }
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
    float ov = 0.f;
    if (t < D) {
        float ks = 0.f, qs = 0.f;
#pragma unroll
        for (int wi = 0; wi < NW; ++wi) {
            ks += s_part[wi][t][0];
            qs += s_part[wi][t][1];
        }
        const float d = __ldg(beta + unit) * (s_y[2][t] - ks);
        s_delta[t] = d;
        ov = qs + kq * d;
        if constexpr (EP == EP_NONE) Elem<T>::store(out + vo + t, ov);
    }
    if constexpr (EP != EP_NONE) {  // the sum of o^2 over the head's D channels, per warp
        float ss = ov * ov;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[warp][0] = ss;
    }
    __syncthreads();
    if constexpr (EP != EP_NONE) {  // y = o / rms(o) * weight * act(gate): the only store of the output
        if (t < D) {
            float ss = 0.f;
#pragma unroll
            for (int wi = 0; wi < NW; ++wi) ss += s_red[wi][0];
            const float den = ss / (float)D + neps;
            const float inv = den > 0.f ? 1.0f / sqrtf(den) : 0.f;
            Elem<T>::store(out + vo + t, ov * inv * nw * gate_act<EP>(gz));
        }
    }

    // 4. S <- Diag(a) S + k^ delta^T, written back once
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

// D = 128: the head's 64 KiB state slice is staged in shared memory by one
// bulk copy that runs while the conv and the norms do, instead of living in
// registers. With 80 registers and 73 KiB of shared memory, three heads are
// resident per SM instead of two. That shortens the tail of a launch of a few
// waves (a 69-layer stack at 8 sequences: 1.70 -> 1.57 ms per step) and keeps
// HBM busier in a launch of many (64 sequences x 96 heads: 131.9 against
// 133.1 us per step for the register kernel). Each thread owns four value
// columns over every eighth row: it reduces S'^T k^ and S'^T q^ from shared
// memory and writes its part of the updated state back with 16-byte stores.
constexpr int BULK_NT = 256;
constexpr uint32_t BULK_SMEM = 128 * 128 * 4 + 16;
constexpr long long WAIT_LIMIT_DECODE = 2000000000LL;  // clock cycles (about 1 s)

template <typename T, int GM, int EP>
__global__ void __launch_bounds__(BULK_NT, 3)
    fused_decode_bulk_kernel(const T *__restrict__ x, T *__restrict__ ring, const float *__restrict__ w,
                             const float *__restrict__ g, const float *__restrict__ beta, float *__restrict__ state,
                             T *__restrict__ out, int H, float eps, unsigned *err, const T *__restrict__ gate_in,
                             const float *__restrict__ nweight, float neps, int mode) {
    using namespace tc;
    constexpr int D = 128, NW = BULK_NT / 32;
    extern __shared__ uint8_t smem_raw[];
    // 16-byte aligned base derived from the shared array itself (accesses compile to shared-memory instructions)
    float *Ss = reinterpret_cast<float *>(
        smem_raw + ((16u - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 15u)) & 15u));
    __shared__ float s_y[3][D];
    __shared__ float s_qa[D], s_ka[D], s_kh[D], s_a[D], s_delta[D];
    __shared__ float s_red[NW][3];
    __shared__ float s_part[NW][D];  // one column sum at a time
    __shared__ uint64_t bar;

    const int unit = blockIdx.x;  // b*H + h
    const int b = unit / H, h = unit % H;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    float *Sg = state + (size_t)unit * D * D;
    // Every launch is a programmatic dependent launch: it may start while the
    // kernel before it on the stream drains, and griddepcontrol.wait below
    // holds the CTA until that kernel has completed. mode 1
    // (KDA_DECODE_OVERLAP_PREV: that kernel does not write this state) issues
    // the state copy before the wait; mode 2 (no promise) issues only L2
    // prefetches before it and the copy after it.
    if (t == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        if (mode != 2) {
            mbar_arrive_expect_tx(&bar, D * D * 4);
            bulk_load(Ss, Sg, D * D * 4, &bar);
        }
    }
    // In mode 1 the state copy above overlaps the previous kernel's tail. In
    // both modes the wait below holds every read of x, ring, g and beta (that
    // kernel's possible outputs), and in mode 2 also the state copy, until it
    // has completed. Dependents are released only after the wait, so a kernel
    // two launches back has always completed before the next one starts.
    // Before the wait, the head's state (mode 2) and its x, ring, tap, g, beta
    // (and output gate) rows are prefetched into L2 only. L2 is where the
    // previous kernel's writes land, and every load of these rows comes after
    // the wait, so a prefetch can bring them closer but never serve a stale
    // value.
    if (mode == 2 && t >= 12 && t < 16) prefetch_l2_bulk(Sg + (t - 12) * (D * D / 4), D * D);  // the state, 4 x 16 KB
    if (t < 12) {
        const size_t row = ((size_t)b * 3 + (t % 3)) * H + h;  // (b*3 + p)*H + h
        if (t < 3) prefetch_l2_bulk(x + row * D, D * sizeof(T));
        else if (t < 6) prefetch_l2_bulk(ring + row * 3 * D, 3 * D * sizeof(T));
        else if (t >= 9) prefetch_l2_bulk(w + ((size_t)(t - 9) * H + h) * D * 4, D * 16);  // taps of projection t - 9
        else if (t == 6) {
            if constexpr (GM == KDA_GATE_CHANNEL) prefetch_l2_bulk(g + (size_t)unit * D, D * 4);
            else if constexpr (GM == KDA_GATE_HEAD) asm volatile("prefetch.global.L2 [%0];" ::"l"(g + unit));
        } else if (t == 7) asm volatile("prefetch.global.L2 [%0];" ::"l"(beta + unit));
        else if constexpr (EP != EP_NONE) prefetch_l2_bulk(gate_in + (size_t)unit * D, D * sizeof(T));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (mode == 2 && t == 0) {
        mbar_arrive_expect_tx(&bar, D * D * 4);
        bulk_load(Ss, Sg, D * D * 4, &bar);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // 1. width-4 causal conv + SiLU for q, k, v; shift the ring
    for (int idx = t; idx < 3 * D; idx += BULK_NT) {
        const int p = idx / D, c = idx % D;
        const size_t row = ((size_t)b * 3 + p) * H + h;
        const size_t xo = row * D + c, ro = row * 3 * D + c;
        const float xv = Elem<T>::load(x + xo);
        const float r0 = Elem<T>::load(ring + ro), r1 = Elem<T>::load(ring + ro + D),
                    r2 = Elem<T>::load(ring + ro + 2 * D);
        const float4 tap = __ldg(reinterpret_cast<const float4 *>(w) + (((size_t)p * H + h) * D + c));
        const float z = tap.x * r0 + tap.y * r1 + tap.z * r2 + tap.w * xv;
        s_y[p][c] = z / (1.0f + expf(-z));
        Elem<T>::store(ring + ro, r1);
        Elem<T>::store(ring + ro + D, r2);
        Elem<T>::store(ring + ro + 2 * D, xv);
    }
    const size_t vo = (size_t)unit * D;
    float av = 0.f, gz = 0.f, nw = 0.f;
    if (t < D) {
        if constexpr (GM == KDA_GATE_CHANNEL) av = expf(__ldg(g + vo + t));
        else if constexpr (GM == KDA_GATE_HEAD) av = expf(__ldg(g + unit));
        else av = 1.f;
        if constexpr (EP != EP_NONE) {
            gz = Elem<T>::load(gate_in + vo + t);
            nw = __ldg(nweight + t);
        }
    }
    __syncthreads();

    // 2. L2 norms of q, k and their dot
    float qv = 0.f, kv = 0.f;
    if (t < D) {
        qv = s_y[0][t];
        kv = s_y[1][t];
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
    for (int wi = 0; wi < NW; ++wi) {
        sqq += s_red[wi][0];
        skk += s_red[wi][1];
        sqk += s_red[wi][2];
    }
    const float rq = inv_norm(sqq, eps), rk = inv_norm(skk, eps);
    const float kq = sqk * rq * rk;
    if (t < D) {
        s_qa[t] = qv * rq * av;
        s_ka[t] = kv * rk * av;
        s_kh[t] = kv * rk;
        s_a[t] = av;
    }
    // 3. the state slice has landed (bounded wait); the barrier also orders
    // every read of s_red above before the epilogue reuses it
    const bool got = mbar_wait(&bar, 0, WAIT_LIMIT_DECODE);
    if (__syncthreads_or(!got)) {
        if (t == 0) {
            atomicOr(err, DEVERR_TIMEOUT);
            mbar_wait(&bar, 0, WAIT_LIMIT_DECODE);  // let the copy land before shared memory goes away
        }
        return;
    }

    // 4. column sums of S'^T k^ and S'^T q^: thread (4 columns c4, rows rg + 8m)
    const int c4 = t & 31, rg = warp;
    const float4 *Ss4 = reinterpret_cast<const float4 *>(Ss);
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = rg + 8 * m;
        const float4 sv = Ss4[i * 32 + c4];
        const float ka = s_ka[i], qa = s_qa[i];
        pk[0] += ka * sv.x; pk[1] += ka * sv.y; pk[2] += ka * sv.z; pk[3] += ka * sv.w;
        pq[0] += qa * sv.x; pq[1] += qa * sv.y; pq[2] += qa * sv.z; pq[3] += qa * sv.w;
    }
    *reinterpret_cast<float4 *>(&s_part[rg][4 * c4]) = make_float4(pk[0], pk[1], pk[2], pk[3]);
    __syncthreads();
    float ks = 0.f;
    if (t < D) {
#pragma unroll
        for (int wi = 0; wi < NW; ++wi) ks += s_part[wi][t];
    }
    __syncthreads();
    *reinterpret_cast<float4 *>(&s_part[rg][4 * c4]) = make_float4(pq[0], pq[1], pq[2], pq[3]);
    __syncthreads();
    float ov = 0.f;
    if (t < D) {
        float qs = 0.f;
#pragma unroll
        for (int wi = 0; wi < NW; ++wi) qs += s_part[wi][t];
        const float d = __ldg(beta + unit) * (s_y[2][t] - ks);
        s_delta[t] = d;
        ov = qs + kq * d;
        if constexpr (EP == EP_NONE) Elem<T>::store(out + vo + t, ov);
    }
    if constexpr (EP != EP_NONE) {  // the sum of o^2 over the head's D channels, per warp
        float ss = ov * ov;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) s_red[warp][0] = ss;
    }
    __syncthreads();
    if constexpr (EP != EP_NONE) {  // y = o / rms(o) * weight * act(gate): the only store of the output
        if (t < D) {
            float ss = 0.f;
#pragma unroll
            for (int wi = 0; wi < NW; ++wi) ss += s_red[wi][0];
            const float den = ss / (float)D + neps;
            const float inv = den > 0.f ? 1.0f / sqrtf(den) : 0.f;
            Elem<T>::store(out + vo + t, ov * inv * nw * gate_act<EP>(gz));
        }
    }

    // 5. S <- Diag(a) S + k^ delta^T, written back once with 16-byte row stores
    const float4 d4 = *reinterpret_cast<const float4 *>(&s_delta[4 * c4]);
    float4 *Sg4 = reinterpret_cast<float4 *>(Sg);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int i = rg + 8 * m;
        const float4 sv = Ss4[i * 32 + c4];
        const float a = s_a[i], kh = s_kh[i];
        __stcs(Sg4 + i * 32 + c4, make_float4(a * sv.x + kh * d4.x, a * sv.y + kh * d4.y, a * sv.z + kh * d4.z,
                                              a * sv.w + kh * d4.w));
    }
}



// Epilogue operands of one launch: the output gate [B, H, D] (storage dtype),
// the norm weight [D] and the norm eps; unused when EP == EP_NONE.
struct EpiArgs {
    const void *gate = nullptr;
    const float *weight = nullptr;
    float eps = 0.f;
};

template <int D, typename T, int GM, int EP>
static void launch_fused(const void *x, void *ring, const float *w, const float *g, const float *beta,
                         float *state, void *out, int B, int H, float eps, bool overlap, const EpiArgs &ea,
                         cudaStream_t s) {
    const T *gi = static_cast<const T *>(ea.gate);
    // d = 128: the staged kernel at every batch size (B=64, H=96: 131.9 us against 133.1 us for the
    // register kernel, once its shared-memory accesses compiled to shared-memory instructions;
    // 124.5 us once every launch became a dependent launch that prefetches its state into L2)
    if constexpr (D == 128) {
        if (smem_attr_once<fused_decode_bulk_kernel<T, GM, EP>>((int)BULK_SMEM) != cudaSuccess)
            return;  // reported by check_launch
        // a programmatic dependent launch: it may start while the previous kernel drains
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)B * H);
        cfg.blockDim = dim3(BULK_NT);
        cfg.dynamicSmemBytes = BULK_SMEM;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, fused_decode_bulk_kernel<T, GM, EP>, static_cast<const T *>(x),
                           static_cast<T *>(ring), w, g, beta, state, static_cast<T *>(out), H, eps,
                           device_error_word(), gi, ea.weight, ea.eps,
                           overlap ? 1 : 2);  // an error is left for check_launch
    } else {
        fused_decode_kernel<D, T, GM, EP><<<(unsigned)B * H, FusedShape<D>::NT, 0, s>>>(
            static_cast<const T *>(x), static_cast<T *>(ring), w, g, beta, state, static_cast<T *>(out), H, eps,
            gi, ea.weight, ea.eps);
    }
}

template <typename T, int GM, int EP>
static void dispatch_fused(int D, const void *x, void *ring, const float *w, const float *g, const float *beta,
                           float *state, void *out, int B, int H, float eps, bool ov, const EpiArgs &ea,
                           cudaStream_t s) {
    switch (D) {
    case 16: launch_fused<16, T, GM, EP>(x, ring, w, g, beta, state, out, B, H, eps, ov, ea, s); break;
    case 32: launch_fused<32, T, GM, EP>(x, ring, w, g, beta, state, out, B, H, eps, ov, ea, s); break;
    case 64: launch_fused<64, T, GM, EP>(x, ring, w, g, beta, state, out, B, H, eps, ov, ea, s); break;
    default: launch_fused<128, T, GM, EP>(x, ring, w, g, beta, state, out, B, H, eps, ov, ea, s); break;
    }
}

template <typename T, int EP>
static void dispatch_fused_gate(kda_gate gate, int D, const void *x, void *ring, const float *w, const float *g,
                                const float *beta, float *state, void *out, int B, int H, float eps, bool ov,
                                const EpiArgs &ea, cudaStream_t s) {
    if (gate == KDA_GATE_HEAD)
        dispatch_fused<T, KDA_GATE_HEAD, EP>(D, x, ring, w, g, beta, state, out, B, H, eps, ov, ea, s);
    else if (gate == KDA_GATE_NONE)
        dispatch_fused<T, KDA_GATE_NONE, EP>(D, x, ring, w, g, beta, state, out, B, H, eps, ov, ea, s);
    else dispatch_fused<T, KDA_GATE_CHANNEL, EP>(D, x, ring, w, g, beta, state, out, B, H, eps, ov, ea, s);
}

// Arguments shared by the fused entry points; KDA_OK when a launch may follow.
static kda_status check_fused_args(const void *x, void *ring, const float *w, const float *g, const float *beta,
                                   float *state, void *out, int B, int H, int D, kda_dtype dtype, kda_gate gate,
                                   float l2_eps, unsigned flags) {
    if (flags & ~(unsigned)KDA_DECODE_OVERLAP_PREV) return invalid("flags: unknown bits");
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE)
        return invalid("gate must be KDA_GATE_CHANNEL, KDA_GATE_HEAD or KDA_GATE_NONE");
    if (B < 0) return invalid("B must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (!(l2_eps >= 0.f)) return invalid("l2_eps must be >= 0");
    if (B == 0) return KDA_OK;
    if ((long long)B * H > 0x7fffffffLL) return invalid("B*H too large for one launch");
    kda_status st;
    if ((st = check_ptr(x, "x")) || (st = check_ptr(ring, "ring")) || (st = check_ptr(w, "w")) ||
        (gate != KDA_GATE_NONE && (st = check_ptr(g, "g"))) || (st = check_ptr(beta, "beta")) ||
        (st = check_ptr(state, "state")) || (st = check_ptr(out, "out")))
        return st;
    if (out == x || out == ring || (const void *)out == (const void *)state)
        return invalid("out must not alias x, ring or state");
    return KDA_OK;
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_shortconv_decode_step_ex(const void *x, void *ring, const float *w, const float *g,
                                                   const float *beta, float *state, void *out, int B, int H, int D,
                                                   kda_dtype dtype, kda_gate gate, float l2_eps, unsigned flags,
                                                   kda_stream_t stream) {
    clear_detail();
    kda_status st = check_fused_args(x, ring, w, g, beta, state, out, B, H, D, dtype, gate, l2_eps, flags);
    if (st != KDA_OK || B == 0) return st;
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool ov = (flags & KDA_DECODE_OVERLAP_PREV) != 0;
    const EpiArgs none;
    if (dtype == KDA_BF16)
        dispatch_fused_gate<__nv_bfloat16, EP_NONE>(gate, D, x, ring, w, g, beta, state, out, B, H, l2_eps, ov, none,
                                                    s);
    else
        dispatch_fused_gate<float, EP_NONE>(gate, D, x, ring, w, g, beta, state, out, B, H, l2_eps, ov, none, s);
    return check_launch("fused_decode_kernel");
}

extern "C" kda_status kda_shortconv_decode_step_epi(const void *x, void *ring, const float *w, const float *g,
                                                    const float *beta, float *state, const void *out_gate,
                                                    const float *norm_weight, void *y, int B, int H, int D,
                                                    kda_dtype dtype, kda_gate gate, kda_gate_act act,
                                                    float l2_eps, float norm_eps, unsigned flags,
                                                    kda_stream_t stream) {
    clear_detail();
    kda_status st = check_fused_args(x, ring, w, g, beta, state, y, B, H, D, dtype, gate, l2_eps, flags);
    if (st != KDA_OK) return st;
    if (act != KDA_ACT_SIGMOID && act != KDA_ACT_SILU) return invalid("act must be KDA_ACT_SIGMOID or KDA_ACT_SILU");
    if (!(norm_eps >= 0.f)) return invalid("norm_eps must be >= 0");
    if (B == 0) return KDA_OK;
    if ((st = check_ptr(out_gate, "out_gate")) || (st = check_ptr(norm_weight, "norm_weight"))) return st;
    if (y == out_gate) return invalid("y must not alias out_gate");
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool ov = (flags & KDA_DECODE_OVERLAP_PREV) != 0;
    EpiArgs ea;
    ea.gate = out_gate;
    ea.weight = norm_weight;
    ea.eps = norm_eps;
    if (dtype == KDA_BF16) {
        if (act == KDA_ACT_SILU)
            dispatch_fused_gate<__nv_bfloat16, KDA_ACT_SILU>(gate, D, x, ring, w, g, beta, state, y, B, H, l2_eps, ov,
                                                             ea, s);
        else
            dispatch_fused_gate<__nv_bfloat16, KDA_ACT_SIGMOID>(gate, D, x, ring, w, g, beta, state, y, B, H, l2_eps,
                                                                ov, ea, s);
    } else {
        if (act == KDA_ACT_SILU)
            dispatch_fused_gate<float, KDA_ACT_SILU>(gate, D, x, ring, w, g, beta, state, y, B, H, l2_eps, ov, ea, s);
        else
            dispatch_fused_gate<float, KDA_ACT_SIGMOID>(gate, D, x, ring, w, g, beta, state, y, B, H, l2_eps, ov, ea,
                                                        s);
    }
    return check_launch("fused_decode_kernel (output epilogue)");
}

extern "C" kda_status kda_shortconv_decode_step_gated(const void *x, void *ring, const float *w, const float *g,
                                                      const float *beta, float *state, void *out, int B, int H,
                                                      int D, kda_dtype dtype, kda_gate gate, float l2_eps,
                                                      kda_stream_t stream) {
    return kda_shortconv_decode_step_ex(x, ring, w, g, beta, state, out, B, H, D, dtype, gate, l2_eps, 0u, stream);
}

extern "C" kda_status kda_shortconv_decode_step(const void *x, void *ring, const float *w, const float *g,
                                                const float *beta, float *state, void *out, int B, int H, int D,
                                                kda_dtype dtype, float l2_eps, kda_stream_t stream) {
    return kda_shortconv_decode_step_gated(x, ring, w, g, beta, state, out, B, H, D, dtype, KDA_GATE_CHANNEL,
                                           l2_eps, stream);
}
