// kda_prefill_scan.cu -- chunked prefill of one long sequence split into
// segments that run in parallel.
//
// The chunked form ("为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构
// 进化", section 5) hands the state from chunk to chunk, so one sequence is a
// serial chain per head. Every step of that chain is affine in the state and
// acts on the key axis only: S <- A_c S + B_c, with A_c a D x D matrix
// (decay, then the delta correction) and B_c collecting the new writes. Over a
// segment of chunks the same holds, S_end = A S_start + B. So:
//   1. B of every segment: the ordinary prefill of the segments as a packed
//      batch, from zero states (its final states).
//   2. A of every segment: the same with identity initial states and v read
//      as zero (S_end = A I + 0).
//   3. the true initial state of each segment, from the first one:
//      S_{p+1} = A_p S_p + B_p (a short serial scan of D x D products);
//   4. the outputs and final state: the prefill once more from those states.
// Three prefill passes for a P-fold wider launch: it pays when a long
// sequence has few heads, so the serial chain leaves most SMs idle.
#include "kda_common.cuh"
#include "kda_prefill.cuh"

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
// Sp[p] = A[p-1] Sp[p-1] + B[p-1] for p = 1..P-1. The 32-column slice of the
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
    for (int p = 1; p < P; ++p) {
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
// register tile of the output; A passes through shared memory transposed, 32
// k at a time, so that a k step is one 8-byte load of A and one 16-byte load
// of S for 8 FMAs.
constexpr int SCAN128_JS = 16;
__global__ void __launch_bounds__(SCAN_NT) segment_scan128_kernel(const float *__restrict__ A,
                                                                   const float *__restrict__ B,
                                                                   const float *__restrict__ S0,
                                                                   float *__restrict__ Sp, int P, int H) {
    constexpr int D = 128, JS = SCAN128_JS, NS = D / JS, KT = 32, LDA = D + 2;
    __shared__ __align__(16) float sS[D][JS];
    __shared__ __align__(16) float sAT[KT][LDA];
    const int h = blockIdx.x / NS, j0 = (blockIdx.x % NS) * JS, tid = threadIdx.x;
    const int i0 = (tid >> 2) * 2, c0 = (tid & 3) * 4;  // rows i0, i0+1; columns c0..c0+3 of the slice
    const size_t DD = (size_t)D * D;
    for (int e = tid; e < D * JS; e += SCAN_NT) {
        const int i = e / JS, j = e % JS;
        const float v = S0 ? S0[(size_t)h * DD + (size_t)i * D + j0 + j] : 0.f;
        sS[i][j] = v;
        Sp[(size_t)h * DD + (size_t)i * D + j0 + j] = v;
    }
    for (int p = 1; p < P; ++p) {
        const float *Ap = A + ((size_t)(p - 1) * H + h) * DD;
        const float *Bp = B + ((size_t)(p - 1) * H + h) * DD;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int k0 = 0; k0 < D; k0 += KT) {
            __syncthreads();
            for (int e = tid; e < D * KT; e += SCAN_NT) {  // row i, k0 + kk: 32 consecutive floats per row
                const int i = e / KT, kk = e % KT;
                sAT[kk][i] = Ap[(size_t)i * D + k0 + kk];
            }
            __syncthreads();
#pragma unroll 8
            for (int kk = 0; kk < KT; ++kk) {
                const float2 a = *reinterpret_cast<const float2 *>(&sAT[kk][i0]);
                const float4 sv = *reinterpret_cast<const float4 *>(&sS[k0 + kk][c0]);
                acc[0][0] = fmaf(a.x, sv.x, acc[0][0]); acc[0][1] = fmaf(a.x, sv.y, acc[0][1]);
                acc[0][2] = fmaf(a.x, sv.z, acc[0][2]); acc[0][3] = fmaf(a.x, sv.w, acc[0][3]);
                acc[1][0] = fmaf(a.y, sv.x, acc[1][0]); acc[1][1] = fmaf(a.y, sv.y, acc[1][1]);
                acc[1][2] = fmaf(a.y, sv.z, acc[1][2]); acc[1][3] = fmaf(a.y, sv.w, acc[1][3]);
            }
        }
        __syncthreads();  // every thread is done reading the old state
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int i = i0 + r, j = c0 + c;
                const float v = acc[r][c] + Bp[(size_t)i * D + j0 + j];
                sS[i][j] = v;
                Sp[((size_t)p * H + h) * DD + (size_t)i * D + j0 + j] = v;
            }
    }
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// segments actually used for P requested over T tokens in chunks of C
static int scan_segments(int64_t T, int C, int P, int64_t *seg_tokens) {
    const int64_t nch = (T + C - 1) / C;
    const int64_t per = (nch + P - 1) / P;  // chunks per segment
    *seg_tokens = per * C;
    return (int)((nch + per - 1) / per);
}

}  // namespace kda

using namespace kda;

extern "C" size_t kda_chunk_prefill_scan_workspace_bytes(int64_t T, int H, int D, int C, int segments) {
    if (T <= 0 || H < 1 || D < 1 || C < 1 || segments < 1) return 0;
    int64_t seg_tokens = 0;
    const int P = scan_segments(T, C, segments, &seg_tokens);
    const size_t states = (size_t)P * H * D * D * sizeof(float);
    return align256((size_t)(P + 1) * sizeof(int64_t)) + 4 * align256(states);
}

extern "C" kda_status kda_chunk_prefill_scan(const void *q, const void *k, const void *v, const float *g,
                                             const float *beta, const float *initial_state, float *final_state,
                                             void *out, int64_t T, int H, int D, int C, kda_dtype dtype,
                                             kda_gate gate, float l2_eps, int segments, void *workspace,
                                             size_t workspace_bytes, kda_stream_t stream) {
    clear_detail();
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE)
        return invalid("gate must be KDA_GATE_CHANNEL, KDA_GATE_HEAD or KDA_GATE_NONE");
    if (segments < 1 || segments > 4096) return invalid("segments must be in 1..4096");
    if (T < 0) return invalid("T must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
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
    const size_t states = align256((size_t)P * H * D * D * sizeof(float));
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int64_t *cu = reinterpret_cast<int64_t *>(ws);
    float *Bs = reinterpret_cast<float *>(ws + align256((size_t)(P + 1) * sizeof(int64_t)));
    float *As = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(Bs) + states);
    float *Id = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(As) + states);
    float *Sp = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(Id) + states);

    scan_bounds_kernel<<<(P + 1 + 255) / 256, 256, 0, s>>>(cu, P, seg_tokens, T);
    if ((st = check_launch("scan_bounds_kernel"))) return st;
    const long long nid = (long long)P * H * D * D;
    identity_states_kernel<<<(unsigned)((nid + 255) / 256), 256, 0, s>>>(Id, nid, D);
    if ((st = check_launch("identity_states_kernel"))) return st;

    // the segments are equally long except the last, so natural order is longest-first enough
    PrefillArgs a{q, k, v, g, beta, nullptr, Bs, out, cu, P, T, H, D, C, dtype == KDA_BF16, l2_eps, nullptr, 0,
                  err, nullptr, (int)gate};
    auto run = [&](const PrefillArgs &x) { return prefill_tc_applicable(x) ? prefill_tc(x, s) : prefill_simt(x, s); };
    if ((st = run(a))) return st;  // 1. B of each segment (outputs overwritten by step 4)
    PrefillArgs ai = a;
    ai.s_init = Id;
    ai.s_final = As;
    ai.v_zero = true;
    if ((st = run(ai))) return st;  // 2. A of each segment
    // 3. true initial state of each segment
    const int ns = D / SCAN_JS < 1 ? 1 : D / SCAN_JS;
    switch (D) {
    case 16: segment_scan_kernel<16><<<H * ns, SCAN_NT, 0, s>>>(As, Bs, initial_state, Sp, P, H); break;
    case 32: segment_scan_kernel<32><<<H * ns, SCAN_NT, 0, s>>>(As, Bs, initial_state, Sp, P, H); break;
    case 64: segment_scan_kernel<64><<<H * ns, SCAN_NT, 0, s>>>(As, Bs, initial_state, Sp, P, H); break;
    default:
        segment_scan128_kernel<<<H * (128 / SCAN128_JS), SCAN_NT, 0, s>>>(As, Bs, initial_state, Sp, P, H);
        break;
    }
    if ((st = check_launch("segment_scan_kernel"))) return st;
    // 4. outputs and final states from the true initial states
    PrefillArgs af = a;
    af.s_init = Sp;
    af.s_final = Bs;
    if ((st = run(af))) return st;
    if (final_state) {
        const size_t one = (size_t)H * D * D * sizeof(float);
        cudaError_t e = cudaMemcpyAsync(final_state, reinterpret_cast<uint8_t *>(Bs) + (size_t)(P - 1) * one, one,
                                        cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("final state copy: ") + cudaGetErrorString(e));
    }
    return KDA_OK;
}
