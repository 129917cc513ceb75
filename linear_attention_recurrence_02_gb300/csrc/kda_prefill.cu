// kda_prefill.cu -- chunked prefill of the KDA recurrence: argument checks,
// dispatch, and the general CUDA-core kernel (any D in {16,32,64,128}, any
// chunk size 1..64, fp32 or bf16 token tensors).
//
// Chunk algebra ("为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化",
// section 5: attention-like work inside a chunk, state handed between chunks;
// section 6: decay between two positions is the product of the gates in
// between, here exp of a difference of cumulative log gates). For a chunk of
// L tokens entering with state S, with G_r = sum_{s<=r} g_s per key channel:
//   A_rs = beta_r sum_i k_ri k_si exp(G_ri - G_si)     (s < r)
//   P_rs = sum_i q_ri k_si exp(G_ri - G_si)             (s <= r)
//   (I + A) U = Diag(beta) (V - Kt S),      Kt_r = exp(G_r) . k_r
//   O = Qt S + P U,                         Qt_r = exp(G_r) . q_r
//   S' = Diag(exp(G_L)) S + Kb^T U,         Kb_s = exp(G_L - G_s) . k_s
// (q, k already L2-normalised). U is found by forward substitution. This is
// exact algebra of the token recurrence, so any chunk size gives the same
// result up to rounding.
//
// One CTA per (sequence, head, slice of JS value columns) walks the chunks of
// its sequence in order. The state slice stays in shared memory for the whole
// sequence. A and P use exact pairwise exponentials, so the kernel is robust
// to any finite gate; it is the reference-grade fp32 path, not the fast one.
#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "kda_common.cuh"
#include "kda_prefill.cuh"

namespace kda {

constexpr int SIMT_NT = 256;
constexpr int SIMT_CMAX = 64;

__host__ __device__ constexpr int simt_js(int D) { return D < 64 ? D : 64; }

__host__ __device__ inline size_t simt_smem_floats(int D, int C) {
    const int LD = D + 1, JS = simt_js(D);
    return (size_t)3 * C * LD + (size_t)D * JS + (size_t)C * JS + 2 * (size_t)C * C + 2 * (size_t)D + C;
}

template <int D, typename T, bool VZ>  // VZ: v is read as all zeros (not loaded)
__global__ void __launch_bounds__(SIMT_NT)
    prefill_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                        const float *__restrict__ g, const float *__restrict__ beta,
                        const float *s_init, float *s_final, T *__restrict__ out,
                        const int64_t *__restrict__ cu_seqlens, int N, int64_t Ttot, int H, int C, float eps,
                        unsigned *err, const int *__restrict__ order, int gate) {
    constexpr int JS = simt_js(D), LD = D + 1, NS = D / JS, NW = SIMT_NT / 32;
    extern __shared__ float smem[];
    float *sQ = smem;                    // [C][LD]  q^, then Qt
    float *sK = sQ + C * LD;             // [C][LD]  k^, then Kt
    float *sG = sK + C * LD;             // [C][LD]  G, then Kb
    float *sS = sG + C * LD;             // [D][JS]  state slice
    float *sU = sS + D * JS;             // [C][JS]  v, rhs, then U
    float *sA = sU + C * JS;             // [C][C]
    float *sP = sA + C * C;              // [C][C]
    float *sGL = sP + C * C;             // [D]      exp(G_L)
    float *sGLl = sGL + D;               // [D]      G_L
    float *sB = sGLl + D;                // [C]      beta

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slice = blockIdx.x % NS;
    const int h = (blockIdx.x / NS) % H;
    const int n = order ? order[blockIdx.x / (NS * H)] : (int)(blockIdx.x / (NS * H));
    const int j0 = slice * JS;
    int64_t start, end;
    if (!seq_range(cu_seqlens, n, N, Ttot, err, start, end)) return;

    const size_t sbase = ((size_t)n * H + h) * D * D;
    for (int p = tid; p < D * JS; p += SIMT_NT) {
        const int i = p / JS, j = p % JS;
        sS[p] = s_init ? s_init[sbase + (size_t)i * D + j0 + j] : 0.f;
    }

    for (int64_t c0 = start; c0 < end; c0 += C) {
        const int L = (int)((end - c0) < (int64_t)C ? (end - c0) : (int64_t)C);
        __syncthreads();
        // q^, k^ rows (one warp per row), beta, v slice
        for (int r = warp; r < L; r += NW) {
            const size_t o = ((size_t)(c0 + r) * H + h) * D;
            float sq = 0.f, sk = 0.f;
            for (int i = lane; i < D; i += 32) {
                const float a = Elem<T>::load(q + o + i), b = Elem<T>::load(k + o + i);
                sQ[r * LD + i] = a;
                sK[r * LD + i] = b;
                sq += a * a;
                sk += b * b;
            }
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, m);
                sk += __shfl_xor_sync(0xffffffffu, sk, m);
            }
            const float rq = inv_norm(sq, eps), rk = inv_norm(sk, eps);
            for (int i = lane; i < D; i += 32) {
                sQ[r * LD + i] *= rq;
                sK[r * LD + i] *= rk;
            }
            if (lane == 0) sB[r] = beta[(size_t)(c0 + r) * H + h];
        }
        for (int p = tid; p < L * JS; p += SIMT_NT) {
            const int r = p / JS, j = p % JS;
            sU[p] = VZ ? 0.f : Elem<T>::load(v + ((size_t)(c0 + r) * H + h) * D + j0 + j);
        }
        // cumulative log decay per key channel
        if (tid < D) {
            float acc = 0.f;
            for (int r = 0; r < L; ++r) {
                acc += gate == KDA_GATE_CHANNEL ? g[((size_t)(c0 + r) * H + h) * D + tid]
                       : gate == KDA_GATE_HEAD  ? g[(size_t)(c0 + r) * H + h]
                                                : 0.f;
                sG[r * LD + tid] = acc;
            }
        }
        __syncthreads();
        // A and P with exact pairwise decays
        for (int p = tid; p < L * L; p += SIMT_NT) {
            const int r = p / L, s = p % L;
            float a = 0.f, pq = 0.f;
            if (s <= r) {
                for (int i = 0; i < D; ++i) {
                    const float e = expf(sG[r * LD + i] - sG[s * LD + i]);
                    const float ks = sK[s * LD + i] * e;
                    a += sK[r * LD + i] * ks;
                    pq += sQ[r * LD + i] * ks;
                }
            }
            sA[r * C + s] = (s < r) ? sB[r] * a : 0.f;
            sP[r * C + s] = pq;
        }
        if (tid < D) {
            sGLl[tid] = sG[(L - 1) * LD + tid];
            sGL[tid] = expf(sGLl[tid]);
        }
        __syncthreads();
        // Qt, Kt, Kb in place
        for (int p = tid; p < L * D; p += SIMT_NT) {
            const int r = p / D, i = p % D;
            const float Gr = sG[r * LD + i], e = expf(Gr);
            const float kh = sK[r * LD + i];
            sQ[r * LD + i] *= e;
            sK[r * LD + i] = kh * e;
            sG[r * LD + i] = kh * expf(sGLl[i] - Gr);
        }
        __syncthreads();
        // rhs = beta (v - Kt S)
        for (int p = tid; p < L * JS; p += SIMT_NT) {
            const int r = p / JS, j = p % JS;
            float acc = 0.f;
            for (int i = 0; i < D; ++i) acc += sK[r * LD + i] * sS[i * JS + j];
            sU[p] = sB[r] * (sU[p] - acc);
        }
        __syncthreads();
        // forward substitution (I + A) U = rhs, one thread per value column
        if (tid < JS) {
            for (int r = 1; r < L; ++r) {
                float acc = sU[r * JS + tid];
                for (int s = 0; s < r; ++s) acc -= sA[r * C + s] * sU[s * JS + tid];
                sU[r * JS + tid] = acc;
            }
        }
        __syncthreads();
        // O = Qt S + P U
        for (int p = tid; p < L * JS; p += SIMT_NT) {
            const int r = p / JS, j = p % JS;
            float acc = 0.f;
            for (int i = 0; i < D; ++i) acc += sQ[r * LD + i] * sS[i * JS + j];
            for (int s = 0; s <= r; ++s) acc += sP[r * C + s] * sU[s * JS + j];
            Elem<T>::store(out + ((size_t)(c0 + r) * H + h) * D + j0 + j, acc);
        }
        __syncthreads();
        // S' = Diag(exp(G_L)) S + Kb^T U
        for (int p = tid; p < D * JS; p += SIMT_NT) {
            const int i = p / JS, j = p % JS;
            float acc = sGL[i] * sS[p];
            for (int s = 0; s < L; ++s) acc += sG[s * LD + i] * sU[s * JS + j];
            sS[p] = acc;
        }
    }
    __syncthreads();
    if (s_final) {
        for (int p = tid; p < D * JS; p += SIMT_NT) {
            const int i = p / JS, j = p % JS;
            s_final[sbase + (size_t)i * D + j0 + j] = sS[p];
        }
    }
}

template <int D, typename T>
static kda_status launch_simt(const PrefillArgs &a, cudaStream_t s) {
    const size_t smem = simt_smem_floats(D, a.C) * sizeof(float);
    auto kern = a.v_zero ? prefill_simt_kernel<D, T, true> : prefill_simt_kernel<D, T, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    const unsigned grid = launch_seqs(a) * a.H * (D / simt_js(D));
    kern<<<grid, SIMT_NT, smem, s>>>(static_cast<const T *>(a.q), static_cast<const T *>(a.k),
                                     static_cast<const T *>(a.v), a.g, a.beta, a.s_init, a.s_final,
                                     static_cast<T *>(a.out), a.cu_seqlens, a.N, a.T, a.H, a.C, a.eps, a.err,
                                     a.order, a.gate);
    return check_launch("prefill_simt_kernel");
}

template <typename T>
static kda_status dispatch_simt(const PrefillArgs &a, cudaStream_t s) {
    switch (a.D) {
    case 16: return launch_simt<16, T>(a, s);
    case 32: return launch_simt<32, T>(a, s);
    case 64: return launch_simt<64, T>(a, s);
    default: return launch_simt<128, T>(a, s);
    }
}

kda_status prefill_simt(const PrefillArgs &a, cudaStream_t s) {
    return a.bf16 ? dispatch_simt<__nv_bfloat16>(a, s) : dispatch_simt<float>(a, s);
}

kda_status prefill_run(const PrefillArgs &a, cudaStream_t s) {
    if (prefill_tc_applicable(a)) return prefill_tc(a, s);
    if (prefill_tf32_applicable(a)) return prefill_tf32(a, s);
    if (prefill_f32_applicable(a)) return prefill_f32(a, s);
    return prefill_simt(a, s);
}

extern "C" const char *kda_chunk_prefill_route(int D, int C, kda_dtype dtype) {
    if (!valid_head_dim(D) || C < 1 || C > SIMT_CMAX || (dtype != KDA_F32 && dtype != KDA_BF16)) return nullptr;
    PrefillArgs a{};
    a.D = D;
    a.C = C;
    a.T = 1;
    a.bf16 = dtype == KDA_BF16;
    if (prefill_tc_applicable(a)) return "prefill_tc_pipe_kernel";
    if (prefill_tf32_applicable(a)) return "prefill_tf32_kernel";
    if (prefill_f32_applicable(a)) return "prefill_f32_kernel";
    return "prefill_simt_kernel";
}

// Longest sequences first: a sequence's chunks are walked serially by its
// CTAs, so starting the long chains first shortens the tail of a mixed-length
// batch (greedy longest-processing-time order). order[rank] = n, where rank
// counts longer sequences and equal-length sequences with a smaller index.
__global__ void __launch_bounds__(1024) prefill_order_kernel(const int64_t *__restrict__ cu, int N,
                                                             int *__restrict__ order) {
    extern __shared__ int64_t s_len[];
    for (int n = threadIdx.x; n < N; n += blockDim.x) s_len[n] = cu[n + 1] - cu[n];
    __syncthreads();
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        const int64_t ln = s_len[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int64_t lm = s_len[m];
            rank += (lm > ln) || (lm == ln && m < n);
        }
        order[rank] = n;
    }
}

kda_status launch_prefill_order(const int64_t *cu_seqlens, int N, int *order, cudaStream_t s) {
    const size_t smem = (size_t)N * sizeof(int64_t);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(prefill_order_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess)
            return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    }
    prefill_order_kernel<<<1, 1024, smem, s>>>(cu_seqlens, N, order);
    return check_launch("prefill_order_kernel");
}

}  // namespace kda

using namespace kda;

// the launch order of a mixed-length batch: int32 per sequence
static size_t order_bytes(int num_seqs) {
    if (num_seqs < 2 || num_seqs > ORDER_MAX_SEQS) return 0;
    return ((size_t)num_seqs * sizeof(int) + 255) & ~(size_t)255;
}

extern "C" size_t kda_chunk_prefill_workspace_bytes(int64_t total_tokens, int num_seqs, int H, int D, int C) {
    // one long sequence with few heads: room for the automatic split
    if (num_seqs == 1) {
        const int P = prefill_auto_segments(total_tokens, H, C);
        if (P > 0) return kda_chunk_prefill_scan_workspace_bytes(total_tokens, H, D, C, P);
    }
    return order_bytes(num_seqs);
}

// The gated prefill, followed by the output epilogue (a pass of
// kda_gated_rmsnorm over out, in place) when epi_gate != NULL. Run inside the
// tensor-core kernel on the staged output tile instead, the epilogue made the
// 4096-token prefill 0.511 ms against 0.389 ms for the two passes: it lands
// on the state-chain warps, which then become the longest stage.
static kda_status prefill_entry(const void *q, const void *k, const void *v, const float *g, const float *beta,
                                const float *initial_state, float *final_state, void *out,
                                const int64_t *cu_seqlens, int N, int64_t T, int H, int D, int C, kda_dtype dtype,
                                kda_gate gate, float l2_eps, void *workspace, size_t workspace_bytes,
                                kda_stream_t stream, const void *epi_gate, const float *epi_w, kda_gate_act epi_act,
                                float epi_eps, const int *ext_order = nullptr, int ext_nlaunch = 0) {
    // ext_order (device, ext_nlaunch entries): launch only these sequences, in this order
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE)
        return invalid("gate must be KDA_GATE_CHANNEL, KDA_GATE_HEAD or KDA_GATE_NONE");
    if (N < 1) return invalid("N must be >= 1");
    if (T < 0) return invalid("T must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (C < 1 || C > SIMT_CMAX) return invalid("C must be in 1..64");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (!(l2_eps >= 0.f)) return invalid("l2_eps must be >= 0");
    if (cu_seqlens == nullptr && N != 1) return invalid("cu_seqlens is NULL but N != 1");
    if ((long long)N * H * 2 > 0x7fffffffLL) return invalid("N*H too large for one launch");
    const size_t need = ext_order ? 0 : order_bytes(N);
    if (workspace_bytes < need) return invalid("workspace too small");
    kda_status st;
    if (T > 0 && ((st = check_ptr(q, "q")) || (st = check_ptr(k, "k")) || (st = check_ptr(v, "v")) ||
                  (gate != KDA_GATE_NONE && (st = check_ptr(g, "g"))) || (st = check_ptr(beta, "beta")) ||
                  (st = check_ptr(out, "out"))))
        return st;
    if (initial_state && (st = check_ptr(initial_state, "initial_state"))) return st;
    if (final_state && (st = check_ptr(final_state, "final_state"))) return st;
    if (cu_seqlens && (reinterpret_cast<uintptr_t>(cu_seqlens) & 7u)) return invalid("cu_seqlens is not 8-byte aligned");
    if (need && (st = check_ptr(workspace, "workspace"))) return st;
    if (T > 0 && (out == q || out == k || out == v)) return invalid("out must not alias q, k or v");
    if (T == 0 && final_state == nullptr) return KDA_OK;
    if ((st = bind_stream_device(stream))) return st;
    // One sequence (no cu_seqlens) whose serial chunk chain would leave most
    // SMs idle: split it into segments when the workspace has room for that
    // (kda_chunk_prefill_workspace_bytes asks for it).
    if (cu_seqlens == nullptr && T > 0 && ext_order == nullptr) {
        const int P = prefill_auto_segments(T, H, C);
        if (P > 0 && workspace != nullptr && workspace_bytes >= kda_chunk_prefill_scan_workspace_bytes(T, H, D, C, P)) {
            st = kda_chunk_prefill_scan(q, k, v, g, beta, initial_state, final_state, out, T, H, D, C, dtype, gate,
                                        l2_eps, P, workspace, workspace_bytes, stream);
            if (st != KDA_OK || epi_gate == nullptr) return st;
            return kda_gated_rmsnorm(out, epi_gate, epi_w, out, T, H, D, dtype, epi_act, epi_eps, stream);
        }
    }
    PrefillArgs a{q, k, v, g, beta, initial_state, final_state, out, cu_seqlens, N, T, H, D, C,
                  dtype == KDA_BF16, l2_eps, workspace, workspace_bytes, device_error_word(), nullptr, (int)gate};
    if (a.err == nullptr) return fail(KDA_ERR_CUDA, "device error word unavailable");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ext_order != nullptr) {
        a.order = ext_order;
        a.nlaunch = ext_nlaunch;
    } else if (need > 0 && cu_seqlens != nullptr) {
        int *order = static_cast<int *>(workspace);
        if ((st = launch_prefill_order(cu_seqlens, N, order, s))) return st;
        a.order = order;
    }
    if ((st = prefill_run(a, s))) return st;
    if (epi_gate == nullptr || T == 0) return KDA_OK;
    return kda_gated_rmsnorm(out, epi_gate, epi_w, out, T, H, D, dtype, epi_act, epi_eps, stream);
}

extern "C" kda_status kda_chunk_prefill_gated(const void *q, const void *k, const void *v, const float *g,
                                              const float *beta, const float *initial_state, float *final_state,
                                              void *out, const int64_t *cu_seqlens, int N, int64_t T, int H, int D,
                                              int C, kda_dtype dtype, kda_gate gate, float l2_eps, void *workspace,
                                              size_t workspace_bytes, kda_stream_t stream) {
    clear_detail();
    return prefill_entry(q, k, v, g, beta, initial_state, final_state, out, cu_seqlens, N, T, H, D, C, dtype, gate,
                         l2_eps, workspace, workspace_bytes, stream, nullptr, nullptr, KDA_ACT_SIGMOID, 0.f);
}

extern "C" kda_status kda_chunk_prefill_epi(const void *q, const void *k, const void *v, const float *g,
                                            const float *beta, const float *initial_state, float *final_state,
                                            void *out, const int64_t *cu_seqlens, int N, int64_t T, int H, int D,
                                            int C, kda_dtype dtype, kda_gate gate, float l2_eps, const void *out_gate,
                                            const float *norm_weight, kda_gate_act act, float norm_eps,
                                            void *workspace, size_t workspace_bytes, kda_stream_t stream) {
    clear_detail();
    if (act != KDA_ACT_SIGMOID && act != KDA_ACT_SILU) return invalid("act must be KDA_ACT_SIGMOID or KDA_ACT_SILU");
    if (!(norm_eps >= 0.f)) return invalid("norm_eps must be >= 0");
    kda_status st;
    if (T > 0 && ((st = check_ptr(out_gate, "out_gate")) || (st = check_ptr(norm_weight, "norm_weight")))) return st;
    if (T > 0 && (out_gate == out || out_gate == q || out_gate == k || out_gate == v))
        return invalid("out_gate must not alias out, q, k or v");
    return prefill_entry(q, k, v, g, beta, initial_state, final_state, out, cu_seqlens, N, T, H, D, C, dtype, gate,
                         l2_eps, workspace, workspace_bytes, stream, T > 0 ? out_gate : nullptr, norm_weight, act,
                         norm_eps);
}

extern "C" kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, const float *g,
                                        const float *beta, const float *initial_state, float *final_state,
                                        void *out, const int64_t *cu_seqlens, int N, int64_t T, int H, int D,
                                        int C, kda_dtype dtype, float l2_eps, void *workspace,
                                        size_t workspace_bytes, kda_stream_t stream) {
    return kda_chunk_prefill_gated(q, k, v, g, beta, initial_state, final_state, out, cu_seqlens, N, T, H, D, C,
                                   dtype, KDA_GATE_CHANNEL, l2_eps, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- batches with long sequences
// Segments per sequence for kda_chunk_prefill_split. The batch's work is W
// chunk-heads (every sequence's chunks times H); spread evenly it keeps each
// of the `sms` SMs busy for ceil(W / sms) chunk steps. A sequence whose serial
// chain of chunks is longer than that (and than 8 chunks) gets
// P = min(chunks / balance, 4096) segments when P >= 4: its two scan passes
// then take 1/P of its chain each, and the scan and the correction pay. The
// sequences that stay whole run beside the first split sequence's passes, one
// CTA per (sequence, head), so P is capped where that leaves them SMs of their
// own: P * H + (whole sequences) * H <= sms, as long as P stays >= 4. The
// per-head arrays of a segment start 16-byte aligned only when H is a
// multiple of 4, so other H are never split. -1 for invalid lengths.
static int split_plan(const int64_t *cu, int N, int H, int C, int sms, int *seg) {
    if (cu == nullptr || seg == nullptr || N < 1 || H < 1 || C < 1 || cu[0] != 0) return -1;
    int64_t W = 0;
    for (int i = 0; i < N; ++i) {
        if (cu[i + 1] < cu[i]) return -1;
        W += (cu[i + 1] - cu[i] + C - 1) / C;
    }
    if (sms <= 0) sms = current_sms();
    const int64_t bal = sms > 0 ? std::max<int64_t>((W * H + sms - 1) / sms, 8) : 0;
    int n = 0;
    int64_t whole = 0;  // sequences with tokens that stay whole
    for (int i = 0; i < N; ++i) {
        const int64_t ch = (cu[i + 1] - cu[i] + C - 1) / C;
        const int64_t P = (bal > 0 && H % 4 == 0) ? std::min<int64_t>(ch / bal, 4096) : 0;
        seg[i] = P >= 4 ? (int)P : 1;
        n += P >= 4 ? 1 : 0;
        whole += (P < 4 && ch > 0) ? 1 : 0;
    }
    const int64_t cap = sms > 0 ? ((int64_t)sms - whole * H) / H : 0;
    if (n > 0 && whole > 0 && cap >= 4)
        for (int i = 0; i < N; ++i)
            if (seg[i] > cap) seg[i] = (int)cap;
    return n;
}

// The launch order of the sequences kda_chunk_prefill_split keeps whole travels
// to the device in kernel parameters, ORDER_SLICE entries per launch, so that a
// captured graph holds the list itself rather than a host address to copy from.
constexpr int ORDER_SLICE = 1000;
struct OrderSlice {
    int offset, n;
    int idx[ORDER_SLICE];
};
__global__ void order_fill_kernel(const __grid_constant__ OrderSlice sl, int *__restrict__ order) {
    for (int i = threadIdx.x; i < sl.n; i += blockDim.x) order[sl.offset + i] = sl.idx[i];
}

// The side stream on which kda_chunk_prefill_split runs the sequences that stay
// whole, and the fork and join events around it: one set per device, created on
// first use and kept for the process. The mutex serialises the calls' enqueueing
// (the events are re-recorded by every call).
struct SplitSide {
    std::mutex mu;
    cudaStream_t side[64] = {};
    cudaEvent_t fork[64] = {}, join[64] = {};
};
static SplitSide g_split_side;

static size_t align256_(size_t x) { return (x + 255) & ~(size_t)255; }

// workspace: the largest split sequence's scan workspace, then the launch order of the rest
static size_t split_ws(const int64_t *cu, const int *seg, int N, int H, int D, int C, size_t *scan_bytes) {
    size_t scan = 0;
    for (int i = 0; i < N; ++i)
        if (seg[i] > 1)
            scan = std::max(scan, kda_chunk_prefill_scan_workspace_bytes(cu[i + 1] - cu[i], H, D, C, seg[i]));
    scan = align256_(scan);
    if (scan_bytes) *scan_bytes = scan;
    return scan + align256_((size_t)N * sizeof(int));
}

extern "C" int kda_chunk_prefill_split_plan(const int64_t *host_cu_seqlens, int N, int H, int C, int sms,
                                            int *segments) {
    return split_plan(host_cu_seqlens, N, H, C, sms, segments);
}

extern "C" size_t kda_chunk_prefill_split_workspace_bytes(const int64_t *host_cu_seqlens, int N, int H, int D,
                                                          int C) {
    if (N < 1 || N > (1 << 24)) return 0;
    std::vector<int> seg((size_t)N);
    if (split_plan(host_cu_seqlens, N, H, C, 0, seg.data()) < 0) return 0;
    return split_ws(host_cu_seqlens, seg.data(), N, H, D, C, nullptr);
}

extern "C" kda_status kda_chunk_prefill_split(const void *q, const void *k, const void *v, const float *g,
                                              const float *beta, const float *initial_state, float *final_state,
                                              void *out, const int64_t *cu_seqlens, const int64_t *host_cu_seqlens,
                                              int N, int64_t T, int H, int D, int C, kda_dtype dtype, kda_gate gate,
                                              float l2_eps, void *workspace, size_t workspace_bytes,
                                              kda_stream_t stream) {
    clear_detail();
    if (gate != KDA_GATE_CHANNEL && gate != KDA_GATE_HEAD && gate != KDA_GATE_NONE)
        return invalid("gate must be KDA_GATE_CHANNEL, KDA_GATE_HEAD or KDA_GATE_NONE");
    if (N < 1 || N > (1 << 24)) return invalid("N must be in 1..2^24");
    if (T < 0) return invalid("T must be >= 0");
    if (H < 1) return invalid("H must be >= 1");
    if (!valid_head_dim(D)) return invalid("D must be one of 16, 32, 64, 128");
    if (C < 1 || C > SIMT_CMAX) return invalid("C must be in 1..64");
    if (dtype != KDA_F32 && dtype != KDA_BF16) return invalid("dtype must be KDA_F32 or KDA_BF16");
    if (cu_seqlens == nullptr || host_cu_seqlens == nullptr)
        return invalid("cu_seqlens and host_cu_seqlens are both required");
    std::vector<int> seg((size_t)N);
    const int nsplit = split_plan(host_cu_seqlens, N, H, C, 0, seg.data());
    if (nsplit < 0) return invalid("host_cu_seqlens must start at 0 and be non-decreasing");
    if (host_cu_seqlens[N] != T) return invalid("host_cu_seqlens[N] must equal T");
    if (nsplit == 0)  // nothing to split: the ordinary prefill
        return kda_chunk_prefill_gated(q, k, v, g, beta, initial_state, final_state, out, cu_seqlens, N, T, H, D, C,
                                       dtype, gate, l2_eps, workspace, workspace_bytes, stream);
    size_t scan_bytes = 0;
    const size_t need = split_ws(host_cu_seqlens, seg.data(), N, H, D, C, &scan_bytes);
    if (workspace_bytes < need) return invalid("workspace too small");
    kda_status st;
    if ((st = check_ptr(workspace, "workspace"))) return st;
    if ((st = bind_stream_device(stream))) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // 1. the sequences that stay whole: one launch, longest first, on a side stream forked from
    // `stream`, so that it runs beside the split sequences' passes; joined back at the end
    std::vector<int> keep;
    for (int i = 0; i < N; ++i)
        if (seg[i] == 1) keep.push_back(i);
    std::stable_sort(keep.begin(), keep.end(), [&](int a, int b) {
        return host_cu_seqlens[a + 1] - host_cu_seqlens[a] > host_cu_seqlens[b + 1] - host_cu_seqlens[b];
    });
    std::unique_lock<std::mutex> lock(g_split_side.mu);
    cudaEvent_t join = nullptr;
    if (!keep.empty()) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess || dev < 0 || dev >= 64)
            return fail(KDA_ERR_CUDA, "cudaGetDevice failed or device index above 63");
        if (g_split_side.side[dev] == nullptr) {
            cudaStream_t ns = nullptr;
            cudaEvent_t ef = nullptr, ej = nullptr;
            if ((e = cudaStreamCreateWithFlags(&ns, cudaStreamNonBlocking)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&ef, cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&ej, cudaEventDisableTiming)) != cudaSuccess)
                return fail(KDA_ERR_CUDA, std::string("side stream: ") + cudaGetErrorString(e));
            g_split_side.side[dev] = ns;
            g_split_side.fork[dev] = ef;
            g_split_side.join[dev] = ej;
        }
        cudaStream_t side = g_split_side.side[dev];
        join = g_split_side.join[dev];
        int *order = reinterpret_cast<int *>(static_cast<uint8_t *>(workspace) + scan_bytes);
        for (size_t o = 0; o < keep.size(); o += ORDER_SLICE) {
            OrderSlice sl;
            sl.offset = (int)o;
            sl.n = (int)std::min<size_t>(ORDER_SLICE, keep.size() - o);
            std::copy(keep.begin() + (ptrdiff_t)o, keep.begin() + (ptrdiff_t)(o + sl.n), sl.idx);
            order_fill_kernel<<<1, 256, 0, s>>>(sl, order);
            if ((st = check_launch("order_fill_kernel"))) return st;
        }
        if ((e = cudaEventRecord(g_split_side.fork[dev], s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(side, g_split_side.fork[dev], 0)) != cudaSuccess)
            return fail(KDA_ERR_CUDA, std::string("fork: ") + cudaGetErrorString(e));
        if ((st = prefill_entry(q, k, v, g, beta, initial_state, final_state, out, cu_seqlens, N, T, H, D, C, dtype,
                                gate, l2_eps, nullptr, 0, reinterpret_cast<kda_stream_t>(side), nullptr, nullptr,
                                KDA_ACT_SIGMOID, 0.f, order, (int)keep.size())))
            return st;
        if ((e = cudaEventRecord(join, side)) != cudaSuccess)
            return fail(KDA_ERR_CUDA, std::string("join: ") + cudaGetErrorString(e));
    }
    // 2. each long sequence through the chunk-state scan over its own rows; `stream` then joins the
    // side stream (also when a launch failed, so that nothing of the call runs unordered after it)
    const size_t elt = dtype == KDA_BF16 ? 2 : 4;
    st = KDA_OK;
    for (int i = 0; i < N && st == KDA_OK; ++i) {
        if (seg[i] == 1) continue;
        const int64_t t0 = host_cu_seqlens[i], len = host_cu_seqlens[i + 1] - t0;
        const size_t row = (size_t)t0 * H * D, sst = (size_t)i * H * D * D;
        const float *gi = g == nullptr ? nullptr
                          : gate == KDA_GATE_CHANNEL ? g + row
                          : gate == KDA_GATE_HEAD ? g + (size_t)t0 * H
                                                  : g;
        st = kda_chunk_prefill_scan(static_cast<const uint8_t *>(q) + row * elt,
                                    static_cast<const uint8_t *>(k) + row * elt,
                                    static_cast<const uint8_t *>(v) + row * elt, gi, beta + (size_t)t0 * H,
                                    initial_state ? initial_state + sst : nullptr,
                                    final_state ? final_state + sst : nullptr,
                                    static_cast<uint8_t *>(out) + row * elt, len, H, D, C, dtype, gate, l2_eps,
                                    seg[i], workspace, scan_bytes, stream);
    }
    if (join != nullptr) {
        cudaError_t e = cudaStreamWaitEvent(s, join, 0);
        if (e != cudaSuccess && st == KDA_OK) return fail(KDA_ERR_CUDA, std::string("join: ") + cudaGetErrorString(e));
    }
    return st;
}
