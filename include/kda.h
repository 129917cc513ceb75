/*
 * kda.h -- C ABI of libkda.so: the Kimi Delta Attention (KDA) gated
 * delta-rule recurrence on one NVIDIA GB300 (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *  [W] "KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析"
 *      - "KDA 递推公式先衰减再差分": per token and head, decay the state along
 *        the key axis, S <- Diag(exp(g_t)) S_{t-1} with g in log space, then
 *        apply the delta rule S_t = S + beta_t k_t (v_t - S^T k_t)^T, then read
 *        out o_t = S_t^T q_t; q and k are L2-normalised inside the kernel; a
 *        width-4 causal short convolution with SiLU precedes q/k/v and needs a
 *        3-token ring per projection at decode, kept as session state.
 *      - "414MB 的 KDA 状态从哪来": state 128 x 128 fp32 per (layer, head);
 *        ring 3 projections x 3 tokens x 128 per head.
 *  [G] "为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化"
 *      - section 5: chunked evaluation (attention-like inside a chunk of C
 *        tokens, state hand-off between chunks, C = 64 or 128 for tensor cores).
 *      - section 7: the per-channel gate Diag(alpha_t) of Kimi Linear.
 *
 * Conventions shared by every call:
 *  - State S of one (sequence, head) is D x D fp32, row i = key channel,
 *    column j = value channel, row-major (d_k = d_v = D).
 *  - Token tensors are token-major and packed: x[t, h, c] at ((t*H)+h)*D + c.
 *  - q, k are L2-normalised as x / sqrt(sum x^2 + l2_eps); a vector whose
 *    sum of squares plus l2_eps is zero normalises to zero. v is not
 *    normalised; q carries no extra 1/sqrt(D) scale.
 *  - g (log-space gate, per key channel) and beta are always fp32; q, k, v,
 *    conv inputs/outputs and the outputs o use `dtype`.
 *  - Every pointer is a DEVICE pointer owned by the caller and must be
 *    16-byte aligned. Buffers must not alias one another except where a
 *    call says so. Calls are asynchronous on `stream` (NULL = the legacy
 *    default stream), launch on the stream's device and allocate nothing.
 *  - Argument checks are synchronous: a failure returns KDA_ERR_INVALID_ARG
 *    (or KDA_ERR_UNSUPPORTED) and launches nothing. A failed launch returns
 *    KDA_ERR_CUDA. kda_last_error_detail() gives the message of the last
 *    failure on the calling thread.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *kda_stream_t;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* bad shape, null or misaligned pointer, short workspace */
    KDA_ERR_UNSUPPORTED = 2, /* valid request this build does not implement */
    KDA_ERR_CUDA = 3,        /* CUDA runtime error (launch, device query) */
    KDA_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up */
    KDA_ERR_DEVICE_CHECK = 5 /* a kernel found invalid data (e.g. non-monotone cu_seqlens) */
} kda_status;

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Form of the decay gate ("为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3
 * 的架构进化", section 7: Kimi Delta Attention decays every key channel by its
 * own factor, Gated DeltaNet by one factor per head; the plain delta rule of
 * section 4 has no decay). g is always in log space, alpha = exp(g).
 *   KDA_GATE_CHANNEL  g [..., H, D]: one log-gate per key channel (KDA)
 *   KDA_GATE_HEAD     g [..., H]:    one log-gate per head (Gated DeltaNet)
 *   KDA_GATE_NONE     g unused, may be NULL: alpha = 1 (DeltaNet)          */
typedef enum { KDA_GATE_CHANNEL = 0, KDA_GATE_HEAD = 1, KDA_GATE_NONE = 2 } kda_gate;

/* Activation of the output gate in kda_gated_rmsnorm:
 *   KDA_ACT_SIGMOID  act(z) = 1 / (1 + exp(-z))
 *   KDA_ACT_SILU     act(z) = z / (1 + exp(-z))                           */
typedef enum { KDA_ACT_SIGMOID = 0, KDA_ACT_SILU = 1 } kda_gate_act;

/* Static description of a status code. Never NULL. */
const char *kda_status_string(kda_status s);

/* Message of the last failed call on the calling thread ("" if none). The
 * pointer stays valid until the next call on this thread. */
const char *kda_last_error_detail(void);

/* ABI version of this library (increments on incompatible changes). */
int kda_abi_version(void);

/* Bytes of recurrent state for `layers` x `heads` states of dk x dv fp32
 * ([W] "414MB 的 KDA 状态从哪来"; 69 x 96 x 128 x 128 x 4 B = 414 MiB). */
size_t kda_state_bytes(int layers, int heads, int dk, int dv);

/* Bytes of short-conv ring for `layers` x `batch` x `heads`: 3 projections
 * x 3 cached tokens x d elements of `elem_bytes` each ([W] same table). */
size_t kda_shortconv_ring_bytes(int layers, int batch, int heads, int d, int elem_bytes);

/*
 * One decode step of the width-4 causal depthwise short convolution with
 * SiLU that precedes q, k and v ([W] "KDA 递推公式先衰减再差分", last
 * paragraph; ring size from "414MB 的 KDA 状态从哪来").
 *
 *   x    [B,3,H,D] dtype   current pre-conv projections, p = 0,1,2 = q,k,v
 *   ring [B,3,H,3,D] dtype in/out: x_{t-3}, x_{t-2}, x_{t-1} (slot 0 oldest);
 *                          on return holds x_{t-2}, x_{t-1}, x_t
 *   w    [3,H,D,4] fp32    taps; w[p,h,c,3] multiplies x_t, w[p,h,c,m] for
 *                          m < 3 multiplies ring slot m
 *   y    [3,B,H,D] dtype   out: SiLU(w0 r0 + w1 r1 + w2 r2 + w3 x), written
 *                          projection-major so that y[0], y[1], y[2] are the
 *                          contiguous [B,H,D] q, k, v of kda_decode_step
 * Requires B >= 0, H >= 1, D in {16,32,64,128}. y may not alias x or ring.
 * B = 0 is a no-op. x and ring are read by TMA tensor copies: KDA_ERR_CUDA
 * if the driver's tensor-map encoder rejects them. A copy that does not land
 * within about a second sets the device error word (KDA_ERR_TIMEOUT from the
 * next kda_sync_status); the sequences of that copy keep their y and ring
 * contents. The launch is a programmatic dependent launch: it may start while
 * the kernel before it on the stream drains, but reads x, ring and w only once
 * that kernel has completed (before that it only prefetches them into L2), so
 * stream order holds as for a plain launch.
 */
kda_status kda_shortconv_step(const void *x, void *ring, const float *w, void *y,
                              int B, int H, int D, kda_dtype dtype, kda_stream_t stream);

/*
 * The same short convolution over a packed batch of prompts, as prefill runs
 * it ([W] "KDA 递推公式先衰减再差分": conv + SiLU in front of q/k/v, with the
 * 3-token ring that decode carries on). For each sequence n, tokens
 * [cu_seqlens[n], cu_seqlens[n+1]) are convolved as if kda_shortconv_step
 * had been called once per token, starting from ring_in[n]; ring_out[n]
 * receives the ring after the last token, ready for kda_shortconv_step or
 * kda_shortconv_decode_step on the same sequences.
 *
 *   x        [T,3,H,D] dtype    pre-conv projections, p = 0,1,2 = q,k,v
 *   ring_in  [N,3,H,3,D] dtype  history before each sequence (slot 0
 *                               oldest), or NULL for zeros
 *   w        [3,H,D,4] fp32     taps, as in kda_shortconv_step
 *   y        [3,T,H,D] dtype    out: post-conv, projection-major, so y[0],
 *                               y[1], y[2] are the [T,H,D] q, k, v of
 *                               kda_chunk_prefill
 *   ring_out [N,3,H,3,D] dtype  out, or NULL; a sequence with no tokens
 *                               gets ring_in[n] (or zeros)
 *   cu_seqlens device int64 [N+1], or NULL for one sequence of T tokens
 * SiLU is evaluated with the fast exponential and division intrinsics.
 * Requires N >= 1, T >= 0, H >= 1, D in {16,32,64,128}; y may not alias x
 * or a ring, and ring_out may not alias ring_in or x. Invalid cu_seqlens
 * (not 0 .. T, or decreasing) set the device error word reported by
 * kda_sync_status; the affected tiles write nothing.
 */
kda_status kda_shortconv_prefill(const void *x, const void *ring_in, const float *w, void *y,
                                 void *ring_out, const int64_t *cu_seqlens, int N, int64_t T,
                                 int H, int D, kda_dtype dtype, kda_stream_t stream);

/*
 * One KDA decode step for B independent sequences ([W] "KDA 递推公式先衰减再差分";
 * per-channel gate as in [G] section 7). For each (b, h):
 *   q^ = L2(q), k^ = L2(k), a = exp(g)
 *   S' = Diag(a) S;  delta = beta (v - S'^T k^);  S <- S' + k^ delta^T
 *   o  = S^T q^  (= S'^T q^ + (k^ . q^) delta)
 * The state is read once and written once.
 *
 *   q, k, v [B,H,D] dtype (post-conv);  g [B,H,D] fp32;  beta [B,H] fp32
 *   state   [B,H,D,D] fp32, in/out (updated in place)
 *   out     [B,H,D] dtype
 * Requires B >= 0, H >= 1, D in {16,32,64,128}, l2_eps >= 0. B = 0 is a no-op.
 */
kda_status kda_decode_step(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, float *state, void *out, int B, int H, int D,
                           kda_dtype dtype, float l2_eps, kda_stream_t stream);

/*
 * kda_decode_step with the gate form chosen by `gate`: g is [B,H,D] for
 * KDA_GATE_CHANNEL, [B,H] for KDA_GATE_HEAD, and unused (may be NULL) for
 * KDA_GATE_NONE. kda_decode_step is this call with KDA_GATE_CHANNEL.
 */
kda_status kda_decode_step_gated(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, float *state, void *out, int B, int H, int D,
                                 kda_dtype dtype, kda_gate gate, float l2_eps, kda_stream_t stream);

/*
 * Short conv + decode step in one launch: the same recurrence as
 * kda_shortconv_step followed by kda_decode_step on its output ([W] "KDA
 * 递推公式先衰减再差分": conv + SiLU in front of q/k/v, then decay, delta,
 * readout), except that the post-conv q, k, v stay in fp32 inside the kernel
 * (never rounded to `dtype` nor written to memory).
 *
 *   x [B,3,H,D] dtype, ring [B,3,H,3,D] dtype (in/out), w [3,H,D,4] fp32,
 *   g [B,H,D] fp32, beta [B,H] fp32, state [B,H,D,D] fp32 (in/out),
 *   out [B,H,D] dtype
 * Same requirements and errors as the two calls it replaces. At D = 128 the
 * launch is a programmatic dependent launch: it may start while the kernel
 * before it on `stream` drains, but before that kernel has completed it only
 * prefetches its state and input rows into L2 (which cannot serve a stale
 * value); every read and write waits. So the results are those of a plain
 * launch, and consecutive steps on one state overlap their launch boundary.
 */
kda_status kda_shortconv_decode_step(const void *x, void *ring, const float *w, const float *g,
                                     const float *beta, float *state, void *out, int B, int H, int D,
                                     kda_dtype dtype, float l2_eps, kda_stream_t stream);

/*
 * kda_shortconv_decode_step with the gate form chosen by `gate` (g as in
 * kda_decode_step_gated). kda_shortconv_decode_step is this call with
 * KDA_GATE_CHANNEL.
 */
kda_status kda_shortconv_decode_step_gated(const void *x, void *ring, const float *w, const float *g,
                                           const float *beta, float *state, void *out, int B, int H,
                                           int D, kda_dtype dtype, kda_gate gate, float l2_eps,
                                           kda_stream_t stream);

/* Launch flags of kda_shortconv_decode_step_ex. */
enum { KDA_DECODE_OVERLAP_PREV = 1 };

/*
 * kda_shortconv_decode_step_gated with launch flags (same arguments, layouts,
 * requirements and errors; flags = 0 is that call). With
 * KDA_DECODE_OVERLAP_PREV the caller promises that the kernel enqueued on
 * `stream` just before this call does not write this call's `state` (for
 * instance, it is the decode step of another layer). The launch may then
 * start while that kernel drains (programmatic dependent launch) and stream
 * its state meanwhile. It reads x, ring, g and beta, and writes anything,
 * only after that kernel has completed. Launch shapes that have no tail to
 * overlap ignore the flag. Unknown flag bits are KDA_ERR_INVALID_ARG.
 */
kda_status kda_shortconv_decode_step_ex(const void *x, void *ring, const float *w, const float *g,
                                        const float *beta, float *state, void *out, int B, int H, int D,
                                        kda_dtype dtype, kda_gate gate, float l2_eps, unsigned flags,
                                        kda_stream_t stream);

/*
 * Output epilogue of a layer: gated RMSNorm of the attention output, per
 * (token, head) row of D value channels. [W] "相关源码与文档导航" names a
 * gated RMSNorm among the KDA kernel's parts and [G] section 6 (the Gated
 * DeltaNet figure) an output gate that scales the features; neither prints a
 * formula, and this is the plainest reading:
 *
 *   y[t,h,j] = o[t,h,j] / sqrt(mean_j' o[t,h,j']^2 + eps) * weight[j]
 *              * act(gate[t,h,j])
 *
 * A row whose mean square plus eps is exactly zero gives zeros.
 *   o, gate, y [T,H,D] dtype (o: the output of a decode step, T = B, or of a
 *   prefill); weight [D] fp32, shared by the heads. y may alias o or gate
 *   (each element is read before it is written by the same thread).
 * Requires T >= 0, H >= 1, D in {16,32,64,128}, eps >= 0. T = 0 is a no-op.
 */
kda_status kda_gated_rmsnorm(const void *o, const void *gate, const float *weight, void *y, int64_t T,
                             int H, int D, kda_dtype dtype, kda_gate_act act, float eps,
                             kda_stream_t stream);

/*
 * Fused short conv + decode step with the output epilogue of
 * kda_gated_rmsnorm applied before the output is stored, in one launch ([W]
 * "KDA 递推公式先衰减再差分" for the step, [W] "相关源码与文档导航" and [G]
 * section 6 for the gated RMSNorm; the reading of kda_gated_rmsnorm):
 *
 *   y[b,h,j] = o[b,h,j] / sqrt(mean_j' o[b,h,j']^2 + norm_eps)
 *              * norm_weight[j] * act(out_gate[b,h,j])
 *
 * where o is the decode step's attention output, kept in fp32 inside the
 * kernel (never rounded to `dtype` nor written to memory). The state and
 * the ring are updated exactly as by kda_shortconv_decode_step_ex.
 *   x, ring, w, g, beta, state: as kda_shortconv_decode_step_gated
 *   out_gate [B,H,D] dtype: the output gate's pre-activation for this token
 *   norm_weight [D] fp32, shared by the heads
 *   y [B,H,D] dtype: receives the epilogue's result; it may not alias x,
 *   ring, state or out_gate
 * flags as kda_shortconv_decode_step_ex (with KDA_DECODE_OVERLAP_PREV the
 * gate too is read only after the previous kernel has completed).
 * Requires act KDA_ACT_SIGMOID or KDA_ACT_SILU and norm_eps >= 0; other
 * requirements and errors as kda_shortconv_decode_step_ex. B = 0 is a no-op.
 */
kda_status kda_shortconv_decode_step_epi(const void *x, void *ring, const float *w, const float *g,
                                         const float *beta, float *state, const void *out_gate,
                                         const float *norm_weight, void *y, int B, int H, int D,
                                         kda_dtype dtype, kda_gate gate, kda_gate_act act, float l2_eps,
                                         float norm_eps, unsigned flags, kda_stream_t stream);

/*
 * Chunked prefill of ONE sequence of T tokens, split into `segments` runs of
 * whole chunks that are processed side by side ([G] section 5: each chunk
 * step is affine in the state, S <- A S + B with A acting on the key axis,
 * and so is a run of them, and so is every readout o_t = S_t^T q_t). Two
 * passes of the ordinary prefill over the segments: from zero states (their
 * B, and the outputs without the carried state's part) and from identity
 * states with v read as zero (their A, and the outputs A_t^T q_t that carry
 * that part); then a serial fp32 scan S_{p+1} = A_p S_p + B_p gives the
 * state at every segment start and the final state, and one product per
 * segment and head adds (A_t^T q_t)^T S_p to every output. The result equals
 * kda_chunk_prefill_gated on the whole sequence up to rounding. It pays when
 * the sequence is long and H is small, so that the serial chunk chain leaves
 * most SMs idle. segments = 0 picks floor(SMs / H) (at least 2): one pass
 * over the segments then fills the GPU once.
 *
 *   q, k, v, out [T,H,D] dtype; g [T,H,D] / [T,H] / unused per `gate`;
 *   beta [T,H] fp32; initial_state [H,D,D] fp32 or NULL (zeros);
 *   final_state [H,D,D] fp32 or NULL.
 *   workspace: kda_chunk_prefill_scan_workspace_bytes(T, H, D, C, segments)
 *   bytes of device memory, 16-byte aligned: four fp32 states per segment and
 *   head and one [T,H,D] output buffer (sized for fp32; with segments = 0 the
 *   size is that of the current device's choice).
 * segments in 0..4096; segments = 1, T = 0 or T <= C run the ordinary
 * prefill (no workspace needed). Other requirements and errors as
 * kda_chunk_prefill_gated.
 */
size_t kda_chunk_prefill_scan_workspace_bytes(int64_t T, int H, int D, int C, int segments);
kda_status kda_chunk_prefill_scan(const void *q, const void *k, const void *v, const float *g,
                                  const float *beta, const float *initial_state, float *final_state,
                                  void *out, int64_t T, int H, int D, int C, kda_dtype dtype, kda_gate gate,
                                  float l2_eps, int segments, void *workspace, size_t workspace_bytes,
                                  kda_stream_t stream);

/*
 * kda_chunk_prefill_gated followed by the output epilogue of
 * kda_gated_rmsnorm on its output, in one call: out receives
 *   RMSNorm(o) * norm_weight * act(out_gate)
 * per (token, head) row, o being the attention output: the prefill, then
 * the epilogue kernel in place over out (run inside the tensor-core prefill
 * kernel instead, it was slower). out_gate [T,H,D] dtype, norm_weight [D]
 * fp32 (16-byte aligned);
 * out_gate may not alias out, q, k or v. Other arguments and errors as
 * kda_chunk_prefill_gated and kda_gated_rmsnorm.
 */
kda_status kda_chunk_prefill_epi(const void *q, const void *k, const void *v, const float *g,
                                 const float *beta, const float *initial_state, float *final_state,
                                 void *out, const int64_t *cu_seqlens, int N, int64_t T, int H, int D,
                                 int C, kda_dtype dtype, kda_gate gate, float l2_eps, const void *out_gate,
                                 const float *norm_weight, kda_gate_act act, float norm_eps,
                                 void *workspace, size_t workspace_bytes, kda_stream_t stream);

/* Chunked prefill of a packed batch in which some sequences are long
 * ("为什么 Kimi K3 敢把 KV Cache 扔掉？" section 5, the chunk-to-chunk state
 * hand-off, which is affine in the state: the same scan as
 * kda_chunk_prefill_scan, applied per sequence). The host-side lengths let
 * the call plan the split without a device round trip:
 * kda_chunk_prefill_split_plan gives each sequence its segment count.
 *   - A sequence is split when its serial chain of chunks is longer than
 *     the batch's work per SM would be with every chunk-head spread evenly
 *     (and than 8 chunks), into P = min(chunks / that balance, 4096)
 *     segments when P >= 4. Sequences are never split when H is not a
 *     multiple of 4. When some sequences stay whole, P is capped at
 *     (SMs - whole sequences x H) / H if that is still >= 4, so that the
 *     whole sequences' CTAs find SMs of their own beside the first split
 *     sequence's passes.
 *   - The sequences kept whole run in one prefill launch, longest first, on
 *     an internal side stream forked from `stream` by an event; each split
 *     one runs through kda_chunk_prefill_scan over its own rows, with its own
 *     initial and final state, on `stream`, which then waits for the side
 *     stream. The side stream and its two events are created on the first
 *     such call on a device and kept for the process (make that first call
 *     outside a stream capture); the enqueueing is serialised across host
 *     threads. The call can be captured into a CUDA graph: the launch order
 *     travels in kernel parameters, and fork and join are events.
 *   - With nothing to split this is kda_chunk_prefill_gated.
 * Arguments as kda_chunk_prefill_gated, plus host_cu_seqlens: a host copy of
 * cu_seqlens (both required; they must agree, which is not checked on the
 * device side). The results equal kda_chunk_prefill_gated's up to rounding.
 *   workspace  device buffer of kda_chunk_prefill_split_workspace_bytes(
 *              host_cu_seqlens, N, H, D, C) bytes.
 * The split uses the current device's SM count; plan, workspace and call
 * must see the same device. Errors: KDA_ERR_INVALID_ARG for bad lengths
 * (host_cu_seqlens[0] != 0, decreasing, host_cu_seqlens[N] != T) or a short
 * workspace, the callees' errors otherwise. */
kda_status kda_chunk_prefill_split(const void *q, const void *k, const void *v, const float *g,
                                   const float *beta, const float *initial_state, float *final_state,
                                   void *out, const int64_t *cu_seqlens, const int64_t *host_cu_seqlens,
                                   int N, int64_t T, int H, int D, int C, kda_dtype dtype, kda_gate gate,
                                   float l2_eps, void *workspace, size_t workspace_bytes, kda_stream_t stream);

/* Workspace bytes kda_chunk_prefill_split needs (0 for invalid lengths). */
size_t kda_chunk_prefill_split_workspace_bytes(const int64_t *host_cu_seqlens, int N, int H, int D, int C);

/* The split kda_chunk_prefill_split makes: segments[i] = the segment count of
 * sequence i (1: kept whole). sms: the SM count to plan for, or <= 0 for the
 * current device's (then no GPU means no split). Returns the number of split
 * sequences, or -1 for invalid lengths. Needs no GPU. */
int kda_chunk_prefill_split_plan(const int64_t *host_cu_seqlens, int N, int H, int C, int sms, int *segments);

/* Name of the kernel kda_chunk_prefill (and the gated, epilogue and scan
 * entry points, per segment) runs for head dimension D, chunk size C and
 * dtype: "prefill_tc_pipe_kernel" (tcgen05, bf16), "prefill_tf32_kernel"
 * (tcgen05 kind::tf32, fp32), "prefill_f32_kernel" (CUDA cores, D = 128) or
 * "prefill_simt_kernel" (CUDA cores, any shape). A static string; NULL when
 * D, C or dtype is not one kda_chunk_prefill accepts. Needs no GPU. */
const char *kda_chunk_prefill_route(int D, int C, kda_dtype dtype);

/* Workspace bytes kda_chunk_prefill needs for these sizes (may be 0). */
size_t kda_chunk_prefill_workspace_bytes(int64_t total_tokens, int num_seqs, int H, int D, int C);

/*
 * Chunked prefill over a packed batch of N sequences ([G] section 5: inside
 * a chunk of C tokens the work is attention-like, the state is handed from
 * chunk to chunk; the result equals the token recurrence of
 * kda_decode_step applied to every token in order).
 *
 *   q, k, v [T,H,D] dtype;  g [T,H,D] fp32;  beta [T,H] fp32
 *   initial_state [N,H,D,D] fp32 or NULL (zeros)
 *   final_state   [N,H,D,D] fp32 or NULL (not written); may equal
 *                 initial_state (read before written per (sequence, head))
 *   out           [T,H,D] dtype
 *   cu_seqlens    device int64 [N+1], cu_seqlens[0] = 0, non-decreasing,
 *                 cu_seqlens[N] = T; or NULL for one sequence of T tokens
 *                 (then N must be 1). Chunks never straddle sequences; a
 *                 sequence's last chunk may be short; empty sequences pass
 *                 their initial state through.
 *   C             chunk size: 1..64. The kernel each shape runs on is what
 *                 kda_chunk_prefill_route names: bf16 with D = 128 or 64 and
 *                 C = 16, 32 or 64 takes the bf16 tensor-core kernel, which
 *                 always works in 64-token chunks (the chunked form is an exact
 *                 rewrite of the recurrence, so the chunk length changes only
 *                 the rounding); fp32 with D = 128 and C >= 16 the tf32
 *                 tensor-core kernel; other D = 128 shapes a register-tiled
 *                 CUDA-core kernel; the rest the general CUDA-core kernel
 *   workspace     device buffer of at least
 *                 kda_chunk_prefill_workspace_bytes(T, N, H, D, C) bytes
 *                 (NULL allowed when that is 0); contents are scratch. For
 *                 one sequence (N = 1) whose serial chunk chain would leave
 *                 most SMs idle (floor(SMs / H) >= 4 and at least 8 chunks
 *                 per segment), that size makes room for the automatic split
 *                 of kda_chunk_prefill_scan, which the call then uses when
 *                 cu_seqlens is NULL; with a smaller workspace (or NULL) the
 *                 same call runs the serial prefill. The size depends on the
 *                 current device.
 * Invalid cu_seqlens contents are found on the device: the affected
 * sequences are skipped and kda_sync_status() reports KDA_ERR_DEVICE_CHECK.
 */
kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const float *initial_state, float *final_state,
                             void *out, const int64_t *cu_seqlens, int N, int64_t T, int H,
                             int D, int C, kda_dtype dtype, float l2_eps, void *workspace,
                             size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_prefill with the gate form chosen by `gate`: g is [T,H,D] for
 * KDA_GATE_CHANNEL, [T,H] for KDA_GATE_HEAD, and unused (may be NULL) for
 * KDA_GATE_NONE. kda_chunk_prefill is this call with KDA_GATE_CHANNEL. The
 * tensor-core path specialises on the gate form: a per-head gate is read as
 * one float per token-head and scanned once per chunk, and no gate skips
 * the decay factors altogether.
 */
kda_status kda_chunk_prefill_gated(const void *q, const void *k, const void *v, const float *g,
                                   const float *beta, const float *initial_state, float *final_state,
                                   void *out, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                   int D, int C, kda_dtype dtype, kda_gate gate, float l2_eps,
                                   void *workspace, size_t workspace_bytes, kda_stream_t stream);

/*
 * kda_chunk_prefill for callers that cannot allocate device memory. The pages
 * have no counterpart: this is a convenience of the library, not part of the
 * method.
 *
 * kda_chunk_prefill needs a small workspace for a mixed-length batch: the
 * longest-first launch order, one int32 per sequence. Some callers cannot call
 * cudaMalloc when they run the prefill. Examples are code inside another
 * framework's allocator or memory-pool callback, where a nested allocation
 * would deadlock or fragment the pool, and serving paths whose policy forbids
 * allocation per request. This entry point takes no workspace. It keeps that
 * order in a fixed array in device memory that the library owns: 16 KiB per
 * GPU, held from the first use until the process exits.
 *
 * Arguments, layouts and results are those of kda_chunk_prefill.
 * Limit: N <= 4096 sequences; a larger N returns KDA_ERR_INVALID_ARG (use
 * kda_chunk_prefill with a workspace instead).
 * The first call on a device looks up the array's device address (once per
 * device, with that device current), so make that first call before any
 * stream capture. The address is kept with the CUDA context it belongs to: if
 * the device's primary context is rebuilt (cudaDeviceReset), the next call
 * looks it up again, so that call too should come before any capture. Every call on a device shares the array, which keeps the
 * previous call's contents. Nothing in it needs clearing, because each call
 * rewrites every entry it reads. Calls that may overlap on the GPU (different
 * streams, no ordering between them) race on the array and must not be issued.
 */
kda_status kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v, const float *g,
                                     const float *beta, const float *initial_state, float *final_state,
                                     void *out, const int64_t *cu_seqlens, int N, int64_t T, int H, int D,
                                     int C, kda_dtype dtype, float l2_eps, kda_stream_t stream);

/* Synchronise `stream`, then report (and clear) any device-side error flag
 * raised by earlier calls on the stream's device: KDA_ERR_DEVICE_CHECK,
 * KDA_ERR_TIMEOUT, KDA_ERR_CUDA for an asynchronous CUDA error, else KDA_OK. */
kda_status kda_sync_status(kda_stream_t stream);

/*
 * Diagnostic of the failure reporting, not part of the method. Launches one
 * CTA whose thread 0 waits on a shared-memory mbarrier that nothing ever
 * completes, with the same clock-bounded wait the tensor-core kernels use,
 * limited to `limit_cycles` SM clock cycles (1 .. 2e9). The wait gives up,
 * sets the device error word and the kernel returns, so the next
 * kda_sync_status on the stream reports KDA_ERR_TIMEOUT and the context
 * stays usable. Lets a caller check, on its own GPU, that an expired wait
 * is reported instead of hanging.
 */
kda_status kda_selftest_bounded_wait(long long limit_cycles, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
