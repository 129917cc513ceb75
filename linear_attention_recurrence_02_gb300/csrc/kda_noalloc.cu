// kda_noalloc.cu -- chunked prefill for callers that cannot allocate.
//
// kda_chunk_prefill asks the caller for a small workspace: the longest-first
// launch order of a mixed-length batch, one int32 per sequence. Some callers
// have no way to provide it. One example is code that runs inside another
// framework's allocator or memory-pool callback, where a nested cudaMalloc
// would deadlock or fragment the pool. Another is a latency-critical serving
// path whose policy forbids allocation per request.
//
// This file holds the scratch for those callers in a fixed-size device
// array. Every GPU that loads the library keeps the array until the process
// exits. The entry point below passes the array's device address as the
// workspace of the ordinary prefill, so the computation is identical to
// kda_chunk_prefill with a caller-provided workspace.
#include <string>

#include "kda_common.cuh"

// Launch-order scratch for up to KDA_NOALLOC_MAX_SEQS sequences (16 KiB).
#define KDA_NOALLOC_MAX_SEQS 4096
static __device__ __align__(256) int g_noalloc_order[KDA_NOALLOC_MAX_SEQS];

namespace kda {

// The symbol's device address on the current device. In host code
// `g_noalloc_order` is only a host-side stand-in, so the kernel must be given
// this address, never the name. It is looked up on a device's first call and
// again whenever the device's context has changed since (a cudaDeviceReset
// rebuilds the primary context, and the array moves with it).
static kda_status noalloc_scratch(void **out) {
    static SymbolCache cache;
    return symbol_address(&g_noalloc_order, cache, out);
}

}  // namespace kda

using namespace kda;

extern "C" kda_status kda_chunk_prefill_noalloc(const void *q, const void *k, const void *v, const float *g,
                                                const float *beta, const float *initial_state, float *final_state,
                                                void *out, const int64_t *cu_seqlens, int N, int64_t T, int H,
                                                int D, int C, kda_dtype dtype, float l2_eps, kda_stream_t stream) {
    clear_detail();
    if (N > KDA_NOALLOC_MAX_SEQS)
        return invalid("N exceeds the allocation-free maximum of " + std::to_string(KDA_NOALLOC_MAX_SEQS) +
                       " sequences; use kda_chunk_prefill with a workspace");
    // only the launch order of a mixed-length batch lives in the static array
    // (a single sequence needs none and then runs the serial prefill)
    const size_t need = N >= 2 ? kda_chunk_prefill_workspace_bytes(T, N, H, D, C) : 0;
    void *ws = nullptr;
    if (need > 0) {
        kda_status st = bind_stream_device(stream);
        if (st != KDA_OK) return st;
        if ((st = noalloc_scratch(&ws))) return st;
        if (need > sizeof(g_noalloc_order)) return invalid("workspace need exceeds the static scratch");
    }
    // The order kernel writes every one of the N entries it uses, so nothing
    // left by an earlier call needs clearing.
    return kda_chunk_prefill(q, k, v, g, beta, initial_state, final_state, out, cu_seqlens, N, T, H, D, C, dtype,
                             l2_eps, ws, ws ? need : 0, stream);
}
