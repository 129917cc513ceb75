// kda_prefill.cu -- chunked prefill (placeholder until the kernels land).
#include "kda_common.cuh"

using namespace kda;

extern "C" size_t kda_chunk_prefill_workspace_bytes(int64_t, int, int, int, int) { return 0; }

extern "C" kda_status kda_chunk_prefill(const void *, const void *, const void *, const float *, const float *,
                                        const float *, float *, void *, const int64_t *, int, int64_t, int, int,
                                        int, kda_dtype, float, void *, size_t, kda_stream_t) {
    clear_detail();
    return fail(KDA_ERR_UNSUPPORTED, "chunked prefill not built yet");
}
