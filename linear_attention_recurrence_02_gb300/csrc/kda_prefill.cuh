// kda_prefill.cuh -- internal interface between the prefill entry point and
// its kernels (CUDA-core general path, tensor-core bf16 path).
#pragma once

#include "kda_common.cuh"

namespace kda {

struct PrefillArgs {
    const void *q, *k, *v;
    const float *g, *beta;
    const float *s_init;
    float *s_final;
    void *out;
    const int64_t *cu_seqlens;
    int N;
    int64_t T;
    int H, D, C;
    bool bf16;
    float eps;
    void *workspace;
    size_t workspace_bytes;
    unsigned *err;
};

kda_status prefill_simt(const PrefillArgs &a, cudaStream_t s);

}  // namespace kda
