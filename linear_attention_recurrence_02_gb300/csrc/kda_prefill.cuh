// kda_prefill.cuh -- internal interface between the prefill entry point and
// its kernels (CUDA-core general path, tensor-core bf16 path).
#pragma once

#include <cuda.h>

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
    const int *order;  // sequences by descending length (device), or NULL = natural order
    int gate;          // kda_gate: g is [T,H,D], [T,H], or unused
    bool v_zero = false;  // read v as all zeros (v is not loaded)
    int nlaunch = 0;      // sequences launched (order[0..nlaunch) when set; 0: all N)
};

// (sequence, head) CTAs per head of a prefill launch
inline unsigned launch_seqs(const PrefillArgs &a) { return (unsigned)(a.nlaunch > 0 ? a.nlaunch : a.N); }

// Largest batch the length sort handles; bigger batches keep their order.
constexpr int ORDER_MAX_SEQS = 4096;

// Launch the length sort of the N sequences into `order` (int32 [N], device).
kda_status launch_prefill_order(const int64_t *cu_seqlens, int N, int *order, cudaStream_t s);

kda_status prefill_simt(const PrefillArgs &a, cudaStream_t s);
bool prefill_tc_applicable(const PrefillArgs &a);
kda_status prefill_tc(const PrefillArgs &a, cudaStream_t s);
bool prefill_f32_applicable(const PrefillArgs &a);
kda_status prefill_f32(const PrefillArgs &a, cudaStream_t s);
bool prefill_tf32_applicable(const PrefillArgs &a);
kda_status prefill_tf32(const PrefillArgs &a, cudaStream_t s);
// The kernel for these arguments: tensor cores (bf16, d = 128, C = 64), the
// register-tiled fp32 kernel (d = 128, any C), else the general CUDA-core one.
kda_status prefill_run(const PrefillArgs &a, cudaStream_t s);

// Segments of the automatic long-sequence split for one sequence of T tokens
// with H heads on the current device, or 0 when the serial prefill is kept.
// Streaming multiprocessors of the current device (0 if unknown).
int current_sms();
int prefill_auto_segments(int64_t T, int H, int C);

namespace tcp {
// 2-D tiled TMA map over a row-major [rows][inner] tensor of `elem`-byte
// elements with a box of box_inner x box_rows; false if the encoder fails.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t elem, uint64_t inner,
              uint64_t rows, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle sw);
}  // namespace tcp

// Validated [start, end) of sequence n; on invalid cu_seqlens sets the
// device error word and returns false (the caller skips the sequence).
__device__ __forceinline__ bool seq_range(const int64_t *cu, int n, int N, int64_t T, unsigned *err,
                                          int64_t &start, int64_t &end) {
    if (n < 0 || n >= N) {  // a launch-order entry that names no sequence
        if (err) atomicOr(err, DEVERR_SEQLENS);
        return false;
    }
    if (cu == nullptr) {
        start = 0;
        end = T;
        return true;
    }
    start = cu[n];
    end = cu[n + 1];
    const bool ok = start >= 0 && start <= end && end <= T && (n != 0 || start == 0) && (n != N - 1 || end == T);
    if (!ok && err) atomicOr(err, DEVERR_SEQLENS);
    return ok;
}

}  // namespace kda
