// kda_prefill_tc.cu -- chunked KDA prefill on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA) for bf16 q/k/v, d_k = d_v = 128 or 64 (the
// latter as zero channels of the 128-channel layout), in chunks of 64 tokens
// (a requested C of 16 or 32 runs the same 64-token algebra).
//
// Method: the chunk algebra of the general kernel (kda_prefill.cu; "为什么 Kimi
// K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化", section 5: attention-
// like work inside a chunk, state hand-off between chunks; section 6:
// cumulative decay as a product of gates; the WY/UT reparameterisation it
// names is realised here as T = (I + A)^-1 Diag(beta)). With G the
// cumulative log decay inside the chunk and a per-channel anchor c:
//   Lk = e^{G-c} k^,  Lq = e^{G-c} q^,  Rk = e^{c-G} k^,  S~ = Diag(e^c) S
//   [A_raw; P_raw] = [Lk; Lq] Rk^T            (G1)   A = mask_<(beta A_raw)
//   T = (I + A)^-1 Diag(beta)                  (CUDA cores, fp32, and tf32 mma.sync merges)
//   W' = T Lk,  U0 = T V                       (G2, G3)
//   U = U0 - W' S~                             (G4)
//   O = Lq S~ + P U                            (G5, G6)
//   S <- Diag(e^{G_L}) S + Kb^T U,  Kb = e^{G_L-G} k^ = Diag(e^{G_L-c}) Rk
// Lk S~ = Diag-folded e^G k^ S, so W' S~ = T Kt S and Lq S~ = Qt S exactly.
// The state is held as S = Diag(sigma) S_st with sigma = e^{G_L-c} of the
// chunk that wrote it, so the update needs no Kb tile:
//   S_st <- Diag(e^c sigma_old) S_st + Rk^T U  (G7),  S~ = Diag(e^c sigma_old) S_st
// c = min(0, G_L + 40) keeps every factor and 1/sigma inside e^[-40, 40]
// whenever the chunk's decay span G_0 - G_L is at most 80; a chunk beyond that
// computes A and P with exact pairwise exponentials on CUDA cores, uses c = 0
// and Kb in place of Rk, and resets sigma to 1.
//
// Layout: every MMA has M = 128 on a channel axis, so TMEM lane = channel
// (key channel i or value channel j) throughout, and the fp32 state S_st^T
// (lane j, column i) never leaves TMEM between chunks. Operands are bf16 in
// 128-byte-swizzled shared memory tiles, loaded by TMA (q, k, v, g) or
// written by the CUDA cores from TMEM read-backs; S~^T and U^T go back to
// TMEM as bf16 pairs and feed G4-G7 as the A operand. TMA drops k and q into
// one 128-row tile that becomes [Lk; Lq] in place; W' is later read back over
// its dead Lk rows, transposed: channel-major, so that each thread stores
// its own 128-byte row, and G4 takes it as an MN-major operand.
//
// One CTA (512 threads) per (sequence, head) walks the chunks of its
// sequence with three warp groups: eight "front" warps build the operand
// tiles of chunk c + 2, four "back" warps run the MMAs and the solve of chunk
// c + 1, and four "chain" warps run the state chain of chunk c (see the
// pipelined kernel below). Every wait is bounded.
#include <cuda.h>

#include <atomic>
#include <cstring>
#include <string>

#include "kda_common.cuh"
#include "kda_prefill.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace tcp {

using namespace tc;

constexpr int C = 64, D = 128;
constexpr int LDB = 20, BLK = 16 * LDB;  // solve scratch: block row stride (bank-conflict free A fragments), block size
constexpr uint32_t QK_BYTES = 2 * 16384, G_BYTES = 32768, V_BYTES = 16384;
constexpr long long WAIT_LIMIT = 4000000000LL;  // clock cycles (about 2 s)
// Anchored factors stay within e^[-ANCHOR, ANCHOR] when the chunk's decay
// span is at most SPAN_MAX; the fp32 state kept as S / sigma then stays
// below e^ANCHOR times |S|.
constexpr float ANCHOR = 40.f, SPAN_MAX = 2.f * ANCHOR;

constexpr uint32_t ID_KK64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_MK64 = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, 0, 1);
constexpr uint32_t ID_KM64 = idesc_bf16(128, 64, 0, 1);

// byte offset of 16-byte chunk cc (channels 8cc..8cc+7) of `row` in a
// 128-byte-swizzled tile whose 64-channel blocks hold `rows` rows each
__device__ __forceinline__ uint32_t swz(int row, int cc, int rows) {
    return (uint32_t)((cc >> 3) * rows * 128 + row * 128 + (((cc & 7) ^ (row & 7)) << 4));
}
// float index of the 4-float group k4 (0..15) of row r in a 64 x 64 fp32
// matrix whose 16-byte groups are XOR-swizzled by the row (bank-conflict free
// for 16-byte accesses by consecutive rows)
__device__ __forceinline__ int fsw(int r, int k4) { return r * 64 + ((k4 ^ (r & 7)) << 2); }

constexpr float LOG2E = 1.4426950408889634f;
// 2^x on the special-function unit (inputs here are within +-128)
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// barrier over the first `n` threads of the CTA only (id > 0)
__device__ __forceinline__ void named_bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// fp32 -> tf32 operand: round to nearest (ties away from zero) on the 10-bit
// mantissa by adding half an ulp of tf32 to the bit pattern and truncating
__device__ __forceinline__ uint32_t to_tf32(float x) { return (__float_as_uint(x) + 0x1000u) & 0xffffe000u; }
// warp-level D(16x8) += A(16x8, row) * B(8x8, col) on tf32 inputs, fp32 accumulate
__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                 "{%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// C fragments c[nt] of a 16 x 16 tile (rows g, g+8; columns 8nt + 2tg, +1) ->
// tf32 B fragments b[kk][nt] (rows 8kk + tg, 8kk + tg + 4; column 8nt + g)
__device__ __forceinline__ void c_to_b(const float (&c)[2][4], uint32_t (&b)[2][2][2], int lane) {
    const int g = lane >> 2, tg = lane & 3;
    const int src0 = 4 * tg + (g >> 1), src1 = src0 + 16;
    const bool odd = g & 1;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float e0 = __shfl_sync(0xffffffffu, c[nt][2 * kk], src0);
            const float o0 = __shfl_sync(0xffffffffu, c[nt][2 * kk + 1], src0);
            const float e1 = __shfl_sync(0xffffffffu, c[nt][2 * kk], src1);
            const float o1 = __shfl_sync(0xffffffffu, c[nt][2 * kk + 1], src1);
            b[kk][nt][0] = to_tf32(odd ? o0 : e0);
            b[kk][nt][1] = to_tf32(odd ? o1 : e1);
        }
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



// ------------------------------------------------- MMA groups, issued by one elected lane
// Each helper is called by a whole warp (warp-uniform control flow). One lane,
// chosen by elect.sync, issues the group's MMAs and commits them to `bar`;
// the shared-memory descriptors of the later K steps are the first ones plus
// immediate offsets (the start-address field counts 16-byte units, and every
// tile here lies below 256 KB, so the additions never carry out of it).
// Issuing from a divergent `if (tid == 0)` with per-call descriptor
// arithmetic cost about 100 cycles per MMA on a busy SM; this form about 60.

// 8 MMAs over K = 128 (two 64-channel blocks of four 16-wide steps), A and B
// K-major in shared memory, blocks ABLK / BBLK bytes apart; the first step
// accumulates when `acc` is nonzero.
template <uint32_t ABLK, uint32_t BBLK>
__device__ __forceinline__ void mma8_ss(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc,
                                        uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred p, a0, t;\n\t.reg .b64 x1, x2, x3, x4, x5, x6, x7, y1, y2, y3, y4, y5, y6, y7;\n\t"
        "setp.ne.u32 a0, %4, 0;\n\tsetp.eq.u32 t, 0, 0;\n\t"
        "add.s64 x1, %1, 2;\n\tadd.s64 x2, %1, 4;\n\tadd.s64 x3, %1, 6;\n\t"
        "add.s64 x4, %1, %6;\n\tadd.s64 x5, %1, %7;\n\tadd.s64 x6, %1, %8;\n\tadd.s64 x7, %1, %9;\n\t"
        "add.s64 y1, %2, 2;\n\tadd.s64 y2, %2, 4;\n\tadd.s64 y3, %2, 6;\n\t"
        "add.s64 y4, %2, %10;\n\tadd.s64 y5, %2, %11;\n\tadd.s64 y6, %2, %12;\n\tadd.s64 y7, %2, %13;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, a0;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x1, y1, %3, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x2, y2, %3, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x3, y3, %3, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x4, y4, %3, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x5, y5, %3, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x6, y6, %3, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x7, y7, %3, t;\n\t"
        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}\n" ::"r"(d),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc), "r"(smem_u32(bar)), "n"(ABLK / 16), "n"(ABLK / 16 + 2),
        "n"(ABLK / 16 + 4), "n"(ABLK / 16 + 6), "n"(BBLK / 16), "n"(BBLK / 16 + 2), "n"(BBLK / 16 + 4),
        "n"(BBLK / 16 + 6)
        : "memory");
}

// Two interleaved groups of four MMAs over K = 64 sharing the B operand
// (K-major, steps 32 bytes apart): D1 = A1 B^T, D2 = A2 B^T with A1, A2
// MN-major, K steps 2048 bytes apart (G2 and G3).
__device__ __forceinline__ void mma44_ss(uint32_t d1, uint64_t a1, uint32_t d2, uint64_t a2, uint64_t bd,
                                         uint32_t idesc, uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred p, f, t;\n\t.reg .b64 x1, x2, x3, z1, z2, z3, y1, y2, y3;\n\t"
        "setp.ne.u32 f, 0, 0;\n\tsetp.eq.u32 t, 0, 0;\n\t"
        "add.s64 x1, %1, 128;\n\tadd.s64 x2, %1, 256;\n\tadd.s64 x3, %1, 384;\n\t"
        "add.s64 z1, %3, 128;\n\tadd.s64 z2, %3, 256;\n\tadd.s64 z3, %3, 384;\n\t"
        "add.s64 y1, %4, 2;\n\tadd.s64 y2, %4, 4;\n\tadd.s64 y3, %4, 6;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %4, %5, f;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%2], %3, %4, %5, f;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x1, y1, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%2], z1, y1, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x2, y2, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%2], z2, y2, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], x3, y3, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%2], z3, y3, %5, t;\n\t"
        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}\n" ::"r"(d1),
        "l"(a1), "r"(d2), "l"(a2), "l"(bd), "r"(idesc), "r"(smem_u32(bar))
        : "memory");
}

// G4 and G5: two interleaved groups of eight MMAs over K = 128 with the same A
// in TMEM (8 columns per K step): D1 = A B1^T with B1 MN-major (K rows of 128
// bytes, 16 per step, 64 rows per piece, pieces 16 KB apart), D2 = A B2^T
// with B2 K-major (steps 32 bytes apart, 64-channel blocks 16 KB apart).
__device__ __forceinline__ void mma88_ts(uint32_t d1, uint64_t b1, uint32_t idesc1, uint32_t d2, uint64_t b2,
                                         uint32_t idesc2, uint32_t at, uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred p, f, t;\n\t.reg .b32 x1, x2, x3, x4, x5, x6, x7;\n\t"
        ".reg .b64 y1, y2, y3, y4, y5, y6, y7, z1, z2, z3, z4, z5, z6, z7;\n\t"
        "setp.ne.u32 f, 0, 0;\n\tsetp.eq.u32 t, 0, 0;\n\t"
        "add.u32 x1, %6, 8;\n\tadd.u32 x2, %6, 16;\n\tadd.u32 x3, %6, 24;\n\tadd.u32 x4, %6, 32;\n\t"
        "add.u32 x5, %6, 40;\n\tadd.u32 x6, %6, 48;\n\tadd.u32 x7, %6, 56;\n\t"
        "add.s64 y1, %1, 128;\n\tadd.s64 y2, %1, 256;\n\tadd.s64 y3, %1, 384;\n\t"
        "add.s64 y4, %1, 1024;\n\tadd.s64 y5, %1, 1152;\n\tadd.s64 y6, %1, 1280;\n\tadd.s64 y7, %1, 1408;\n\t"
        "add.s64 z1, %4, 2;\n\tadd.s64 z2, %4, 4;\n\tadd.s64 z3, %4, 6;\n\t"
        "add.s64 z4, %4, 1024;\n\tadd.s64 z5, %4, 1026;\n\tadd.s64 z6, %4, 1028;\n\tadd.s64 z7, %4, 1030;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %1, %2, f;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [%6], %4, %5, f;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x1], y1, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x1], z1, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x2], y2, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x2], z2, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x3], y3, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x3], z3, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x4], y4, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x4], z4, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x5], y5, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x5], z5, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x6], y6, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x6], z6, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x7], y7, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x7], z7, %5, t;\n\t"
        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}\n" ::"r"(d1),
        "l"(b1), "r"(idesc1), "r"(d2), "l"(b2), "r"(idesc2), "r"(at), "r"(smem_u32(bar))
        : "memory");
}

// Two interleaved groups of four accumulating MMAs over K = 64 with the same
// A in TMEM (8 columns per K step): D1 += A B1^T with B1 K-major (steps 32
// bytes apart), D2 += A B2^T with B2 MN-major (steps 2048 bytes apart) (G6, G7).
__device__ __forceinline__ void mma44_ts(uint32_t d1, uint64_t b1, uint32_t idesc1, uint32_t d2, uint64_t b2,
                                         uint32_t idesc2, uint32_t at, uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b32 x1, x2, x3;\n\t.reg .b64 y1, y2, y3, z1, z2, z3;\n\t"
        "setp.eq.u32 t, 0, 0;\n\t"
        "add.u32 x1, %6, 8;\n\tadd.u32 x2, %6, 16;\n\tadd.u32 x3, %6, 24;\n\t"
        "add.s64 y1, %1, 2;\n\tadd.s64 y2, %1, 4;\n\tadd.s64 y3, %1, 6;\n\t"
        "add.s64 z1, %4, 128;\n\tadd.s64 z2, %4, 256;\n\tadd.s64 z3, %4, 384;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %1, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [%6], %4, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x1], y1, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x1], z1, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x2], y2, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x2], z2, %5, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%0], [x3], y3, %2, t;\n\t"
        "@p tcgen05.mma.cta_group::1.kind::f16 [%3], [x3], z3, %5, t;\n\t"
        "@p tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}\n" ::"r"(d1),
        "l"(b1), "r"(idesc1), "r"(d2), "l"(b2), "r"(idesc2), "r"(at), "r"(smem_u32(bar))
        : "memory");
}

// ------------------------------------------------- the kernel
// Three warp groups work on three consecutive chunks at once:
//   front, warps 4-11: chunk c + 2's norms, cumulative decay, anchors and the
//     operand tiles [Lk; Lq] and Rk (everything that needs no MMA);
//   back, warps 0-3: chunk c + 1's G1, A/P read-back, the solve for T, G2/G3
//     and the W' read-back;
//   chain, warps 12-15: the state chain of chunk c (S~ conversion, G4/G5, U,
//     G6/G7, output).
// The hand-offs are mbarriers in shared memory:
//   fr[b]     front -> back: operand tiles of chunk parity b built (with the
//             per-channel gate the chain waits on it too: the S~ factors)
//   ready[b]  back -> chain: chunk of parity b fully prepared
//   c45[b]    G4/G5 of chunk parity b done (tcgen05.commit): its W' / Lq
//             tile may be reloaded; the chain itself then issues the q/k
//             loads of the chunk two ahead into it
//   ofree[b]  chain -> front, right after G6/G7 of chunk parity b: U0[b],
//             Rk[b], P[b] and the per-chunk factors may be reused (the back
//             warps, which reach them only through fr[b], are done too). The
//             output is staged in its own tile, which the chain rewrites
//             once the bulk store of the chunk before has read it.
// Code size: the three groups run three different loop bodies at once, so the
// outer loops of the read-backs, the conversions and the operand build are
// kept rolled (`#pragma unroll 1`). Fully unrolled, instruction-fetch stalls
// grew fourfold once every SM was busy and a 152-head launch ran 30% slower.
namespace pipe {
constexpr int NTP = 512;
// Register split between the warp groups (setmaxnreg, one value per warpgroup):
// the two front warpgroups shrink to FRONT_REGS, the back and chain warpgroups
// grow to BACK_REGS and CHAIN_REGS. The shares must add up to exactly what the
// CTA was launched with, 4 BACK + 8 FRONT + 4 CHAIN = 16 R (R = registers per
// thread at launch, 128 for 512 threads), or a grow would wait for registers
// that never come; the host checks this before launching. The per-channel
// gate's chain needs fewer registers than the others' (its S~ factors are
// vectors read from shared memory), so its back warps get more.
template <int GM> struct Regs {
    static constexpr int BACK = GM == KDA_GATE_CHANNEL ? 168 : 160;
    static constexpr int FRONT = 104;
    static constexpr int CHAIN = GM == KDA_GATE_CHANNEL ? 136 : 144;
    static_assert(4 * BACK + 8 * FRONT + 4 * CHAIN == 16 * 128, "register split");
};
constexpr uint32_t X0 = 0;              // [k; q] -> [Lk; Lq], chunk parity 0 (32 KB); parity 1 at X0 + 32768
constexpr uint32_t V_ = 65536;          // v tile (16 KB): loaded for chunk c + 1 once G3 of chunk c is done
constexpr uint32_t OST = 81920;         // O staging of the chain's bulk output store (16 KB)
constexpr uint32_t G_ = 98304;          // g fp32 [64][128] -> G (log2 units) (32 KB)
constexpr uint32_t RK0 = 131072;        // Rk (Kb on the exact path) per parity (16 KB each)
constexpr uint32_t P0 = 163840;         // P per parity (8 KB each)
constexpr uint32_t T_ = 180224;         // T (8 KB)
constexpr uint32_t A_ = 188416;         // A fp32 (16 KB)
constexpr uint32_t DV = 204800;         // solve scratch: D_0..D_3, M_10, M_32 (7.5 KB)
constexpr uint32_t YV = 212992;         // solve scratch: Y blocks (5 KB)
constexpr uint32_t SMALL = 218112;      // per-row / per-channel vectors, barriers, counters (6 KB)
constexpr uint32_t SMEM = SMALL + 6144 + 1024;
// TMEM columns
constexpr uint32_t T_S = 0, T_SB = 128, T_X = 192, T_O = 256, T_U0 = 320, T_AP = 448;  // U0 parity b at 320 + 64 b
}  // namespace pipe

// Bounded wait that also gives up once the other warp group has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t *bar, uint32_t parity, volatile uint32_t *abort_flag) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > WAIT_LIMIT) {
            *abort_flag = 1u;
            return false;
        }
    }
    return true;
}
// OR of `pred` over the `n` threads of named barrier `id` (also a barrier).
__device__ __forceinline__ bool group_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

template <int GM>
__global__ void __launch_bounds__(pipe::NTP, 1)
    prefill_tc_pipe_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                           const __grid_constant__ CUtensorMap tm_o,
                           const float *__restrict__ g_head, const float *__restrict__ beta, const float *s_init,
                           float *s_final, __nv_bfloat16 *__restrict__ out, const int64_t *__restrict__ cu_seqlens,
                           int N, int64_t Ttot, int H, float eps, unsigned *err, const int *__restrict__ order,
                           int v_zero, int dg) {
    // dg: the head dimension in memory (128, or 64 with channels 64..127 zero-filled by the loads)
    using namespace pipe;
    constexpr bool GCH = GM == KDA_GATE_CHANNEL, GHD = GM == KDA_GATE_HEAD, GNO = GM == KDA_GATE_NONE;
    constexpr int BAR_CHAIN = 2, BAR_BACK = 3, BAR_FRONT = 4;
    constexpr int BAR_FRONT_N = 5, BAR_FRONT_S = 6;  // the front's norm half (ft < 128) and scan half
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base derived from the shared array itself (accesses compile to shared-memory instructions)
    uint8_t *sm = smem_raw + ((1024u - ((uint32_t)__cvta_generic_to_shared(smem_raw) & 1023u)) & 1023u);
    float *s_rq = reinterpret_cast<float *>(sm + SMALL);
    float *s_rk = s_rq + 64;
    float *s_beta = s_rk + 64;
    float *s_gl = s_beta + 128;     // G at the chunk's last row (natural log)
    float *s_c = s_gl + 128;        // anchor c
    float *s_g1 = s_c + 128;        // per-head gate: g per row, then G per row (log2 units)
    float *s_sigp = s_g1 + 64;      // sigma of the chunk prep finished last
    float *s_sf = s_sigp + 128;     // [2][128] S~ factor e^c sigma_old, per chunk parity
    float *s_pf = s_sf + 256;       // [2][128] rescale of the stored state before G7
    float *s_sig = s_pf + 256;      // [2][128] sigma after the chunk
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_sig + 256);
    uint64_t *bar_qk = bars;        // [2]
    uint64_t *bar_g = bars + 2;
    uint64_t *bar_v = bars + 3;
    uint64_t *bar_mp = bars + 5;    // prep MMA commits
    uint64_t *bar_c45 = bars + 6;   // [2]
    uint64_t *bar_c67 = bars + 8;
    uint64_t *bar_ready = bars + 9; // [2]
    uint64_t *bar_ofree = bars + 11;// [2]
    uint64_t *bar_fr = bars + 13;   // [2] front -> back: operand tiles of chunk parity b built
    volatile uint32_t *s_abort = reinterpret_cast<volatile uint32_t *>(bars + 15);
    uint32_t *s_taddr = reinterpret_cast<uint32_t *>(bars + 16);
    // TMA barriers qk0, qk1, g, v: phases armed and phases waited for, so that
    // an aborted launch can let every copy in flight land before exiting
    uint32_t *s_armed = reinterpret_cast<uint32_t *>(bars + 17);
    uint32_t *s_waited = s_armed + 5;
    uint32_t *s_exact = reinterpret_cast<uint32_t *>(bars + 22);  // [2] chunk parity b takes the exact path
    float *gt = reinterpret_cast<float *>(sm + G_);
    float *Am = reinterpret_cast<float *>(sm + A_);
    float *Dv = reinterpret_cast<float *>(sm + DV);
    float *Yv = reinterpret_cast<float *>(sm + YV);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q4 = warp & 3;
    const bool is_prep = tid < 384;  // back (warps 0-3) and front (warps 4-11)
    const int h = blockIdx.x % H, n = order ? order[blockIdx.x / H] : (int)(blockIdx.x / H);
    int64_t start, end;
    if (!seq_range(cu_seqlens, n, N, Ttot, err, start, end)) return;
    const int nchunks = (int)((end - start + C - 1) / C);

    auto issue_qk = [&](int y, int b) {
        uint8_t *xb = sm + X0 + 32768 * b;
        s_armed[b] += 1;
        mbar_arrive_expect_tx(bar_qk + b, QK_BYTES);
        tma_load_3d(xb, &tm_k, bar_qk + b, 0, h, y);
        tma_load_3d(xb + 16384, &tm_k, bar_qk + b, 64, h, y);
        tma_load_3d(xb + 8192, &tm_q, bar_qk + b, 0, h, y);
        tma_load_3d(xb + 24576, &tm_q, bar_qk + b, 64, h, y);
    };
    auto issue_g = [&](int y) {
        s_armed[2] += 1;
        mbar_arrive_expect_tx(bar_g, G_BYTES);
        tma_load_3d(sm + G_, &tm_g, bar_g, 0, h, y);
    };
    auto issue_v = [&](int y) {
        s_armed[3] += 1;
        if (v_zero) {  // nothing to load: release the tile; the back warps zero it
            mbar_arrive(bar_v);
            return;
        }
        mbar_arrive_expect_tx(bar_v, V_BYTES);
        tma_load_3d(sm + V_, &tm_v, bar_v, 0, h, y);
        tma_load_3d(sm + V_ + 8192, &tm_v, bar_v, 64, h, y);
    };

    if (tid == 0) {
        for (int i = 0; i < 15; ++i) mbar_init(bars + i, 1);
        for (int i = 0; i < 10; ++i) s_armed[i] = 0u;
        *s_abort = 0u;
        fence_mbar_init();
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        if constexpr (GCH) tma_prefetch_desc(&tm_g);
        if (nchunks > 0) {
            issue_qk((int)start, 0);
            if constexpr (GCH) issue_g((int)start);
            issue_v((int)start);
        }
        if (nchunks > 1) issue_qk((int)(start + C), 1);
    }
    if (tid < 128) s_sigp[tid] = 1.f;
    if (warp == 0) {
        tmem_alloc(s_taddr, 512);
        tmem_relinquish();
    }
    sync_tc();
    const uint32_t tbase = *s_taddr;
    const uint32_t lrow = (uint32_t)(32 * q4) << 16;  // this warp's TMEM lane quarter
    const uint32_t sbase = smem_u32(sm);
    const int jl = 32 * q4 + lane;                    // this thread's TMEM lane (channel)
    const size_t soff = ((size_t)n * H + h) * dg * dg;  // the state of this (sequence, head): [dg][dg]
    bool ok = true;

    if (is_prep) {
        if (tid >= 128) {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(Regs<GM>::FRONT));
            // ======================= front: warps 4-11 ======================
            // Chunk c: waits for its q/k (and g) tiles, norms, cumulative decay,
            // anchors and the operand tiles [Lk; Lq] and Rk, one chunk ahead of
            // the back warps; fr[c & 1] hands the chunk over.
            const int ft = tid - 128;  // 0..255
            float beta_reg = 0.f, gh_reg = 0.f;  // next chunk's beta / per-head gate, loaded one chunk ahead
            if (ft < C && start + ft < end) {
                beta_reg = beta[(size_t)(start + ft) * H + h];
                if constexpr (GHD) gh_reg = g_head[(size_t)(start + ft) * H + h];
            }
            for (int ci = 0; ci < nchunks; ++ci) {
                const int b = ci & 1;
                const int64_t c0 = start + (int64_t)ci * C;
                const int L = (int)((end - c0) < (int64_t)C ? (end - c0) : (int64_t)C);
                const bool has_next = ci + 1 < nchunks;
                uint8_t *xb = sm + X0 + 32768 * b;
                bool bad = false, got = true;
                float *sb = s_beta + 64 * b;
                if constexpr (GCH) {
                    // the decay scan needs only g, which comes on its own barrier well ahead: the scan half
                    // (ft >= 128) starts on it at once, while the norm half waits for q/k, computes the
                    // norms, and only then waits for ofree[b] (the chain is done with chunk ci - 2, hence
                    // the back warps too). One warp per half spins; the others wait in the half's named
                    // barrier at no issue cost.
                    if (ft < 128) {
                        if (ft < 32) got = wait_or_abort(bar_qk + b, (ci >> 1) & 1, s_abort);
                        got = !group_or(BAR_FRONT_N, 128, !got);
                        if (got) {
                            if (ft == 0) {
                                s_waited[b] += 1;
                                // the loads of chunk ci + 2 are issued one to two chunks from now,
                                // inside the pipeline's dependency cycle: stage their tiles in L2
                                if (ci + 2 < nchunks) {
                                    const int y2 = (int)(c0 + 2 * C);
                                    tma_prefetch_l2_3d(&tm_k, 0, h, y2);
                                    tma_prefetch_l2_3d(&tm_q, 0, h, y2);
                                    tma_prefetch_l2_3d(&tm_v, 0, h, y2);
                                    if (dg > 64) {
                                        tma_prefetch_l2_3d(&tm_k, 64, h, y2);
                                        tma_prefetch_l2_3d(&tm_q, 64, h, y2);
                                        tma_prefetch_l2_3d(&tm_v, 64, h, y2);
                                    }
                                    if constexpr (GCH) tma_prefetch_l2_3d(&tm_g, 0, h, y2);
                                }
                            }
                            if (ft < C) sb[ft] = beta_reg;
                            if (L < C) {  // rows past the end of the sequence contribute nothing
                                const uint4 z4 = make_uint4(0, 0, 0, 0);
                                for (int p = ft; p < (C - L) * 16; p += 128) {
                                    const int r = L + (p >> 4), cc = p & 15;
                                    *reinterpret_cast<uint4 *>(xb + swz(r, cc, 128)) = z4;
                                    *reinterpret_cast<uint4 *>(xb + swz(r + 64, cc, 128)) = z4;
                                }
                            }
                            named_bar_sync(BAR_FRONT_N, 128);
                            // L2 norm of one row (q rows for ft < 64, k rows after)
                            const int r = ft & 63;
                            const int row = ft < 64 ? r + 64 : r;  // q rows follow the k rows
                            float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                            for (int cc = 0; cc < 16; ++cc) {
                                float f[8];
                                unpack8(*reinterpret_cast<const uint4 *>(xb + swz(row, cc, 128)), f);
#pragma unroll
                                for (int e = 0; e < 8; ++e) ss[e & 3] = fmaf(f[e], f[e], ss[e & 3]);
                            }
                            (ft < 64 ? s_rq : s_rk)[r] = inv_norm((ss[0] + ss[1]) + (ss[2] + ss[3]), eps);
                            // The norms above need only the q/k tile and write factors the front alone
                            // reads; the rest of the front rewrites this parity's tiles, so it waits for
                            // the chain to release them (ofree). Norms first: 4K 288.7 -> 280.1 us.
                            if (ft < 32) got = ci < 2 || wait_or_abort(bar_ofree + b, ((ci - 2) >> 1) & 1, s_abort);
                            got = !group_or(BAR_FRONT_N, 128, !got);
                        }
                    } else {
                        if (ft < 160) got = wait_or_abort(bar_g, ci & 1, s_abort);
                        got = !group_or(BAR_FRONT_S, 128, !got);
                        if (got) {
                            if (ft == 128) s_waited[2] += 1;
                            if (L < C) {
                                const uint4 z4 = make_uint4(0, 0, 0, 0);
                                for (int p = ft - 128; p < (C - L) * 32; p += 128)
                                    *reinterpret_cast<uint4 *>(sm + G_ + (L + (p >> 5)) * 512 + (p & 31) * 16) = z4;
                            }
                            named_bar_sync(BAR_FRONT_S, 128);
                            // cumulative decay of key channel ft - 128
                            const int i = ft - 128;
                            // running sum down the 64 rows, 16 rows at a time
                            float run = 0.f, G0 = 0.f;
#pragma unroll 1
                            for (int r0 = 0; r0 < 64; r0 += 16) {
                                float gv[16];
#pragma unroll
                                for (int r = 0; r < 16; ++r) gv[r] = gt[(r0 + r) * 128 + i];
#pragma unroll
                                for (int r = 0; r < 16; ++r) {
                                    run = r0 + r == 0 ? gv[r] : run + gv[r];
                                    gv[r] = run;
                                }
                                if (r0 == 0) G0 = gv[0];
#pragma unroll
                                for (int r = 0; r < 16; ++r) gt[(r0 + r) * 128 + i] = gv[r] * LOG2E;
                            }
                            const float GL = run;
                            bad = !(G0 - GL <= SPAN_MAX);
                            s_gl[i] = GL;
                        }
                    }
                    if (group_or(BAR_FRONT, 256, !got)) {
                        ok = false;
                        break;
                    }
                } else {
                    // One warp spins on the barriers; the others wait in the named barrier,
                    // which costs them no issue slots.
                    if (ft < 32)
                        got = wait_or_abort(bar_qk + b, (ci >> 1) & 1, s_abort) &&
                              (!GCH || wait_or_abort(bar_g, ci & 1, s_abort));
                    if (group_or(BAR_FRONT, 256, !got)) {
                        ok = false;
                        break;
                    }
                    if (ft == 0) {
                        s_waited[b] += 1;
                        if constexpr (GCH) s_waited[2] += 1;
                        // the loads of chunk ci + 2 are issued one to two chunks from now,
                        // inside the pipeline's dependency cycle: stage their tiles in L2
                        if (ci + 2 < nchunks) {
                            const int y2 = (int)(c0 + 2 * C);
                            tma_prefetch_l2_3d(&tm_k, 0, h, y2);
                            tma_prefetch_l2_3d(&tm_q, 0, h, y2);
                            tma_prefetch_l2_3d(&tm_v, 0, h, y2);
                            if (dg > 64) {
                                tma_prefetch_l2_3d(&tm_k, 64, h, y2);
                                tma_prefetch_l2_3d(&tm_q, 64, h, y2);
                                tma_prefetch_l2_3d(&tm_v, 64, h, y2);
                            }
                            if constexpr (GCH) tma_prefetch_l2_3d(&tm_g, 0, h, y2);
                        }
                    }
                    if (ft < C) {
                        sb[ft] = beta_reg;
                        if constexpr (GHD) s_g1[ft] = gh_reg;
                    }
                    if (L < C) {  // rows past the end of the sequence contribute nothing
                        const uint4 z4 = make_uint4(0, 0, 0, 0);
                        for (int p = ft; p < (C - L) * 16; p += 256) {
                            const int r = L + (p >> 4), cc = p & 15;
                            *reinterpret_cast<uint4 *>(xb + swz(r, cc, 128)) = z4;
                            *reinterpret_cast<uint4 *>(xb + swz(r + 64, cc, 128)) = z4;
                        }
                        if constexpr (GCH)
                            for (int p = ft; p < (C - L) * 32; p += 256)
                                *reinterpret_cast<uint4 *>(sm + G_ + (L + (p >> 5)) * 512 + (p & 31) * 16) = z4;
                    }
                    named_bar_sync(BAR_FRONT, 256);

                    // ft < 128: L2 norm of one row (q rows for ft < 64, k rows after);
                    // ft >= 128: the decay of the per-head gate, or nothing
                    if (ft < 128) {
                        const int r = ft & 63;
                        const int row = ft < 64 ? r + 64 : r;  // q rows follow the k rows
                        float ss[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                        for (int cc = 0; cc < 16; ++cc) {
                            float f[8];
                            unpack8(*reinterpret_cast<const uint4 *>(xb + swz(row, cc, 128)), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) ss[e & 3] = fmaf(f[e], f[e], ss[e & 3]);
                        }
                        (ft < 64 ? s_rq : s_rk)[r] = inv_norm((ss[0] + ss[1]) + (ss[2] + ss[3]), eps);
                    } else if constexpr (GCH) {
                        const int i = ft - 128;
                        // running sum down the 64 rows, 16 rows at a time
                        float run = 0.f, G0 = 0.f;
#pragma unroll 1
                        for (int r0 = 0; r0 < 64; r0 += 16) {
                            float gv[16];
#pragma unroll
                            for (int r = 0; r < 16; ++r) gv[r] = gt[(r0 + r) * 128 + i];
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                run = r0 + r == 0 ? gv[r] : run + gv[r];
                                gv[r] = run;
                            }
                            if (r0 == 0) G0 = gv[0];
#pragma unroll
                            for (int r = 0; r < 16; ++r) gt[(r0 + r) * 128 + i] = gv[r] * LOG2E;
                        }
                        const float GL = run;
                        bad = !(G0 - GL <= SPAN_MAX);
                        s_gl[i] = GL;
                    } else if constexpr (GHD) {
                        if (warp == 8) {
                            const float g0 = s_g1[2 * lane], g1 = s_g1[2 * lane + 1];
                            float incl = g0 + g1;
#pragma unroll
                            for (int o = 1; o < 32; o <<= 1) {
                                const float y = __shfl_up_sync(0xffffffffu, incl, o);
                                if (lane >= o) incl += y;
                            }
                            const float G1v = incl, G0v = incl - g1;
                            const float GL = __shfl_sync(0xffffffffu, incl, 31);
                            const float Gfirst = __shfl_sync(0xffffffffu, G0v, 0);
                            bad = !(Gfirst - GL <= SPAN_MAX);
                            s_g1[2 * lane] = G0v * LOG2E;
                            s_g1[2 * lane + 1] = G1v * LOG2E;
#pragma unroll
                            for (int e = 0; e < 4; ++e) s_gl[4 * lane + e] = GL;
                        }
                    } else {
                        s_gl[ft - 128] = 0.f;
                    }
                    // as in the per-channel form: the norms and the per-head decay first, then wait for
                    // the chain to release this parity's tiles (4K per-head 261.8 -> 258.2 us)
                    if (ft < 32) got = ci < 2 || wait_or_abort(bar_ofree + b, ((ci - 2) >> 1) & 1, s_abort);
                    if (group_or(BAR_FRONT, 256, !got)) {
                        ok = false;
                        break;
                    }
                }
                const bool exact = GNO ? (named_bar_sync(BAR_FRONT, 256), false) : group_or(BAR_FRONT, 256, bad);
                // per-channel anchor c and state scale sigma
                if (ft < 128) {
                    const float GL = s_gl[ft], so = s_sigp[ft];
                    const float c = exact ? 0.f : fminf(0.f, GL + ANCHOR);
                    const float ec = expf(c);
                    const float sn = exact ? 1.f : expf(GL - c);
                    s_c[ft] = c;
                    s_sf[128 * b + ft] = ec * so;
                    s_pf[128 * b + ft] = exact ? expf(GL) * so : ec * so;
                    s_sig[128 * b + ft] = sn;
                    s_sigp[ft] = sn;
                }
                if (ft == 0) s_exact[b] = exact ? 1u : 0u;
                named_bar_sync(BAR_FRONT, 256);

                uint8_t *pb = sm + P0 + 8192 * b;
                if (exact) {  // A and P with exact pairwise decays
                    // A goes to the back warps' solve buffer: wait until they are done with chunk ci - 1
                    if (ci > 0) {
                        if (ft < 32) got = wait_or_abort(bar_ready + (b ^ 1), ((ci - 1) >> 1) & 1, s_abort);
                        if (group_or(BAR_FRONT, 256, !got)) {
                            ok = false;
                            break;
                        }
                    }
                    for (int p = ft; p < C * C; p += 256) {
                        const int r = p & 63, s = p >> 6;
                        float a = 0.f, pq = 0.f;
                        if (s <= r) {
                            const float rkr = s_rk[r], rks = s_rk[s], rqr = s_rq[r];
                            for (int cc = 0; cc < 16; ++cc) {
                                float kr[8], ks[8], qr[8];
                                unpack8(*reinterpret_cast<const uint4 *>(xb + swz(r, cc, 128)), kr);
                                unpack8(*reinterpret_cast<const uint4 *>(xb + swz(s, cc, 128)), ks);
                                unpack8(*reinterpret_cast<const uint4 *>(xb + swz(r + 64, cc, 128)), qr);
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    const int i = cc * 8 + e;
                                    float x = ks[e] * rks;
                                    if constexpr (GCH) x *= ex2(gt[r * 128 + i] - gt[s * 128 + i]);
                                    a += kr[e] * rkr * x;
                                    pq += qr[e] * rqr * x;
                                }
                            }
                        }
                        if constexpr (GHD) {
                            const float f = s <= r ? ex2(s_g1[r] - s_g1[s]) : 0.f;
                            a *= f;
                            pq *= f;
                        }
                        Am[fsw(r, s >> 2) + (s & 3)] = (s < r) ? sb[r] * a : 0.f;
                        *reinterpret_cast<__nv_bfloat16 *>(pb + r * 128 + ((((s >> 3) ^ (r & 7))) << 4) + (s & 7) * 2) =
                            __float2bfloat16_rn(pq);
                    }
                    named_bar_sync(BAR_FRONT, 256);
                }

                // operand tiles: [Lk; Lq] in place, and Rk (Kb on the exact path)
                uint8_t *rkb = sm + RK0 + 16384 * b;
                {
                    const int cc = ft & 15, rb = ft >> 4;  // rb 0..15
                    float cv[8], glv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        cv[e] = s_c[GCH ? cc * 8 + e : 0] * LOG2E;
                        glv[e] = s_gl[GCH ? cc * 8 + e : 0] * LOG2E;
                    }
#pragma unroll 1
                    for (int m = 0; m < 4; ++m) {
                        const int r = rb + 16 * m;
                        const uint32_t ok_ = swz(r, cc, 128), oq = swz(r + 64, cc, 128);
                        float qf[8], kf[8];
                        unpack8(*reinterpret_cast<const uint4 *>(xb + oq), qf);
                        unpack8(*reinterpret_cast<const uint4 *>(xb + ok_), kf);
                        const float rq = s_rq[r], rk = s_rk[r];
                        float G[8];
                        if constexpr (GCH) {
                            const float4 ga = *reinterpret_cast<const float4 *>(gt + r * 128 + cc * 8);
                            const float4 gb = *reinterpret_cast<const float4 *>(gt + r * 128 + cc * 8 + 4);
                            G[0] = ga.x; G[1] = ga.y; G[2] = ga.z; G[3] = ga.w;
                            G[4] = gb.x; G[5] = gb.y; G[6] = gb.z; G[7] = gb.w;
                        } else {
                            const float gr = GHD ? s_g1[r] : 0.f;
#pragma unroll
                            for (int e = 0; e < 8; ++e) G[e] = gr;
                        }
                        float lk[8], lq[8], rkv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float kh = kf[e] * rk, qh = qf[e] * rq;
                            if constexpr (GNO) {
                                lk[e] = kh;
                                lq[e] = qh;
                                rkv[e] = kh;
                            } else {
                                const float e1 = ex2(G[e] - cv[e]);
                                lk[e] = e1 * kh;
                                lq[e] = e1 * qh;
                                rkv[e] = (exact ? ex2(glv[e] - G[e]) : ex2(cv[e] - G[e])) * kh;
                            }
                        }
                        *reinterpret_cast<uint4 *>(xb + ok_) = pack8(lk);
                        *reinterpret_cast<uint4 *>(xb + oq) = pack8(lq);
                        *reinterpret_cast<uint4 *>(rkb + swz(r, cc, 64)) = pack8(rkv);
                    }
                }
                fence_async_smem();
                named_bar_sync(BAR_FRONT, 256);
                if (ft == 0) {
                    mbar_arrive(bar_fr + b);
                    // g of this chunk is consumed
                    if constexpr (GCH)
                        if (has_next) issue_g((int)(c0 + C));
                }
                if (ft < C) {
                    const bool in = has_next && c0 + C + ft < end;
                    beta_reg = in ? beta[(size_t)(c0 + C + ft) * H + h] : 0.f;
                    if constexpr (GHD) gh_reg = in ? g_head[(size_t)(c0 + C + ft) * H + h] : 0.f;
                }
            }
            if (!ok) *s_abort = 1u;
        } else {
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Regs<GM>::BACK));
            // ======================= back: warps 0-3 ========================
            // Chunk c: G1, A/P read-back, the solve for T, G2/G3 and the W'
            // read-back; ready[c & 1] hands the chunk to the chain.
            uint32_t ph_mp = 0;
            bool pend_mp = false;
            for (int ci = 0; ci < nchunks; ++ci) {
                const int b = ci & 1;
                const int64_t c0 = start + (int64_t)ci * C;
                const int L = (int)((end - c0) < (int64_t)C ? (end - c0) : (int64_t)C);
                uint8_t *xb = sm + X0 + 32768 * b;
                const uint32_t xs = sbase + X0 + 32768 * b;
                bool got = warp != 0 || wait_or_abort(bar_fr + b, (ci >> 1) & 1, s_abort);
                if (group_or(BAR_BACK, 128, !got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool exact = s_exact[b] != 0u;
                const float *sb = s_beta + 64 * b;
                uint8_t *pb = sm + P0 + 8192 * b;
                // G1: [A_raw; P_raw] = [Lk; Lq] Rk^T
                if (warp == 0 && !exact)
                    mma8_ss<16384, 8192>(tbase + T_AP, sdesc_sw128(xs, 16, 1024),
                                         sdesc_sw128(sbase + RK0 + 16384 * b, 16, 1024), ID_KK64, 0u, bar_mp);
                pend_mp = !exact;
                // warps 0, 1: A read-back; warps 2, 3: P read-back; then the solve
                got = true;
                if (!exact) {
                    if (warp == 0) got = wait_or_abort(bar_mp, ph_mp, s_abort);
                    got = !group_or(BAR_BACK, 128, !got);
                    tc_fence_after();
                }
                if (!exact && got && q4 < 2) {  // A: TMEM lanes 0-63, masked (s < r), times beta
                    const int r = 32 * q4 + lane;
                    const float br = sb[r];
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t r32[32];
                        tmem_ld32(tbase + lrow + T_AP + 32 * half, r32);
                        tmem_ld_wait();
#pragma unroll
                        for (int g4 = 0; g4 < 8; ++g4) {
                            float4 a4;
                            const int sc = 32 * half + 4 * g4;
                            a4.x = (sc + 0 < r) ? br * __uint_as_float(r32[4 * g4 + 0]) : 0.f;
                            a4.y = (sc + 1 < r) ? br * __uint_as_float(r32[4 * g4 + 1]) : 0.f;
                            a4.z = (sc + 2 < r) ? br * __uint_as_float(r32[4 * g4 + 2]) : 0.f;
                            a4.w = (sc + 3 < r) ? br * __uint_as_float(r32[4 * g4 + 3]) : 0.f;
                            *reinterpret_cast<float4 *>(Am + fsw(r, sc >> 2)) = a4;
                        }
                    }
                }
                if (!exact && got && q4 >= 2) {  // P: TMEM lanes 64-127, masked (s <= r)
                    const int r = 32 * (q4 - 2) + lane;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t r32[32];
                        tmem_ld32(tbase + lrow + T_AP + 32 * half, r32);
                        tmem_ld_wait();
                        float pv[32];
#pragma unroll
                        for (int m = 0; m < 32; ++m) pv[m] = (32 * half + m <= r) ? __uint_as_float(r32[m]) : 0.f;
#pragma unroll
                        for (int qd = 0; qd < 4; ++qd) {
                            const int cc = 4 * half + qd;
                            *reinterpret_cast<uint4 *>(pb + r * 128 + ((cc ^ (r & 7)) << 4)) = pack8(pv + 8 * qd);
                        }
                    }
                }
                named_bar_sync(BAR_BACK, 128);
                // M^-1 = (I + A)^-1 with A strictly lower, by 16 x 16 blocks.
                // Step 1: warp S inverts the diagonal block, D_S = (I + A_SS)^-1, by
                // forward substitution (lane = column; lanes 16-31 repeat 0-15).
                {
                    const int S = warp, b0 = 16 * S, cl = lane & 15;
                    float x[16];
#pragma unroll
                    for (int rl = 0; rl < 16; ++rl) x[rl] = (rl == cl) ? 1.f : 0.f;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float4 a4[16];
#pragma unroll
                        for (int rl = 4 * j + 1; rl < 16; ++rl)
                            a4[rl] = *reinterpret_cast<const float4 *>(Am + fsw(b0 + rl, 4 * S + j));
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int kl = 4 * j + e;
#pragma unroll
                            for (int rl = kl + 1; rl < 16; ++rl) {
                                const float a = e == 0 ? a4[rl].x : e == 1 ? a4[rl].y : e == 2 ? a4[rl].z : a4[rl].w;
                                x[rl] = fmaf(-a, x[kl], x[rl]);
                            }
                        }
                    }
                    if (lane < 16) {
                        const int s = b0 + cl;
                        const float bs = sb[s];
                        __nv_bfloat16 *tcol = reinterpret_cast<__nv_bfloat16 *>(sm + T_) + (s & 7);
#pragma unroll
                        for (int rl = 0; rl < 16; ++rl) {
                            const int r = b0 + rl;
                            Dv[S * BLK + rl * LDB + cl] = x[rl];
                            tcol[r * 64 + (((s >> 3) ^ (r & 7)) << 3)] = __float2bfloat16_rn(x[rl] * bs);
                        }
                    }
                    const uint4 z4 = make_uint4(0, 0, 0, 0);
                    for (int R = 0; R < S; ++R) {  // T blocks above the diagonal are zero
                        const int r = 16 * R + (lane >> 1), cc = 2 * S + (lane & 1);
                        *reinterpret_cast<uint4 *>(sm + T_ + r * 128 + ((cc ^ (r & 7)) << 4)) = z4;
                    }
                }
                named_bar_sync(BAR_BACK, 128);
                // Step 2, by doubling: M_10 = -D_1 A_10 D_0 and M_32 = -D_3 A_32 D_2
                // (warps 0, 1) while warps 2, 3 start Y_RS = sum_K A_RK M_KS for the
                // lower-left 32 x 32 block (R = 2, 3) with the parts that need no M_10.
                // Step 3 adds A_R1 M_10; step 4: M_2S = -D_2 Y_2S, M_3S = -(M_32 Y_2S + D_3 Y_3S).
                {
                    const int g = lane >> 2, tg = lane & 3;
                    // 16 x 16 block products on m16n8k8 tf32 tiles; X row-major with row stride LDB
                    auto a_blk = [&](const float *X, int kk, uint32_t (&a)[4]) {
                        a[0] = to_tf32(X[g * LDB + 8 * kk + tg]);
                        a[1] = to_tf32(X[(g + 8) * LDB + 8 * kk + tg]);
                        a[2] = to_tf32(X[g * LDB + 8 * kk + tg + 4]);
                        a[3] = to_tf32(X[(g + 8) * LDB + 8 * kk + tg + 4]);
                    };
                    auto a_am = [&](int R, int K, int kk, uint32_t (&a)[4]) {
                        const int k4 = 4 * K + 2 * kk, r0 = 16 * R + g;
                        a[0] = to_tf32(Am[fsw(r0, k4) + tg]);
                        a[1] = to_tf32(Am[fsw(r0 + 8, k4) + tg]);
                        a[2] = to_tf32(Am[fsw(r0, k4 + 1) + tg]);
                        a[3] = to_tf32(Am[fsw(r0 + 8, k4 + 1) + tg]);
                    };
                    auto b_blk = [&](const float *X, int kk, int nt, uint32_t (&b)[2]) {
                        b[0] = to_tf32(X[(8 * kk + tg) * LDB + 8 * nt + g]);
                        b[1] = to_tf32(X[(8 * kk + tg + 4) * LDB + 8 * nt + g]);
                    };
                    // acc += A_RK (from Am) * X
                    auto mm_am = [&](float (&acc)[2][4], int R, int K, const float *X) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            uint32_t a[4];
                            a_am(R, K, kk, a);
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt) {
                                uint32_t b[2];
                                b_blk(X, kk, nt, b);
                                mma_tf32_16x8x8(acc[nt], a, b);
                            }
                        }
                    };
                    // acc += Xa * Xb (both row-major blocks)
                    auto mm_blk = [&](float (&acc)[2][4], const float *Xa, const float *Xb) {
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            uint32_t a[4];
                            a_blk(Xa, kk, a);
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt) {
                                uint32_t b[2];
                                b_blk(Xb, kk, nt, b);
                                mma_tf32_16x8x8(acc[nt], a, b);
                            }
                        }
                    };
                    auto st_blk = [&](float *X, const float (&c)[2][4]) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            *reinterpret_cast<float2 *>(X + g * LDB + 8 * nt + 2 * tg) = make_float2(c[nt][0], c[nt][1]);
                            *reinterpret_cast<float2 *>(X + (g + 8) * LDB + 8 * nt + 2 * tg) = make_float2(c[nt][2], c[nt][3]);
                        }
                    };
                    // T_RS = -c Diag(beta_S) as bf16 pairs
                    auto st_t = [&](int R, int S, const float (&c)[2][4]) {
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt) {
                            const int s = 16 * S + 8 * nt + 2 * tg;
                            const float b0s = -sb[s], b1s = -sb[s + 1];
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const int r = 16 * R + g + 8 * hf;
                                *reinterpret_cast<__nv_bfloat162 *>(sm + T_ + r * 128 + (((s >> 3) ^ (r & 7)) << 4) +
                                                                    (s & 7) * 2) =
                                    __floats2bfloat162_rn(c[nt][2 * hf] * b0s, c[nt][2 * hf + 1] * b1s);
                            }
                        }
                    };
                    const float *D0 = Dv, *D1 = Dv + BLK, *D2 = Dv + 2 * BLK, *D3 = Dv + 3 * BLK;
                    float *M10 = Dv + 4 * BLK, *M32 = Dv + 5 * BLK;
                    float *Y20 = Yv, *Y21 = Yv + BLK, *Y30 = Yv + 2 * BLK, *Y31 = Yv + 3 * BLK;
                    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    float y1[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    if (warp < 2) {
                        const int R = warp == 0 ? 1 : 3;  // block (R, R-1)
                        mm_am(acc, R, R - 1, warp == 0 ? D0 : D2);
                        uint32_t yb[2][2][2];
                        c_to_b(acc, yb, lane);
                        const float *dr = warp == 0 ? D1 : D3;
                        float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            uint32_t a[4];
                            a_blk(dr, kk, a);
#pragma unroll
                            for (int nt = 0; nt < 2; ++nt) mma_tf32_16x8x8(z[nt], a, yb[kk][nt]);
                        }
                        st_t(R, R - 1, z);  // T = -z Diag(beta)
#pragma unroll
                        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) z[nt][e] = -z[nt][e];
                        st_blk(warp == 0 ? M10 : M32, z);
                    } else {
                        const int R = warp;  // 2 or 3
                        mm_am(acc, R, 1, D1);              // Y_R1 = A_R1 D_1 (final)
                        st_blk(R == 2 ? Y21 : Y31, acc);
                        mm_am(y1, R, 0, D0);               // Y_R0 partial: A_R0 D_0
                    }
                    named_bar_sync(BAR_BACK, 128);
                    if (warp >= 2) {
                        const int R = warp;
                        mm_am(y1, R, 1, M10);              // Y_R0 += A_R1 M_10
                        st_blk(R == 2 ? Y20 : Y30, y1);
                    }
                    named_bar_sync(BAR_BACK, 128);
                    {
                        // warp 0: (2,0), 1: (2,1), 2: (3,0), 3: (3,1)
                        const int R = 2 + (warp >> 1), S = warp & 1;
                        const float *y2 = S == 0 ? Y20 : Y21;
                        float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                        if (R == 2) {
                            mm_blk(z, D2, y2);
                        } else {
                            mm_blk(z, M32, y2);
                            mm_blk(z, D3, S == 0 ? Y30 : Y31);
                        }
                        st_t(R, S, z);
                    }
                }
                // the v tile is needed from G3 on (loaded right after G3 of the
                // chunk before)
                if (warp == 0) got = got && wait_or_abort(bar_v, ci & 1, s_abort);
                if (tid == 0 && got) s_waited[3] += 1;
                const int z0 = v_zero ? 0 : L;  // v read as zeros: every row
                // rows past the end of the sequence contribute nothing: zeroed
                // once every back thread knows the tile has landed
                if (z0 < C) got = !group_or(BAR_BACK, 128, !got);
                if (z0 < C && got) {
                    const uint4 z4 = make_uint4(0, 0, 0, 0);
                    for (int p = tid; p < (C - z0) * 16; p += 128) {
                        const int r = z0 + (p >> 4), cc = p & 15;
                        *reinterpret_cast<uint4 *>(sm + V_ + swz(r, cc, 64)) = z4;
                    }
                }
                fence_async_smem();
                tc_fence_before();
                if (group_or(BAR_BACK, 128, !got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (!exact) {
                    ph_mp ^= 1;
                    pend_mp = false;
                }

                // G2: W'^T = Lk^T T^T (over A/P in TMEM),  G3: U0^T = V^T T^T
                if (warp == 0)
                    mma44_ss(tbase + T_AP, sdesc_sw128(xs, 16384, 1024), tbase + T_U0 + 64 * b,
                             sdesc_sw128(sbase + V_, 8192, 1024), sdesc_sw128(sbase + T_, 16, 1024), ID_MK64, bar_mp);
                pend_mp = true;
                got = warp != 0 || wait_or_abort(bar_mp, ph_mp, s_abort);
                if (group_or(BAR_BACK, 128, !got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                ph_mp ^= 1;
                pend_mp = false;
                // G3 has read the v tile: load the next chunk's v into it
                if (tid == 0 && ci + 1 < nchunks) issue_v((int)(c0 + C));
                // W'^T (lane i, column r) -> row i of an MN-major W' operand (128 rows of
                // 64 tokens, 128 bytes each) over the Lk rows of this chunk's tile (dead
                // after G2): rows 0-63 over block 0's, rows 64-127 over block 1's. Each
                // thread stores its own row with 16-byte stores.
                {
                    const int i = jl;
                    uint8_t *wrow = xb + (i >> 6) * 16384 + (i & 63) * 128;
#pragma unroll 1
                    for (int half = 0; half < 2; ++half) {
                        uint32_t r32[32];
                        tmem_ld32(tbase + lrow + T_AP + 32 * half, r32);
                        tmem_ld_wait();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int cc = 4 * half + q;
                            float f[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(r32[8 * q + e]);
                            *reinterpret_cast<uint4 *>(wrow + ((cc ^ (i & 7)) << 4)) = pack8(f);
                        }
                    }
                }
                fence_async_smem();
                tc_fence_before();
                named_bar_sync(BAR_BACK, 128);
                if (tid == 0) mbar_arrive(bar_ready + b);
            }
            if (!ok) {  // let this group's own MMAs land before shared memory goes away
                *s_abort = 1u;
                if (pend_mp) mbar_wait(bar_mp, ph_mp, WAIT_LIMIT);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(Regs<GM>::CHAIN));
        // ============================ chain: warps 12-15 ==========================
        const int ct = tid - 384;  // 0..127
        // initial state -> TMEM (S^T: lane j, column i); sigma = 1
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            uint32_t r[32];
            // dg is 64 or 128, so a 32-row part lies wholly inside or outside the stored state
            const bool in = s_init != nullptr && jl < dg && 32 * part < dg;
#pragma unroll
            for (int m = 0; m < 32; ++m)
                r[m] = in ? __float_as_uint(s_init[soff + (size_t)(32 * part + m) * dg + jl]) : 0u;
            tmem_st32(tbase + lrow + T_S + 32 * part, r);
        }
        tmem_st_wait();
        uint32_t ph67 = 0;
        bool pend67 = false;
        int pend45 = -1;  // chunk whose G4/G5 are issued but not yet waited for
        int last_b = -1;
        for (int ci = 0; ci < nchunks; ++ci) {
            const int b = ci & 1;
            const int64_t c0 = start + (int64_t)ci * C;
            const int L = (int)((end - c0) < (int64_t)C ? (end - c0) : (int64_t)C);
            // S~ needs only the front's factors of this chunk, published with its operand
            // tiles. With the per-channel gate the chain converts it while the back still
            // works on the chunk (4K 283 -> 280 us, 8 x 8192 tokens 3.21 -> 3.15 ms). With a
            // per-head gate or none the early conversion competes with the back's solve and
            // is slower (259 -> 265 us, 240 -> 252 us), so those forms wait for the back first.
            bool got = ct >= 32 || wait_or_abort((GCH ? bar_fr : bar_ready) + b, (ci >> 1) & 1, s_abort);
            if (group_or(BAR_CHAIN, 128, !got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // the previous chunk's bulk output store has had a whole back phase to
            // read the output staging; the barrier after the S~ conversion
            // publishes that to the other chain threads before they rewrite it
            if (ct == 0 && ci > 0) bulk_wait_read();
            // S = Diag(sigma) S_st. S~^T = S_st^T Diag(sf) -> TMEM bf16 pairs; S_st^T <- S_st^T Diag(pf)
            const float *sf = s_sf + 128 * b, *pf = s_pf + 128 * b;
#pragma unroll 1
            for (int q32 = 0; q32 < 4; ++q32) {
                const int i0 = 32 * q32;
                uint32_t r[32], pk[16];
                tmem_ld32(tbase + lrow + T_S + i0, r);
                tmem_ld_wait();
                {
#pragma unroll
                    for (int g4 = 0; g4 < 8; ++g4) {
                        const float4 fc = GCH ? *reinterpret_cast<const float4 *>(sf + i0 + 4 * g4)
                                              : make_float4(sf[0], sf[0], sf[0], sf[0]);
                        const float4 fl = GCH ? *reinterpret_cast<const float4 *>(pf + i0 + 4 * g4)
                                              : make_float4(pf[0], pf[0], pf[0], pf[0]);
                        const float fcv[4] = {fc.x, fc.y, fc.z, fc.w}, flv[4] = {fl.x, fl.y, fl.z, fl.w};
                        float so[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float sv = __uint_as_float(r[4 * g4 + e]);
                            so[e] = sv * fcv[e];
                            r[4 * g4 + e] = __float_as_uint(sv * flv[e]);
                        }
                        __nv_bfloat162 t0 = __floats2bfloat162_rn(so[0], so[1]);
                        __nv_bfloat162 t1 = __floats2bfloat162_rn(so[2], so[3]);
                        pk[2 * g4] = *reinterpret_cast<uint32_t *>(&t0);
                        pk[2 * g4 + 1] = *reinterpret_cast<uint32_t *>(&t1);
                    }
                    // without a gate the rescale is by 1: S_st stays as it is
                    if constexpr (!GNO) tmem_st32(tbase + lrow + T_S + i0, r);
                }
                tmem_st16(tbase + lrow + T_SB + 16 * q32, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            if constexpr (GCH) {
                got = ct >= 32 || wait_or_abort(bar_ready + b, (ci >> 1) & 1, s_abort);
                if (group_or(BAR_CHAIN, 128, !got)) {
                    ok = false;
                    break;
                }
            } else {
                named_bar_sync(BAR_CHAIN, 128);
            }
            tc_fence_after();
            // G4: X^T = S~^T W'^T (W' channel-major), G5: O^T = S~^T Lq^T, one commit
            if (ct < 32)
                mma88_ts(tbase + T_X, sdesc_sw128(sbase + X0 + 32768 * b, 8192, 1024), ID_KM64, tbase + T_O,
                         sdesc_sw128(sbase + X0 + 32768 * b + 8192, 16, 1024), ID_KK64, tbase + T_SB, bar_c45 + b);
            pend45 = ci;
            got = ct >= 32 || wait_or_abort(bar_c45 + b, (ci >> 1) & 1, s_abort);
            if (group_or(BAR_CHAIN, 128, !got)) {
                ok = false;
                break;
            }
            pend45 = -1;
            tc_fence_after();
            // this chunk's W' / Lq tile is consumed: load the chunk two ahead into it
            if (ct == 0 && ci + 2 < nchunks) issue_qk((int)(c0 + 2 * C), b);
            // U^T = U0^T - X^T -> bf16 pairs in TMEM over S~ (dead after G4/G5)
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t u0[32], x[32], pk[16];
                tmem_ld32(tbase + lrow + T_U0 + 64 * b + 32 * half, u0);
                tmem_ld32(tbase + lrow + T_X + 32 * half, x);
                tmem_ld_wait();
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(u0[2 * m]) - __uint_as_float(x[2 * m]),
                                                             __uint_as_float(u0[2 * m + 1]) - __uint_as_float(x[2 * m + 1]));
                    pk[m] = *reinterpret_cast<uint32_t *>(&t);
                }
                tmem_st16(tbase + lrow + T_SB + 16 * half, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            named_bar_sync(BAR_CHAIN, 128);
            tc_fence_after();
            // G6: O^T += U^T P^T,  G7: S_st^T += U^T Rk (Kb on the exact path)
            if (ct < 32)
                mma44_ts(tbase + T_O, sdesc_sw128(sbase + P0 + 8192 * b, 16, 1024), ID_KK64, tbase + T_S,
                         sdesc_sw128(sbase + RK0 + 16384 * b, 8192, 1024), ID_KM128, tbase + T_SB, bar_c67);
            pend67 = true;
            got = ct >= 32 || wait_or_abort(bar_c67, ph67, s_abort);
            if (group_or(BAR_CHAIN, 128, !got)) {
                ok = false;
                break;
            }
            ph67 ^= 1;
            pend67 = false;
            tc_fence_after();
            // U0[b], Rk[b], P[b] and the factors of this parity are consumed
            if (ct == 0) mbar_arrive(bar_ofree + b);
            // O^T (lane j, column r) -> the output staging: two [64 rows][64
            // channels] bf16 boxes
            uint8_t *ost = sm + OST;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t o32[32];
                tmem_ld32(tbase + lrow + T_O + 32 * half, o32);
                tmem_ld_wait();
                __nv_bfloat16 *col = reinterpret_cast<__nv_bfloat16 *>(ost + (jl >> 6) * 8192) + (jl & 63);
#pragma unroll
                for (int m = 0; m < 32; ++m) col[(32 * half + m) * 64] = __float2bfloat16_rn(__uint_as_float(o32[m]));
            }
            fence_async_smem();
            tc_fence_before();
            named_bar_sync(BAR_CHAIN, 128);
            if (L == C) {
                // a whole chunk: one bulk store per 64-channel box; the staging is
                // rewritten once the copy engine has read it (next chunk)
                if (ct == 0) {
                    tma_store_3d(&tm_o, ost, 0, h, (int)c0);
                    if (dg > 64) tma_store_3d(&tm_o, ost + 8192, 64, h, (int)c0);
                    bulk_commit();
                }
            } else {
                // a sequence's short last chunk: plain stores of its rows only (the rows
                // after it belong to the next sequence)
                uint4 orow[8];
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    const int p = ct + 128 * k8, r = p >> 4, c16 = p & 15;
                    orow[k8] = *reinterpret_cast<const uint4 *>(ost + (c16 >> 3) * 8192 + r * 128 + (c16 & 7) * 16);
                }
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    const int p = ct + 128 * k8, r = p >> 4, c16 = p & 15;
                    if (r < L && 8 * c16 < dg)
                        *reinterpret_cast<uint4 *>(out + ((size_t)(c0 + r) * H + h) * dg + c16 * 8) = orow[k8];
                }
            }
            last_b = b;
        }
        if (ct == 0) bulk_wait_all();  // output copies complete before the CTA's shared memory goes away
        if (ok && s_final) {  // S = Diag(sigma) S_st
            const float *sg = last_b >= 0 ? s_sig + 128 * last_b : nullptr;
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                uint32_t r[32];
                tmem_ld32(tbase + lrow + T_S + 32 * part, r);
                tmem_ld_wait();
                if (jl < dg && 32 * part < dg)
#pragma unroll
                    for (int m = 0; m < 32; ++m)
                        s_final[soff + (size_t)(32 * part + m) * dg + jl] =
                            __uint_as_float(r[m]) * (sg ? sg[32 * part + m] : 1.f);
            }
        }
        if (!ok) {
            *s_abort = 1u;
            if (pend45 >= 0) mbar_wait(bar_c45 + (pend45 & 1), (pend45 >> 1) & 1, WAIT_LIMIT);
            if (pend67) mbar_wait(bar_c67, ph67, WAIT_LIMIT);
        }
    }
    if (!ok && (tid == 0 || tid == 384)) atomicOr(err, DEVERR_TIMEOUT);
    sync_tc();
    // after an abort: every copy still in flight must land before exit
    if (tid == 0 && *s_abort) {
        uint64_t *tb[4] = {bar_qk, bar_qk + 1, bar_g, bar_v};
        for (int i = 0; i < 4; ++i)
            for (uint32_t w = s_waited[i]; w < s_armed[i]; ++w)
                if (!mbar_wait(tb[i], w & 1, WAIT_LIMIT)) break;
    }
    sync_tc();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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

bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t elem, uint64_t inner,
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

// 3-D map over [T][H][d] (dims innermost first: d, H, T), box box_d x 1 x box_t. A box reaching
// past d (d = 64, box_d = 128) reads zeros there.
static bool make_map3(CUtensorMap *m, const void *base, CUtensorMapDataType dt, uint32_t elem, uint64_t d, uint64_t H,
                      uint64_t T, uint32_t box_d, uint32_t box_t, CUtensorMapSwizzle sw) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d, H, T};
    const cuuint64_t strides[2] = {d * elem, H * d * elem};
    const cuuint32_t box[3] = {box_d, 1, box_t};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tcp

namespace tc {
bool make_map_nd(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int rank, const uint64_t *dims,
                 const uint64_t *strides, const uint32_t *box) {
    tcp::EncodeTiledFn fn = tcp::encode_fn();
    if (!fn || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return fn(m, dt, (cuuint32_t)rank, const_cast<void *>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}
}  // namespace tc

// bf16, d = 128 or 64 (64: the kernel's channels 64..127 read as zeros, which leaves every
// product of the chunk algebra unchanged), C = 16, 32 or 64. The kernel always works in chunks of
// 64 tokens: the chunked form is an exact rewrite of the recurrence, so the chunk length changes
// only the rounding.
bool prefill_tc_applicable(const PrefillArgs &a) {
    return a.bf16 && (a.D == 128 || a.D == 64) && (a.C == 64 || a.C == 32 || a.C == 16) && a.T > 0 &&
           a.T <= 0x7fffffffLL;
}

// The pipelined kernel runs every gate form (4K workload, per-channel gate:
// 0.420 ms against 0.473 ms for the sequential kernel).
template <int GM>
static kda_status launch_tc(const PrefillArgs &a, const CUtensorMap &mq, const CUtensorMap &mk,
                            const CUtensorMap &mv, const CUtensorMap &mg, cudaStream_t s) {
    using namespace tcp;
    const float *gh = GM == KDA_GATE_HEAD ? a.g : nullptr;
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(a.out);
    // the kernel stores whole output chunks through this map
    CUtensorMap mo;
    if (!make_map3(&mo, a.out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)a.D, (uint64_t)a.H, (uint64_t)a.T, 64,
                   64, CU_TENSOR_MAP_SWIZZLE_NONE))
        return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    // the register split only adds up for the launch register count it was made for
    static std::atomic<int> regs_ok{0};  // 0 unknown, 1 checked, -1 mismatch
    if (regs_ok.load(std::memory_order_acquire) == 0) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, prefill_tc_pipe_kernel<GM>);
        if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncGetAttributes: ") + cudaGetErrorString(e));
        using RG = pipe::Regs<GM>;
        const bool okr = 4 * RG::BACK + 8 * RG::FRONT + 4 * RG::CHAIN == 16 * fa.numRegs &&
                         RG::FRONT <= fa.numRegs && fa.numRegs <= RG::BACK && fa.numRegs <= RG::CHAIN;
        regs_ok.store(okr ? 1 : -1, std::memory_order_release);
    }
    if (regs_ok.load(std::memory_order_acquire) < 0)
        return fail(KDA_ERR_UNSUPPORTED, "prefill kernel built with a register count its warp split was not made for");
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_pipe_kernel<GM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)pipe::SMEM);
    if (e != cudaSuccess) return fail(KDA_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    prefill_tc_pipe_kernel<GM><<<launch_seqs(a) * a.H, pipe::NTP, pipe::SMEM, s>>>(
        mq, mk, mv, mg, mo, gh, a.beta, a.s_init, a.s_final, o, a.cu_seqlens, a.N, a.T, a.H, a.eps, a.err, a.order,
        a.v_zero ? 1 : 0, a.D);
    return check_launch("prefill_tc_pipe_kernel");
}

kda_status prefill_tc(const PrefillArgs &a, cudaStream_t s) {
    using namespace tcp;
    CUtensorMap mq, mk, mv, mg;
    memset(&mg, 0, sizeof(mg));  // not read unless the gate is per channel
    const uint64_t d = (uint64_t)a.D, hh = (uint64_t)a.H, rows = (uint64_t)a.T;
    const auto bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!make_map3(&mq, a.q, bf, 2, d, hh, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map3(&mk, a.k, bf, 2, d, hh, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map3(&mv, a.v, bf, 2, d, hh, rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        (a.gate == KDA_GATE_CHANNEL && !make_map3(&mg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, hh, rows, 128, 64,
                                                  CU_TENSOR_MAP_SWIZZLE_NONE)))
        return fail(KDA_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    if (a.gate == KDA_GATE_HEAD) return launch_tc<KDA_GATE_HEAD>(a, mq, mk, mv, mg, s);
    if (a.gate == KDA_GATE_NONE) return launch_tc<KDA_GATE_NONE>(a, mq, mk, mv, mg, s);
    return launch_tc<KDA_GATE_CHANNEL>(a, mq, mk, mv, mg, s);
}

}  // namespace kda
