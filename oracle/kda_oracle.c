/*
 * kda_oracle.c -- TEST INFRASTRUCTURE ONLY. Not part of the product path.
 *
 * A plain, slow, sequential fp64 CPU statement of the Kimi Delta Attention
 * (KDA) gated delta-rule recurrence and of the width-4 causal short
 * convolution that feeds it. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *  [W]  "KV缓存从11.25GB缩到0.21GB: WARP中Kimi Delta Attention线性注意力原理剖析",
 *       section "KDA 递推公式先衰减再差分": per token, first decay the state along
 *       the key axis, S <- Diag(exp(g_t)) S_{t-1} (g kept in log space and
 *       exponentiated inside the kernel), then correct it by the delta rule,
 *       S_t = S + beta_t k_t (v_t - S^T k_t)^T, then read out o_t = S_t^T q_t;
 *       q and k are L2-normalised inside the kernel; a width-4 causal short
 *       convolution with SiLU precedes q/k/v and needs a 3-token ring at decode.
 *  [G]  "为什么 Kimi K3 敢把 KV Cache 扔掉？一篇讲透 GPT-2 到 K3 的架构进化",
 *       section 5 (chunked training): inside a chunk of size C the work is
 *       attention-like, across chunks the state is handed on; C=1 is the plain
 *       recurrence and C=N the quadratic form. Section 6: the cumulative decay
 *       between a write at x and a read at x+t is the product of the gates in
 *       between. Section 7: the Kimi Linear update in product form
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T.
 *
 * Conventions (readings where the pages are silent; each is also listed in
 * the design notes):
 *  - State S is d_k x d_v, row i = key channel, column j = value channel,
 *    row-major, as in [W].
 *  - L2 normalisation: xhat = x / sqrt(sum x^2 + eps); a vector whose
 *    sum of squares plus eps is exactly zero normalises to zero.
 *  - No extra 1/sqrt(d) scale on q.
 *  - Short conv: depthwise, no bias; tap 3 multiplies the current token, taps
 *    0..2 multiply x_{t-3}, x_{t-2}, x_{t-1}; the ring is chronological
 *    (slot 0 = oldest) and is shifted after each step.
 *
 * Parity pins: every function here is checked by the not-gpu tests against
 * the worked example of [G] section 4, closed forms (beta=0, g=0, very
 * negative g, orthonormal keys), the product form of [G] section 7, the
 * scalar-gate form of [G] section 6, a norm invariant, library convolution
 * and the chunk-equivalence property of [G] section 5.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* L2 normalisation of one length-D vector; [W] section "KDA 递推公式先衰减再差分"
 * states that q and k are normalised inside the kernel. */
static void l2_normalise(const double *x, double *out, int D, double eps)
{
    double ss = 0.0;
    for (int i = 0; i < D; ++i)
        ss += x[i] * x[i];
    double den = ss + eps;
    if (den == 0.0) {
        for (int i = 0; i < D; ++i)
            out[i] = 0.0;
        return;
    }
    double inv = 1.0 / sqrt(den);
    for (int i = 0; i < D; ++i)
        out[i] = x[i] * inv;
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/*
 * One decode step of the width-4 causal depthwise short convolution + SiLU
 * ([W] last paragraph of "KDA 递推公式先衰减再差分"; ring size per the
 * "414MB 的 KDA 状态从哪来" table: 3 projections x 3 tokens x d per head).
 *
 *   x    [B,3,H,D]    current pre-conv projections (q,k,v)
 *   ring [B,3,H,3,D]  x_{t-3}, x_{t-2}, x_{t-1} (in/out, shifted by one)
 *   w    [3,H,D,4]    taps; w[..,3] multiplies x_t
 *   y    [B,3,H,D]    SiLU(conv)
 */
void oracle_shortconv_step(const double *x, double *ring, const double *w,
                           double *y, int B, int H, int D)
{
    for (int b = 0; b < B; ++b)
        for (int p = 0; p < 3; ++p)
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < D; ++c) {
                    size_t xi = (((size_t)b * 3 + p) * H + h) * D + c;
                    size_t rb = ((((size_t)b * 3 + p) * H + h) * 3) * D + c;
                    const double *wt = w + (((size_t)p * H + h) * D + c) * 4;
                    double r0 = ring[rb], r1 = ring[rb + D], r2 = ring[rb + 2 * (size_t)D];
                    double xt = x[xi];
                    double z = wt[0] * r0 + wt[1] * r1 + wt[2] * r2 + wt[3] * xt;
                    y[xi] = silu(z);
                    ring[rb] = r1;
                    ring[rb + D] = r2;
                    ring[rb + 2 * (size_t)D] = xt;
                }
}

/*
 * The same short convolution over a packed batch of sequences, as a prefill
 * would run it ([W] "KDA 递推公式先衰减再差分": conv + SiLU in front of q/k/v,
 * with the 3-token ring that decode carries on). Sequence n covers tokens
 * [cu_seqlens[n], cu_seqlens[n+1]); its history before the first token is
 * ring_in[n] (zeros if ring_in is NULL). Each token is one application of
 * the step above to a batch of one; ring_out[n] (if not NULL) receives the
 * ring after the sequence's last token, so an empty sequence passes ring_in
 * through unchanged.
 *   x        [T,3,H,D]     pre-conv projections
 *   ring_in  [N,3,H,3,D]   or NULL
 *   y        [3,T,H,D]     post-conv q, k, v (projection-major)
 *   ring_out [N,3,H,3,D]   or NULL
 */
void oracle_shortconv_seq(const double *x, const double *ring_in, const double *w, double *y,
                          double *ring_out, const int64_t *cu_seqlens, int N, int64_t T, int H, int D)
{
    const size_t row = (size_t)3 * H * D;       /* one token of x */
    const size_t rsz = (size_t)3 * H * 3 * D;   /* one sequence's ring */
    double *ring = malloc(rsz * sizeof(double));
    double *yt = malloc(row * sizeof(double));
    if (!ring || !yt) {
        free(ring);
        free(yt);
        return;
    }
    for (int n = 0; n < N; ++n) {
        for (size_t e = 0; e < rsz; ++e) ring[e] = ring_in ? ring_in[(size_t)n * rsz + e] : 0.0;
        for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            oracle_shortconv_step(x + (size_t)t * row, ring, w, yt, 1, H, D);
            for (int p = 0; p < 3; ++p)
                for (int h = 0; h < H; ++h)
                    for (int c = 0; c < D; ++c)
                        y[(((size_t)p * T + t) * H + h) * D + c] = yt[((size_t)p * H + h) * D + c];
        }
        if (ring_out)
            for (size_t e = 0; e < rsz; ++e) ring_out[(size_t)n * rsz + e] = ring[e];
    }
    free(ring);
    free(yt);
}

/*
 * The KDA recurrence, token by token ([W] "KDA 递推公式先衰减再差分").
 *
 * Packed variable-length layout: tokens of all sequences are concatenated;
 * sequence n covers tokens [cu_seqlens[n], cu_seqlens[n+1]).
 *   q,k,v,g  [T,H,D]   (g is the log-space per-key-channel gate)
 *   beta     [T,H]
 *   s_init   [N,H,D,D] or NULL (zeros)
 *   s_final  [N,H,D,D] or NULL
 *   out      [T,H,D]
 * A decode step is the special case of N sequences of one token each.
 * Independent (sequence, head) units are spread over nthreads threads.
 */
void oracle_recurrence(const double *q, const double *k, const double *v,
                       const double *g, const double *beta,
                       const double *s_init, double *s_final, double *out,
                       const int64_t *cu_seqlens, int N, int H, int D,
                       double eps, int nthreads)
{
    long units = (long)N * H;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long u = 0; u < units; ++u) {
        int n = (int)(u / H), h = (int)(u % H);
        double *S = (double *)malloc(sizeof(double) * (size_t)D * D);
        double *qh = (double *)malloc(sizeof(double) * (size_t)D * 4);
        double *kh = qh + D, *kv = qh + 2 * D, *dl = qh + 3 * D;
        size_t soff = ((size_t)n * H + h) * (size_t)D * D;
        if (s_init)
            memcpy(S, s_init + soff, sizeof(double) * (size_t)D * D);
        else
            memset(S, 0, sizeof(double) * (size_t)D * D);
        for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            size_t o = ((size_t)t * H + h) * D;
            double b = beta[(size_t)t * H + h];
            l2_normalise(q + o, qh, D, eps);
            l2_normalise(k + o, kh, D, eps);
            /* (1) forget along the key axis: S <- Diag(exp(g_t)) S */
            for (int i = 0; i < D; ++i) {
                double a = exp(g[o + i]);
                for (int j = 0; j < D; ++j)
                    S[(size_t)i * D + j] *= a;
            }
            /* (2) delta correction: S <- S + beta k (v - S^T k)^T */
            for (int j = 0; j < D; ++j) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i)
                    acc += S[(size_t)i * D + j] * kh[i];
                kv[j] = acc;
            }
            for (int j = 0; j < D; ++j)
                dl[j] = b * (v[o + j] - kv[j]);
            for (int i = 0; i < D; ++i)
                for (int j = 0; j < D; ++j)
                    S[(size_t)i * D + j] += kh[i] * dl[j];
            /* (3) read out: o = S^T q */
            for (int j = 0; j < D; ++j) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i)
                    acc += S[(size_t)i * D + j] * qh[i];
                out[o + j] = acc;
            }
        }
        if (s_final)
            memcpy(s_final + soff, S, sizeof(double) * (size_t)D * D);
        free(S);
        free(qh);
    }
}

/*
 * Chunked evaluation of the same recurrence, used only to pin the chunk
 * equivalence property ([G] section 5: C=1 is the recurrence, C=N the
 * quadratic form; section 6: decay between positions is the product of the
 * gates in between, here exp of a difference of cumulative log gates).
 *
 * Within a chunk of L tokens with state S at its start, write
 * G_r = sum_{s<=r} g_s (per key channel), and let u_r be the value that the
 * delta rule writes at position r, u_r = beta_r (v_r - (Diag(e^{g_r}) S_{r-1})^T k_r).
 * Unrolling the recurrence over the chunk gives
 *   u_r + sum_{s<r} A_rs u_s = beta_r (v_r - S^T (e^{G_r} . k_r)),
 *   A_rs = beta_r sum_i k_ri k_si exp(G_ri - G_si)           (s < r)
 *   o_r  = S^T (e^{G_r} . q_r) + sum_{s<=r} P_rs u_s,
 *   P_rs = sum_i q_ri k_si exp(G_ri - G_si)                   (s <= r)
 *   S'   = Diag(e^{G_L}) S + sum_s (e^{G_L - G_s} . k_s) u_s^T
 * and the first line is solved for u by forward substitution.
 */
void oracle_chunked(const double *q, const double *k, const double *v,
                    const double *g, const double *beta,
                    const double *s_init, double *s_final, double *out,
                    const int64_t *cu_seqlens, int N, int H, int D,
                    double eps, int C, int nthreads)
{
    long units = (long)N * H;
    if (C < 1)
        C = 1;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long u = 0; u < units; ++u) {
        int n = (int)(u / H), h = (int)(u % H);
        size_t DD = (size_t)D * D, CD = (size_t)C * D, CC = (size_t)C * C;
        double *S = (double *)malloc(sizeof(double) * DD);
        double *Sn = (double *)malloc(sizeof(double) * DD);
        double *Q = (double *)malloc(sizeof(double) * CD);
        double *K = (double *)malloc(sizeof(double) * CD);
        double *G = (double *)malloc(sizeof(double) * CD);
        double *U = (double *)malloc(sizeof(double) * CD);
        double *A = (double *)malloc(sizeof(double) * CC);
        double *P = (double *)malloc(sizeof(double) * CC);
        double *bt = (double *)malloc(sizeof(double) * C);
        size_t soff = ((size_t)n * H + h) * DD;
        if (s_init)
            memcpy(S, s_init + soff, sizeof(double) * DD);
        else
            memset(S, 0, sizeof(double) * DD);
        for (int64_t c0 = cu_seqlens[n]; c0 < cu_seqlens[n + 1]; c0 += C) {
            int L = (int)((cu_seqlens[n + 1] - c0) < C ? (cu_seqlens[n + 1] - c0) : C);
            for (int r = 0; r < L; ++r) {
                size_t o = ((size_t)(c0 + r) * H + h) * D;
                l2_normalise(q + o, Q + (size_t)r * D, D, eps);
                l2_normalise(k + o, K + (size_t)r * D, D, eps);
                bt[r] = beta[(size_t)(c0 + r) * H + h];
                for (int i = 0; i < D; ++i)
                    G[(size_t)r * D + i] = g[o + i] + (r ? G[(size_t)(r - 1) * D + i] : 0.0);
            }
            for (int r = 0; r < L; ++r)
                for (int s = 0; s <= r; ++s) {
                    double ak = 0.0, pq = 0.0;
                    for (int i = 0; i < D; ++i) {
                        double e = exp(G[(size_t)r * D + i] - G[(size_t)s * D + i]);
                        ak += K[(size_t)r * D + i] * K[(size_t)s * D + i] * e;
                        pq += Q[(size_t)r * D + i] * K[(size_t)s * D + i] * e;
                    }
                    A[(size_t)r * C + s] = (s < r) ? bt[r] * ak : 0.0;
                    P[(size_t)r * C + s] = pq;
                }
            /* forward substitution for u */
            for (int r = 0; r < L; ++r) {
                for (int j = 0; j < D; ++j) {
                    double ks = 0.0;
                    for (int i = 0; i < D; ++i)
                        ks += exp(G[(size_t)r * D + i]) * K[(size_t)r * D + i] * S[(size_t)i * D + j];
                    size_t o = ((size_t)(c0 + r) * H + h) * D;
                    double rhs = bt[r] * (v[o + j] - ks);
                    for (int s = 0; s < r; ++s)
                        rhs -= A[(size_t)r * C + s] * U[(size_t)s * D + j];
                    U[(size_t)r * D + j] = rhs;
                }
            }
            /* outputs */
            for (int r = 0; r < L; ++r) {
                size_t o = ((size_t)(c0 + r) * H + h) * D;
                for (int j = 0; j < D; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < D; ++i)
                        acc += exp(G[(size_t)r * D + i]) * Q[(size_t)r * D + i] * S[(size_t)i * D + j];
                    for (int s = 0; s <= r; ++s)
                        acc += P[(size_t)r * C + s] * U[(size_t)s * D + j];
                    out[o + j] = acc;
                }
            }
            /* state hand-off to the next chunk */
            const double *GL = G + (size_t)(L - 1) * D;
            for (int i = 0; i < D; ++i)
                for (int j = 0; j < D; ++j) {
                    double acc = exp(GL[i]) * S[(size_t)i * D + j];
                    for (int s = 0; s < L; ++s)
                        acc += exp(GL[i] - G[(size_t)s * D + i]) * K[(size_t)s * D + i] * U[(size_t)s * D + j];
                    Sn[(size_t)i * D + j] = acc;
                }
            memcpy(S, Sn, sizeof(double) * DD);
        }
        if (s_final)
            memcpy(s_final + soff, S, sizeof(double) * DD);
        free(S); free(Sn); free(Q); free(K); free(G); free(U); free(A); free(P); free(bt);
    }
}

/*
 * Output epilogue of a layer: gated RMSNorm of the attention output, one row
 * of D value channels per (token, head). [W] section "相关源码与文档导航" lists a
 * gated RMSNorm among the parts of the KDA kernel, and [G] section 6 (the
 * Gated DeltaNet architecture figure) says the output passes a gate that
 * scales its features; neither prints the formula. The reading taken (and
 * listed in the design notes) is the plainest one:
 *   y_j = o_j / sqrt(mean_j' o_j'^2 + eps) * weight_j * act(gate_j)
 * with act the logistic sigmoid (act = 0) or SiLU, z * sigmoid(z) (act = 1).
 * A row whose mean square plus eps is exactly zero maps to zero.
 *
 *   o, gate [R, D] (R = tokens x heads rows), weight [D], y [R, D]
 */
void oracle_gated_rmsnorm(const double *o, const double *gate, const double *weight, double *y,
                          int64_t R, int D, double eps, int act)
{
    for (int64_t r = 0; r < R; ++r) {
        const double *orow = o + r * D, *grow = gate + r * D;
        double ss = 0.0;
        for (int j = 0; j < D; ++j)
            ss += orow[j] * orow[j];
        /* a row whose mean square plus eps is exactly zero maps to zero, as in
         * the L2 normalisation above */
        const double den = ss / D + eps;
        const double inv = den > 0.0 ? 1.0 / sqrt(den) : 0.0;
        for (int j = 0; j < D; ++j) {
            const double z = grow[j];
            const double sg = 1.0 / (1.0 + exp(-z));
            y[r * D + j] = orow[j] * inv * weight[j] * (act == 1 ? z * sg : sg);
        }
    }
}

/* Number of threads the OpenMP runtime would use by default (for reporting). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
