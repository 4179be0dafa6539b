/*
 * fa_oracle.c - plain, slow FP64 CPU oracle for exact scaled-dot-product
 * attention and its gradient.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  It shares no code, header, table
 * or helper with the CUDA path; it is not a fallback for it.
 *
 * What it computes is the plain definition of attention, written out without
 * blocking, fusion or reordering:
 *
 *   S_ij = scale * sum_c Q_ic K_jc                  (standard attention, page 4
 *                                                     "standard_attention";
 *                                                     page 3 section 1, steps 1-3)
 *   S_ij = -inf for j > i when causal               (key j visible to query i
 *                                                     iff j <= i)
 *   m_i  = max_j S_ij,  P_ij = exp(S_ij - m_i) / sum_j exp(S_ij - m_i)
 *                                                    (safe softmax, page 4
 *                                                     "softmax decomposition")
 *   O_i  = sum_j P_ij V_j
 *   LSE_i = m_i + ln sum_j exp(S_ij - m_i)          (natural log, per query row)
 *
 * The backward is the textbook gradient of the forward above, with explicit
 * N x N matrices per (batch, head):
 *
 *   dV = P^T dO,   dP = dO V^T,   D_i = sum_c dO_ic O_ic,
 *   dS = P o (dP - D 1^T),   dQ = scale dS K,   dK = scale dS^T Q.
 *
 * The pages only say that the backward recomputes the attention matrix
 * instead of storing it (page 4, "recomputation"); these formulas are the
 * plainest reading and are pinned by finite differences in the tests.
 *
 * D is the row sum of dO o O over the output O the backward is handed.  The
 * method stores O in the output precision (bf16 for bf16 inputs, fp32 for
 * fp32 inputs) and its backward forms D from that stored tensor, so the
 * backward takes o_storage: 0 uses the exact FP64 O (the true gradient of the
 * exact function), 1 rounds the FP64 O to bf16 (nearest, ties to even) and 2
 * rounds it to fp32 before D is formed.  Nothing else changes.
 *
 * All inputs are float64 arrays in [B, H, N, d] row-major layout (the caller
 * converts bf16 / fp32 inputs exactly).  Work is spread over query rows (and,
 * in the backward, over the rows of each output) with OpenMP; every output
 * element is one sum in a fixed order, so the thread count never changes a
 * result.
 *
 * Return value of every entry point: 0 on success, -1 on a bad argument,
 * -2 when a scratch allocation fails.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int bad_shape(int64_t B, int64_t H, int64_t N, int64_t d) {
    return B < 1 || H < 1 || N < 1 || d < 1;
}

/* One query row i of one head with N keys: builds the row of S, its softmax,
 * O_i and LSE_i.  srow is caller scratch of N doubles; on return srow holds
 * P_i. */
static void attention_row(const double* q_i, const double* kh, const double* vh,
                          int64_t i, int64_t N, int64_t d, int causal, double scale,
                          double* srow, double* o_i, double* lse_i) {
    int64_t last = (causal && i < N - 1) ? i : N - 1; /* keys 0..last are visible */
    double m = -INFINITY;
    for (int64_t j = 0; j <= last; ++j) {
        const double* k_j = kh + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += q_i[c] * k_j[c];
        srow[j] = scale * acc;
        if (srow[j] > m) m = srow[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j <= last; ++j) {
        srow[j] = exp(srow[j] - m);
        l += srow[j];
    }
    for (int64_t j = 0; j <= last; ++j) srow[j] /= l;
    for (int64_t j = last + 1; j < N; ++j) srow[j] = 0.0;
    for (int64_t c = 0; c < d; ++c) o_i[c] = 0.0;
    for (int64_t j = 0; j <= last; ++j) {
        const double* v_j = vh + j * d;
        double p = srow[j];
        for (int64_t c = 0; c < d; ++c) o_i[c] += p * v_j[c];
    }
    *lse_i = m + log(l);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward over every (b, h) head: q [B,H,N,d], k and v [B,H,Nk,d];
 * o [B,H,N,d], lse [B,H,N].  The method itself has Nk == N; a different key
 * count only serves tests that attend to one block of keys at a time. */
int oracle_fwd(const double* q, const double* k, const double* v,
               int64_t B, int64_t H, int64_t N, int64_t Nk, int64_t d, int causal,
               double scale, double* o, double* lse) {
    if (!q || !k || !v || !o || !lse || bad_shape(B, H, N, d) || Nk < 1) return -1;
    int64_t rows = B * H * N;
    int failed = 0;
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)Nk);
        if (!srow) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t r = 0; r < rows; ++r) {
            if (!srow) continue;
            int64_t bh = r / N, i = r % N;
            attention_row(q + r * d, k + bh * Nk * d, v + bh * Nk * d, i, Nk, d, causal, scale,
                          srow, o + r * d, lse + r);
        }
        free(srow);
    }
    return failed ? -2 : 0;
}

/* Forward on sampled rows: sample s is query row rows[s] of head heads[s]
 * (head index = b * H + h).  o_rows [n, d], lse_rows [n]. */
int oracle_fwd_rows(const double* q, const double* k, const double* v,
                    int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
                    const int64_t* heads, const int64_t* rows, int64_t n,
                    double* o_rows, double* lse_rows) {
    if (!q || !k || !v || !heads || !rows || !o_rows || !lse_rows || bad_shape(B, H, N, d) ||
        n < 0)
        return -1;
    for (int64_t s = 0; s < n; ++s)
        if (heads[s] < 0 || heads[s] >= B * H || rows[s] < 0 || rows[s] >= N) return -1;
    int failed = 0;
#pragma omp parallel
    {
        double* srow = (double*)malloc(sizeof(double) * (size_t)N);
        if (!srow) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t s = 0; s < n; ++s) {
            if (!srow) continue;
            int64_t bh = heads[s], i = rows[s];
            attention_row(q + (bh * N + i) * d, k + bh * N * d, v + bh * N * d, i, N, d,
                          causal, scale, srow, o_rows + s * d, lse_rows + s);
        }
        free(srow);
    }
    return failed ? -2 : 0;
}

/* Attention probabilities P [N, N] of one head (q, k are [N, d]). */
int oracle_probs(const double* q, const double* k, int64_t N, int64_t d, int causal,
                 double scale, double* p) {
    if (!q || !k || !p || bad_shape(1, 1, N, d)) return -1;
    double* o_i = (double*)malloc(sizeof(double) * (size_t)d);
    double* v0 = (double*)calloc((size_t)(N * d), sizeof(double));
    if (!o_i || !v0) {
        free(o_i);
        free(v0);
        return -2;
    }
    double lse;
    for (int64_t i = 0; i < N; ++i)
        attention_row(q + i * d, k, v0, i, N, d, causal, scale, p + i * N, o_i, &lse);
    free(o_i);
    free(v0);
    return 0;
}

/* x rounded to the nearest bfloat16 value (8 significant bits), ties to even.
 * Written for the normal range; zero, infinities and NaN pass through. */
double oracle_round_bf16(double x) {
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    double m = frexp(x, &e);          /* x = m 2^e, 0.5 <= |m| < 1 */
    double r = nearbyint(ldexp(m, 8)); /* default rounding mode: nearest, ties to even */
    return ldexp(r, e - 8);
}

/* x[i] rounded as oracle_round_bf16 rounds it, for i < n. */
int oracle_round_bf16_array(const double* x, int64_t n, double* out) {
    if (n < 0 || (n > 0 && (!x || !out))) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i]);
    return 0;
}

static double stored_output(double x, int o_storage) {
    if (o_storage == 1) return oracle_round_bf16(x);
    if (o_storage == 2) return (double)(float)x;
    return x;
}

/* Backward of one head with explicit N x N matrices.  All pointers are the
 * head's own [N, d] (or [N]) slices.  Scratch: 2 N^2 + N d doubles.  Each
 * loop below is spread over threads by output row; every output element is
 * still one sum in a fixed order, so the result does not depend on the
 * thread count. */
static int backward_head(const double* qh, const double* kh, const double* vh,
                         const double* doh, int64_t N, int64_t d, int causal, double scale,
                         int o_storage, double* dqh, double* dkh, double* dvh, double* dh) {
    double* P = (double*)malloc(sizeof(double) * (size_t)(N * N));
    double* dS = (double*)malloc(sizeof(double) * (size_t)(N * N));
    double* O = (double*)malloc(sizeof(double) * (size_t)(N * d));
    if (!P || !dS || !O) {
        free(P);
        free(dS);
        free(O);
        return -2;
    }
    /* Forward again, keeping P and O (FP64). */
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t i = 0; i < N; ++i) {
        double lse;
        attention_row(qh + i * d, kh, vh, i, N, d, causal, scale, P + i * N, O + i * d, &lse);
    }
    /* dV = P^T dO */
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t i = 0; i < N; ++i) acc += P[i * N + j] * doh[i * d + c];
            dvh[j * d + c] = acc;
        }
    /* D_i = dO_i . O_i, then dS = P o (dP - D), dP_ij = dO_i . V_j */
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t i = 0; i < N; ++i) {
        double Di = 0.0;
        for (int64_t c = 0; c < d; ++c) Di += doh[i * d + c] * stored_output(O[i * d + c], o_storage);
        if (dh) dh[i] = Di;
        for (int64_t j = 0; j < N; ++j) {
            double dP = 0.0;
            for (int64_t c = 0; c < d; ++c) dP += doh[i * d + c] * vh[j * d + c];
            dS[i * N + j] = P[i * N + j] * (dP - Di);
        }
    }
    /* dQ = scale dS K */
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t i = 0; i < N; ++i)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < N; ++j) acc += dS[i * N + j] * kh[j * d + c];
            dqh[i * d + c] = scale * acc;
        }
    /* dK = scale dS^T Q */
#pragma omp parallel for schedule(dynamic, 8)
    for (int64_t j = 0; j < N; ++j)
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int64_t i = 0; i < N; ++i) acc += dS[i * N + j] * qh[i * d + c];
            dkh[j * d + c] = scale * acc;
        }
    free(P);
    free(dS);
    free(O);
    return 0;
}

/* Backward on a list of whole heads.  heads[s] (b * H + h) selects the s-th
 * head computed; heads == NULL means all B*H heads in order.  Outputs are
 * packed per computed head: dq/dk/dv [n, N, d], dvec [n, N] (D, may be NULL).
 * o_storage selects the O that D is formed from (0 exact, 1 bf16, 2 fp32). */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dO,
               int64_t B, int64_t H, int64_t N, int64_t d, int causal, double scale,
               int o_storage, const int64_t* heads, int64_t n, double* dq, double* dk,
               double* dv, double* dvec) {
    if (!q || !k || !v || !dO || !dq || !dk || !dv || bad_shape(B, H, N, d)) return -1;
    if (o_storage < 0 || o_storage > 2) return -1;
    if (!heads) n = B * H;
    if (n < 0) return -1;
    if (heads)
        for (int64_t s = 0; s < n; ++s)
            if (heads[s] < 0 || heads[s] >= B * H) return -1;
    /* Heads one after the other; the threads work inside each head. */
    for (int64_t s = 0; s < n; ++s) {
        int64_t bh = heads ? heads[s] : s;
        int64_t off = bh * N * d;
        int rc = backward_head(q + off, k + off, v + off, dO + off, N, d, causal, scale,
                               o_storage, dq + s * N * d, dk + s * N * d, dv + s * N * d,
                               dvec ? dvec + s * N : NULL);
        if (rc) return rc;
    }
    return 0;
}
