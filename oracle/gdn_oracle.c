/*
 * Gated DeltaNet forward recurrence -- plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the checker, not the product: only
 * the tests, the smoke check and the CPU-baseline leg of the benchmark load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (per sequence n and value head h, independently):
 *
 *   The gated delta rule, as described in words in the podcast episode
 *   "Qwen3.8-Next design: hybrid attention, residuals and n-gram embeddings",
 *   transcript segment 14: a decay alpha first erases part of the whole state,
 *   then the rule reads what is stored under the current key, subtracts it from
 *   the new value and writes only that error (so the same key written twice
 *   leaves one corrected entry). Segment 4 of the same transcript adds that the
 *   state has a fixed size and the cost is linear in the sequence length.
 *
 *   Written out, with the state S of shape d_k x d_v (rows = key dimension):
 *
 *     S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *         = alpha_t S_{t-1} + beta_t k_t (v_t - alpha_t S_{t-1}^T k_t)^T
 *     o_t = scale * S_t^T q_t,            scale = 1/sqrt(d_k) by default
 *
 *   alpha_t = exp(g_t) with g the log-decay input; beta_t is the write
 *   strength. q/k head of value head h is h / (H_v / H_qk) (contiguous
 *   groups). The orientation of S (d_k x d_v, read out through S^T) is the one
 *   reading of the rule under which a written value is retrieved under its key
 *   (S^T k = v for alpha = beta = 1 and a unit key).
 *
 * Two forms are provided:
 *   gdn_oracle_recurrent -- the token-by-token definition above (the oracle).
 *   gdn_oracle_chunked   -- the chunkwise algebra (cumulative log-decay, the
 *                           unit-lower-triangular system (I + A) T = I solved by
 *                           forward substitution, W/U, inter-chunk state) used
 *                           only to pin that algebra against the definition.
 *
 * Inputs: q, k, v are fp32 (dtype 0) or raw bf16 bit patterns (dtype 1,
 * upcast exactly to fp32 then fp64 element by element); g, beta, h0 are fp32.
 * All arithmetic is fp64. Work is split over the requested (n, h) pairs with
 * OpenMP; within a pair it is strictly sequential.
 *
 * Outputs are compact per requested pair p = (n, h): o_out holds, pair after
 * pair, a [len_n, d_v] block; s_out holds a [d_k, d_v] block per pair.
 * o_offsets[p] gives the first row of pair p's block in o_out (the caller
 * computes it as the running sum of the pair lengths).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double elem(const void* p, int dtype, size_t i) {
    if (dtype == 0) return (double)((const float*)p)[i];
    uint32_t bits = ((uint32_t)((const uint16_t*)p)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

typedef struct {
    const void* q; const void* k; const void* v; int dtype;
    const float* g; const float* beta; const float* h0;
    const int32_t* cu; int32_t h_qk, h_v, d_k, d_v; double scale;
} problem;

/* Load the initial state of pair (n, h) into S (zeros when h0 is NULL). */
static void load_state(const problem* P, int n, int h, double* S) {
    size_t sz = (size_t)P->d_k * P->d_v;
    if (!P->h0) { memset(S, 0, sz * sizeof(double)); return; }
    const float* src = P->h0 + ((size_t)n * P->h_v + h) * sz;
    for (size_t i = 0; i < sz; ++i) S[i] = (double)src[i];
}

/* Token-by-token gated delta rule for one (n, h) pair. */
static void run_recurrent(const problem* P, int n, int h, double* o, double* S) {
    const int dk = P->d_k, dv = P->d_v, grp = P->h_v / P->h_qk, hk = h / grp;
    double* kv = (double*)malloc(sizeof(double) * (2 * (size_t)dk + 2 * (size_t)dv));
    double *kk = kv, *qq = kv + dk, *vv = kv + 2 * dk, *err = kv + 2 * dk + dv;
    load_state(P, n, h, S);
    int32_t t0 = P->cu[n], t1 = P->cu[n + 1];
    for (int32_t t = t0; t < t1; ++t) {
        size_t qk_base = ((size_t)t * P->h_qk + hk) * dk;
        size_t v_base = ((size_t)t * P->h_v + h) * dv;
        for (int i = 0; i < dk; ++i) { kk[i] = elem(P->k, P->dtype, qk_base + i); qq[i] = elem(P->q, P->dtype, qk_base + i); }
        for (int j = 0; j < dv; ++j) vv[j] = elem(P->v, P->dtype, v_base + j);
        double alpha = exp((double)P->g[(size_t)t * P->h_v + h]);
        double beta = (double)P->beta[(size_t)t * P->h_v + h];
        /* error = v - (alpha S)^T k : what the decayed state stores under k, subtracted from v */
        for (int j = 0; j < dv; ++j) {
            double read = 0.0;
            for (int i = 0; i < dk; ++i) read += S[(size_t)i * dv + j] * kk[i];
            err[j] = vv[j] - alpha * read;
        }
        /* S = alpha S + beta k error^T */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j)
                S[(size_t)i * dv + j] = alpha * S[(size_t)i * dv + j] + beta * kk[i] * err[j];
        /* o = scale S^T q */
        double* orow = o + (size_t)(t - t0) * dv;
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qq[i];
            orow[j] = P->scale * acc;
        }
    }
    free(kv);
}

/* Chunkwise form for one (n, h) pair. Within a chunk, positions r = 0..L-1,
 * G_r = g_0 + ... + g_r (cumulative log-decay), gamma_r = exp(G_r),
 * Gamma_rs = exp(G_r - G_s) for r >= s (only differences with r >= s are ever
 * exponentiated, so no factor exceeds 1 when g <= 0).
 *   A_rs  = beta_r Gamma_rs k_r.k_s  (s < r), strictly lower
 *   T     = (I + A)^{-1}             (forward substitution, column by column)
 *   W     = T diag(beta gamma) K,    U = T diag(beta) V
 *   Delta = U - W S                  (the written errors of the chunk)
 *   O     = scale (diag(gamma) Q S + (Q K^T o Gamma o [r>=s]) Delta)
 *   S'    = gamma_{L-1} S + (diag(Gamma_{L-1,.}) K)^T Delta
 * A partial last chunk simply has L < C (the same as padding it with rows of
 * g = 0, beta = 0, k = v = 0, which are exact no-ops). */
static void run_chunked(const problem* P, int n, int h, int C, double* o, double* S) {
    const int dk = P->d_k, dv = P->d_v, grp = P->h_v / P->h_qk, hk = h / grp;
    size_t need = (size_t)C * dk * 2 + (size_t)C * dv * 4 + (size_t)C * C * 2 + (size_t)C * 4 + (size_t)C * dk;
    double* buf = (double*)malloc(sizeof(double) * need);
    double *K = buf, *Q = K + (size_t)C * dk, *V = Q + (size_t)C * dk, *U = V + (size_t)C * dv;
    double *D = U + (size_t)C * dv, *OO = D + (size_t)C * dv, *A = OO + (size_t)C * dv, *T = A + (size_t)C * C;
    double *G = T + (size_t)C * C, *B = G + C, *gam = B + C, *x = gam + C, *W = x + C;
    load_state(P, n, h, S);
    int32_t t0 = P->cu[n], t1 = P->cu[n + 1];
    for (int32_t c0 = t0; c0 < t1; c0 += C) {
        int L = (t1 - c0) < C ? (int)(t1 - c0) : C;
        double acc = 0.0;
        for (int r = 0; r < L; ++r) {
            int32_t t = c0 + r;
            size_t qk_base = ((size_t)t * P->h_qk + hk) * dk, v_base = ((size_t)t * P->h_v + h) * dv;
            for (int i = 0; i < dk; ++i) { K[(size_t)r * dk + i] = elem(P->k, P->dtype, qk_base + i); Q[(size_t)r * dk + i] = elem(P->q, P->dtype, qk_base + i); }
            for (int j = 0; j < dv; ++j) V[(size_t)r * dv + j] = elem(P->v, P->dtype, v_base + j);
            acc += (double)P->g[(size_t)t * P->h_v + h];
            G[r] = acc;
            gam[r] = exp(acc);
            B[r] = (double)P->beta[(size_t)t * P->h_v + h];
        }
        /* A (strictly lower) */
        for (int r = 0; r < L; ++r)
            for (int s = 0; s < L; ++s) {
                double a = 0.0;
                if (s < r) {
                    double dot = 0.0;
                    for (int i = 0; i < dk; ++i) dot += K[(size_t)r * dk + i] * K[(size_t)s * dk + i];
                    a = B[r] * exp(G[r] - G[s]) * dot;
                }
                A[(size_t)r * C + s] = a;
            }
        /* T = (I + A)^{-1}: column c solves (I + A) x = e_c by forward substitution */
        for (int c = 0; c < L; ++c) {
            for (int r = 0; r < L; ++r) {
                double xr = (r == c) ? 1.0 : 0.0;
                for (int s = 0; s < r; ++s) xr -= A[(size_t)r * C + s] * x[s];
                x[r] = xr;
            }
            for (int r = 0; r < L; ++r) T[(size_t)r * C + c] = x[r];
        }
        /* W = T diag(beta gamma) K ; U = T diag(beta) V */
        for (int r = 0; r < L; ++r) {
            for (int i = 0; i < dk; ++i) {
                double w = 0.0;
                for (int s = 0; s < L; ++s) w += T[(size_t)r * C + s] * B[s] * gam[s] * K[(size_t)s * dk + i];
                W[(size_t)r * dk + i] = w;
            }
            for (int j = 0; j < dv; ++j) {
                double u = 0.0;
                for (int s = 0; s < L; ++s) u += T[(size_t)r * C + s] * B[s] * V[(size_t)s * dv + j];
                U[(size_t)r * dv + j] = u;
            }
        }
        /* Delta = U - W S */
        for (int r = 0; r < L; ++r)
            for (int j = 0; j < dv; ++j) {
                double ws = 0.0;
                for (int i = 0; i < dk; ++i) ws += W[(size_t)r * dk + i] * S[(size_t)i * dv + j];
                D[(size_t)r * dv + j] = U[(size_t)r * dv + j] - ws;
            }
        /* O = scale (diag(gamma) Q S + (Q K^T o Gamma o causal) Delta) */
        for (int r = 0; r < L; ++r) {
            for (int j = 0; j < dv; ++j) {
                double qs = 0.0;
                for (int i = 0; i < dk; ++i) qs += Q[(size_t)r * dk + i] * S[(size_t)i * dv + j];
                OO[(size_t)r * dv + j] = gam[r] * qs;
            }
            for (int s = 0; s <= r; ++s) {
                double dot = 0.0;
                for (int i = 0; i < dk; ++i) dot += Q[(size_t)r * dk + i] * K[(size_t)s * dk + i];
                double p = dot * exp(G[r] - G[s]);
                for (int j = 0; j < dv; ++j) OO[(size_t)r * dv + j] += p * D[(size_t)s * dv + j];
            }
            double* orow = o + (size_t)(c0 - t0 + r) * dv;
            for (int j = 0; j < dv; ++j) orow[j] = P->scale * OO[(size_t)r * dv + j];
        }
        /* S = gamma_last S + (diag(Gamma_last,.) K)^T Delta */
        double gl = gam[L - 1];
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                double s_new = gl * S[(size_t)i * dv + j];
                for (int s = 0; s < L; ++s) s_new += exp(G[L - 1] - G[s]) * K[(size_t)s * dk + i] * D[(size_t)s * dv + j];
                S[(size_t)i * dv + j] = s_new;
            }
    }
    free(buf);
}

static int check(const problem* P, int32_t N, const int32_t* pairs, int32_t n_pairs) {
    if (!P->q || !P->k || !P->v || !P->g || !P->beta || !P->cu) return 1;
    if (P->h_qk <= 0 || P->h_v <= 0 || P->h_v % P->h_qk || P->d_k <= 0 || P->d_v <= 0) return 2;
    if (P->dtype != 0 && P->dtype != 1) return 3;
    for (int32_t n = 0; n < N; ++n) if (P->cu[n + 1] < P->cu[n]) return 4;
    for (int32_t p = 0; p < n_pairs; ++p)
        if (pairs[2 * p] < 0 || pairs[2 * p] >= N || pairs[2 * p + 1] < 0 || pairs[2 * p + 1] >= P->h_v) return 5;
    return 0;
}

static int run(int chunk, const void* q, const void* k, const void* v, int dtype,
               const float* g, const float* beta, const float* h0, const int32_t* cu, int32_t N,
               int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v, double scale,
               const int32_t* pairs, int32_t n_pairs, const int64_t* o_offsets,
               double* o_out, double* s_out, int32_t n_threads) {
    problem P = {q, k, v, dtype, g, beta, h0, cu, h_qk, h_v, d_k, d_v, scale};
    int bad = check(&P, N, pairs, n_pairs);
    if (bad) return bad;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int32_t p = 0; p < n_pairs; ++p) {
        int n = pairs[2 * p], h = pairs[2 * p + 1];
        double* o = o_out + (size_t)o_offsets[p] * d_v;
        double* S = s_out + (size_t)p * d_k * d_v;
        if (chunk <= 0) run_recurrent(&P, n, h, o, S);
        else run_chunked(&P, n, h, chunk, o, S);
    }
    return 0;
}

int gdn_oracle_recurrent(const void* q, const void* k, const void* v, int dtype,
                         const float* g, const float* beta, const float* h0, const int32_t* cu, int32_t N,
                         int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v, double scale,
                         const int32_t* pairs, int32_t n_pairs, const int64_t* o_offsets,
                         double* o_out, double* s_out, int32_t n_threads) {
    return run(0, q, k, v, dtype, g, beta, h0, cu, N, h_qk, h_v, d_k, d_v, scale,
               pairs, n_pairs, o_offsets, o_out, s_out, n_threads);
}

int gdn_oracle_chunked(const void* q, const void* k, const void* v, int dtype,
                       const float* g, const float* beta, const float* h0, const int32_t* cu, int32_t N,
                       int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v, double scale, int32_t chunk,
                       const int32_t* pairs, int32_t n_pairs, const int64_t* o_offsets,
                       double* o_out, double* s_out, int32_t n_threads) {
    if (chunk <= 0) return 6;
    return run(chunk, q, k, v, dtype, g, beta, h0, cu, N, h_qk, h_v, d_k, d_v, scale,
               pairs, n_pairs, o_offsets, o_out, s_out, n_threads);
}

int gdn_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
