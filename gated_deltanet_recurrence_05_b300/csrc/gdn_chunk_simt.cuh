// Chunkwise-parallel prefill on CUDA cores, all arithmetic in fp32.
//
// Serves fp32 inputs (whose tolerance a bf16/tf32 tensor-core path cannot
// meet), head sizes other than 128, and cross-checks of the tensor-core
// kernel. One CTA per (sequence, value head, d_v tile of up to 64 columns);
// state columns evolve independently, so tiling d_v only repeats the
// d_v-independent work (K K^T, the triangular solve, W).
//
// Per chunk of C tokens (positions r, s in 0..C-1, G = cumulative log-decay
// within the chunk, gamma_r = exp(G_r), Gamma_rs = exp(G_r - G_s) for r >= s):
//   A     = strictly-lower( diag(beta) (Gamma o K K^T) )
//   T     = (I + A)^{-1}                     (forward substitution, per column)
//   W     = T diag(beta gamma) K,  U = T diag(beta) V
//   Delta = U - W S                          (errors written by the chunk)
//   O     = scale (diag(gamma) Q S + (Q K^T o Gamma o causal) Delta)
//   S    <- gamma_{last} S + (diag(Gamma_{last,.}) K)^T Delta
// This unrolls the per-token rule (the decay erases the whole state, the
// delta term writes only the error under the current key; "Qwen3.8-Next
// design" podcast transcript, segment 14) over one chunk: with
// delta_r = beta_r (v_r - alpha_r S_{r-1}^T k_r) one gets
// (I + A) Delta = diag(beta) V - diag(beta gamma) K S. Only exponentials of
// G_r - G_s with r >= s are formed, so no factor exceeds 1 for g <= 0.
// A ragged last chunk is handled as if padded with rows g = 0, beta = 0,
// k = v = 0 (exact no-ops); padded outputs are not stored.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

struct SimtArgs {
    const void* q; const void* k; const void* v;
    const float* g; const float* beta; const float* h0;
    const int32_t* cu; const int32_t* order;
    void* o; float* hT;
    int num_seqs; long long total; long long eq_len;
    int h_qk, h_v, d_k, d_v, grp, C, dvt, n_tiles;
    float scale;
};

// Shared-memory footprint in floats for (C, d_k, dvt).
__host__ __device__ inline size_t simt_smem_floats(int C, int d_k, int dvt) {
    const int ldk = d_k + 1;
    return (size_t)d_k * dvt            // S tile
         + 2 * (size_t)C * ldk          // K, Q (padded rows)
         + (size_t)C * dvt              // V tile
         + 3 * (size_t)C * C            // A, P, T
         + (size_t)C * d_k              // W
         + (size_t)C * dvt              // U / Delta
         + 3 * (size_t)C;               // G, gamma, beta
}

template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256)
chunk_simt_kernel(SimtArgs p) {
    extern __shared__ float smem[];
    const int C = p.C, d_k = p.d_k, d_v = p.d_v, dvt = p.dvt, ldk = d_k + 1;
    const int tile = blockIdx.x % p.n_tiles;
    const int unit = blockIdx.x / p.n_tiles;
    const int h = unit % p.h_v;
    const int pos = unit / p.h_v;
    int n;
    if (!seq_of(p.order, pos, p.num_seqs, n)) return;
    long long t0, t1;
    if (!seq_bounds(p.cu, n, p.num_seqs, p.total, p.eq_len, t0, t1)) return;
    const int hk = h / p.grp;
    const int j0 = tile * dvt;
    const int nj = min(dvt, d_v - j0);
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    const TIn* v = static_cast<const TIn*>(p.v);
    TOut* o = static_cast<TOut*>(p.o);

    float* S = smem;                       // [d_k][dvt]
    float* K = S + (size_t)d_k * dvt;      // [C][ldk]
    float* Q = K + (size_t)C * ldk;        // [C][ldk]
    float* V = Q + (size_t)C * ldk;        // [C][dvt]
    float* A = V + (size_t)C * dvt;        // [C][C]
    float* P = A + (size_t)C * C;          // [C][C]
    float* T = P + (size_t)C * C;          // [C][C]
    float* W = T + (size_t)C * C;          // [C][d_k]
    float* U = W + (size_t)C * d_k;        // [C][dvt]  (U, then Delta)
    float* G = U + (size_t)C * dvt;        // [C]
    float* gam = G + C;                    // [C]
    float* bet = gam + C;                  // [C]
    const int tid = threadIdx.x, nth = blockDim.x;

    // initial state tile
    const size_t sbase = ((size_t)n * p.h_v + h) * d_k * d_v;
    for (int e = tid; e < d_k * dvt; e += nth) {
        const int i = e / dvt, j = e % dvt;
        S[e] = (p.h0 && j < nj) ? p.h0[sbase + (size_t)i * d_v + j0 + j] : 0.f;
    }

    for (long long c0 = t0; c0 < t1; c0 += C) {
        const int L = (int)min((long long)C, t1 - c0);
        __syncthreads();
        for (int e = tid; e < C * d_k; e += nth) {
            const int r = e / d_k, i = e % d_k;
            float kv = 0.f, qv = 0.f;
            if (r < L) {
                const size_t a = ((size_t)(c0 + r) * p.h_qk + hk) * d_k + i;
                kv = to_f32(k[a]);
                qv = to_f32(q[a]);
            }
            K[r * ldk + i] = kv;
            Q[r * ldk + i] = qv;
        }
        for (int e = tid; e < C * dvt; e += nth) {
            const int r = e / dvt, j = e % dvt;
            V[e] = (r < L && j < nj) ? to_f32(v[((size_t)(c0 + r) * p.h_v + h) * d_v + j0 + j]) : 0.f;
        }
        if (tid < C) {
            const int r = tid;
            G[r] = r < L ? p.g[(size_t)(c0 + r) * p.h_v + h] : 0.f;
            bet[r] = r < L ? p.beta[(size_t)(c0 + r) * p.h_v + h] : 0.f;
        }
        __syncthreads();
        if (tid == 0) {  // cumulative log-decay (C <= 64 terms)
            float acc = 0.f;
            for (int r = 0; r < C; ++r) { acc += G[r]; G[r] = acc; }
        }
        __syncthreads();
        if (tid < C) gam[tid] = expf(G[tid]);
        // A (strictly lower, decayed, beta-scaled) and P (causal, decayed)
        for (int e = tid; e < C * C; e += nth) {
            const int r = e / C, s = e % C;
            float a = 0.f, pp = 0.f;
            if (s <= r) {
                float kk = 0.f, qk = 0.f;
                for (int i = 0; i < d_k; ++i) {
                    const float ks = K[s * ldk + i];
                    kk = fmaf(K[r * ldk + i], ks, kk);
                    qk = fmaf(Q[r * ldk + i], ks, qk);
                }
                const float dec = expf(G[r] - G[s]);
                pp = qk * dec;
                if (s < r) a = bet[r] * dec * kk;
            }
            A[e] = a;
            P[e] = pp;
        }
        __syncthreads();
        // T = (I + A)^{-1}: thread c solves column c by forward substitution
        if (tid < C) {
            const int c = tid;
            for (int r = 0; r < C; ++r) {
                float x = (r == c) ? 1.f : 0.f;
                for (int s = c; s < r; ++s) x = fmaf(-A[r * C + s], T[s * C + c], x);
                T[r * C + c] = x;
            }
        }
        __syncthreads();
        // W = T diag(beta gamma) K ; U = T diag(beta) V
        for (int e = tid; e < C * d_k; e += nth) {
            const int r = e / d_k, i = e % d_k;
            float w = 0.f;
            for (int s = 0; s <= r; ++s) w = fmaf(T[r * C + s] * bet[s] * gam[s], K[s * ldk + i], w);
            W[e] = w;
        }
        for (int e = tid; e < C * dvt; e += nth) {
            const int r = e / dvt, j = e % dvt;
            float u = 0.f;
            for (int s = 0; s <= r; ++s) u = fmaf(T[r * C + s] * bet[s], V[s * dvt + j], u);
            U[e] = u;
        }
        __syncthreads();
        // Delta = U - W S
        for (int e = tid; e < C * dvt; e += nth) {
            const int r = e / dvt, j = e % dvt;
            float ws = 0.f;
            for (int i = 0; i < d_k; ++i) ws = fmaf(W[r * d_k + i], S[i * dvt + j], ws);
            U[e] -= ws;
        }
        __syncthreads();
        // O = scale (diag(gamma) Q S + P Delta)
        for (int e = tid; e < C * dvt; e += nth) {
            const int r = e / dvt, j = e % dvt;
            if (r >= L || j >= nj) continue;
            float qs = 0.f;
            for (int i = 0; i < d_k; ++i) qs = fmaf(Q[r * ldk + i], S[i * dvt + j], qs);
            float acc = gam[r] * qs;
            for (int s = 0; s <= r; ++s) acc = fmaf(P[r * C + s], U[s * dvt + j], acc);
            o[((size_t)(c0 + r) * p.h_v + h) * d_v + j0 + j] = from_f32<TOut>(p.scale * acc);
        }
        __syncthreads();
        // S <- gamma_last S + (diag(Gamma_last,.) K)^T Delta; beta is no longer
        // needed this chunk, so its slot holds Gamma_last,s.
        const float gl = gam[L - 1];
        if (tid < C) bet[tid] = tid < L ? expf(G[L - 1] - G[tid]) : 0.f;
        __syncthreads();
        for (int e = tid; e < d_k * dvt; e += nth) {
            const int i = e / dvt, j = e % dvt;
            float acc = gl * S[e];
            for (int s = 0; s < L; ++s) acc = fmaf(bet[s] * K[s * ldk + i], U[s * dvt + j], acc);
            S[e] = acc;
        }
    }
    __syncthreads();
    if (p.hT) {
        for (int e = tid; e < d_k * dvt; e += nth) {
            const int i = e / dvt, j = e % dvt;
            if (j < nj) p.hT[sbase + (size_t)i * d_v + j0 + j] = S[e];
        }
    }
}

}  // namespace gdn
