// Decode step of the gated delta rule: one token for N independent sequences.
//
// Per (sequence n, value head h), with S the d_k x d_v fp32 state:
//   kS = S^T k, qS = S^T q                     (one read of S)
//   u  = beta (v - alpha kS)                   (the written error)
//   S' = alpha S + k u^T                       (written back in place)
//   o  = scale S'^T q = scale (alpha qS + (k.q) u)
// The last identity lets the output come from the same single pass over S.
// This is the gated delta rule of "Qwen3.8-Next design: hybrid attention,
// residuals and n-gram embeddings" (podcast transcript, segment 14) applied
// to one token; the decode cost axis is the one named in the abstract of
// "On the Design of Qwen3.8-Next Architecture".
#pragma once

#include "gdn_common.cuh"
#include "gdn_epilogue.cuh"

namespace gdn {

// d_k = d_v = 128 fast path. One CTA of 8 warps per (n, h); warp w owns state
// columns [16w, 16w + 16). Lane l holds the 4 columns 16w + 4(l % 4) .. +3 of
// rows (l / 4) + 8m, m = 0..15, i.e. 64 fp32 state values in registers. Every
// state access is a 128-bit load/store; a warp instruction touches 8 rows x
// 64 contiguous bytes. The reductions over rows finish with 3 xor-shuffles
// over the lane bits that select the row; no shared-memory reduction and no
// block-wide barrier beyond the one that publishes k and q.
// GATED: o is written through the epilogue of gdn_epilogue.cuh (zero-centred
// RMSNorm over the 128 features of the head, times sigmoid(z)); its sum of
// squares takes two more shuffles and one block barrier.
template <typename TIn, typename TOut, bool GATED = false>
__global__ void __launch_bounds__(256, 2)
decode_d128_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                   const TIn* __restrict__ v, const float* __restrict__ g,
                   const float* __restrict__ beta, float* __restrict__ state,
                   TOut* __restrict__ o, int h_qk, int h_v, int grp, float scale,
                   const TIn* __restrict__ zg = nullptr, const float* __restrict__ wn = nullptr,
                   float eps = 0.f) {
    constexpr int D = 128;
    const int nh = blockIdx.x;
    const int n = nh / h_v;
    const int h = nh - n * h_v;
    const int hk = h / grp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = lane >> 2;
    const int col = warp * 16 + (lane & 3) * 4;

    float* S = state + (size_t)nh * D * D;
    float4 s[16];
#pragma unroll
    for (int m = 0; m < 16; ++m)
        s[m] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(r0 + 8 * m) * D + col));

    __shared__ float sk[D], sq[D];
    {
        const size_t base = ((size_t)n * h_qk + hk) * D;
        const int t = threadIdx.x & (D - 1);
        if (threadIdx.x < D) sk[t] = to_f32(k[base + t]);
        else sq[t] = to_f32(q[base + t]);
    }
    const float a = expf(g[nh]);
    const float b = beta[nh];
    float vv[4];
    {
        const TIn* vp = v + (size_t)nh * D + col;
#pragma unroll
        for (int c = 0; c < 4; ++c) vv[c] = to_f32(vp[c]);
    }
    __syncthreads();

    float ks[4] = {0.f, 0.f, 0.f, 0.f}, qs[4] = {0.f, 0.f, 0.f, 0.f}, kq = 0.f;
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float ki = sk[r0 + 8 * m], qi = sq[r0 + 8 * m];
        ks[0] = fmaf(s[m].x, ki, ks[0]); ks[1] = fmaf(s[m].y, ki, ks[1]);
        ks[2] = fmaf(s[m].z, ki, ks[2]); ks[3] = fmaf(s[m].w, ki, ks[3]);
        qs[0] = fmaf(s[m].x, qi, qs[0]); qs[1] = fmaf(s[m].y, qi, qs[1]);
        qs[2] = fmaf(s[m].z, qi, qs[2]); qs[3] = fmaf(s[m].w, qi, qs[3]);
        kq = fmaf(ki, qi, kq);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            ks[c] += __shfl_xor_sync(0xffffffffu, ks[c], off);
            qs[c] += __shfl_xor_sync(0xffffffffu, qs[c], off);
        }
        kq += __shfl_xor_sync(0xffffffffu, kq, off);
    }
    float u[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = b * (vv[c] - a * ks[c]);

#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float ki = sk[r0 + 8 * m];
        float4 t;
        t.x = fmaf(a, s[m].x, ki * u[0]);
        t.y = fmaf(a, s[m].y, ki * u[1]);
        t.z = fmaf(a, s[m].z, ki * u[2]);
        t.w = fmaf(a, s[m].w, ki * u[3]);
        __stcs(reinterpret_cast<float4*>(S + (size_t)(r0 + 8 * m) * D + col), t);
    }
    float ov[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) ov[c] = scale * fmaf(a, qs[c], kq * u[c]);
    if constexpr (GATED) {
        // lanes with equal lane % 4 hold the same columns: the warp's 16
        // columns are summed over lane bits 0-1, the 8 warps through smem
        __shared__ float red[8];
        float ss = ov[0] * ov[0] + ov[1] * ov[1] + ov[2] * ov[2] + ov[3] * ov[3];
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) tot += red[i];
        const float rinv = rsqrtf(fmaf(tot, 1.0f / D, eps));
        if (r0 == 0) {
            const TIn* zp = zg + (size_t)nh * D + col;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float sc = wn ? 1.0f + wn[col + c] : 1.0f;
                ov[c] = ov[c] * rinv * sc * sigmoid_f(to_f32(zp[c]));
            }
        }
    }
    if (r0 == 0) {
        TOut* op = o + (size_t)nh * D + col;
#pragma unroll
        for (int c = 0; c < 4; ++c) op[c] = from_f32<TOut>(ov[c]);
    }
}

// Any d_k, d_v <= 128: one CTA per (n, h), thread j owns state column j and
// walks the rows (column accesses are coalesced across the threads). Two
// passes over S (read for the reductions, then read-modify-write).
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(128)
decode_generic_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                      const TIn* __restrict__ v, const float* __restrict__ g,
                      const float* __restrict__ beta, float* __restrict__ state,
                      TOut* __restrict__ o, int h_qk, int h_v, int grp, int d_k, int d_v,
                      float scale) {
    const int nh = blockIdx.x;
    const int n = nh / h_v;
    const int h = nh - n * h_v;
    const int hk = h / grp;
    __shared__ float sk[128], sq[128], red[128];
    const size_t base = ((size_t)n * h_qk + hk) * d_k;
    for (int i = threadIdx.x; i < d_k; i += blockDim.x) {
        sk[i] = to_f32(k[base + i]);
        sq[i] = to_f32(q[base + i]);
    }
    __syncthreads();
    // k.q (block reduction over d_k)
    float part = 0.f;
    for (int i = threadIdx.x; i < d_k; i += blockDim.x) part += sk[i] * sq[i];
    red[threadIdx.x] = part;
    __syncthreads();
    for (int w = 64; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    const float kq = red[0];
    const float a = expf(g[nh]);
    const float b = beta[nh];
    float* S = state + (size_t)nh * d_k * d_v;
    for (int j = threadIdx.x; j < d_v; j += blockDim.x) {
        float ks = 0.f, qs = 0.f;
        for (int i = 0; i < d_k; ++i) {
            const float sij = S[(size_t)i * d_v + j];
            ks = fmaf(sij, sk[i], ks);
            qs = fmaf(sij, sq[i], qs);
        }
        const float u = b * (to_f32(v[(size_t)nh * d_v + j]) - a * ks);
        for (int i = 0; i < d_k; ++i) {
            float* p = S + (size_t)i * d_v + j;
            *p = fmaf(a, *p, sk[i] * u);
        }
        o[(size_t)nh * d_v + j] = from_f32<TOut>(scale * fmaf(a, qs, kq * u));
    }
}

}  // namespace gdn
