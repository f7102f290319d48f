// Input prologue of a GDN layer: short causal depthwise convolution over the
// tokens of each sequence, SiLU, and (for q and k) an L2 norm per head,
//     u[t, c] = sum_{i<K} w[c, i] x[t - (K-1) + i, c],  s = silu(u),
//     y[t, head] = s[t, head] / sqrt(sum_head s^2 + eps).
// The pages say only that GDN adds "short causal convolutions" ("Qwen3.8-Next
// design: hybrid attention, residuals and n-gram embeddings", transcript
// segment 14) and feed the rule L2-normalised q and k. The past of a
// sequence's first tokens is the caller's conv state (its K-1 preceding
// inputs, oldest first) or zero; the final state is the last K-1 inputs.
//
// One warp per (token, block of 128 channels): lane l owns channels
// 128 b + 4 l .. + 3 (one vector load per tap), so a head of up to 128
// channels is reduced inside the warp. Both kernels are HBM-bound: x is read
// once from DRAM (the K taps of neighbouring tokens hit L1/L2) and y written
// once.
#pragma once

#include "gdn_common.cuh"
#include "gdn_epilogue.cuh"  // sigmoid_fast

namespace gdn {

__device__ __forceinline__ float silu_f(float u) { return u * sigmoid_fast(u); }

__device__ __forceinline__ void load4f(const __nv_bfloat16* p, float* v) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xffff0000u);
    v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void load4f(const float* p, float* v) {
    const float4 f = *reinterpret_cast<const float4*>(p);
    v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
}
__device__ __forceinline__ void store4f(__nv_bfloat16* p, const float* v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), b = __floats2bfloat162_rn(v[2], v[3]);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void store4f(float* p, const float* v) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

// V consecutive elements (V = 4 or 8) as fp32.
template <int V, typename T> __device__ __forceinline__ void loadVf(const T* p, float* v) {
#pragma unroll
    for (int h = 0; h < V / 4; ++h) load4f(p + 4 * h, v + 4 * h);
}
template <int V, typename T> __device__ __forceinline__ void storeVf(T* p, const float* v) {
#pragma unroll
    for (int h = 0; h < V / 4; ++h) store4f(p + 4 * h, v + 4 * h);
}

// silu, then the L2 norm over groups of `ng` channels (ng = 0: none; else a
// power of two, at least V, dividing 32 V: the group spans ng / V lanes)
template <int V>
__device__ __forceinline__ void silu_norm(float* s, int ng, float eps) {
#pragma unroll
    for (int j = 0; j < V; ++j) s[j] = silu_f(s[j]);
    if (ng) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j) ss = fmaf(s[j], s[j], ss);
        for (int off = 1; off < ng / V; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float r = rsqrtf(ss + eps);
#pragma unroll
        for (int j = 0; j < V; ++j) s[j] *= r;
    }
}

// Sequence of token t: cu == nullptr means num_seqs sequences of eq_len.
__device__ __forceinline__ int seq_of_token(const int32_t* cu, int num_seqs, long long eq_len, long long t) {
    if (cu == nullptr) return (int)(t / eq_len);
    int lo = 0, hi = num_seqs;  // cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

// Each warp filters a run of RUN consecutive tokens for one block of 32 V
// channels (V per lane: 4, or 8 when C and the head size allow): the taps
// slide through registers (one load and one store per token), the weights are
// loaded once per run, and a run crossing into the next sequence restarts its
// window from that sequence's state.
template <typename T, int K, int V>
__global__ void __launch_bounds__(256)
short_conv_kernel(const T* __restrict__ x, const float* __restrict__ w, T* __restrict__ y,
                  const int32_t* __restrict__ cu, const float* __restrict__ st_in, float* __restrict__ st_out,
                  int num_seqs, long long total, long long eq_len, int C, int ng, float eps) {
    constexpr int RUN = 32;
    const int lane = threadIdx.x & 31;
    const int c = (int)blockIdx.y * (32 * V) + V * lane;
    const bool live = c < C;  // C % V == 0: a lane's V channels are all in or all out
    float wv[V][K];
#pragma unroll
    for (int j = 0; j < V; ++j)
#pragma unroll
        for (int i = 0; i < K; ++i) wv[j][i] = live ? w[(size_t)(c + j) * K + i] : 0.f;
    const long long runs = (total + RUN - 1) / RUN;
    for (long long rr = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); rr < runs; rr += (long long)gridDim.x * 8) {
        const long long ta = rr * RUN, tb = ta + RUN < total ? ta + RUN : total;
        int n = seq_of_token(cu, num_seqs, eq_len, ta);
        long long t0 = cu ? cu[n] : (long long)n * eq_len;
        long long t1 = cu ? cu[n + 1] : t0 + eq_len;
        float win[K][V];  // win[i] = input at t - (K-1) + i
        bool bad = false;
        auto restart = [&](long long t) {  // window for token t of sequence n
#pragma unroll
            for (int i = 0; i < K - 1; ++i) {
                const long long p = t - (K - 1) + i;
                if (!live) {
#pragma unroll
                    for (int j = 0; j < V; ++j) win[i][j] = 0.f;
                } else if (p >= t0) {
                    loadVf<V>(x + p * C + c, win[i]);
                } else if (st_in) {  // the caller's past: entry p - t0 + K - 1
                    const float* sp = st_in + ((size_t)n * C + c) * (K - 1) + (p - t0 + K - 1);
#pragma unroll
                    for (int j = 0; j < V; ++j) win[i][j] = sp[j * (K - 1)];
                } else {
#pragma unroll
                    for (int j = 0; j < V; ++j) win[i][j] = 0.f;
                }
            }
        };
        if (ta < t0 || ta >= t1 || t0 < 0 || t1 > total) bad = true;
        if (!bad) restart(ta);
        // the run's inputs in batches of 8 tokens, loaded before they are used
        constexpr int BATCH = V == 4 ? 8 : 4;
        float xb[BATCH][V];
        for (long long tq = ta; tq < tb && !bad; tq += BATCH) {
#pragma unroll
            for (int k = 0; k < BATCH; ++k) {
                if (live && tq + k < tb) loadVf<V>(x + (tq + k) * C + c, xb[k]);
                else {
#pragma unroll
                    for (int j = 0; j < V; ++j) xb[k][j] = 0.f;
                }
            }
#pragma unroll
            for (int k = 0; k < BATCH; ++k) {
                const long long t = tq + k;
                if (t >= tb || bad) break;
                while (t >= t1) {  // next non-empty sequence (warp-uniform)
                    ++n;
                    if (n >= num_seqs) { bad = true; break; }
                    t0 = cu ? cu[n] : (long long)n * eq_len;
                    t1 = cu ? cu[n + 1] : t0 + eq_len;
                    if (t0 != t || t1 > total) { bad = true; break; }
                    if (t < t1) restart(t);
                }
                if (bad) break;
#pragma unroll
                for (int j = 0; j < V; ++j) win[K - 1][j] = xb[k][j];
                float acc[V];
#pragma unroll
                for (int j = 0; j < V; ++j) {
                    float a = 0.f;
#pragma unroll
                    for (int i = 0; i < K; ++i) a = fmaf(wv[j][i], win[i][j], a);
                    acc[j] = a;
                }
                silu_norm<V>(acc, ng, eps);  // every lane takes part in the shuffles
                if (live) {
                    storeVf<V>(y + t * C + c, acc);
                    if (st_out && t == t1 - 1) {  // the K-1 newest inputs become the state
                        float* so = st_out + ((size_t)n * C + c) * (K - 1);
#pragma unroll
                        for (int i = 1; i < K; ++i)
#pragma unroll
                            for (int j = 0; j < V; ++j) so[j * (K - 1) + (i - 1)] = win[i][j];
                    }
                }
#pragma unroll
                for (int i = 0; i < K - 1; ++i)
#pragma unroll
                    for (int j = 0; j < V; ++j) win[i][j] = win[i + 1][j];
            }
        }
        if (bad && lane == 0) set_device_error(1u);  // cu_seqlens not ascending or out of range
    }
}

// Empty sequences keep their state (st_out = st_in, or zero); cu == nullptr:
// every sequence is empty.
__global__ void conv_state_carry_kernel(const int32_t* __restrict__ cu, const float* __restrict__ st_in,
                                        float* __restrict__ st_out, int num_seqs, long long per_seq) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)num_seqs * per_seq) return;
    const int n = (int)(i / per_seq);
    if (cu && cu[n + 1] != cu[n]) return;
    st_out[i] = st_in ? st_in[i] : 0.f;
}

// One token per sequence: state [N, C, K-1] fp32 (oldest first) is read and
// shifted in place.
template <typename T, int K>
__global__ void __launch_bounds__(256)
short_conv_step_kernel(const T* __restrict__ x, const float* __restrict__ w, float* __restrict__ st,
                       T* __restrict__ y, int num_seqs, int C, int ng, float eps) {
    const int lane = threadIdx.x & 31;
    const int nblk = (C + 127) >> 7;
    const long long units = (long long)num_seqs * nblk;
    for (long long u = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); u < units; u += (long long)gridDim.x * 8) {
        const int n = (int)(u / nblk);
        const int c = ((int)(u - (long long)n * nblk) << 7) + 4 * lane;
        const bool live = c < C;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (live) {
            float xv[4];
            load4f(x + (size_t)n * C + c, xv);
            float* sp = st + ((size_t)n * C + c) * (K - 1);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float s[K];
#pragma unroll
                for (int i = 0; i < K - 1; ++i) s[i] = sp[j * (K - 1) + i];
                s[K - 1] = xv[j];
                const float* wr = w + (size_t)(c + j) * K;
#pragma unroll
                for (int i = 0; i < K; ++i) acc[j] = fmaf(wr[i], s[i], acc[j]);
#pragma unroll
                for (int i = 0; i < K - 1; ++i) sp[j * (K - 1) + i] = s[i + 1];
            }
        }
        silu_norm<4>(acc, ng, eps);
        if (live) store4f(y + (size_t)n * C + c, acc);
    }
}

}  // namespace gdn
