// Per-channel-decay variant of the gated delta rule (KDA). The pages name KDA
// only as the alternative linear mixer ("Qwen3.8 attention gate" page,
// blueprint component "Gated DeltaNet / KDA"); the rule implemented is the
// gated delta rule of "Qwen3.8-Next design: hybrid attention, residuals and
// n-gram embeddings" (podcast transcript, segment 14) with one decay per key
// channel, S of shape d_k x d_v:
//
//   S~  = diag(a_t) S_{t-1},  a_t = exp(g_t) in R^{d_k}
//   e_t = v_t - S~^T k_t,     S_t = S~ + b_t k_t e_t^T,     o_t = scale S_t^T q_t
//
// Since S~^T x = S^T (a o x), the reads use a o k and a o q, and
// S_t^T q = S^T (a o q) + (k . q) u with u = b e: one pass over S for both
// reads, one for the update. d_k = d_v = 128.
#pragma once

#include "gdn_common.cuh"
#include "gdn_epilogue.cuh"
#include "gdn_backward.cuh"

namespace gdn {
namespace kda {

constexpr int D = 128;
constexpr int BLK = 32;        // tokens staged per block
constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int RED = 132;

// Decode step: one CTA of 8 warps per (n, h), the layout of decode_d128_kernel
// (warp w owns columns 16w..16w+15; lane l holds 4 columns of rows
// (l / 4) + 8m, m = 0..15), one read and one write of each state.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(256, 2)
kda_decode_d128_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k, const TIn* __restrict__ v,
                       const float* __restrict__ g, const float* __restrict__ beta, float* __restrict__ state,
                       TOut* __restrict__ o, int h_qk, int h_v, int grp, float scale) {
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

    __shared__ float sk[D], sak[D], saq[D], sa[D];
    if (threadIdx.x < D) {
        const int i = threadIdx.x;
        const size_t base = ((size_t)n * h_qk + hk) * D + i;
        const float a = expf(g[(size_t)nh * D + i]);
        const float ki = to_f32(k[base]);
        sk[i] = ki;
        sa[i] = a;
        sak[i] = a * ki;
        saq[i] = a * to_f32(q[base]);
    }
    const float b = beta[nh];
    float vv[4];
    {
        const TIn* vp = v + (size_t)nh * D + col;
#pragma unroll
        for (int c = 0; c < 4; ++c) vv[c] = to_f32(vp[c]);
    }
    float kq = 0.f;  // k . q, from the unscaled q
    {
        const size_t base = ((size_t)n * h_qk + hk) * D + 4 * lane;
        const float4 k4 = load4(k + base), q4 = load4(q + base);
        kq = warp_sum(k4.x * q4.x + k4.y * q4.y + k4.z * q4.z + k4.w * q4.w);
    }
    __syncthreads();

    float ks[4] = {0.f, 0.f, 0.f, 0.f}, qs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float ki = sak[r0 + 8 * m], qi = saq[r0 + 8 * m];
        ks[0] = fmaf(s[m].x, ki, ks[0]); ks[1] = fmaf(s[m].y, ki, ks[1]);
        ks[2] = fmaf(s[m].z, ki, ks[2]); ks[3] = fmaf(s[m].w, ki, ks[3]);
        qs[0] = fmaf(s[m].x, qi, qs[0]); qs[1] = fmaf(s[m].y, qi, qs[1]);
        qs[2] = fmaf(s[m].z, qi, qs[2]); qs[3] = fmaf(s[m].w, qi, qs[3]);
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            ks[c] += __shfl_xor_sync(0xffffffffu, ks[c], off);
            qs[c] += __shfl_xor_sync(0xffffffffu, qs[c], off);
        }
    }
    float u[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) u[c] = b * (vv[c] - ks[c]);
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const float ki = sk[r0 + 8 * m], ai = sa[r0 + 8 * m];
        float4 t;
        t.x = fmaf(ai, s[m].x, ki * u[0]);
        t.y = fmaf(ai, s[m].y, ki * u[1]);
        t.z = fmaf(ai, s[m].z, ki * u[2]);
        t.w = fmaf(ai, s[m].w, ki * u[3]);
        __stcs(reinterpret_cast<float4*>(S + (size_t)(r0 + 8 * m) * D + col), t);
    }
    if (r0 == 0) {
        TOut* op = o + (size_t)nh * D + col;
#pragma unroll
        for (int c = 0; c < 4; ++c) op[c] = from_f32<TOut>(scale * fmaf(kq, u[c], qs[c]));
    }
}

// Prefill: one CTA of 256 threads per (sequence, value head) walks the
// sequence token by token with the state in registers (thread: rows
// 16w..16w+15, columns 4l..4l+3); blocks of 32 tokens are staged in shared
// memory with a o k, a o q, a and k . q precomputed. Two block barriers per
// token (one column-sum exchange for both reads, one to publish u).
constexpr int OFF_K = 0;
constexpr int OFF_AK = OFF_K + BLK * D;
constexpr int OFF_AQ = OFF_AK + BLK * D;
constexpr int OFF_A = OFF_AQ + BLK * D;
constexpr int OFF_V = OFF_A + BLK * D;
constexpr int OFF_U = OFF_V + BLK * D;
constexpr int OFF_RED = OFF_U + D;
constexpr int OFF_B = OFF_RED + 2 * NW * RED;
constexpr int OFF_KQ = OFF_B + BLK;
constexpr int SMEM_FLOATS = OFF_KQ + BLK;
constexpr size_t SMEM_BYTES = (size_t)SMEM_FLOATS * sizeof(float);

struct Args {
    const void* q; const void* k; const void* v;
    const float* g; const float* beta; const float* h0;
    const int32_t* cu; const int32_t* order;
    void* o; float* hT;
    long long total, eq_len;
    int num_seqs, h_qk, h_v, grp;
    float scale;
    int nseg;          // segments per sequence (one CTA each; 1 = the whole sequence)
    long long bal_tokens;  // > 0: equal lengths; every grp CTAs take this many consecutive tokens of the
                           // (sequence, q/k head) groups in order, one CTA per value head of the group
                           // (at most two pieces of units each); nseg = 1
};

// First token to process for a segment whose outputs start at token a of a
// sequence starting at s0 (one warp; every lane returns it). Token t maps a
// difference of states D to (I - beta_t k_t k_t^T) diag(alpha_t) D, whose
// spectral norm is at most max_i alpha_ti max(1, |1 - beta_t |k_t|^2|) times
// that of D; the result is the nearest ts at which the product of these
// factors over ts .. a - 1 is below 2^-40, or s0 (exact) if it never is.
template <typename TIn>
__device__ __forceinline__ long long segment_prefix_start(const Args& p, long long s0, long long a, int h, int hk,
                                                          int lane) {
    constexpr float LN_EPS = -27.7258872f;  // 40 ln 2
    const TIn* k = static_cast<const TIn*>(p.k);
    float acc = 0.f;
    for (long long p0 = a; p0 > s0; p0 -= 32) {
        const long long tok = p0 - 1 - lane;
        const bool valid = tok >= s0;
        float c = 0.f;
        if (valid) {
            const float* gp = p.g + ((size_t)tok * p.h_v + h) * D;
            const TIn* kp = k + ((size_t)tok * p.h_qk + hk) * D;
            float gmax = -INFINITY, ss = 0.f;
#pragma unroll 4
            for (int i = 0; i < D; i += 4) {
                const float4 g4 = *reinterpret_cast<const float4*>(gp + i);
                gmax = fmaxf(gmax, fmaxf(fmaxf(g4.x, g4.y), fmaxf(g4.z, g4.w)));
                const float4 k4 = load4(kp + i);
                ss = fmaf(k4.x, k4.x, fmaf(k4.y, k4.y, fmaf(k4.z, k4.z, fmaf(k4.w, k4.w, ss))));
            }
            const float f = fabsf(1.f - p.beta[(size_t)tok * p.h_v + h] * ss);
            c = gmax + (f > 1.f ? logf(f) : 0.f);
        }
        float incl = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, valid && acc + incl <= LN_EPS);
        if (hit) return p0 - 1 - (__ffs(hit) - 1);
        acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    return s0;
}

template <typename TIn>
__device__ __forceinline__ void kda_stage(float* sm, const Args& p, long long tb0, int n, int h, int hk) {
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    const TIn* v = static_cast<const TIn*>(p.v);
    for (int idx = threadIdx.x; idx < BLK * (D / 4); idx += NT) {
        const int j = idx >> 5, c = (idx & 31) * 4;
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), qq = kk, vv = kk, aa = make_float4(1.f, 1.f, 1.f, 1.f);
        if (j < n) {
            const long long t = tb0 + j;
            const size_t qk_off = ((size_t)t * p.h_qk + hk) * D + c;
            const size_t v_off = ((size_t)t * p.h_v + h) * D + c;
            kk = load4(k + qk_off);
            qq = load4(q + qk_off);
            vv = load4(v + v_off);
            const float4 gg = *reinterpret_cast<const float4*>(p.g + v_off);
            aa = make_float4(expf(gg.x), expf(gg.y), expf(gg.z), expf(gg.w));
        }
        *reinterpret_cast<float4*>(sm + OFF_K + j * D + c) = kk;
        *reinterpret_cast<float4*>(sm + OFF_AK + j * D + c) =
            make_float4(aa.x * kk.x, aa.y * kk.y, aa.z * kk.z, aa.w * kk.w);
        *reinterpret_cast<float4*>(sm + OFF_AQ + j * D + c) =
            make_float4(aa.x * qq.x, aa.y * qq.y, aa.z * qq.z, aa.w * qq.w);
        *reinterpret_cast<float4*>(sm + OFF_A + j * D + c) = aa;
        *reinterpret_cast<float4*>(sm + OFF_V + j * D + c) = vv;
    }
    // k . q per token: warp w takes tokens w, w + 8, ... (lanes: 4 channels each)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < BLK; j += NW) {
        float x = 0.f;
        if (j < n) {
            const size_t qk_off = ((size_t)(tb0 + j) * p.h_qk + hk) * D + 4 * lane;
            const float4 kk = load4(k + qk_off), qq = load4(q + qk_off);
            x = kk.x * qq.x + kk.y * qq.y + kk.z * qq.z + kk.w * qq.w;
        }
        x = warp_sum(x);
        if (lane == 0) sm[OFF_KQ + j] = x;
    }
    if (threadIdx.x < BLK) sm[OFF_B + threadIdx.x] = threadIdx.x < n ? p.beta[(size_t)(tb0 + threadIdx.x) * p.h_v + h] : 0.f;
}

// Two CTAs fit on an SM (at most 128 registers per thread, 91 KB of shared
// memory): when the (sequence, value head) units are fewer than twice the
// SMs, each sequence is split into segments (one CTA each), started a few
// tokens early from a zero state where the decay allows it
// (segment_prefix_start), so that more warps share each SM.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NT, 2) kda_prefill_kernel(const Args p) {
    extern __shared__ float4 smem_f4[];
    __shared__ long long seg_start;
    float* sm = reinterpret_cast<float*>(smem_f4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = warp * 16, c0 = lane * 4;
    TOut* o = static_cast<TOut*>(p.o);
    // this CTA's work: a segment of one (sequence, value head) unit, or with
    // bal_tokens the end of one unit and the start of the next (pieces): it
    // stores the outputs of tokens [seg_a, t1) of sequence n, value head h
    struct Piece { long long seg_a, t1, s0, s1; int n, h; };
    Piece pc0{}, pc1{};
    int npieces = 0;
    if (p.bal_tokens == 0) {
        const int seg = blockIdx.x % p.nseg, unit = blockIdx.x / p.nseg;
        const int pos = unit / p.h_v, h = unit - pos * p.h_v;
        int n = 0;
        long long s0 = 0, s1 = 0;
        if (!seq_of(p.order, pos, p.num_seqs, n)) return;
        if (!seq_bounds(p.cu, n, p.num_seqs, p.total, p.eq_len, s0, s1)) return;
        const long long seg_len = ((s1 - s0 + p.nseg - 1) / p.nseg + BLK - 1) / BLK * BLK;
        const long long seg_a = s0 + seg * seg_len;
        if (seg > 0 && seg_a >= s1) return;  // an empty segment
        pc0 = Piece{seg_a, seg_len > 0 && seg_a + seg_len < s1 ? seg_a + seg_len : s1, s0, s1, n, h};
        npieces = 1;
    } else {
        // tokens of the (sequence, q/k head) groups in order; the grp value
        // heads of a group take the same share in neighbouring CTAs
        const long long gtot = (long long)p.num_seqs * p.h_qk * p.eq_len;
        const int r = blockIdx.x % p.grp;
        long long a = (long long)(blockIdx.x / p.grp) * p.bal_tokens;
        const long long b = min(a + p.bal_tokens, gtot);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (a >= b) break;
            const long long u = a / p.eq_len, lo = a - u * p.eq_len, hi = min(p.eq_len, lo + (b - a));
            const int h = (int)(u % p.h_qk) * p.grp + r, pos = (int)(u / p.h_qk);
            int n = 0;
            long long s0 = 0, s1 = 0;
            if (!seq_of(p.order, pos, p.num_seqs, n)) return;
            if (!seq_bounds(p.cu, n, p.num_seqs, p.total, p.eq_len, s0, s1)) return;
            const Piece x{s0 + lo, min(s0 + hi, s1), s0, s1, n, h};
            if (i == 0) pc0 = x; else pc1 = x;
            ++npieces;
            a += hi - lo;
        }
        if (npieces == 0) return;
    }
    for (int ip = 0; ip < npieces; ++ip) {
        const Piece pc = pc0;  // the current piece (pc1 moves up at the end)
        const long long seg_a = pc.seg_a, t1 = pc.t1, s0 = pc.s0, s1 = pc.s1;
        const int n = pc.n, h = pc.h, hk = h / p.grp;
        __syncthreads();  // seg_start and the stage of the previous piece are free
        if (warp == 0) {
            const long long ts = seg_a > s0 ? segment_prefix_start<TIn>(p, s0, seg_a, h, hk, lane) : s0;
            if (lane == 0) seg_start = ts;
        }
        __syncthreads();
        const long long t0 = seg_start;  // first token processed
        const size_t st_off = ((size_t)n * p.h_v + h) * D * D;

        float S[16][4];
        if (p.h0 && t0 == s0) bwd::load_state(S, p.h0 + st_off, r0, c0);
        else bwd::zero_state(S);
        for (long long tb0 = t0; tb0 < t1; tb0 += BLK) {
            const int nt = (int)min((long long)BLK, t1 - tb0);
            __syncthreads();
            kda_stage<TIn>(sm, p, tb0, nt, h, hk);
            __syncthreads();
            for (int j = 0; j < nt; ++j) {
                float ak[16], aq[16];
#pragma unroll
                for (int r = 0; r < 16; r += 4) {
                    const float4 x = *reinterpret_cast<const float4*>(sm + OFF_AK + j * D + r0 + r);
                    ak[r] = x.x; ak[r + 1] = x.y; ak[r + 2] = x.z; ak[r + 3] = x.w;
                    const float4 y = *reinterpret_cast<const float4*>(sm + OFF_AQ + j * D + r0 + r);
                    aq[r] = y.x; aq[r + 1] = y.y; aq[r + 2] = y.z; aq[r + 3] = y.w;
                }
                float ks[4] = {0.f, 0.f, 0.f, 0.f}, qs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int r = 0; r < 16; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        ks[c] = fmaf(S[r][c], ak[r], ks[c]);
                        qs[c] = fmaf(S[r][c], aq[r], qs[c]);
                    }
                float* red = sm + OFF_RED;
                *reinterpret_cast<float4*>(red + warp * RED + c0) = make_float4(ks[0], ks[1], ks[2], ks[3]);
                *reinterpret_cast<float4*>(red + (NW + warp) * RED + c0) = make_float4(qs[0], qs[1], qs[2], qs[3]);
                __syncthreads();
                {
                    const int colx = threadIdx.x >> 1, part = threadIdx.x & 1;
                    float sk = 0.f, sq = 0.f;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        sk += red[(part * 4 + m) * RED + colx];
                        sq += red[(NW + part * 4 + m) * RED + colx];
                    }
                    sk += __shfl_xor_sync(0xffffffffu, sk, 1);
                    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
                    if (part == 0) {
                        const float uu = sm[OFF_B + j] * (sm[OFF_V + j * D + colx] - sk);
                        sm[OFF_U + colx] = uu;
                        if (tb0 + j >= seg_a)  // the piece's prefix tokens are not stored
                            o[((size_t)(tb0 + j) * p.h_v + h) * D + colx] = from_f32<TOut>(p.scale * fmaf(sm[OFF_KQ + j], uu, sq));
                    }
                }
                __syncthreads();
                const float4 u4 = *reinterpret_cast<const float4*>(sm + OFF_U + c0);
                const float u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int r = 0; r < 16; r += 4) {
                    const float4 a4 = *reinterpret_cast<const float4*>(sm + OFF_A + j * D + r0 + r);
                    const float4 k4 = *reinterpret_cast<const float4*>(sm + OFF_K + j * D + r0 + r);
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                        for (int c = 0; c < 4; ++c) S[r + rr][c] = fmaf(av[rr], S[r + rr][c], kv[rr] * u[c]);
                }
            }
        }
        if (p.hT && t1 == s1) bwd::store_state(S, p.hT + st_off, r0, c0);  // the piece ends its sequence
        pc0 = pc1;
    }
}

}  // namespace kda
}  // namespace gdn
