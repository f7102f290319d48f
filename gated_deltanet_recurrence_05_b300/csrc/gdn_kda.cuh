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
// The decode step uses S~^T x = S^T (a o x): the reads use a o k and a o q,
// and S_t^T q = S^T (a o q) + (k . q) u with u = b e, one pass over S for both
// reads and one for the update. The prefill takes chunks of 16 tokens in the
// WY form (below). d_k = d_v = 128.
#pragma once

#include "gdn_common.cuh"
#include "gdn_epilogue.cuh"
#include "gdn_backward.cuh"

namespace gdn {
namespace kda {

constexpr int D = 128;
constexpr int BLK = 32;        // granularity of prefill segments and shares (tokens)
constexpr int NT = 256;
constexpr int NW = NT / 32;

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

// Prefill: chunks of C = 16 tokens in the WY form of the rule. Within a
// chunk, with G_t = sum_{u <= t} g_u per key channel (from the chunk start)
// and S0 the state before the chunk, the unrolled rule gives S~_t =
// diag(exp(G_t)) S0 + sum_{s<t} diag(exp(G_t - G_s)) beta_s k_s e_s^T, so the
// errors e_t, outputs and next state are
//
//   A_ts = beta_s sum_i k_si k_ti exp(G_ti - G_si)   (s < t)
//   P_ts = beta_s sum_i k_si q_ti exp(G_ti - G_si)   (s <= t)
//   E    = (I + A)^{-1} (V - K_G S0),   K_G = rows k_t o exp(G_t)
//   O    = scale (Q_G S0 + P E),        Q_G = rows q_t o exp(G_t)
//   S_L  = diag(exp(G_L)) S0 + K_T^T diag(beta) E,  K_T = rows k_t o exp(G_L - G_t)
//
// Every decay factor is the exponential of a difference G_t - G_s <= 0 (or
// G_t <= 0), so none exceeds 1. A and P fold the factor into rows scaled by
// exp(G_t) and exp(-G_s) while every running sum of the chunk is within
// 2^+-100, and take it per element otherwise.
//
// One CTA of 256 threads per piece; warp w owns state columns 16w..16w+15
// and keeps S^T (16 columns x 128 rows) in fp32 registers as the accumulator
// fragments of the warp MMA (m16n8k8, tf32): lane (g, c) = (lane / 4,
// lane % 4) holds rows 8j + 2c, 8j + 2c + 1 of columns 16w + g, 16w + g + 8,
// j = 0..15. The three state products of a chunk, S0^T K_G^T, S0^T Q_G^T and
// U^T K_T (U = diag(beta) E), run on the tensor cores with fp32 accuracy:
// each fp32 operand x is split into tf32 parts x = hi + lo and the product
// taken as hi hi + hi lo + lo hi (fp32 accumulation). The contraction index
// of each 8-wide step is taken in the order (2c, 2c + 1 for c = 0..3) on both
// operands, which makes the state's accumulator fragments its A fragments
// without any data movement. The triangular solve and the outputs run per
// column on lanes 0-15 of each warp; the chunk's tiles (k, q, v, the decays,
// A and P) are shared through shared memory.
constexpr int C = 16;                  // tokens per chunk
constexpr int XS = D + 8;              // row stride of K_G, Q_G, K_I ([token][channel]): conflict-free fragments
constexpr int KS = C + 8;              // row stride of K_T^T ([channel][token])
// |running log2-decay| up to which exp(-G) and exp(G) stay normal fp32
// numbers (2^100 and 2^-100) and their product keeps full precision
constexpr float G2_MAX = 100.f;
constexpr int OFF_K = 0;               // k   [C][D]
constexpr int OFF_Q = OFF_K + C * D;   // q   [C][D]
constexpr int OFF_V = OFF_Q + C * D;   // v   [C][D]
constexpr int OFF_G2 = OFF_V + C * D;  // g as loaded, then G / ln 2 [C][D] (running sums, base 2)
constexpr int OFF_KG = OFF_G2 + C * D; // K_G [C][XS], tf32 high parts
constexpr int OFF_KGL = OFF_KG + C * XS; // and the low parts (K_G = high + low)
constexpr int OFF_QG = OFF_KGL + C * XS; // Q_G likewise
constexpr int OFF_QGL = OFF_QG + C * XS;
constexpr int OFF_KI = OFF_QGL + C * XS; // K_I = rows k_t o exp(-G_t) [C][XS]
constexpr int OFF_KTT = OFF_KI + C * XS; // K_T^T [D][KS]
constexpr int OFF_GL = OFF_KTT + D * KS; // exp(G_L) [D]
constexpr int OFF_AM = OFF_GL + D;       // A [C][C]
constexpr int OFF_PM = OFF_AM + C * C;   // P [C][C]
constexpr int OFF_BT = OFF_PM + C * C;   // beta [C]
constexpr int OFF_WS = OFF_BT + C;       // per warp: S0^T K_G (then beta E), S0^T Q_G [2][C][16]
constexpr int WS_FLOATS = 2 * C * 16;
constexpr int SMEM_FLOATS = OFF_WS + NW * WS_FLOATS;
constexpr size_t SMEM_BYTES = (size_t)SMEM_FLOATS * sizeof(float);
static_assert(OFF_KG % 4 == 0 && OFF_KTT % 4 == 0 && OFF_WS % 4 == 0 && XS % 4 == 0 && KS % 2 == 0,
              "vector alignment");
static_assert(2 * SMEM_BYTES + 2048 <= 232448, "two CTAs per SM");

__device__ __forceinline__ float ex2f(float x) {  // 2^x on the special-function unit
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// x = hi + lo with hi, lo tf32 (round to nearest): hi holds the top 11 bits
// of the significand and lo the next 11, so hi hi + hi lo + lo hi carries
// about 22 bits of each product
__device__ __forceinline__ void split_tf32(float x, uint32_t& hi, uint32_t& lo) {
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
    const float r = x - __uint_as_float(hi);
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(lo) : "f"(r));
}
// D += A B on the warp MMA, m16n8k8, tf32 operands, fp32 accumulators
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// D += A B to about fp32 accuracy from split operands (small terms first)
__device__ __forceinline__ void mma3(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                     const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
    mma_tf32(d, al, bh[0], bh[1]);
    mma_tf32(d, ah, bl[0], bl[1]);
    mma_tf32(d, ah, bh[0], bh[1]);
}

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

// Stage tokens [tb0, tb0 + n) of the piece into shared memory as fp32 (rows
// j >= n: k = q = v = 0, g = 0, beta = 0, which leave the state unchanged),
// then the running sums of g (one thread per channel, in place) and the
// chunk's decayed rows (thread (half hf, channel i): the tokens of its half).
// Returns whether some running sum is beyond +-G2_MAX (a block-wide OR).
template <typename TIn>
__device__ __forceinline__ bool kda_stage_chunk(float* sm, const Args& p, long long tb0, int n, int h, int hk) {
    constexpr float LOG2E = 1.4426950408889634f;
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    const TIn* v = static_cast<const TIn*>(p.v);
    for (int idx = threadIdx.x; idx < C * (D / 4); idx += NT) {
        const int j = idx >> 5, c = (idx & 31) * 4;
        float4 kk = make_float4(0.f, 0.f, 0.f, 0.f), qq = kk, vv = kk, gg = kk;
        if (j < n) {
            const long long t = tb0 + j;
            const size_t qk_off = ((size_t)t * p.h_qk + hk) * D + c;
            const size_t v_off = ((size_t)t * p.h_v + h) * D + c;
            kk = load4(k + qk_off);
            qq = load4(q + qk_off);
            vv = load4(v + v_off);
            gg = *reinterpret_cast<const float4*>(p.g + v_off);
        }
        *reinterpret_cast<float4*>(sm + OFF_K + j * D + c) = kk;
        *reinterpret_cast<float4*>(sm + OFF_Q + j * D + c) = qq;
        *reinterpret_cast<float4*>(sm + OFF_V + j * D + c) = vv;
        *reinterpret_cast<float4*>(sm + OFF_G2 + j * D + c) = gg;
    }
    if (threadIdx.x < C) sm[OFF_BT + threadIdx.x] = threadIdx.x < n ? p.beta[(size_t)(tb0 + threadIdx.x) * p.h_v + h] : 0.f;
    __syncthreads();
    const int hf = threadIdx.x >> 7, i = threadIdx.x & (D - 1);
    if (hf == 0) {  // running sums of g, in place, one thread per channel
        float gv[C];
#pragma unroll
        for (int j = 0; j < C; ++j) gv[j] = sm[OFF_G2 + j * D + i];
        float acc = 0.f;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            acc = fmaf(gv[j], LOG2E, acc);
            sm[OFF_G2 + j * D + i] = acc;
        }
        sm[OFF_GL + i] = ex2f(acc);
    }
    __syncthreads();
    const float acc = sm[OFF_G2 + (C - 1) * D + i];
    bool wide = false;  // a running sum outside [-G2_MAX, G2_MAX]: exp(-G) could overflow
#pragma unroll
    for (int jj = 0; jj < C / 2; ++jj) {
        const int j = (C / 2) * hf + jj;
        const float gm = sm[OFF_G2 + j * D + i];
        const float e = ex2f(gm), kj = sm[OFF_K + j * D + i];
        wide |= fabsf(gm) > G2_MAX;
        uint32_t hi, lo;
        split_tf32(kj * e, hi, lo);
        sm[OFF_KG + j * XS + i] = __uint_as_float(hi);
        sm[OFF_KGL + j * XS + i] = __uint_as_float(lo);
        split_tf32(sm[OFF_Q + j * D + i] * e, hi, lo);
        sm[OFF_QG + j * XS + i] = __uint_as_float(hi);
        sm[OFF_QGL + j * XS + i] = __uint_as_float(lo);
        sm[OFF_KTT + i * KS + j] = kj * ex2f(acc - gm);
        sm[OFF_KI + j * XS + i] = kj * ex2f(-gm);
    }
    return __syncthreads_or(wide) != 0;
}

// A and P of the staged chunk on the warp MMA when the decay factors fold
// into the rows (no running sum beyond +-G2_MAX): warps 0-3 take one 16 x 8
// block each (A or P; the columns s = 0-7 or 8-15) of K_G K_I^T or Q_G K_I^T
// over the 128 channels, in fp32 accuracy (split tf32 operands), and store it
// scaled by beta_s. Entries outside s < t (A) or s <= t (P) are stored too and
// never read.
__device__ __forceinline__ void kda_chunk_ap_mma(float* sm, int warp, int lane) {
    const int fg = lane >> 2, fc = lane & 3;
    const int isP = warp >> 1, nb = warp & 1;
    const float* Xh = sm + (isP ? OFF_QG : OFF_KG);
    const float* Xl = sm + (isP ? OFF_QGL : OFF_KGL);
    const float* Ki = sm + OFF_KI + (8 * nb + fg) * XS;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int kt = 0; kt < D / 8; ++kt) {
        const int o0 = fg * XS + 8 * kt + 2 * fc, o1 = o0 + 8 * XS;
        const uint2 h0 = *reinterpret_cast<const uint2*>(Xh + o0), h1 = *reinterpret_cast<const uint2*>(Xh + o1);
        const uint2 l0 = *reinterpret_cast<const uint2*>(Xl + o0), l1 = *reinterpret_cast<const uint2*>(Xl + o1);
        const float2 bv = *reinterpret_cast<const float2*>(Ki + 8 * kt + 2 * fc);
        const uint32_t ah[4] = {h0.x, h1.x, h0.y, h1.y}, al[4] = {l0.x, l1.x, l0.y, l1.y};
        uint32_t bh[2], bl[2];
        split_tf32(bv.x, bh[0], bl[0]);
        split_tf32(bv.y, bh[1], bl[1]);
        mma3(d, ah, al, bh, bl);
    }
    float* M = sm + (isP ? OFF_PM : OFF_AM);
    const int s0 = 8 * nb + 2 * fc;
    const float b0 = sm[OFF_BT + s0], b1 = sm[OFF_BT + s0 + 1];
    M[fg * C + s0] = b0 * d[0];
    M[fg * C + s0 + 1] = b1 * d[1];
    M[(fg + 8) * C + s0] = b0 * d[2];
    M[(fg + 8) * C + s0 + 1] = b1 * d[3];
}

// A (thread tid < 120) or P (the other 136) entry of the staged chunk with
// the decay factors taken per element (a chunk whose running decays pass
// +-G2_MAX, where exp(-G) could overflow): one dot product over the 128
// channels, the channels rotated by lane so that the lanes' 16-byte reads
// spread over all banks.
__device__ __forceinline__ void kda_chunk_ap_wide(float* sm, int lane) {
    const bool isA = threadIdx.x < (C * (C - 1)) / 2;
    int jj = isA ? (int)threadIdx.x : (int)threadIdx.x - (C * (C - 1)) / 2, t = 0;
    while (jj >= (isA ? t : t + 1)) {  // entries of row t: s < t (A) or s <= t (P)
        jj -= isA ? t : t + 1;
        ++t;
    }
    const int s = jj;
    const float* X = sm + (isA ? OFF_K : OFF_Q) + t * D;
    const float* Ks = sm + OFF_K + s * D;
    const float* Gt = sm + OFF_G2 + t * D;
    const float* Gs = sm + OFF_G2 + s * D;
    float acc = 0.f;
#pragma unroll 4
    for (int m = 0; m < D / 4; ++m) {
        const int i = ((m + lane) & (D / 4 - 1)) * 4;
        const float4 x = *reinterpret_cast<const float4*>(X + i), kk = *reinterpret_cast<const float4*>(Ks + i);
        const float4 gt = *reinterpret_cast<const float4*>(Gt + i), gs = *reinterpret_cast<const float4*>(Gs + i);
        acc = fmaf(x.x * kk.x, ex2f(gt.x - gs.x), acc);
        acc = fmaf(x.y * kk.y, ex2f(gt.y - gs.y), acc);
        acc = fmaf(x.z * kk.z, ex2f(gt.z - gs.z), acc);
        acc = fmaf(x.w * kk.w, ex2f(gt.w - gs.w), acc);
    }
    sm[(isA ? OFF_AM : OFF_PM) + t * C + s] = sm[OFF_BT + s] * acc;
}

// Two CTAs fit on an SM (at most 128 registers per thread, 99 KB of shared
// memory): when the (sequence, value head) units are fewer than twice the
// SMs, each sequence is split into segments (one CTA each), started a few
// tokens early from a zero state where the decay allows it
// (segment_prefix_start), or, for equal lengths, into balanced shares, so
// that more warps share each SM.
template <typename TIn, typename TOut>
__global__ void __launch_bounds__(NT, 2) kda_prefill_kernel(const Args p) {
    extern __shared__ float4 smem_f4[];
    __shared__ long long seg_start;
    float* sm = reinterpret_cast<float*>(smem_f4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int fg = lane >> 2, fc = lane & 3;  // fragment row group and column pair
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

        // S^T fragments: Sd[j] = S[8j + 2c][cg], S[8j + 2c + 1][cg], S[8j + 2c][cg + 8],
        // S[8j + 2c + 1][cg + 8] with cg = 16 warp + g (lane = 4 g + c)
        float Sd[D / 8][4];
        {
            const float* src = p.h0 + st_off;
            const bool from_h0 = p.h0 && t0 == s0;
#pragma unroll
            for (int j = 0; j < D / 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    Sd[j][e] = from_h0 ? src[(size_t)(8 * j + 2 * fc + (e & 1)) * D + 16 * warp + fg + 8 * (e >> 1)]
                                       : 0.f;
        }
        float* ws = sm + OFF_WS + warp * WS_FLOATS;
        for (long long tb0 = t0; tb0 < t1; tb0 += C) {
            const int nt = (int)min((long long)C, t1 - tb0);
            __syncthreads();  // the previous chunk's tiles are free
            const bool wide = kda_stage_chunk<TIn>(sm, p, tb0, nt, h, hk);  // ends with a block barrier
            if (wide) kda_chunk_ap_wide(sm, lane);
            else if (warp < 4) kda_chunk_ap_mma(sm, warp, lane);
            // S0^T K_G^T and S0^T Q_G^T (16 columns x 16 tokens each) on the warp MMA
            {
                float Y[2][2][4];
#pragma unroll
                for (int x = 0; x < 2; ++x)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) Y[x][n][e] = 0.f;
#pragma unroll
                for (int kt = 0; kt < D / 8; ++kt) {
                    uint32_t ah[4], al[4];
                    split_tf32(Sd[kt][0], ah[0], al[0]);
                    split_tf32(Sd[kt][2], ah[1], al[1]);
                    split_tf32(Sd[kt][1], ah[2], al[2]);
                    split_tf32(Sd[kt][3], ah[3], al[3]);
#pragma unroll
                    for (int x = 0; x < 2; ++x)
#pragma unroll
                        for (int n = 0; n < 2; ++n) {
                            const int ob = (8 * n + fg) * XS + 8 * kt + 2 * fc;
                            const uint2 h = *reinterpret_cast<const uint2*>(sm + (x ? OFF_QG : OFF_KG) + ob);
                            const uint2 l = *reinterpret_cast<const uint2*>(sm + (x ? OFF_QGL : OFF_KGL) + ob);
                            const uint32_t bh[2] = {h.x, h.y}, bl[2] = {l.x, l.y};
                            mma3(Y[x][n], ah, al, bh, bl);
                        }
                }
                // to the warp's scratch as [kind][token][column]
#pragma unroll
                for (int x = 0; x < 2; ++x)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            ws[x * C * 16 + (8 * n + 2 * fc + (e & 1)) * 16 + fg + 8 * (e >> 1)] = Y[x][n][e];
            }
            __syncthreads();  // A and P of the chunk; the warp's scratch
            // per column (lanes 0-15 of the warp): E = (I + A)^{-1} (V - K_G S0) by forward
            // substitution, over S0^T K_G in the warp's scratch
            if (lane < 16) {
                const int col = 16 * warp + lane;
                float e[C];
#pragma unroll
                for (int t = 0; t < C; ++t) {
                    float r = sm[OFF_V + t * D + col] - ws[t * 16 + lane];
#pragma unroll
                    for (int s4 = 0; s4 < t; s4 += 4) {
                        const float4 a4 = *reinterpret_cast<const float4*>(sm + OFF_AM + t * C + s4);
                        r = fmaf(-a4.x, e[s4], r);
                        if (s4 + 1 < t) r = fmaf(-a4.y, e[s4 + 1], r);
                        if (s4 + 2 < t) r = fmaf(-a4.z, e[s4 + 2], r);
                        if (s4 + 3 < t) r = fmaf(-a4.w, e[s4 + 3], r);
                    }
                    e[t] = r;
                }
#pragma unroll
                for (int t = 0; t < C; ++t) ws[t * 16 + lane] = e[t];
            }
            __syncwarp();
            {  // O = scale (Q_G S0 + P E) for column cl and the tokens t = hp, hp + 2, ..., stored
                const int cl = lane & 15, hp = lane >> 4;
                float e[C];
#pragma unroll
                for (int u = 0; u < C; ++u) e[u] = ws[u * 16 + cl];
                TOut* ob = o + ((size_t)tb0 * p.h_v + h) * D + 16 * warp + cl;
                const size_t ostride = (size_t)p.h_v * D;
#pragma unroll
                for (int m = 0; m < C / 2; ++m) {
                    const int t = 2 * m + hp;
                    float y = ws[C * 16 + t * 16 + cl];
#pragma unroll
                    for (int s4 = 0; s4 <= 2 * m + 1; s4 += 4) {  // s <= t; P vanishes above the diagonal
                        const float4 p4 = *reinterpret_cast<const float4*>(sm + OFF_PM + t * C + s4);
                        if (s4 <= t) y = fmaf(p4.x, e[s4], y);
                        if (s4 + 1 <= t) y = fmaf(p4.y, e[s4 + 1], y);
                        if (s4 + 2 <= t) y = fmaf(p4.z, e[s4 + 2], y);
                        if (s4 + 3 <= t) y = fmaf(p4.w, e[s4 + 3], y);
                    }
                    if (t < nt && tb0 + t >= seg_a)  // the piece's prefix tokens are not stored
                        ob[(size_t)t * ostride] = from_f32<TOut>(p.scale * y);
                }
            }
            // S^T <- S^T diag(exp(G_L)) + U^T K_T on the warp MMA (U = diag(beta) E)
            {
                uint32_t uh[2][4], ul[2][4];
#pragma unroll
                for (int kt = 0; kt < 2; ++kt) {
                    const float* u = ws + (8 * kt + 2 * fc) * 16 + fg;  // E
                    const float b0 = sm[OFF_BT + 8 * kt + 2 * fc], b1 = sm[OFF_BT + 8 * kt + 2 * fc + 1];
                    split_tf32(b0 * u[0], uh[kt][0], ul[kt][0]);
                    split_tf32(b0 * u[8], uh[kt][1], ul[kt][1]);
                    split_tf32(b1 * u[16], uh[kt][2], ul[kt][2]);
                    split_tf32(b1 * u[24], uh[kt][3], ul[kt][3]);
                }
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    const float2 gl = *reinterpret_cast<const float2*>(sm + OFF_GL + 8 * j + 2 * fc);
                    Sd[j][0] *= gl.x; Sd[j][1] *= gl.y; Sd[j][2] *= gl.x; Sd[j][3] *= gl.y;
#pragma unroll
                    for (int kt = 0; kt < 2; ++kt) {
                        const float2 bv = *reinterpret_cast<const float2*>(sm + OFF_KTT + (8 * j + fg) * KS + 8 * kt + 2 * fc);
                        uint32_t bh[2], bl[2];
                        split_tf32(bv.x, bh[0], bl[0]);
                        split_tf32(bv.y, bh[1], bl[1]);
                        mma3(Sd[j], uh[kt], ul[kt], bh, bl);
                    }
                }
            }
        }
        if (p.hT && t1 == s1) {  // the piece ends its sequence
            float* dst = p.hT + st_off;
#pragma unroll
            for (int j = 0; j < D / 8; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    dst[(size_t)(8 * j + 2 * fc + (e & 1)) * D + 16 * warp + fg + 8 * (e >> 1)] = Sd[j][e];
        }
        pc0 = pc1;
    }
}

}  // namespace kda
}  // namespace gdn
