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
// fragments of the warp MMA: lane (g, c) = (lane / 4, lane % 4) holds rows
// 8j + 2c, 8j + 2c + 1 of columns 16w + g, 16w + g + 8, j = 0..15, which are
// also the A fragments of an m16n8k16 product over rows 16i .. 16i + 15
// (fragments 2i, 2i + 1), so the state feeds its own reads with no data
// movement. The three state products of a chunk, S0^T K_G^T, S0^T Q_G^T and
// U^T K_T (U = diag(beta) E), run in fp32 accuracy on fp16 m16n8k16: each
// operand is scaled by a power of two into [2^14, 2^15) at its maximum (per
// warp for S and U, per chunk for K_G, Q_G, K_T), split into fp16 parts
// x = hi + lo 2^-11 (the low part stored scaled so that it stays a normal
// fp16 number: unscaled, many low parts are subnormal, and the products then
// missed fp32 accuracy on the tensor cores), and the product taken as
// hi hi + (hi lo + lo hi) 2^-11 with fp32 accumulation; the scales are undone
// exactly. A and P (K_G K_I^T, Q_G K_I^T) pair exp(G_t) with exp(-G_s), whose
// ranges only fp32 holds: they run on m16n8k8 tf32 with each operand split
// into tf32 parts (the contraction order 2c, 2c + 1 within each 8-wide step).
// The triangular solve runs per column on lanes 0-15 of each warp, the
// outputs on all lanes; the chunk's tiles (k, q, v, the decays, A and P) are
// shared through shared memory.
constexpr int C = 16;                  // tokens per chunk
constexpr int XS = D + 8;              // row stride (floats) of K_I ([token][channel]): conflict-free fragments
constexpr int RW = (D + 8) / 2;        // row stride (32-bit words of two fp16) of K_G, Q_G ([token][channel])
constexpr int RT = (C + 8) / 2;        // row stride (words) of K_T^T ([channel][token])
// |running log2-decay| up to which exp(-G) and exp(G) stay normal fp32
// numbers (2^100 and 2^-100) and their product keeps full precision
constexpr float G2_MAX = 100.f;
constexpr int OFF_K = 0;               // k   [C][D]
constexpr int OFF_Q = OFF_K + C * D;   // q   [C][D]
constexpr int OFF_V = OFF_Q + C * D;   // v   [C][D]
constexpr int OFF_G2 = OFF_V + C * D;  // g as loaded, then G / ln 2 [C][D] (running sums, base 2)
// K_G, Q_G, K_T^T are kept as fp16 pairs (high, low) scaled by the chunk's
// powers of two 2^ek, 2^eq (x = high + low to about 22 bits)
constexpr int OFF_KG = OFF_G2 + C * D;   // K_G 2^ek, high parts [C][RW words]
constexpr int OFF_KGL = OFF_KG + C * RW; // and the low parts
constexpr int OFF_QG = OFF_KGL + C * RW; // Q_G 2^eq likewise
constexpr int OFF_QGL = OFF_QG + C * RW;
constexpr int OFF_KTT = OFF_QGL + C * RW;  // K_T^T 2^ek, high parts [D][RT words]
constexpr int OFF_KTL = OFF_KTT + D * RT;  // and the low parts
constexpr int OFF_KI = OFF_KTL + D * RT;   // K_I = rows k_t o exp(-G_t) [C][XS] fp32
// K_G and Q_G in fp32 for A and P, where they meet K_I: exp(G_t) can be far
// below the fp16 range while exp(G_t - G_s) is not
constexpr int OFF_KG32 = OFF_KI + C * XS;
constexpr int OFF_QG32 = OFF_KG32 + C * XS;
constexpr int OFF_GL = OFF_QG32 + C * XS;  // exp(G_L) [D]
constexpr int OFF_MX = OFF_GL + D;         // per warp max |k|, max |q|, max growth of the chunk [3][NW]
constexpr int OFF_AM = OFF_MX + 3 * NW;  // A [C][C]
constexpr int OFF_PM = OFF_AM + C * C;   // P [C][C]
constexpr int OFF_BT = OFF_PM + C * C;   // beta [C]
constexpr int OFF_WS = OFF_BT + C;       // per warp: S0^T K_G (then beta E), S0^T Q_G [2][C][16]
constexpr int WS_FLOATS = 2 * C * 16;
constexpr int SMEM_FLOATS = OFF_WS + NW * WS_FLOATS;
constexpr size_t SMEM_BYTES = (size_t)SMEM_FLOATS * sizeof(float);
static_assert(OFF_KG % 4 == 0 && OFF_KI % 4 == 0 && OFF_WS % 4 == 0 && XS % 4 == 0,
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
// 2^e, exact for e in [-126, 127] (clamped outside, which only extreme
// magnitudes of the state or the inputs reach)
__device__ __forceinline__ float pow2i(int e) { return __int_as_float((127 + max(-126, min(127, e))) << 23); }
// the power of two 2^e that brings max |x| = m into [2^14, 2^15) (1 for m = 0)
__device__ __forceinline__ int scale_exp(float m) {
    return m > 0.f ? max(-60, min(60, 14 - ilogbf(m))) : 0;
}
// fp16 pairs (x0, x1) = high + low 2^-11, packed as two half2 words: the low
// part is stored scaled by 2^11 so that it stays a normal fp16 number
// wherever x itself is (unscaled, it falls into the subnormal range, where
// the tensor-core products lost precision)
constexpr float LO_UP = 2048.f, LO_DOWN = 1.f / 2048.f;
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn((x0 - hf.x) * LO_UP, (x1 - hf.y) * LO_UP);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}
// D += A B on the warp MMA, m16n8k16, fp16 operands, fp32 accumulators
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// the cross terms high x low of split operands (both scaled by 2^11)
__device__ __forceinline__ void mma_cross(float (&d)[4], const uint32_t (&ah)[4], const uint32_t (&al)[4],
                                          const uint32_t (&bh)[2], const uint32_t (&bl)[2]) {
    mma_f16(d, al, bh[0], bh[1]);
    mma_f16(d, ah, bl[0], bl[1]);
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
__device__ __forceinline__ bool kda_stage_chunk(float* sm, const Args& p, long long tb0, int n, int h, int hk,
                                                int& ek, int& eq) {
    constexpr float LOG2E = 1.4426950408889634f;
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    const TIn* v = static_cast<const TIn*>(p.v);
    float mk = 0.f, mq = 0.f;  // max |k|, |q| of the thread's part of the chunk
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
        mk = fmaxf(mk, fmaxf(fmaxf(fabsf(kk.x), fabsf(kk.y)), fmaxf(fabsf(kk.z), fabsf(kk.w))));
        mq = fmaxf(mq, fmaxf(fmaxf(fabsf(qq.x), fabsf(qq.y)), fmaxf(fabsf(qq.z), fabsf(qq.w))));
        *reinterpret_cast<float4*>(sm + OFF_K + j * D + c) = kk;
        *reinterpret_cast<float4*>(sm + OFF_Q + j * D + c) = qq;
        *reinterpret_cast<float4*>(sm + OFF_V + j * D + c) = vv;
        *reinterpret_cast<float4*>(sm + OFF_G2 + j * D + c) = gg;
    }
    if (threadIdx.x < C) sm[OFF_BT + threadIdx.x] = threadIdx.x < n ? p.beta[(size_t)(tb0 + threadIdx.x) * p.h_v + h] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, off));
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, off));
    }
    if ((threadIdx.x & 31) == 0) {
        sm[OFF_MX + (threadIdx.x >> 5)] = mk;
        sm[OFF_MX + NW + (threadIdx.x >> 5)] = mq;
    }
    __syncthreads();
    // the chunk's scales 2^ek, 2^eq: max |K_G|, |K_T| <= max |k|, max |Q_G| <= max |q|
    {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            a = fmaxf(a, sm[OFF_MX + w]);
            b = fmaxf(b, sm[OFF_MX + NW + w]);
        }
        ek = scale_exp(a);
        eq = scale_exp(b);
    }
    const int hf = threadIdx.x >> 7, i = threadIdx.x & (D - 1);
    if (hf == 0) {  // running sums of g, in place, one thread per channel
        float gv[C];
#pragma unroll
        for (int j = 0; j < C; ++j) gv[j] = sm[OFF_G2 + j * D + i];
        float acc = 0.f, gmax = 0.f, gmin = 0.f;
#pragma unroll
        for (int j = 0; j < C; ++j) {
            acc = fmaf(gv[j], LOG2E, acc);
            sm[OFF_G2 + j * D + i] = acc;
            gmax = fmaxf(gmax, acc);
            gmin = fminf(gmin, acc);
        }
        sm[OFF_GL + i] = ex2f(acc);
        // largest log2 factor by which a row of K_G, Q_G or K_T exceeds |k| or |q|
        // (0 for decays; positive only where some g > 0)
        float up = fmaxf(gmax, acc - gmin);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) up = fmaxf(up, __shfl_xor_sync(0xffffffffu, up, off));
        if ((threadIdx.x & 31) == 0) sm[OFF_MX + 2 * NW + (threadIdx.x >> 5)] = up;
    }
    __syncthreads();
    {
        float up = 0.f;
#pragma unroll
        for (int w = 0; w < D / 32; ++w) up = fmaxf(up, sm[OFF_MX + 2 * NW + w]);
        const int sh = (int)ceilf(fminf(up, 60.f));
        ek = max(-100, ek - sh);
        eq = max(-100, eq - sh);
    }
    const float acc = sm[OFF_G2 + (C - 1) * D + i];
    const float sk = pow2i(ek), sq = pow2i(eq);
    __half* kgh = reinterpret_cast<__half*>(sm + OFF_KG);
    __half* kgl = reinterpret_cast<__half*>(sm + OFF_KGL);
    __half* qgh = reinterpret_cast<__half*>(sm + OFF_QG);
    __half* qgl = reinterpret_cast<__half*>(sm + OFF_QGL);
    __half* kth = reinterpret_cast<__half*>(sm + OFF_KTT);
    __half* ktl = reinterpret_cast<__half*>(sm + OFF_KTL);
    bool wide = false;  // a running sum outside [-G2_MAX, G2_MAX]: exp(-G) could overflow
#pragma unroll
    for (int jj = 0; jj < C / 2; ++jj) {
        const int j = (C / 2) * hf + jj;
        const float gm = sm[OFF_G2 + j * D + i];
        const float e = ex2f(gm), kj = sm[OFF_K + j * D + i];
        wide |= fabsf(gm) > G2_MAX;
        const float kg1 = kj * e, qg1 = sm[OFF_Q + j * D + i] * e;
        sm[OFF_KG32 + j * XS + i] = kg1;
        sm[OFF_QG32 + j * XS + i] = qg1;
        const float kg = kg1 * sk, qg = qg1 * sq, kt = kj * ex2f(acc - gm) * sk;
        const __half kgh_ = __float2half_rn(kg), qgh_ = __float2half_rn(qg), kth_ = __float2half_rn(kt);
        kgh[j * 2 * RW + i] = kgh_;
        kgl[j * 2 * RW + i] = __float2half_rn((kg - __half2float(kgh_)) * LO_UP);
        qgh[j * 2 * RW + i] = qgh_;
        qgl[j * 2 * RW + i] = __float2half_rn((qg - __half2float(qgh_)) * LO_UP);
        kth[i * 2 * RT + j] = kth_;
        ktl[i * 2 * RT + j] = __float2half_rn((kt - __half2float(kth_)) * LO_UP);
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
    const float* X = sm + (isP ? OFF_QG32 : OFF_KG32);
    const float* Ki = sm + OFF_KI + (8 * nb + fg) * XS;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int kt = 0; kt < D / 8; ++kt) {
        // channels 8kt + 2c, 8kt + 2c + 1 of tokens g and g + 8 (the k order 2c, 2c + 1)
        const float2 x0 = *reinterpret_cast<const float2*>(X + fg * XS + 8 * kt + 2 * fc);
        const float2 x1 = *reinterpret_cast<const float2*>(X + (fg + 8) * XS + 8 * kt + 2 * fc);
        const float2 bv = *reinterpret_cast<const float2*>(Ki + 8 * kt + 2 * fc);
        uint32_t ah[4], al[4], bh[2], bl[2];
        split_tf32(x0.x, ah[0], al[0]);
        split_tf32(x1.x, ah[1], al[1]);
        split_tf32(x0.y, ah[2], al[2]);
        split_tf32(x1.y, ah[3], al[3]);
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
            int ek, eq;
            const bool wide = kda_stage_chunk<TIn>(sm, p, tb0, nt, h, hk, ek, eq);  // ends with a block barrier
            if (wide) kda_chunk_ap_wide(sm, lane);
            else if (warp < 4) kda_chunk_ap_mma(sm, warp, lane);
            // S0^T K_G^T and S0^T Q_G^T (16 columns x 16 tokens each) on the warp MMA
            {
                float Y[2][2][4], Yx[2][2][4];  // high x high; the cross terms (scaled by 2^11)
#pragma unroll
                for (int x = 0; x < 2; ++x)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e) Y[x][n][e] = Yx[x][n][e] = 0.f;
                // the warp's slice of S scaled by 2^es into the fp16 range
                float m = 0.f;
#pragma unroll
                for (int j = 0; j < D / 8; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) m = fmaxf(m, fabsf(Sd[j][e]));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                const int es = scale_exp(m);
                const float ss = pow2i(es);
                const uint32_t* Kh = reinterpret_cast<const uint32_t*>(sm + OFF_KG);
                const uint32_t* Kl = reinterpret_cast<const uint32_t*>(sm + OFF_KGL);
                const uint32_t* Qh = reinterpret_cast<const uint32_t*>(sm + OFF_QG);
                const uint32_t* Ql = reinterpret_cast<const uint32_t*>(sm + OFF_QGL);
#pragma unroll
                for (int kt = 0; kt < D / 16; ++kt) {  // rows 16 kt .. 16 kt + 15 = fragments 2kt, 2kt + 1
                    uint32_t ah[4], al[4];
                    split_f16x2(Sd[2 * kt][0] * ss, Sd[2 * kt][1] * ss, ah[0], al[0]);
                    split_f16x2(Sd[2 * kt][2] * ss, Sd[2 * kt][3] * ss, ah[1], al[1]);
                    split_f16x2(Sd[2 * kt + 1][0] * ss, Sd[2 * kt + 1][1] * ss, ah[2], al[2]);
                    split_f16x2(Sd[2 * kt + 1][2] * ss, Sd[2 * kt + 1][3] * ss, ah[3], al[3]);
#pragma unroll
                    for (int x = 0; x < 2; ++x)
#pragma unroll
                        for (int n = 0; n < 2; ++n) {
                            const int ob = (8 * n + fg) * RW + 8 * kt + fc;
                            const uint32_t* H = x ? Qh : Kh;
                            const uint32_t* L = x ? Ql : Kl;
                            const uint32_t bh[2] = {H[ob], H[ob + 4]}, bl[2] = {L[ob], L[ob + 4]};
                            mma_cross(Yx[x][n], ah, al, bh, bl);
                            mma_f16(Y[x][n], ah, bh[0], bh[1]);
                        }
                }
                // to the warp's scratch as [kind][token][column], scales undone
                const float rk = pow2i(-es - ek), rq = pow2i(-es - eq);
#pragma unroll
                for (int x = 0; x < 2; ++x)
#pragma unroll
                    for (int n = 0; n < 2; ++n)
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            ws[x * C * 16 + (8 * n + 2 * fc + (e & 1)) * 16 + fg + 8 * (e >> 1)] =
                                fmaf(Yx[x][n][e], LO_DOWN, Y[x][n][e]) * (x ? rq : rk);
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
            // S^T <- S^T diag(exp(G_L)) + U^T K_T on the warp MMA (U = diag(beta) E); U scaled by
            // 2^eu into the fp16 range, K_T by 2^ek, and S^T by both for the accumulation
            {
                float uv[8];
                {
                    const float* u = ws + 2 * fc * 16 + fg;  // E[token][column]
                    const float b0 = sm[OFF_BT + 2 * fc], b1 = sm[OFF_BT + 2 * fc + 1];
                    const float b8 = sm[OFF_BT + 2 * fc + 8], b9 = sm[OFF_BT + 2 * fc + 9];
                    uv[0] = b0 * u[0];   uv[1] = b1 * u[16];       // column g, tokens 2c, 2c + 1
                    uv[2] = b0 * u[8];   uv[3] = b1 * u[24];       // column g + 8
                    uv[4] = b8 * u[128]; uv[5] = b9 * u[144];      // column g, tokens 2c + 8, 2c + 9
                    uv[6] = b8 * u[136]; uv[7] = b9 * u[152];      // column g + 8
                }
                float m = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(uv[e]));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                const int eu = scale_exp(m);
                const float su = pow2i(eu), sup = pow2i(eu + ek), rup = pow2i(-eu - ek);
                uint32_t uh[4], ul[4];
                split_f16x2(uv[0] * su, uv[1] * su, uh[0], ul[0]);
                split_f16x2(uv[2] * su, uv[3] * su, uh[1], ul[1]);
                split_f16x2(uv[4] * su, uv[5] * su, uh[2], ul[2]);
                split_f16x2(uv[6] * su, uv[7] * su, uh[3], ul[3]);
                const uint32_t* Th = reinterpret_cast<const uint32_t*>(sm + OFF_KTT);
                const uint32_t* Tl = reinterpret_cast<const uint32_t*>(sm + OFF_KTL);
#pragma unroll
                for (int j = 0; j < D / 8; ++j) {
                    const float2 gl = *reinterpret_cast<const float2*>(sm + OFF_GL + 8 * j + 2 * fc);
                    const float g0 = gl.x * sup * LO_UP, g1 = gl.y * sup * LO_UP;
                    Sd[j][0] *= g0; Sd[j][1] *= g1; Sd[j][2] *= g0; Sd[j][3] *= g1;
                    const int ob = (8 * j + fg) * RT + fc;  // tokens 2c, 2c + 1 (and + 8) of row 8j + g
                    const uint32_t bh[2] = {Th[ob], Th[ob + 4]}, bl[2] = {Tl[ob], Tl[ob + 4]};
                    mma_cross(Sd[j], uh, ul, bh, bl);  // at the scale 2^11 of the low parts
                    Sd[j][0] *= LO_DOWN; Sd[j][1] *= LO_DOWN; Sd[j][2] *= LO_DOWN; Sd[j][3] *= LO_DOWN;
                    mma_f16(Sd[j], uh, bh[0], bh[1]);
                    Sd[j][0] *= rup; Sd[j][1] *= rup; Sd[j][2] *= rup; Sd[j][3] *= rup;
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
