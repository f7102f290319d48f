// Backward pass of the gated delta rule (the gradient needed to train the
// token mixer: "On the Design of Qwen3.8-Next Architecture", arXiv abstract,
// which weighs every change by its training cost next to its prefill and
// decode cost). The forward rule is the one of "Qwen3.8-Next design: hybrid
// attention, residuals and n-gram embeddings" (podcast transcript, segment 14):
//
//   e_t = v_t - a_t S_{t-1}^T k_t,  S_t = a_t S_{t-1} + b_t k_t e_t^T,  o_t = scale S_t^T q_t
//
// with a_t = exp(g_t), b_t = beta_t, S of shape d_k x d_v. Given dO and
// dS_T, the gradient follows the reverse-order chain rule, carrying
// D = dL/dS_t from the last token to the first:
//
//   D    += scale q_t dO_t^T          dq_t = scale S_t dO_t
//   de    = b_t D^T k_t = dv_t        dbeta_t = (D^T k_t) . e_t
//   dk_t  = b_t D e_t - a_t S_{t-1} de
//   D     = a_t (D - k_t de^T)        dS_0 = D after the first token
//
// and the decay gradient has the exact closed form
//
//   dg_t = <dS_T, S_T> + sum_{r >= t} (q_r . dq_r - v_r . dv_r)
//
// (<D_t, S_t> - dv_t.v_t = <D_t, a_t (I - b_t k_t k_t^T) S_{t-1}> = dg_t, and
// q_t . dq_t = dO_t . o_t), so no inner product with a whole state is needed.
//
// Design (one CTA of 256 threads per (sequence, value head), d_k = d_v = 128):
//  * Phase 1 runs the recurrence forward in fp32 registers. It stores the
//    state at the start of every block of BLK = 32 tokens (the checkpoints,
//    64 KB each) and, per token, the error e_t and q_t . dq_t in the caller's
//    workspace, and writes dq_t = scale S_t dO_t (it holds S_t).
//  * Phase 2 walks the blocks last to first. For a block it stages the
//    block's q, k, v, dO, g, beta and the stored e_t in shared memory, loads
//    the block's checkpoint S_b and runs the reverse steps with D in
//    registers.
//  * S_{t-1} is never stored per token: inside a block
//      S_{t-1} = gam_{t-1} S_b + sum_{s<t} Gam_{t-1,s} b_s k_s e_s^T
//    (gam, Gam: products of the block's decays), so the one state product of
//    the reverse step, S_{t-1} de, is S_b de (a pass over registers) plus a
//    block-local correction sum_{s<t} Gam_{t-1,s} b_s (e_s . de_t) k_s that is
//    applied to all tokens of the block at its end (two small products over
//    shared memory).
//  * Thread (warp w, lane l) holds rows 16w..16w+15, columns 4l..4l+3 of the
//    state (64 registers for S or S_b, 64 for D); state traffic is 128-bit
//    and coalesced. Column sums (S^T k, D^T k) go through one 8 x 128
//    shared-memory exchange; row sums (S dO, D e, S_b de) stay inside the warp
//    (a 16-value reduce-scatter over the lanes, 16 shuffles).
// Two block barriers per forward or reverse step.
#pragma once

#include "gdn_common.cuh"
#include "gdn_epilogue.cuh"

namespace gdn {
namespace bwd {

constexpr int D = 128;          // d_k = d_v
constexpr int BLK = 32;         // tokens per checkpoint block (= one warp's lanes)
constexpr int NT = 256;         // threads per CTA
constexpr int NW = NT / 32;     // warps; warp w owns 16 state rows
constexpr int RED = 132;        // padded row stride of the column-sum exchange
constexpr int SD = D * D;       // state elements

// Shared-memory layout (floats).
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + BLK * D;
constexpr int OFF_V = OFF_K + BLK * D;
constexpr int OFF_DO = OFF_V + BLK * D;
constexpr int OFF_E = OFF_DO + BLK * D;
constexpr int OFF_DE = OFF_E + BLK * D;
constexpr int OFF_DK = OFF_DE + BLK * D;
constexpr int OFF_RED = OFF_DK + BLK * D;
constexpr int OFF_CM = OFF_RED + NW * RED;
constexpr int OFF_G = OFF_CM + BLK * BLK;
constexpr int OFF_B = OFF_G + BLK;
constexpr int OFF_L = OFF_B + BLK;
constexpr int OFF_QDQ = OFF_L + BLK;
constexpr int OFF_VDV = OFF_QDQ + BLK * NW;
constexpr int OFF_DB = OFF_VDV + BLK * NW;
constexpr int OFF_QT = OFF_DB + BLK * NW;        // q_t . dq_t of the block's tokens
constexpr int OFF_MISC = OFF_QT + BLK;
constexpr int SMEM_FLOATS = OFF_MISC + 16;
constexpr size_t SMEM_BYTES = (size_t)SMEM_FLOATS * sizeof(float);
static_assert(OFF_RED % 4 == 0 && RED % 4 == 0, "float4 column-sum stores");

struct Args {
    const void* q; const void* k; const void* v; const void* dout;
    const float* g; const float* beta; const float* h0; const float* dht;
    const int32_t* cu; const int32_t* order;
    float* dq; float* dk;          // [T, H_v, 128]: final when H_v == H_qk, else per value head
    float* dv; float* dg; float* dbeta; float* dh0;
    float* ckpt;                   // [H_v, nslots, 128, 128]
    float* e_ws;                   // [T, H_v, 128]: e_t of every token (phase 1 -> phase 2)
    float* qdq_ws;                 // [T, H_v]: q_t . dq_t
    long long nslots;
    long long total, eq_len;
    int num_seqs, h_qk, h_v, grp;
    float scale;
};

// Sum over the 32 lanes of x[0..15] (row r of the thread's 16 rows), left in
// the lanes whose bits 1..4 give r: lane l holds the total of row (l >> 1) & 15.
__device__ __forceinline__ float row_reduce16(const float (&x)[16], int lane) {
    const unsigned F = 0xffffffffu;
    float y[8], z[4], w[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const float keep = b4 ? x[m + 8] : x[m], send = b4 ? x[m] : x[m + 8];
        y[m] = keep + __shfl_xor_sync(F, send, 16);      // row 8*b4 + m
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float keep = b3 ? y[m + 4] : y[m], send = b3 ? y[m] : y[m + 4];
        z[m] = keep + __shfl_xor_sync(F, send, 8);       // row 8*b4 + 4*b3 + m
    }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        const float keep = b2 ? z[m + 2] : z[m], send = b2 ? z[m] : z[m + 2];
        w[m] = keep + __shfl_xor_sync(F, send, 4);       // row 8*b4 + 4*b3 + 2*b2 + m
    }
    float s = (b1 ? w[1] : w[0]) + __shfl_xor_sync(F, b1 ? w[0] : w[1], 2);
    s += __shfl_xor_sync(F, s, 1);
    return s;
}

// The thread's 16 x 4 block of a row-major 128 x 128 fp32 state.
__device__ __forceinline__ void load_state(float (&S)[16][4], const float* src, int r0, int c0) {
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float4 v = *reinterpret_cast<const float4*>(src + (size_t)(r0 + r) * D + c0);
        S[r][0] = v.x; S[r][1] = v.y; S[r][2] = v.z; S[r][3] = v.w;
    }
}
__device__ __forceinline__ void store_state(const float (&S)[16][4], float* dst, int r0, int c0) {
#pragma unroll
    for (int r = 0; r < 16; ++r)
        *reinterpret_cast<float4*>(dst + (size_t)(r0 + r) * D + c0) = make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
}
__device__ __forceinline__ void zero_state(float (&S)[16][4]) {
#pragma unroll
    for (int r = 0; r < 16; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) S[r][c] = 0.f;
}

// Stage tokens [tb0, tb0 + n) of the sequence into shared memory as fp32
// (rows j >= n are zero, g = beta = 0), and the running sum of g in the block.
template <typename TIn, typename TdO>
__device__ __forceinline__ void load_block(float* sm, const Args& p, long long tb0, int n, int h, int hk) {
    const TIn* q = static_cast<const TIn*>(p.q);
    const TIn* k = static_cast<const TIn*>(p.k);
    const TIn* v = static_cast<const TIn*>(p.v);
    const TdO* dO = static_cast<const TdO*>(p.dout);
    for (int idx = threadIdx.x; idx < BLK * (D / 4); idx += NT) {
        const int j = idx >> 5, c = (idx & 31) * 4;
        float4 kq = make_float4(0.f, 0.f, 0.f, 0.f), kk = kq, kv = kq, kd = kq;
        if (j < n) {
            const long long t = tb0 + j;
            const size_t qk_off = ((size_t)t * p.h_qk + hk) * D + c;
            const size_t v_off = ((size_t)t * p.h_v + h) * D + c;
            kk = load4(k + qk_off);
            kv = load4(v + v_off);
            kq = load4(q + qk_off);
            kd = load4(dO + v_off);
        }
        *reinterpret_cast<float4*>(sm + OFF_K + j * D + c) = kk;
        *reinterpret_cast<float4*>(sm + OFF_V + j * D + c) = kv;
        *reinterpret_cast<float4*>(sm + OFF_Q + j * D + c) = kq;
        *reinterpret_cast<float4*>(sm + OFF_DO + j * D + c) = kd;
    }
    if (threadIdx.x < 32) {
        const int j = threadIdx.x;
        float gj = 0.f, bj = 0.f;
        if (j < n) {
            const size_t o = (size_t)(tb0 + j) * p.h_v + h;
            gj = p.g[o];
            bj = p.beta[o];
        }
        sm[OFF_G + j] = gj;
        sm[OFF_B + j] = bj;
        float L = gj;  // inclusive running sum over the block's lanes
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, L, off);
            if (j >= off) L += y;
        }
        sm[OFF_L + j] = L;
    }
}

// Column sums over all 128 rows of the per-thread partials c[4] (columns
// c0..c0+3): thread tid returns the total of column tid >> 1 (both threads of
// a pair hold it). Ends with the block barrier that publishes nothing else.
__device__ __forceinline__ float column_sum(float* sm, const float (&c)[4], int warp, int c0) {
    float* red = sm + OFF_RED;
    *reinterpret_cast<float4*>(red + warp * RED + c0) = make_float4(c[0], c[1], c[2], c[3]);
    __syncthreads();
    const int col = threadIdx.x >> 1, part = threadIdx.x & 1;
    float s = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) s += red[(part * 4 + m) * RED + col];
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    return s;
}

// One forward token j of the staged block: S <- a S + b k e^T with
// e = v - a S^T k stored to shared memory; then dq = scale S dO from the new
// state (written to p.dq) and the per-warp parts of q . dq.
__device__ __forceinline__ void forward_token(float* sm, float (&S)[16][4], const Args& p, int j,
                                              long long t, int h, int warp, int lane, int r0, int c0) {
    float kr[16];
#pragma unroll
    for (int r = 0; r < 16; r += 4) {
        const float4 x = *reinterpret_cast<const float4*>(sm + OFF_K + j * D + r0 + r);
        kr[r] = x.x; kr[r + 1] = x.y; kr[r + 2] = x.z; kr[r + 3] = x.w;
    }
    const float a = expf(sm[OFF_G + j]), b = sm[OFF_B + j];
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 16; ++r)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) c[cc] = fmaf(S[r][cc], kr[r], c[cc]);
    const float s = column_sum(sm, c, warp, c0);
    if ((threadIdx.x & 1) == 0) {
        const int col = threadIdx.x >> 1;
        sm[OFF_E + j * D + col] = sm[OFF_V + j * D + col] - a * s;
    }
    __syncthreads();
    const float4 e4 = *reinterpret_cast<const float4*>(sm + OFF_E + j * D + c0);
    const float u[4] = {b * e4.x, b * e4.y, b * e4.z, b * e4.w};
    const float4 d4 = *reinterpret_cast<const float4*>(sm + OFF_DO + j * D + c0);
    const float dov[4] = {d4.x, d4.y, d4.z, d4.w};
    float rr[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        rr[r] = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            S[r][cc] = fmaf(a, S[r][cc], kr[r] * u[cc]);
            rr[r] = fmaf(S[r][cc], dov[cc], rr[r]);
        }
    }
    const float srow = row_reduce16(rr, lane);
    float x = 0.f;
    if ((lane & 1) == 0) {
        const int i = r0 + (lane >> 1);
        const float dqv = p.scale * srow;
        p.dq[((size_t)t * p.h_v + h) * D + i] = dqv;
        x = sm[OFF_Q + j * D + i] * dqv;
    }
    x = warp_sum(x);
    if (lane == 0) sm[OFF_QDQ + j * NW + warp] = x;
}

// One reverse token j of the staged block (see the header for the algebra).
// Sb holds the block's checkpoint state. Writes dv; leaves in shared memory
// de_j, the partial dk_j = b D e - a gam_{j-1} S_b de (the in-block
// correction is added at the block's end) and the per-warp parts of
// v . dv and dbeta.
__device__ __forceinline__ void reverse_token(float* sm, float (&Dm)[16][4], const float (&Sb)[16][4],
                                              const Args& p, int j, long long t, int h, int warp, int lane,
                                              int r0, int c0) {
    float kr[16], qr[16];
#pragma unroll
    for (int r = 0; r < 16; r += 4) {
        const float4 x = *reinterpret_cast<const float4*>(sm + OFF_K + j * D + r0 + r);
        kr[r] = x.x; kr[r + 1] = x.y; kr[r + 2] = x.z; kr[r + 3] = x.w;
        const float4 y = *reinterpret_cast<const float4*>(sm + OFF_Q + j * D + r0 + r);
        qr[r] = p.scale * y.x; qr[r + 1] = p.scale * y.y; qr[r + 2] = p.scale * y.z; qr[r + 3] = p.scale * y.w;
    }
    const float a = expf(sm[OFF_G + j]), b = sm[OFF_B + j];
    const float4 d4 = *reinterpret_cast<const float4*>(sm + OFF_DO + j * D + c0);
    const float dov[4] = {d4.x, d4.y, d4.z, d4.w};
    float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < 16; ++r)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            Dm[r][cc] = fmaf(qr[r], dov[cc], Dm[r][cc]);
            c[cc] = fmaf(Dm[r][cc], kr[r], c[cc]);
        }
    const float s = column_sum(sm, c, warp, c0);   // (D^T k)_col
    float vd = 0.f, dbp = 0.f;
    if ((threadIdx.x & 1) == 0) {
        const int col = threadIdx.x >> 1;
        const float de = b * s;
        sm[OFF_DE + j * D + col] = de;
        p.dv[((size_t)t * p.h_v + h) * D + col] = de;
        vd = sm[OFF_V + j * D + col] * de;
        dbp = s * sm[OFF_E + j * D + col];
    }
    vd = warp_sum(vd);
    dbp = warp_sum(dbp);
    if (lane == 0) {
        sm[OFF_VDV + j * NW + warp] = vd;
        sm[OFF_DB + j * NW + warp] = dbp;
    }
    __syncthreads();
    const float4 e4 = *reinterpret_cast<const float4*>(sm + OFF_E + j * D + c0);
    const float4 f4 = *reinterpret_cast<const float4*>(sm + OFF_DE + j * D + c0);
    const float ev[4] = {e4.x, e4.y, e4.z, e4.w}, dev[4] = {f4.x, f4.y, f4.z, f4.w};
    float r2[16], r3[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        r2[r] = 0.f;
        r3[r] = 0.f;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            r2[r] = fmaf(Dm[r][cc], ev[cc], r2[r]);
            r3[r] = fmaf(Sb[r][cc], dev[cc], r3[r]);
            Dm[r][cc] = a * fmaf(-kr[r], dev[cc], Dm[r][cc]);
        }
    }
    const float s2 = row_reduce16(r2, lane);
    const float s3 = row_reduce16(r3, lane);
    if ((lane & 1) == 0) {
        const int i = r0 + (lane >> 1);
        const float gprev = j > 0 ? expf(sm[OFF_L + j - 1]) : 1.f;
        sm[OFF_DK + j * D + i] = b * s2 - a * gprev * s3;
    }
}

// End of a block (n tokens staged, reverse steps done): add the in-block
// correction to dk, write dk, dbeta and dg (reverse running sum with `carry`,
// held by warp 0).
__device__ __forceinline__ void finish_block(float* sm, const Args& p, long long tb0, int n, int h,
                                             int warp, int lane, float& carry) {
    __syncthreads();
    // Cm[t][s] = Gam_{t-1,s} b_s (e_s . de_t), s < t
    for (int t = warp; t < n; t += NW) {
        const float4 f4 = *reinterpret_cast<const float4*>(sm + OFF_DE + t * D + 4 * lane);
        const float Lt = sm[OFF_L + t - (t > 0 ? 1 : 0)];
        for (int s = 0; s < t; ++s) {
            const float4 e4 = *reinterpret_cast<const float4*>(sm + OFF_E + s * D + 4 * lane);
            float x = e4.x * f4.x + e4.y * f4.y + e4.z * f4.z + e4.w * f4.w;
            x = warp_sum(x);
            if (lane == 0) sm[OFF_CM + t * BLK + s] = expf(Lt - sm[OFF_L + s]) * sm[OFF_B + s] * x;
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < n * D; idx += NT) {
        const int t = idx >> 7, i = idx & (D - 1);
        float corr = 0.f;
        for (int s = 0; s < t; ++s) corr = fmaf(sm[OFF_CM + t * BLK + s], sm[OFF_K + s * D + i], corr);
        const float a = expf(sm[OFF_G + t]);
        p.dk[((size_t)(tb0 + t) * p.h_v + h) * D + i] = sm[OFF_DK + t * D + i] - a * corr;
    }
    if (warp == 0) {
        float x = 0.f, dbv = 0.f;
        if (lane < n) {
            x = sm[OFF_QT + lane];
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                x -= sm[OFF_VDV + lane * NW + w];
                dbv += sm[OFF_DB + lane * NW + w];
            }
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {   // suffix sums: x_t <- sum_{r >= t} x_r
            const float y = __shfl_down_sync(0xffffffffu, x, off);
            if (lane + off < 32) x += y;
        }
        if (lane < n) {
            const size_t o = (size_t)(tb0 + lane) * p.h_v + h;
            p.dg[o] = carry + x;
            p.dbeta[o] = dbv;
        }
        carry += __shfl_sync(0xffffffffu, x, 0);
    }
}

template <typename TIn, typename TdO>
__global__ void __launch_bounds__(NT, 1) backward_kernel(const Args p) {
    extern __shared__ float4 smem_f4[];
    float* sm = reinterpret_cast<float*>(smem_f4);
    const int pos = blockIdx.x / p.h_v, h = blockIdx.x - pos * p.h_v, hk = h / p.grp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = warp * 16, c0 = lane * 4;
    int n = 0;
    long long t0 = 0, t1 = 0;
    if (!seq_of(p.order, pos, p.num_seqs, n)) return;
    if (!seq_bounds(p.cu, n, p.num_seqs, p.total, p.eq_len, t0, t1)) return;
    const long long len = t1 - t0;
    const int nb = (int)((len + BLK - 1) / BLK);
    const long long slot0 = t0 / BLK + n;
    if (slot0 + nb > p.nslots) {  // unreachable with valid cu_seqlens; never index past the workspace
        if (threadIdx.x == 0) set_device_error(1u);
        return;
    }
    float* ck = p.ckpt + ((size_t)h * p.nslots + slot0) * SD;
    const size_t st_off = ((size_t)n * p.h_v + h) * SD;

    // ---- phase 1: forward, checkpoint at every block start
    float S[16][4];
    if (p.h0) load_state(S, p.h0 + st_off, r0, c0);
    else zero_state(S);
    for (int bi = 0; bi < nb; ++bi) {
        const long long tb0 = t0 + (long long)bi * BLK;
        const int nt = (int)min((long long)BLK, t1 - tb0);
        store_state(S, ck + (size_t)bi * SD, r0, c0);
        __syncthreads();
        load_block<TIn, TdO>(sm, p, tb0, nt, h, hk);
        __syncthreads();
        for (int j = 0; j < nt; ++j) forward_token(sm, S, p, j, tb0 + j, h, warp, lane, r0, c0);
        __syncthreads();
        // hand e_t and q_t . dq_t of the block to phase 2
        for (int idx = threadIdx.x; idx < nt * (D / 4); idx += NT) {
            const int j = idx >> 5, c = (idx & 31) * 4;
            *reinterpret_cast<float4*>(p.e_ws + ((size_t)(tb0 + j) * p.h_v + h) * D + c) =
                *reinterpret_cast<const float4*>(sm + OFF_E + j * D + c);
        }
        if (warp == 0 && lane < nt) {
            float x = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) x += sm[OFF_QDQ + lane * NW + w];
            p.qdq_ws[(size_t)(tb0 + lane) * p.h_v + h] = x;
        }
    }
    // <dS_T, S_T> starts the decay gradient's running sum
    float carry = 0.f;
    float Dm[16][4];
    if (p.dht) {
        load_state(Dm, p.dht + st_off, r0, c0);
        float x = 0.f;
#pragma unroll
        for (int r = 0; r < 16; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) x = fmaf(Dm[r][c], S[r][c], x);
        x = warp_sum(x);
        __syncthreads();
        if (lane == 0) sm[OFF_MISC + warp] = x;
        __syncthreads();
        if (warp == 0) {
            float y = lane < NW ? sm[OFF_MISC + lane] : 0.f;
            carry = warp_sum(y);
        }
    } else {
        zero_state(Dm);
    }

    // ---- phase 2: blocks last to first
    for (int bi = nb - 1; bi >= 0; --bi) {
        const long long tb0 = t0 + (long long)bi * BLK;
        const int nt = (int)min((long long)BLK, t1 - tb0);
        __syncthreads();
        load_block<TIn, TdO>(sm, p, tb0, nt, h, hk);
        for (int idx = threadIdx.x; idx < nt * (D / 4); idx += NT) {
            const int j = idx >> 5, c = (idx & 31) * 4;
            *reinterpret_cast<float4*>(sm + OFF_E + j * D + c) =
                *reinterpret_cast<const float4*>(p.e_ws + ((size_t)(tb0 + j) * p.h_v + h) * D + c);
        }
        if (threadIdx.x < nt) sm[OFF_QT + threadIdx.x] = p.qdq_ws[(size_t)(tb0 + threadIdx.x) * p.h_v + h];
        __syncthreads();
        load_state(S, ck + (size_t)bi * SD, r0, c0);   // S_b for the reverse steps
        for (int j = nt - 1; j >= 0; --j) reverse_token(sm, Dm, S, p, j, tb0 + j, h, warp, lane, r0, c0);
        finish_block(sm, p, tb0, nt, h, warp, lane, carry);
    }
    if (p.dh0) store_state(Dm, p.dh0 + st_off, r0, c0);
}

// dq, dk of a q/k head = sum over the grp value heads that read it:
// out[t, hk, :] = sum_g part[t, hk * grp + g, :], for both tensors.
__global__ void group_sum_kernel(const float* __restrict__ dq_part, const float* __restrict__ dk_part,
                                 float* __restrict__ dq, float* __restrict__ dk, long long units, int h_qk,
                                 int grp) {
    const int h_v = h_qk * grp;
    for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < units;
         u += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(u & 31) * 4;
        const long long th = u >> 5;              // t * h_qk + hk
        const long long t = th / h_qk;
        const int hk = (int)(th - t * h_qk);
        const size_t src = ((size_t)t * h_v + (size_t)hk * grp) * D + c;
        float4 aq = make_float4(0.f, 0.f, 0.f, 0.f), ak = aq;
        for (int gi = 0; gi < grp; ++gi) {
            const float4 x = *reinterpret_cast<const float4*>(dq_part + src + (size_t)gi * D);
            const float4 y = *reinterpret_cast<const float4*>(dk_part + src + (size_t)gi * D);
            aq.x += x.x; aq.y += x.y; aq.z += x.z; aq.w += x.w;
            ak.x += y.x; ak.y += y.y; ak.z += y.z; ak.w += y.w;
        }
        *reinterpret_cast<float4*>(dq + (size_t)th * D + c) = aq;
        *reinterpret_cast<float4*>(dk + (size_t)th * D + c) = ak;
    }
}

}  // namespace bwd
}  // namespace gdn
