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
// One warp per (tile of 8 tokens, block of 32 V channels): lane l owns V = 4
// or 8 consecutive channels (one 8- or 16-byte load per row), so a head of up
// to 32 V channels is reduced inside the warp. Both kernels are HBM-bound: x
// is read once from DRAM (the K-1 halo rows of a tile hit L2) and y written
// once.
#pragma once

#include "gdn_common.cuh"
#include "gdn_epilogue.cuh"  // sigmoid_fast
#include "gdn_tc_ptx.cuh"    // mbarrier, TMA

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
    if constexpr (V == 8 && sizeof(T) == 2) {  // eight bf16: one 16-byte store
        uint4 u;
        uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * h], v[2 * h + 1]);
            w[h] = *reinterpret_cast<uint32_t*>(&b);
        }
        *reinterpret_cast<uint4*>(p) = u;
    } else {
#pragma unroll
        for (int h = 0; h < V / 4; ++h) store4f(p + 4 * h, v + 4 * h);
    }
}

// silu, then the L2 norm over groups of `ng` channels (ng = 0: none; else a
// power of two, at least V, dividing 32 V: the group spans ng / V lanes). NG
// fixes the group at compile time: 0 (no norm), a group size, or -1 (ng).
template <int V, int NG = -1>
__device__ __forceinline__ void silu_norm(float* s, int ng, float eps) {
#pragma unroll
    for (int j = 0; j < V; ++j) s[j] = silu_f(s[j]);
    const int g = NG >= 0 ? NG : ng;
    if (g) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < V; ++j) ss = fmaf(s[j], s[j], ss);
        if constexpr (NG > 0) {
#pragma unroll
            for (int off = 1; off < NG / V; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        } else {
            for (int off = 1; off < g / V; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        }
        const float r = rsqrtf(ss + eps);
#pragma unroll
        for (int j = 0; j < V; ++j) s[j] *= r;
    }
}

// silu_norm on P pairs of channels with the packed fp32 operations: silu is
// bit-identical to silu_norm's; the squares of a norm group are summed as two
// interleaved partial sums (even and odd channels) before the shuffles.
template <int P, int NG = -1>
__device__ __forceinline__ void silu_norm2(float2* s, int ng, float eps) {
    const float2 m = make_float2(-1.4426950408889634f, -1.4426950408889634f), one = make_float2(1.f, 1.f);
#pragma unroll
    for (int q = 0; q < P; ++q) {
        const float2 z = __fmul2_rn(m, s[q]);
        float2 e, r;
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.x) : "f"(z.x));
        asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e.y) : "f"(z.y));
        const float2 d = __fadd2_rn(one, e);
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.x) : "f"(d.x));
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r.y) : "f"(d.y));
        s[q] = __fmul2_rn(s[q], r);
    }
    constexpr int V = 2 * P;
    const int g = NG >= 0 ? NG : ng;
    if (g) {
        float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < P; ++q) ss2 = __ffma2_rn(s[q], s[q], ss2);
        float ss = ss2.x + ss2.y;
        if constexpr (NG > 0) {
#pragma unroll
            for (int off = 1; off < NG / V; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        } else {
            for (int off = 1; off < g / V; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        }
        const float r = rsqrtf(ss + eps);
        const float2 r2 = make_float2(r, r);
#pragma unroll
        for (int q = 0; q < P; ++q) s[q] = __fmul2_rn(s[q], r2);
    }
}

// Sequence of token t: cu == nullptr means num_seqs sequences of eq_len.
__device__ __forceinline__ int seq_of_token(const int32_t* cu, int num_seqs, long long eq_len, long long t) {
    if (cu == nullptr) return (int)((uint32_t)t / (uint32_t)eq_len);  // token counts fit 31 bits
    int lo = 0, hi = num_seqs;  // cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

// V consecutive elements of a row as raw 32-bit words (bf16 pairs or fp32),
// kept packed in registers until a tap uses them.
template <typename T, int V> struct RawRow {
    static constexpr int W = V * (int)sizeof(T) / 4;
    uint32_t u[W];
};
template <typename T, int V>
__device__ __forceinline__ RawRow<T, V> load_row(const T* p) {
    RawRow<T, V> r;
    constexpr int W = RawRow<T, V>::W;  // 2 (8-byte load), 4 or 8 (one or two 16-byte loads)
    if constexpr (W == 2) {
        const uint2 a = *reinterpret_cast<const uint2*>(p);
        r.u[0] = a.x; r.u[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < W; i += 4) {
            const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(p) + i);
            r.u[i] = a.x; r.u[i + 1] = a.y; r.u[i + 2] = a.z; r.u[i + 3] = a.w;
        }
    }
    return r;
}
template <typename T, int V> __device__ __forceinline__ RawRow<T, V> zero_row() {
    RawRow<T, V> r;
#pragma unroll
    for (int i = 0; i < RawRow<T, V>::W; ++i) r.u[i] = 0u;
    return r;
}
__device__ __forceinline__ float raw_val(const uint32_t* u, int j, const __nv_bfloat16*) {
    return __uint_as_float((j & 1) ? (u[j >> 1] & 0xffff0000u) : (u[j >> 1] << 16));
}
__device__ __forceinline__ float raw_val(const uint32_t* u, int j, const float*) { return __uint_as_float(u[j]); }

// The TT tokens [tb, tb + nt) of one block of 32 V channels, for the lane's
// V channels c .. c + V - 1, from row(r) = the input of token tb - H + r
// (zero outside the tensor) and the weights as channel pairs w2[q][i] = (w[c +
// 2q][i], w[c + 2q + 1][i]): the taps of a token that fall before its
// sequence's first token come from the caller's conv state (or are zero), and
// the tokens may span several sequences. The lane that holds a sequence's
// last token writes that sequence's final conv state.
template <typename T, int K, int V, int NG, int TT, typename RowFn>
__device__ __forceinline__ void conv_tokens(RowFn row, const float2 (&w2)[V / 2][K],
                                            long long tb, int nt, int c, bool live, const T* x, T* __restrict__ y,
                                            const int32_t* __restrict__ cu, const float* __restrict__ st_in,
                                            float* __restrict__ st_out, int num_seqs, long long total,
                                            long long eq_len, int C, int ng, float eps, int lane) {
    constexpr int H = K - 1;
    auto wsc = [&](int j, int i) { return (j & 1) ? w2[j >> 1][i].y : w2[j >> 1][i].x; };
    int n = seq_of_token(cu, num_seqs, eq_len, tb);
    long long t0 = cu ? cu[n] : (long long)n * eq_len;
    long long t1 = cu ? cu[n + 1] : t0 + eq_len;
    bool bad = tb < t0 || tb >= t1 || t0 < 0 || t1 > total;
    if (!bad && nt == TT && tb - H >= t0 && tb + TT <= t1) {
        // Common case: the tile and its halo lie inside one sequence. Straight-line
        // code on pairs of channels (the packed fp32 multiply, add and FMA of
        // sm_100 give the scalar operations' IEEE results with half the
        // instructions): each row is widened to fp32 once and slides through the
        // window.
        constexpr int P = V / 2;
        float2 win[K][P];
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const RawRow<T, V> ri = row(i);
#pragma unroll
            for (int q = 0; q < P; ++q) win[i][q] = make_float2(raw_val(ri.u, 2 * q, x), raw_val(ri.u, 2 * q + 1, x));
        }
        T* yp = y + tb * C + c;
#pragma unroll
        for (int k = 0; k < TT; ++k) {
            const RawRow<T, V> rk = row(k + H);
#pragma unroll
            for (int q = 0; q < P; ++q) win[H][q] = make_float2(raw_val(rk.u, 2 * q, x), raw_val(rk.u, 2 * q + 1, x));
            float2 acc[P];
#pragma unroll
            for (int q = 0; q < P; ++q) {
                float2 a = __fmul2_rn(w2[q][0], win[0][q]);
#pragma unroll
                for (int i = 1; i < K; ++i) a = __ffma2_rn(w2[q][i], win[i][q], a);
                acc[q] = a;
            }
            silu_norm2<P, NG>(acc, ng, eps);
            if (live) storeVf<V>(yp, reinterpret_cast<const float*>(acc));
            yp += C;
#pragma unroll
            for (int i = 0; i < H; ++i)
#pragma unroll
                for (int q = 0; q < P; ++q) win[i][q] = win[i + 1][q];
        }
        if (st_out && live && tb + TT == t1) {  // the tile ends the sequence: its H newest inputs
            float* so = st_out + ((size_t)n * C + c) * H;
#pragma unroll
            for (int i = 0; i < H; ++i)
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    so[(2 * q) * H + i] = win[i][q].x;
                    so[(2 * q + 1) * H + i] = win[i][q].y;
                }
        }
        return;
    }
    // input at position p of sequence n (p < t0: the caller's past, or zero)
    auto past = [&](long long p, int j) -> float {
        return st_in ? st_in[((size_t)n * C + c + j) * H + (p - t0 + H)] : 0.f;
    };
#pragma unroll
    for (int k = 0; k < TT; ++k) {
        if (k >= nt || bad) break;
        const long long t = tb + k;
        while (t >= t1) {  // the next non-empty sequence starts here (warp-uniform)
            ++n;
            if (n >= num_seqs) { bad = true; break; }
            t0 = cu ? cu[n] : (long long)n * eq_len;
            t1 = cu ? cu[n + 1] : t0 + eq_len;
            if (t0 != t || t1 > total) { bad = true; break; }
        }
        if (bad) break;
        float acc[V];
#pragma unroll
        for (int j = 0; j < V; ++j) acc[j] = wsc(j, K - 1) * raw_val(row(k + H).u, j, x);
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const long long p = t - H + i;
            if (p >= t0) {
#pragma unroll
                for (int j = 0; j < V; ++j) acc[j] = fmaf(wsc(j, i), raw_val(row(k + i).u, j, x), acc[j]);
            } else if (live) {
#pragma unroll
                for (int j = 0; j < V; ++j) acc[j] = fmaf(wsc(j, i), past(p, j), acc[j]);
            }
        }
        silu_norm<V, NG>(acc, ng, eps);  // every lane takes part in the shuffles
        if (live) {
            storeVf<V>(y + t * C + c, acc);
            if (st_out && t == t1 - 1) {  // the H newest inputs become the state
                float* so = st_out + ((size_t)n * C + c) * H;
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const long long p = t - (H - 1) + i;
#pragma unroll
                    for (int j = 0; j < V; ++j)
                        so[j * H + i] = p >= t0 ? raw_val(row(k + 1 + i).u, j, x) : past(p, j);
                }
            }
        }
    }
    if (bad && lane == 0) set_device_error(1u);  // cu_seqlens not ascending or out of range
}

// Tiled filter: each warp takes a tile of TT consecutive tokens for one block
// of 32 V channels (V per lane, 16-byte loads). It loads the tile's rows and
// the K-1 rows before it in one batch (all loads in flight together; the
// halo rows are re-read from L2 by the neighbouring tile), then evaluates the
// tokens one by one from registers (conv_tokens).
template <typename T, int K, int V, int NG>
__global__ void __launch_bounds__(256)
short_conv_kernel(const T* __restrict__ x, const float* __restrict__ w, T* __restrict__ y,
                  const int32_t* __restrict__ cu, const float* __restrict__ st_in, float* __restrict__ st_out,
                  int num_seqs, long long total, long long eq_len, int C, int ng, float eps) {
    constexpr int TT = 8, H = K - 1, NR = TT + H;
    const int lane = threadIdx.x & 31;
    const int c = (int)blockIdx.y * (32 * V) + V * lane;
    const bool live = c < C;  // C % V == 0: a lane's V channels are all in or all out
    float2 w2[V / 2][K];
#pragma unroll
    for (int q = 0; q < V / 2; ++q)
#pragma unroll
        for (int i = 0; i < K; ++i)
            w2[q][i] = live ? make_float2(w[(size_t)(c + 2 * q) * K + i], w[(size_t)(c + 2 * q + 1) * K + i])
                            : make_float2(0.f, 0.f);
    const long long tiles = (total + TT - 1) / TT;
    for (long long tile = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); tile < tiles;
         tile += (long long)gridDim.x * 8) {
        const long long tb = tile * TT;
        const int nt = (int)(total - tb < TT ? total - tb : TT);
        // row r holds the input of token tb - H + r
        RawRow<T, V> rows[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const long long p = tb - H + r;
            rows[r] = (live && p >= 0 && r < H + nt) ? load_row<T, V>(x + p * C + c) : zero_row<T, V>();
        }
        conv_tokens<T, K, V, NG, TT>([&](int r) { return rows[r]; }, w2, tb, nt, c, live, x, y, cu, st_in, st_out,
                                     num_seqs, total, eq_len, C, ng, eps, lane);
    }
}

// The same filter fed by TMA: a persistent CTA of 8 warps takes tiles of 64
// tokens x 32 V channels (V = 16 bytes per lane: 8 bf16 or 4 fp32). One thread
// loads each tile's 64 + K - 1 rows (512 bytes each, the K - 1 rows before
// the tile included; rows outside the tensor read as zeros) into a ring of
// STAGES shared-memory stages, STAGES tiles ahead; each warp evaluates its 8
// tokens with conv_tokens, reading their rows (and the halo) from the stage,
// then releases the stage. Every tile of a CTA has the same channel
// block (the grid is a multiple of the channel blocks), so the weights are
// loaded once. Waits are bounded: on a timeout the CTA records
// GDN_DEVERR_TIMEOUT, waits (bounded) for the loads it issued and returns.
namespace pro {
constexpr int TW = 8;                 // tokens per warp
constexpr int TILE = 8 * TW;          // tokens per tile
constexpr int STAGES = 3;
constexpr uint32_t ROW_BYTES = 512;   // 32 lanes x 16 bytes
template <int K> constexpr uint32_t stage_bytes() { return (uint32_t)(TILE + K - 1) * ROW_BYTES; }
template <int K> constexpr uint32_t smem_bytes() { return STAGES * stage_bytes<K>() + 2 * STAGES * 8 + 1024; }
}  // namespace pro

template <typename T, int K, int NG>
__global__ void __launch_bounds__(256, 2)
short_conv_tma_kernel(const __grid_constant__ CUtensorMap mapX, const T* __restrict__ x, const float* __restrict__ w,
                      T* __restrict__ y, const int32_t* __restrict__ cu, const float* __restrict__ st_in,
                      float* __restrict__ st_out, int num_seqs, long long total, long long eq_len, int C, int ng,
                      float eps, uint32_t max_polls) {
    using namespace tc;
    constexpr int V = 16 / (int)sizeof(T), H = K - 1;
    constexpr uint32_t SB = pro::stage_bytes<K>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(sm + pro::STAGES * SB);
    uint64_t* empty = full + pro::STAGES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ncb = C / (32 * V);
    const long long ntiles = (total + pro::TILE - 1) / pro::TILE * ncb;
    const int cb = (int)(blockIdx.x % (unsigned)ncb);  // gridDim.x is a multiple of ncb
    const int c = cb * (32 * V) + V * lane;
    float2 w2[V / 2][K];
#pragma unroll
    for (int q = 0; q < V / 2; ++q)
#pragma unroll
        for (int i = 0; i < K; ++i) w2[q][i] = make_float2(w[(size_t)(c + 2 * q) * K + i], w[(size_t)(c + 2 * q + 1) * K + i]);
    if (threadIdx.x == 0) {
        for (int i = 0; i < pro::STAGES; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], 8); }
        mbar_fence_init();
        tma_prefetch_desc(&mapX);
    }
    __syncthreads();
    // tile u: tokens (u / ncb) * TILE .., channel block u % ncb
    auto issue = [&](long long i) {  // local tile i of this CTA into stage i % STAGES
        const long long u = blockIdx.x + i * gridDim.x;
        const int s = (int)(i % pro::STAGES);
        mbar_arrive_expect_tx(&full[s], SB);
        tma_load_2d(sm + s * SB, &mapX, &full[s], cb * 32 * V, (int)((u / ncb) * pro::TILE - H));
    };
    long long issued = 0;
    if (threadIdx.x == 0)
        for (; issued < pro::STAGES && blockIdx.x + issued * gridDim.x < ntiles; ++issued) issue(issued);
    bool ok = true;
    long long consumed = 0;  // tiles whose load this thread has seen land
    for (long long i = 0; blockIdx.x + i * gridDim.x < ntiles; ++i) {
        const int s = (int)(i % pro::STAGES);
        const uint32_t ph = (uint32_t)(i / pro::STAGES) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph, nullptr, max_polls))) { ok = false; break; }
        consumed = i + 1;
        const long long tb = (blockIdx.x + i * gridDim.x) / ncb * pro::TILE + warp * pro::TW;
        // this warp's rows (tokens tb - H .. tb + TW - 1), read from the stage as needed
        const uint8_t* srow = sm + s * SB + (uint32_t)(warp * pro::TW) * pro::ROW_BYTES + 16u * lane;
        auto row = [&](int r) { return *reinterpret_cast<const RawRow<T, V>*>(srow + (uint32_t)r * pro::ROW_BYTES); };
        if (tb < total) {
            const int nt = (int)(total - tb < pro::TW ? total - tb : pro::TW);
            conv_tokens<T, K, V, NG, pro::TW>(row, w2, tb, nt, c, true, x, y, cu, st_in, st_out, num_seqs, total,
                                             eq_len, C, ng, eps, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (threadIdx.x == 0 && blockIdx.x + issued * gridDim.x < ntiles) {
            // refill stage s once every warp is done with tile i
            if (!mbar_wait(&empty[s], ph, nullptr, max_polls)) ok = false;
            else issue(issued++);
        }
        if (!__all_sync(0xffffffffu, ok)) break;
    }
    if (threadIdx.x == 0) {
        // never leave with loads in flight: the stages issued beyond the tiles consumed
        for (long long j = consumed; j < issued; ++j)
            mbar_wait(&full[(int)(j % pro::STAGES)], (uint32_t)(j / pro::STAGES) & 1u, nullptr, 10000u);
        if (!ok) set_device_error(2u);
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
