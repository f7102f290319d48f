// Chunkwise-parallel prefill on the 5th-generation tensor cores (tcgen05 +
// TMEM), fed by TMA, for bf16 q/k/v and d_k = d_v = 128, chunk C = 64.
//
// The recurrence (gated delta rule, described in words in "Qwen3.8-Next
// design: hybrid attention, residuals and n-gram embeddings", podcast
// transcript segment 14) is advanced one chunk at a time. Per chunk, with the
// cumulative log-decay G, gamma_r = exp(G_r), Gamma_rs = exp(G_r - G_s):
//   A      = strictly-lower(diag(beta) (Gamma o K K^T)),  T = (I + A)^{-1}
//   W      = T diag(beta gamma) K,     U = T diag(beta) V
//   Delta  = U - W S                   (errors written by the chunk)
//   O      = scale diag(gamma) Q S + (scale Q K^T o Gamma o causal) Delta
//   S     <- gamma_last S + (diag(Gamma_last,.) K)^T Delta
//
// Everything is computed in the transposed frame so that every tensor-core
// product has M = 128 and the state's value dimension lands on TMEM lanes:
//   X      = [K; Q] K^T                                  (M1, 128x64x128)
//   -W^T   = K^T Bw^T,  Bw = -T diag(beta gamma)         (M2, 128x64x64)
//   U^T    = V^T Bu^T,  Bu = T diag(beta)                (M2, 128x64x64)
//   D^T    = U^T + S^T (-W)^T                            (M3a, 128x64x128)
//   O^T    = S^T (gamma scale Q)^T + D^T P^T             (M3b + M4)
//   Sacc   = (D^T diag(Gamma_last,.)) K                  (M5, 128x128x64)
//   S^T   <- gamma_last S^T + Sacc                       (fp32, registers)
// where D^T = Delta^T. Thread (j, half) of the state warps owns half of column
// j of S (TMEM lane j) in fp32 registers for the whole sequence; fp16 copies
// of S^T and of Delta^T (plain and decay-scaled) are written to TMEM and read
// there as the A operand of the next products. Only exponentials of G_r - G_s
// with r >= s are formed, so no factor exceeds 1 for g <= 0.
//
// T = (I + A)^{-1} is solved per 16 x 16 block: diagonal blocks by forward
// substitution in fp32, off-diagonal blocks on the warp-level tensor-core MMA
// (fp16 operands, fp32 accumulation), one block-row per warp.
//
// Operand precision: every product after X takes fp16 operands (10-bit
// mantissa) with fp32 accumulation; the bf16 inputs K, Q, V convert to fp16
// exactly (their magnitudes are far inside the fp16 range), so only the
// computed operands (S, Delta, T, W, P and the decay-scaled Q and Delta) are
// rounded, at 2^-11 instead of bf16's 2^-8. Decay-scaled values that fall
// below the fp16 range contribute less than 1e-7 of the largest terms. The
// path therefore needs |v|, |S| and the errors Delta to stay below 65504 (the
// fp16 range). A value beyond it becomes an infinity in the products and
// leaves a non-finite fp32 state behind; every unit checks its final state
// and records GDN_DEVERR_RANGE, so such inputs are reported, not silently
// wrong (the fp32 CUDA-core kernel serves them).
//
// Warp roles (512 threads) are listed where they branch (chunk_tc_kernel).
// One group of four prep warps builds T for every chunk (A/P pass, then the
// blocked solve); the state warps convert operands two chunks ahead in the
// time they would otherwise wait. The instruction footprint is kept small on
// purpose (rolled issue and conversion loops, one copy of each step): with 16
// warps running different code the instruction cache was the first
// bottleneck. All waits are bounded (a timeout raises an abort flag, records
// GDN_DEVERR_TIMEOUT and every role unwinds). On the way out nothing is left
// in flight: the TMA producer waits for the last load of each ring stage it
// filled, both MMA issuers commit a final barrier (B_DONE) that completes
// only when every product they issued has finished, and TMEM is freed after
// that barrier.
#pragma once

#include <cudaTypedefs.h>

#include "gdn_common.cuh"
#include "gdn_tc_ptx.cuh"

namespace gdn {

struct TcArgs {
    const void* q; const void* k; const void* v;
    const float* g; const float* beta; const float* h0;
    const int32_t* cu; const int32_t* order;
    void* o; float* hT;
    int num_seqs; long long total; long long eq_len;
    int h_qk, h_v, grp;
    float scale;
    uint32_t max_polls;    // poll limit of every mbarrier wait
    int withhold_chunk;    // test of the failure path: the g/beta arrival of this chunk is never made (-1: none)
    int nseg;              // segments per sequence (one CTA each; 1 = the whole sequence in one CTA)
    int bal_chunks;        // > 0: equal-length sequences, every grp CTAs take this many consecutive chunks of
                           // the (sequence, q/k head) groups in order, one CTA per value head of the group
                           // (at most two pieces of units each); nseg = 1
};

// A CTA's piece of a (sequence, value head) unit: it stores the outputs of
// tokens [seg_a, t1) and processes tokens [t0, t1), t0 <= seg_a (a prefix
// started from a zero state, or the sequence start s0 with the initial state)
struct Piece {
    long long t0, seg_a, t1, s0;
    int h, hk, n_seq, nc, len, from_start, last_seg, pad;
};

namespace tck {
constexpr int C = 64, D = 128;
constexpr int KQ_STAGES = 3, V_STAGES = 2, GB_SLOTS = 3;
constexpr int NTHREADS = 512;
// Registers: launched with REGS_LAUNCH per thread (512 x 128 = 65536). The
// single-thread roles give some up; the prep warps and the two state
// warpgroups (64 fp32 state values per thread) take them:
// 128 x (48 + 160 + 152 + 152) = 65536.
constexpr int REGS_LAUNCH = 128, REGS_ROLES = 48, REGS_PREP = 160, REGS_STATE = 152;
static_assert(128 * (REGS_ROLES + REGS_PREP + 2 * REGS_STATE) <= NTHREADS * REGS_LAUNCH,
              "register rebalancing exceeds the launch allocation");
// TMEM columns
constexpr uint32_t T_SACC = 0, T_DU = 128, T_O = 192, T_X = 256, T_W = 320, T_ST = 384, T_DT = 448,
                   T_DTD = 480;
constexpr uint32_t TMEM_COLS = 512;
// shared memory layout (byte offsets from a 1024-aligned base)
constexpr uint32_t KQ_BYTES = 32768;  // K kb0 | Q kb0 | K kb1 | Q kb1, 8 KB each (64 rows x 128 B)
constexpr uint32_t V_BYTES = 16384;   // V kb0 | V kb1
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_V = OFF_KQ + KQ_STAGES * KQ_BYTES;
constexpr uint32_t OFF_WT = OFF_V + V_STAGES * V_BYTES;  // -W^T, MN-major B: 128 rows (i) x 128 B (r)
constexpr uint32_t OFF_BW = OFF_WT + 16384;              // Bw x 2 buffers, K-major B: 64 rows (r) x 128 B (s)
constexpr uint32_t OFF_BU = OFF_BW + 16384;              // Bu x 2 buffers
constexpr uint32_t OFF_P = OFF_BU + 16384;               // P x 2 buffers, K-major B
// prep: A fp16 (64 rows x 128 B, 128-byte swizzle), the diagonal 16x16
// blocks of A in fp32 (column-major), those of T in fp16
constexpr uint32_t OFF_AS = OFF_P + 16384;
constexpr uint32_t OFF_AD = OFF_AS + 8192;
constexpr uint32_t OFF_TS = OFF_AD + 4096;
constexpr uint32_t OFF_GB = OFF_TS + 2048;
constexpr uint32_t GB_FLOATS = 6 * 64 + 4;               // G, gam, bet, bg, dec, qsc, gC
constexpr uint32_t GB_SLOT_BYTES = GB_FLOATS * 4;
constexpr uint32_t OFF_BAR = OFF_GB + GB_SLOTS * GB_SLOT_BYTES;
constexpr uint32_t NUM_BARS = 40;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t OFF_PIECES = OFF_MISC + 16;          // two Piece records
constexpr uint32_t SMEM_BYTES = OFF_PIECES + 2 * 64 + 1024;  // + alignment slack
static_assert(OFF_WT % 1024 == 0 && OFF_BW % 1024 == 0 && OFF_P % 1024 == 0 && OFF_AS % 1024 == 0,
              "tile alignment");
static_assert(GB_SLOT_BYTES % 16 == 0 && OFF_GB % 16 == 0, "gb slot alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// barrier indices
enum {
    B_FULL_KQ = 0, B_EMPTY_KQ = 3, B_FULL_V = 6, B_EMPTY_V = 8, B_GB_FULL = 10, B_GB_EMPTY = 13,
    B_XREADY0 = 16, B_XREADY1, B_XFREE, B_BWU0, B_BWU1, B_M2W0, B_M2W1, B_WREADY, B_DREADY, B_DELTA,
    B_SREADY, B_STREADY, B_OREADY, B_OFREE, B_PFREE0, B_PFREE1, B_DONE, B_CONV0, B_CONV1, B_M2U0, B_M2U1,
    B_VCONV0, B_VCONV1
};
static_assert(B_VCONV1 < (int)NUM_BARS, "barrier count");

// gb slot fields (float offsets)
constexpr int GB_G = 0, GB_GAM = 64, GB_BET = 128, GB_BG = 192, GB_DEC = 256, GB_QSC = 320, GB_GC = 384;

__device__ __forceinline__ uint32_t h2(float lo, float hi) { return tc::pack_f16x2(lo, hi); }
__device__ __forceinline__ float2 unbf2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
__device__ __forceinline__ float2 unh2(uint32_t u) {
    __half2 v = *reinterpret_cast<__half2*>(&u);
    return __half22float2(v);
}
// Write 64 floats v[0..63] as fp16 into row `row` of a 128B-swizzled tile.
__device__ __forceinline__ void store_row_sw128(uint8_t* tile, uint32_t row, const float* v) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 u;
        u.x = h2(v[8 * c + 0], v[8 * c + 1]); u.y = h2(v[8 * c + 2], v[8 * c + 3]);
        u.z = h2(v[8 * c + 4], v[8 * c + 5]); u.w = h2(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(tile + row * 128u + ((((uint32_t)c ^ row) & 7u) << 4)) = u;
    }
}

// Write 32 floats as fp16 into logical 16-byte chunks [4h, 4h + 4) of row
// `row` of a 128B-swizzled tile.
__device__ __forceinline__ void store_half_row_sw128(uint8_t* tile, uint32_t row, const float* v, int h) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint4 u;
        u.x = h2(v[8 * c + 0], v[8 * c + 1]); u.y = h2(v[8 * c + 2], v[8 * c + 3]);
        u.z = h2(v[8 * c + 4], v[8 * c + 5]); u.w = h2(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(tile + row * 128u + (((((uint32_t)(4 * h + c)) ^ row) & 7u) << 4)) = u;
    }
}

// Optional timeline instrumentation (compiled in only with -DGDN_TRACE):
// CTA 0 stores clock64() at fixed points of each role, per chunk, into a
// caller-provided buffer of 64 x 128 timestamps.
#ifdef GDN_TRACE
__device__ unsigned long long* g_trace;
#define GDN_TRACE_AT(point, n)                                                      \
    do {                                                                            \
        if (tb_ && (n) < 128) tb_[(point) * 128 + (n)] = clock64(); \
    } while (0)
#define GDN_TRACE_CTA(point)                                                        \
    do {                                                                            \
        if (g_trace && blockIdx.x < 128) g_trace[(point) * 128 + blockIdx.x] = globaltimer_ns(); \
    } while (0)
#else
#define GDN_TRACE_AT(point, n) \
    do {                       \
    } while (0)
#define GDN_TRACE_CTA(point) \
    do {                     \
    } while (0)
#endif
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// Named barrier that also ORs a predicate over its participants, so that a
// decision to leave a loop is taken by all of them together.
__device__ __forceinline__ bool named_sync_or(int id, int n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}


// Off-diagonal blocks of block-row bi (1..3) of T = (I + A)^{-1} (4 x 4
// blocks of 16 x 16), right-looking: T_ij = -(sum_{k=j+1..bi} T_ik A_kj) T_jj
// for j = bi-1 .. 0. One warp; T_ik stay in registers as fp16 A fragments,
// A_kj and T_jj come from shared memory through ldmatrix (fp16 operands, fp32
// accumulation). Each finished block is written, scaled by the column
// factors, into Bw = T diag(-beta gamma) and Bu = T diag(beta). The loops run
// over the largest case (bi = 3) with warp-uniform guards, so that the
// fragment registers keep compile-time indices and one copy of the code
// serves all three block-rows.
__device__ __forceinline__ void solve_block_row(int bi, uint32_t as_u, uint32_t ts_u, uint8_t* bw, uint8_t* bu,
                                                const float* gb, int lane) {
    using namespace tc;
    const int m = lane >> 3, lr = (lane & 7) + 8 * (m & 1), lc8 = m >> 1;
    auto a_addr = [&](int bk, int bj) {
        const uint32_t R = (uint32_t)(16 * bk + lr), ch = (uint32_t)(2 * bj + lc8);
        return as_u + R * 128u + (((ch ^ R) & 7u) << 4);
    };
    auto t_addr = [&](int bb) {
        return ts_u + (uint32_t)bb * 512u + (uint32_t)lr * 32u + (((uint32_t)lc8 ^ ((uint32_t)lr >> 2)) & 1u) * 16u;
    };
    const int g = lane >> 2, q = lane & 3;
    uint32_t Tf[4][4];  // Tf[k] = fragment of T_{bi,k}, k = j+1 .. bi
#pragma unroll
    for (int k = 1; k < 4; ++k)
        if (k == bi) ldsm_x4(t_addr(k), Tf[k]);
#pragma unroll
    for (int j = 2; j >= 0; --j) {
        if (j >= bi) continue;
        float y0[4] = {0.f, 0.f, 0.f, 0.f}, y1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = j + 1; k < 4; ++k) {
            if (k > bi) break;
            uint32_t b[4];
            ldsm_x4_t(a_addr(k, j), b);
            mma16816(y0, Tf[k], b[0], b[1]);
            mma16816(y1, Tf[k], b[2], b[3]);
        }
        const uint32_t ya[4] = {h2(y0[0], y0[1]), h2(y0[2], y0[3]), h2(y1[0], y1[1]), h2(y1[2], y1[3])};
        uint32_t bt[4];
        ldsm_x4_t(t_addr(j), bt);
        float z0[4] = {0.f, 0.f, 0.f, 0.f}, z1[4] = {0.f, 0.f, 0.f, 0.f};
        mma16816(z0, ya, bt[0], bt[1]);
        mma16816(z1, ya, bt[2], bt[3]);
        // T_{bi,j} = -z
        Tf[j][0] = h2(-z0[0], -z0[1]); Tf[j][1] = h2(-z0[2], -z0[3]);
        Tf[j][2] = h2(-z1[0], -z1[1]); Tf[j][3] = h2(-z1[2], -z1[3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const float* z = nt ? z1 : z0;
            const int S_ = 16 * j + 8 * nt + 2 * q;
            const float2 fbg = *reinterpret_cast<const float2*>(gb + GB_BG + S_);
            const float2 fbe = *reinterpret_cast<const float2*>(gb + GB_BET + S_);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint32_t R = (uint32_t)(16 * bi + g + 8 * hh);
                const uint32_t off = R * 128u + (((((uint32_t)S_ >> 3) ^ R) & 7u) << 4) + (uint32_t)(S_ & 7) * 2u;
                *reinterpret_cast<uint32_t*>(bw + off) = h2(z[2 * hh] * fbg.x, z[2 * hh + 1] * fbg.y);
                *reinterpret_cast<uint32_t*>(bu + off) = h2(-z[2 * hh] * fbe.x, -z[2 * hh + 1] * fbe.y);
            }
        }
    }
}

// A/P pass of the prep warps on chunk n of the CTA (the A and Ad tiles and P
// buffer n & 1; `rows` of its rows are tokens): from X = [K; Q] K^T in TMEM,
// row r of A (rows 0-63, TMEM lanes 0-63) or of P (lanes 64-127) per thread;
// gt = the thread's TMEM lane.
__device__ __forceinline__ void ap_pass(uint8_t* sm, uint32_t tmem, const float* gb, int n, int rows, float scale,
                                        int gt, unsigned long long* tb_) {
    using namespace tc;
    const int wq = gt >> 5;
    const int grp = n & 1;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    uint8_t* As = sm + OFF_AS;
    float* Ad = reinterpret_cast<float*>(sm + OFF_AD);
    // ---- A = strictly-lower(diag(beta) Gamma o K K^T) (fp16 tile + fp32
    //      diagonal blocks) and P = scale (Gamma o Q K^T) masked r >= s
    //      (fp16 B tile). Rows 0-31 only have columns 0-31.
    {
        const bool isA = wq < 2;
        const int r = isA ? gt : gt - 64;
        // beta_r and the output scale enter as exponent offsets (log2 of 0 is -inf: row of zeros)
        const float base = gb[GB_G + r] + (isA ? lg2(gb[GB_BET + r]) : lg2(scale));
        // kept columns: s < r (A), s <= r on live rows (P)
        const int lim = isA ? r : (r < rows ? r + 1 : 0);
        uint8_t* row = isA ? As + r * 128 : sm + OFF_P + (uint32_t)grp * 8192 + r * 128;
        const bool wide = (wq & 1) != 0;  // rows 32-63
        // quarters of 16 columns (rows 0-31 need only 0-31); rows 32-63 take
        // columns 32-63 first: once they are stored, the diagonal blocks 2 and
        // 3 of A are complete and the warp of P rows 0-31 (done early) solves
        // them while this warp finishes columns 0-31
#pragma unroll 1
        for (int qi = 0; qi < 4; ++qi) {
            if (qi >= 2 && !wide) break;
            const int qc = wide ? ((qi + 2) & 3) : qi;
            uint32_t x[16];
            if (qc == 0 && gt == 0) GDN_TRACE_AT(7, n);
            tmem_ld16(tmem + lane_base + T_X + 16 * qc, x);
            tmem_ld_wait();
            if (qc == 0 && gt == 0) GDN_TRACE_AT(8, n);
            // in place: x[e] becomes the fp32 value of column 16 qc + e
            const uint32_t src = smem_u32(gb + GB_G) + 64u * (uint32_t)qc;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 g4 = lds_f4(src + 16u * (uint32_t)q4);
                const float gq[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    const int e = 4 * q4 + e4;
                    // Gamma_rs = exp(G_r - G_s) <= 1 for s <= r (beta_r / scale folded in)
                    x[e] = __float_as_uint((16 * qc + e < lim) ? ex2(base - gq[e4]) * __uint_as_float(x[e]) : 0.f);
                }
            }
            if (qc == 0 && gt == 0) GDN_TRACE_AT(9, n);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const int c = 2 * qc + c2;
                uint4 u;
                u.x = h2(__uint_as_float(x[8 * c2 + 0]), __uint_as_float(x[8 * c2 + 1]));
                u.y = h2(__uint_as_float(x[8 * c2 + 2]), __uint_as_float(x[8 * c2 + 3]));
                u.z = h2(__uint_as_float(x[8 * c2 + 4]), __uint_as_float(x[8 * c2 + 5]));
                u.w = h2(__uint_as_float(x[8 * c2 + 6]), __uint_as_float(x[8 * c2 + 7]));
                *reinterpret_cast<uint4*>(row + ((((uint32_t)c ^ (uint32_t)r) & 7u) << 4)) = u;
            }
            if (isA && ((r >> 4) == qc)) {  // diagonal 16x16 block in fp32, column-major
                float* dcol = Ad + (r >> 4) * 256 + (r & 15);
#pragma unroll
                for (int e = 0; e < 16; ++e) dcol[16 * e] = __uint_as_float(x[e]);
            }
            if (qc == 0 && gt == 0) GDN_TRACE_AT(6, n);
            if (isA && wide && qi == 1) {  // A rows 32-63: diagonal blocks 2, 3 stored
                __syncwarp();
                named_arrive(2, 64);
            }
        }
        if (!isA) fence_async_smem();
    }
}

// First token that a CTA must process for a segment whose outputs start at
// token a of a sequence that starts at s0 (one warp; every lane returns it).
// Each token t maps a difference of two states D to alpha_t (I - beta_t k_t
// k_t^T) D, whose spectral norm is at most c_t = alpha_t max(1, |1 - beta_t
// |k_t|^2|) times that of D. Starting from a zero state at token ts changes
// the state at token a - 1 by at most prod_{t=ts}^{a-1} c_t times the true
// state before ts. The result is the nearest ts with that product below
// 2^-40 (far below fp32 rounding), or s0 (exact: the sequence's own start)
// when the decay never gets there, e.g. for alpha = 1.
__device__ __forceinline__ long long segment_prefix_start(const TcArgs& p, long long s0, long long a, int h,
                                                          int hk, int lane) {
    constexpr float LN_EPS = -27.7258872f;  // 40 ln 2
    const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(p.k);
    float acc = 0.f;  // log of the product over the tokens scanned so far
    for (long long p0 = a; p0 > s0; p0 -= 32) {
        const long long tok = p0 - 1 - lane;  // lane 0: the token nearest to a
        const bool valid = tok >= s0;
        float c = 0.f;
        if (valid) {
            // all loads of the token in flight together (one memory round trip)
            const float gt = p.g[(size_t)tok * p.h_v + h], bt = p.beta[(size_t)tok * p.h_v + h];
            const uint4* kp = reinterpret_cast<const uint4*>(kb + ((size_t)tok * p.h_qk + hk) * D);
            uint4 u[D / 8];
#pragma unroll
            for (int i = 0; i < D / 8; ++i) u[i] = kp[i];
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float lo = __uint_as_float(w[e] << 16), hi = __uint_as_float(w[e] & 0xffff0000u);
                    ss = fmaf(lo, lo, fmaf(hi, hi, ss));
                }
            }
            const float f = fabsf(1.f - bt * ss);
            c = gt + (f > 1.f ? logf(f) : 0.f);
        }
        float incl = c;  // sum over tokens p0 - 1 .. tok
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

template <typename TOut>
__global__ void __launch_bounds__(NTHREADS, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV, TcArgs p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic (not through an
    // integer) so that the compiler keeps every access in the shared space
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC + 4);

    // ---- work of this CTA: one or two pieces of (sequence, value head) units.
    //      A piece stores the outputs of tokens [seg_a, t1); it starts from a
    //      zero state a few tokens earlier (segment_prefix_start), or from the
    //      sequence's initial state at its first token. Either a segment of a
    //      unit (nseg segments per sequence), or, with bal_chunks, the CTA's
    //      share of the chunks of all units taken in order (equal lengths: a
    //      share ends at most one unit after the one it starts in).
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    Piece* pieces = reinterpret_cast<Piece*>(sm + OFF_PIECES);
    // (seq_a: first stored token, t1: end, s0, s1: the sequence, h: value head)
    struct Spec { long long seg_a, t1, s0, s1; int h, n_seq; };
    Spec sp0{}, sp1{};
    int npieces = 0;
    if (p.bal_chunks == 0) {
        const int seg = blockIdx.x % p.nseg;
        const int h = (blockIdx.x / p.nseg) % p.h_v;
        const int pos = blockIdx.x / p.nseg / p.h_v;
        int n_seq;
        if (!seq_of(p.order, pos, p.num_seqs, n_seq)) return;
        long long s0, s1;  // the sequence's tokens
        if (!seq_bounds(p.cu, n_seq, p.num_seqs, p.total, p.eq_len, s0, s1)) return;
        const long long seg_len = ((s1 - s0 + p.nseg - 1) / p.nseg + C - 1) / C * C;
        const long long seg_a = s0 + seg * seg_len;
        if (seg > 0 && seg_a >= s1) return;  // an empty segment
        sp0 = Spec{seg_a, seg_len > 0 && seg_a + seg_len < s1 ? seg_a + seg_len : s1, s0, s1, h, n_seq};
        npieces = 1;
    } else {
        // shares of the chunks of the (sequence, q/k head) groups in order; the
        // grp value heads of a group take the same share in grp neighbouring
        // CTAs, so that they read the group's q and k tiles at the same time
        const long long nch = (p.eq_len + C - 1) / C;  // chunks per unit
        const long long ctot = (long long)p.num_seqs * p.h_qk * nch;
        const int r = blockIdx.x % p.grp;  // value head within the group
        long long a = (long long)(blockIdx.x / p.grp) * p.bal_chunks;
        const long long b = min(a + (long long)p.bal_chunks, ctot);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (a >= b) break;
            const long long u = a / nch, c_lo = a - u * nch, c_hi = min(nch, c_lo + (b - a));
            const int h = (int)(u % p.h_qk) * p.grp + r, pos = (int)(u / p.h_qk);
            int n_seq;
            if (!seq_of(p.order, pos, p.num_seqs, n_seq)) return;
            long long s0, s1;
            if (!seq_bounds(p.cu, n_seq, p.num_seqs, p.total, p.eq_len, s0, s1)) return;
            const Spec x{s0 + c_lo * C, min(s0 + c_hi * C, s1), s0, s1, h, n_seq};
            if (i == 0) sp0 = x; else sp1 = x;
            ++npieces;
            a += c_hi - c_lo;
        }
        if (npieces == 0) return;
    }
    if (warp == 3) {
        auto fill = [&](Piece& P, const Spec x) {
            const int hk_i = x.h / p.grp;
            const long long ts = x.seg_a > x.s0 ? segment_prefix_start(p, x.s0, x.seg_a, x.h, hk_i, lane) : x.s0;
            if (lane == 0) {
                P.t0 = ts; P.seg_a = x.seg_a; P.t1 = x.t1; P.s0 = x.s0;
                P.h = x.h; P.hk = hk_i; P.n_seq = x.n_seq;
                P.len = (int)(x.t1 - ts); P.nc = (P.len + C - 1) / C;
                P.from_start = ts == x.s0;
                P.last_seg = x.t1 == x.s1;  // the piece ends the sequence: it writes the final state
                P.pad = 0;
            }
        };
        fill(pieces[0], sp0);
        if (npieces > 1) fill(pieces[1], sp1);
    }
#ifdef GDN_TRACE
    unsigned long long* const tb_ = blockIdx.x == 0 ? g_trace : nullptr;  // traced block
#else
    unsigned long long* const tb_ = nullptr;
    (void)tb_;
#endif
    if (threadIdx.x == 0) GDN_TRACE_CTA(62);
#ifdef GDN_TRACE
    if (threadIdx.x == 0 && g_trace && blockIdx.x < 128) {
        unsigned int smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        g_trace[61 * 128 + blockIdx.x] = smid;
    }
#endif

    if (threadIdx.x == 0) {
        for (int i = 0; i < KQ_STAGES; ++i) { mbar_init(&bars[B_FULL_KQ + i], 1); mbar_init(&bars[B_EMPTY_KQ + i], 1); }
        for (int i = 0; i < V_STAGES; ++i) { mbar_init(&bars[B_FULL_V + i], 1); mbar_init(&bars[B_EMPTY_V + i], 1); }
        for (int i = 0; i < GB_SLOTS; ++i) { mbar_init(&bars[B_GB_FULL + i], 1); mbar_init(&bars[B_GB_EMPTY + i], 12); }
        mbar_init(&bars[B_XREADY0], 1); mbar_init(&bars[B_XREADY1], 1); mbar_init(&bars[B_XFREE], 4);
        mbar_init(&bars[B_BWU0], 4); mbar_init(&bars[B_BWU1], 4);
        mbar_init(&bars[B_M2W0], 1); mbar_init(&bars[B_M2W1], 1); mbar_init(&bars[B_WREADY], 8);
        mbar_init(&bars[B_M2U0], 1); mbar_init(&bars[B_M2U1], 1);
        mbar_init(&bars[B_VCONV0], 1); mbar_init(&bars[B_VCONV1], 1);
        mbar_init(&bars[B_DREADY], 1); mbar_init(&bars[B_DELTA], 8); mbar_init(&bars[B_SREADY], 1);
        mbar_init(&bars[B_STREADY], 8); mbar_init(&bars[B_OREADY], 1); mbar_init(&bars[B_OFREE], 8);
        mbar_init(&bars[B_PFREE0], 1); mbar_init(&bars[B_PFREE1], 1); mbar_init(&bars[B_DONE], 2);
        mbar_init(&bars[B_CONV0], 8); mbar_init(&bars[B_CONV1], 8);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mapQ); tma_prefetch_desc(&mapK); tma_prefetch_desc(&mapV);
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    // Bw, Bu (both buffers) and P (both buffers) start as zeros: their blocks
    // above the diagonal are never written afterwards
    for (uint32_t i = threadIdx.x; i < (3u * 16384u) / 16u; i += NTHREADS)
        reinterpret_cast<uint4*>(sm + OFF_BW)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int nc0 = pieces[0].nc;
    const int nc = nc0 + (npieces > 1 ? pieces[1].nc : 0);  // chunks of the CTA
    // the piece of the CTA's chunk m, and m's chunk index n within it
    auto piece_of = [&](int m, int& n) -> const Piece& {
        const int i = (npieces > 1 && m >= nc0) ? 1 : 0;
        n = m - (i ? nc0 : 0);
        return pieces[i];
    };
    if (lane == 0) GDN_TRACE_AT(60, warp);

    auto kq_tile = [&](int n) { return sm + OFF_KQ + (uint32_t)(n % KQ_STAGES) * KQ_BYTES; };
    auto v_tile = [&](int n) { return sm + OFF_V + (uint32_t)(n % V_STAGES) * V_BYTES; };
    auto gb_slot = [&](int n) { return reinterpret_cast<float*>(sm + OFF_GB + (uint32_t)(n % GB_SLOTS) * GB_SLOT_BYTES); };
    const uint32_t max_polls = p.max_polls;
    auto WAIT = [&](int b, uint32_t parity) { return mbar_wait(&bars[b], parity, abort_flag, max_polls); };
    // warp-uniform wait (every lane polls; the warp proceeds only if all saw it)
    auto WAITW = [&](int b, uint32_t parity) { return __all_sync(0xffffffffu, WAIT(b, parity)) != 0; };

    // Roles (16 warps). Each role's register budget is set at the top of its
    // own branch, so that the compiler allocates that role's code within it.
    //   warp 0        TMA producer (K, Q, V tiles; L2 prefetch 3 chunks ahead)
    //   warp 1        chunk-order products M2u, M3a, M3b, M5, M4; owns TMEM
    //   warp 2        look-ahead products M1, M2w
    //   warp 3        g, beta -> cumulative decay and factors per chunk
    //   warps 4-7     prep: A/P and the triangular solve (Bw, Bu)
    //   warps 8-15    state: thread (j, half) holds half of column j of S (fp32);
    //                 the -W^T hand-off one chunk ahead while M5 runs, and the
    //                 bf16 -> fp16 operands two chunks ahead between chunks
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        regs_dec<REGS_ROLES>();
        if (lane == 0) {
            int issued_kq = 0, issued_v = 0;
            for (int n = 0; n < nc && !*abort_flag; ++n) {
                int nl;  // chunk n's index within its piece
                const Piece& P = piece_of(n, nl);
                const int t = (int)(P.t0 + (long long)nl * C), hk = P.hk, h = P.h;
                if (nl + 3 < P.nc) {  // warm L2 for chunk n + 3 of the same piece (its stage is still in use)
                    const int tp = t + 3 * C;
                    tma_prefetch_l2_3d(&mapK, 0, hk, tp); tma_prefetch_l2_3d(&mapK, 64, hk, tp);
                    tma_prefetch_l2_3d(&mapQ, 0, hk, tp); tma_prefetch_l2_3d(&mapQ, 64, hk, tp);
                    tma_prefetch_l2_3d(&mapV, 0, h, tp); tma_prefetch_l2_3d(&mapV, 64, h, tp);
                }
                const int s = n % KQ_STAGES;
                if (n >= KQ_STAGES && !WAIT(B_EMPTY_KQ + s, ((n / KQ_STAGES) - 1) & 1)) break;
                uint8_t* kq = kq_tile(n);
                GDN_TRACE_AT(40, n);
                mbar_arrive_expect_tx(&bars[B_FULL_KQ + s], KQ_BYTES);
                tma_load_3d(kq + 0, &mapK, &bars[B_FULL_KQ + s], 0, hk, t);
                tma_load_3d(kq + 8192, &mapQ, &bars[B_FULL_KQ + s], 0, hk, t);
                tma_load_3d(kq + 16384, &mapK, &bars[B_FULL_KQ + s], 64, hk, t);
                tma_load_3d(kq + 24576, &mapQ, &bars[B_FULL_KQ + s], 64, hk, t);
                issued_kq = n + 1;
                const int vs = n % V_STAGES;
                if (n >= V_STAGES && !WAIT(B_EMPTY_V + vs, ((n / V_STAGES) - 1) & 1)) break;
                uint8_t* vt = v_tile(n);
                mbar_arrive_expect_tx(&bars[B_FULL_V + vs], V_BYTES);
                tma_load_3d(vt + 0, &mapV, &bars[B_FULL_V + vs], 0, h, t);
                tma_load_3d(vt + 8192, &mapV, &bars[B_FULL_V + vs], 64, h, t);
                issued_v = n + 1;
            }
            // never leave with copies in flight: wait for the last loads of each
            // ring (they land whether or not anyone consumed them; no abort check)
            for (int n = issued_kq - 1; n >= 0 && n >= issued_kq - KQ_STAGES; --n)
                mbar_wait(&bars[B_FULL_KQ + n % KQ_STAGES], (n / KQ_STAGES) & 1, nullptr, 10000u);
            for (int n = issued_v - 1; n >= 0 && n >= issued_v - V_STAGES; --n)
                mbar_wait(&bars[B_FULL_V + n % V_STAGES], (n / V_STAGES) & 1, nullptr, 10000u);
        }
    } else if (warp == 1) {
        // -------------------------------------------- state-dependent products
        regs_dec<REGS_ROLES>();
        if (lane == 0) {
            const uint32_t id_n64_mn = idesc_f16(128, 64, false, true);
            const uint32_t id_n64_k = idesc_f16(128, 64, false, false);
            const uint32_t id_n128_mn = idesc_f16(128, 128, false, true);
            const uint32_t id_wu = idesc_f16(128, 64, true, false);
            const uint32_t wt = smem_u32(sm + OFF_WT);
            for (int n = 0; n < nc; ++n) {
                // M2u: U^T = V^T Bu^T into the Delta accumulator. Issued here, in
                // program order after M5(n-1) (so Delta(n-1) has been read out)
                // and before M3a(n), which accumulates onto it; needs T of chunk
                // n (BWU) and the fp16 V (CONV).
                if (!WAIT(B_CONV0 + (n & 1), (n >> 1) & 1) || !WAIT(B_VCONV0 + (n & 1), (n >> 1) & 1) ||
                    !WAIT(B_BWU0 + (n & 1), (n >> 1) & 1))
                    break;
                tc_fence_after();
                {
                    const uint32_t vt = smem_u32(v_tile(n));
                    const uint32_t bu = smem_u32(sm + OFF_BU + (uint32_t)(n & 1) * 8192);
#pragma unroll 1
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tmem + T_DU, sdesc_sw128(vt + kk * 2048, 8192, 1024),
                                 sdesc_sw128(bu + kk * 32, 16, 1024), id_wu, kk > 0 ? 1u : 0u);
                    mma_commit(&bars[B_M2U0 + (n & 1)]);
                    mma_commit(&bars[B_EMPTY_V + n % V_STAGES]);
                }
                if (!WAIT(B_WREADY, n & 1) || !WAIT(B_STREADY, n & 1)) break;
                GDN_TRACE_AT(20, n);
                tc_fence_after();
                // M3a: D^T = U^T + S^T (-W)^T  (accumulates onto U^T written by M2u)
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tmem + T_DU, tmem + T_ST + 8 * kk, sdesc_sw128(wt + kk * 2048, 16384, 1024), id_n64_mn, 1u);
                mma_commit(&bars[B_DREADY]);
                if (n >= 1 && !WAIT(B_OFREE, (n - 1) & 1)) break;
                tc_fence_after();
                // M3b: O^T = S^T (gamma scale Q)^T
                const uint32_t kq = smem_u32(kq_tile(n));
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tmem + T_O, tmem + T_ST + 8 * kk,
                                sdesc_sw128(kq + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), id_n64_k,
                                kk > 0 ? 1u : 0u);
                if (!WAIT(B_DELTA, n & 1)) break;
                GDN_TRACE_AT(21, n);
                tc_fence_after();
                // M5: Sacc = (D^T diag(Gamma_last,.)) K
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ts(tmem + T_SACC, tmem + T_DTD + 8 * kk, sdesc_sw128(kq + kk * 2048, 16384, 1024),
                                id_n128_mn, kk > 0 ? 1u : 0u);
                mma_commit(&bars[B_SREADY]);
                // M4: O^T += D^T P^T
                const uint32_t pt = smem_u32(sm + OFF_P + (uint32_t)(n & 1) * 8192);
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ts(tmem + T_O, tmem + T_DT + 8 * kk, sdesc_sw128(pt + kk * 32, 16, 1024), id_n64_k, 1u);
                mma_commit(&bars[B_OREADY]);
                mma_commit(&bars[B_PFREE0 + (n & 1)]);
                mma_commit(&bars[B_EMPTY_KQ + n % KQ_STAGES]);
            }
            mma_commit(&bars[B_DONE]);
        }
    } else if (warp == 2) {
        // ------------------------------------------------- look-ahead products
        // Issue order M1(0), then per chunk m: M1(m+1), M2w(m). M1(m+1) needs the
        // stage and X released by the prep group of m (A/P done); M2w(m) (-W^T,
        // the W half of M2) needs the prep group of m done (T: BWU), chunk m
        // converted (fp16 K: CONV) and the W region read out for chunk m-1.
        // The state warps wait for M1(c) before converting chunk c; the next
        // phase of that XREADY barrier is M1(c+2), which this order issues after
        // M2w(c), i.e. after conversion c was seen.
        regs_dec<REGS_ROLES>();
        if (lane == 0) {
            const uint32_t id_x = idesc_bf16(128, 64, false, false);  // raw bf16 K, Q
            const uint32_t id_wu = idesc_f16(128, 64, true, false);
            auto issue_m1 = [&](int n) {
                const uint32_t kq = smem_u32(kq_tile(n));
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + T_X, sdesc_sw128(kq + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024), id_x,
                             kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars[B_XREADY0 + (n & 1)]);
            };
            auto issue_m2w = [&](int n) {
                const uint32_t kq = smem_u32(kq_tile(n));
                const uint32_t bw = smem_u32(sm + OFF_BW + (uint32_t)(n & 1) * 8192);
#pragma unroll 1
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_W, sdesc_sw128(kq + kk * 2048, 16384, 1024), sdesc_sw128(bw + kk * 32, 16, 1024),
                             id_wu, kk > 0 ? 1u : 0u);
                mma_commit(&bars[B_M2W0 + (n & 1)]);
            };
            if (nc > 0 && WAIT(B_FULL_KQ, 0)) {
                tc_fence_after();
                GDN_TRACE_AT(30, 0);
                issue_m1(0);
                for (int m = 0; m < nc; ++m) {
                    if (m + 1 < nc) {
                        if (!WAIT(B_FULL_KQ + (m + 1) % KQ_STAGES, ((m + 1) / KQ_STAGES) & 1) ||
                            !WAIT(B_XFREE, m & 1))
                            break;
                        tc_fence_after();
                        GDN_TRACE_AT(30, m + 1);
                        issue_m1(m + 1);
                    }
                    if (!WAIT(B_CONV0 + (m & 1), (m >> 1) & 1) || !WAIT(B_BWU0 + (m & 1), (m >> 1) & 1)) break;
                    if (m >= 1 && !WAIT(B_WREADY, (m - 1) & 1)) break;
                    tc_fence_after();
                    GDN_TRACE_AT(31, m);
                    issue_m2w(m);
                }
            }
            mma_commit(&bars[B_DONE]);
        }
    } else if (warp == 3) {
        // ------------------------------------- g, beta -> decay factors per chunk
        regs_dec<REGS_ROLES>();
        // V of chunk m (bf16 -> fp16 in place, the B operand of M2u) once its
        // TMA load has landed: 1024 16-byte units, 32 per lane
        auto convert_v = [&](int m) -> bool {
            if (!WAITW(B_FULL_V + m % V_STAGES, (m / V_STAGES) & 1)) return false;
            uint4* base = reinterpret_cast<uint4*>(v_tile(m));
#pragma unroll 1
            for (int k = 0; k < 32; k += 4) {
                uint4 u[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) u[i] = base[lane + 32 * (k + i)];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 a = unbf2(u[i].x), b2 = unbf2(u[i].y), c = unbf2(u[i].z), d = unbf2(u[i].w);
                    base[lane + 32 * (k + i)] = make_uint4(h2(a.x, a.y), h2(b2.x, b2.y), h2(c.x, c.y), h2(d.x, d.y));
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_VCONV0 + (m & 1)]);
            return true;
        };
        // chunk n's decay factors, then the V tile of chunk n - 1 (one more
        // chunk of time for its load to land)
        for (int n = 0; n <= nc; ++n) {
          if (n < nc) {
            const int slot = n % GB_SLOTS;
            if (n >= GB_SLOTS && !WAITW(B_GB_EMPTY + slot, ((n / GB_SLOTS) - 1) & 1)) break;
            float* gb = gb_slot(n);
            int nl;
            const Piece& P = piece_of(n, nl);
            const long long t = P.t0 + (long long)nl * C;
            const int L = min(C, P.len - nl * C), h = P.h;
            const int r0 = 2 * lane, r1 = 2 * lane + 1;
            const float g0 = r0 < L ? p.g[(t + r0) * p.h_v + h] : 0.f;
            const float g1 = r1 < L ? p.g[(t + r1) * p.h_v + h] : 0.f;
            const float b0 = r0 < L ? p.beta[(t + r0) * p.h_v + h] : 0.f;
            const float b1 = r1 < L ? p.beta[(t + r1) * p.h_v + h] : 0.f;
            float incl = g0 + g1;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            // cumulative log-decay, kept in log2 units (G2 = G log2 e) for ex2
            const float G0 = (incl - g1) * 1.4426950408889634f, G1 = incl * 1.4426950408889634f;
            const float GL0 = __shfl_sync(0xffffffffu, G0, (L - 1) >> 1);
            const float GL1 = __shfl_sync(0xffffffffu, G1, (L - 1) >> 1);
            const float GL = ((L - 1) & 1) ? GL1 : GL0;
            const float e0 = ex2(G0), e1 = ex2(G1);
            gb[GB_G + r0] = G0; gb[GB_G + r1] = G1;
            gb[GB_GAM + r0] = e0; gb[GB_GAM + r1] = e1;
            gb[GB_BET + r0] = b0; gb[GB_BET + r1] = b1;
            gb[GB_BG + r0] = b0 * e0; gb[GB_BG + r1] = b1 * e1;
            gb[GB_DEC + r0] = r0 < L ? ex2(GL - G0) : 0.f;
            gb[GB_DEC + r1] = r1 < L ? ex2(GL - G1) : 0.f;
            gb[GB_QSC + r0] = r0 < L ? p.scale * e0 : 0.f;
            gb[GB_QSC + r1] = r1 < L ? p.scale * e1 : 0.f;
            if (lane == 0) gb[GB_GC] = ex2(GL);
            __syncwarp();
            // (a failure-path test withholds one arrival: every wait on it runs out)
            if (lane == 0 && n != p.withhold_chunk) mbar_arrive(&bars[B_GB_FULL + slot]);
            if (lane == 0) GDN_TRACE_AT(41, n);
          }
          if (n >= 1 && !convert_v(n - 1)) break;
        }
    } else if (warp < 8) {
        // ----------------------------------------------------------------- prep
        // all chunks in order; the Bw/Bu and P buffers and the per-parity
        // barriers of chunk n are those of index g = n & 1
        regs_inc<REGS_PREP>();
        const int gt = threadIdx.x - 128;  // 0..127 = TMEM lane
        const int wq = gt >> 5;
        const int bar_id = 1;
        uint8_t* As = sm + OFF_AS;
        float* Ad = reinterpret_cast<float*>(sm + OFF_AD);
        uint8_t* Ts = sm + OFF_TS;
        for (int n = 0; n < nc; ++n) {
            const int g = n & 1;
            uint8_t* bw = sm + OFF_BW + (uint32_t)g * 8192;
            uint8_t* bu = sm + OFF_BU + (uint32_t)g * 8192;
            const float* gb = gb_slot(n);
            const uint32_t ph = (uint32_t)(n >> 1) & 1u;  // phase parity of the per-parity barriers
            bool ok = WAITW(B_GB_FULL + n % GB_SLOTS, (n / GB_SLOTS) & 1) && WAITW(B_XREADY0 + g, ph);
            // P and Bw/Bu buffers g were last read by the products of chunk n - 2:
            // M2w(n - 2) was issued before M1(n) by the same thread (XREADY(n)
            // completes after it), M2u(n - 2) before M4(n - 2) (PFREE)
            if (ok && n >= 2) ok = WAITW(B_PFREE0 + g, ph ^ 1u);
            if (named_sync_or(bar_id, 128, !ok)) break;
            if (gt == 0) GDN_TRACE_AT(0, n);
            tc_fence_after();
            int nl;
            const Piece& P = piece_of(n, nl);
            ap_pass(sm, tmem, gb, n, min(C, P.len - nl * C), p.scale, gt, tb_);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_XFREE]);
            if (gt == 0) GDN_TRACE_AT(1, n);
            // ---- diagonal blocks T_bb = (I + A_bb)^{-1} by forward substitution
            //      in fp32, lane c of a half-warp solving column c; written to Ts
            //      (fp16) and, scaled, to the diagonal blocks of Bw and Bu. The
            //      warp of A rows 0-31 solves blocks 0, 1 (its own rows) at once;
            //      the warp of P rows 0-31 solves blocks 2, 3 once the warp of A
            //      rows 32-63 has stored them (barrier 2)
            if (wq == 2) named_sync(2, 64);
            if (wq == 0 || wq == 2) {
                const int b = (wq == 0 ? 0 : 2) + (lane >> 4), c = lane & 15;
                // right-looking: once x_ss is final, subtract its column from the rest
                float xs[16];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) xs[rr] = (rr == c) ? 1.f : 0.f;
                const float4* acol = reinterpret_cast<const float4*>(Ad + b * 256);
#pragma unroll
                for (int ss = 0; ss < 15; ++ss) {
#pragma unroll
                    for (int q4 = (ss + 1) >> 2; q4 < 4; ++q4) {
                        const float4 a4 = acol[ss * 4 + q4];
                        if (4 * q4 + 0 > ss) xs[4 * q4 + 0] = fmaf(-a4.x, xs[ss], xs[4 * q4 + 0]);
                        if (4 * q4 + 1 > ss) xs[4 * q4 + 1] = fmaf(-a4.y, xs[ss], xs[4 * q4 + 1]);
                        if (4 * q4 + 2 > ss) xs[4 * q4 + 2] = fmaf(-a4.z, xs[ss], xs[4 * q4 + 2]);
                        if (4 * q4 + 3 > ss) xs[4 * q4 + 3] = fmaf(-a4.w, xs[ss], xs[4 * q4 + 3]);
                    }
                }
                const int S_ = 16 * b + c;
                const float fw = -gb[GB_BG + S_], fu = gb[GB_BET + S_];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    const uint32_t R = (uint32_t)(16 * b + rr);
                    *reinterpret_cast<__half*>(Ts + b * 512 + rr * 32 + ((((uint32_t)c >> 3) ^ ((uint32_t)rr >> 2)) & 1u) * 16 +
                                               (c & 7) * 2) = __float2half_rn(xs[rr]);
                    const uint32_t off = R * 128u + (((((uint32_t)S_ >> 3) ^ R) & 7u) << 4) + (uint32_t)(S_ & 7) * 2u;
                    *reinterpret_cast<__half*>(bw + off) = __float2half_rn(xs[rr] * fw);
                    *reinterpret_cast<__half*>(bu + off) = __float2half_rn(xs[rr] * fu);
                }
            }
            if (gt == 0) GDN_TRACE_AT(2, n);
            named_sync(bar_id, 128);
            // ---- off-diagonal blocks, block-row i = wq by warp wq (right-looking:
            //      T_ij = -(sum_{k=j+1..i} T_ik A_kj) T_jj), on the warp MMA
            if (wq >= 1) solve_block_row(wq, smem_u32(As), smem_u32(Ts), bw, bu, gb, lane);
            if (lane == 0) GDN_TRACE_AT(56 + wq, n);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_BWU0 + g]);
                mbar_arrive(&bars[B_GB_EMPTY + n % GB_SLOTS]);
            }
            if (gt == 0) GDN_TRACE_AT(4, n);
        }
    } else {
        // ---------------------------------------------------------------- state
        // warps 8-15: thread (j, hf) holds rows 64 hf .. 64 hf + 63 of column j
        // of S in fp32 for the whole sequence; handles chunk rows 32 hf .. + 31
        // of Delta^T and of the output
        regs_inc<REGS_STATE>();
        const int ws = warp - 8, q4 = warp & 3, hf = ws >> 2;
        const int j = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        auto sbase_of = [&](const Piece& P) { return ((size_t)P.n_seq * p.h_v + P.h) * (size_t)(D * D); };
        float S[64];
        // a piece starts from the sequence's initial state at its first token,
        // else from zeros
        auto load_initial = [&](const Piece& P) {
            if (p.h0 && P.from_start) {
                const float* hp = p.h0 + sbase_of(P) + (size_t)(64 * hf) * D + j;
#pragma unroll
                for (int c = 0; c < 64; ++c) S[c] = hp[c * D];
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) S[c] = 0.f;
            }
        };
        // end of a piece: fp16 range check; the final state if the piece ends
        // its sequence. A value beyond the range of the fp16 operands (v, the
        // state or a chunk's errors above 65504) became an infinity in a
        // product and has left a non-finite value in the fp32 state, where it
        // stays (decay keeps infinities, sums keep NaNs)
        auto finish_piece = [&](const Piece& P) {
            bool finite = true;
#pragma unroll
            for (int c = 0; c < 64; ++c) finite = finite && (fabsf(S[c]) < INFINITY);
            if (__any_sync(0xffffffffu, !finite) && lane == 0) set_device_error(4u);
            if (p.hT && P.last_seg) {
                float* hp = p.hT + sbase_of(P) + (size_t)(64 * hf) * D + j;
#pragma unroll
                for (int c = 0; c < 64; ++c) hp[c * D] = S[c];
            }
        };
        load_initial(pieces[0]);
        auto put_state_f16 = [&]() {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) pk[c] = h2(S[32 * q + 2 * c], S[32 * q + 2 * c + 1]);
                tmem_st16(tmem + lane_base + T_ST + 32 * hf + 16 * q, pk);
            }
            tmem_st_wait();
        };
        put_state_f16();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_STREADY]);
        // bf16 -> fp16 operands of chunk m, in place (K as it is and Q times
        // gamma scale once M1(m) has consumed the bf16 K and Q): 2 tiles x
        // 128 row halves of 64 values over the 256 state threads
        const int ts = 32 * ws + lane;
        auto convert = [&](int m) -> bool {
            if (!WAITW(B_GB_FULL + m % GB_SLOTS, (m / GB_SLOTS) & 1) ||
                !WAITW(B_XREADY0 + (m & 1), (m >> 1) & 1))
                return false;
            // 16-byte units u = ts + 256 k, k = 0..7 of the K, Q stage (K kb0 | Q kb0
            // | K kb1 | Q kb1, 512 units each: Q for k = 2, 3, 6, 7; tile row
            // (ts >> 3) + 32 (k & 1)). Four loads before their stores in each
            // group. (V is converted by the g/beta warp.)
            const float* qsc = gb_slot(m) + GB_QSC;
            const float q0 = qsc[ts >> 3], q1 = qsc[(ts >> 3) + 32];
#pragma unroll 1
            for (int i = 0; i < 2; ++i) {
                uint4* base = reinterpret_cast<uint4*>(kq_tile(m)) + 1024 * i;
                uint4 u[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) u[j] = base[ts + 256 * j];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint4 w = u[j];
                    if (j >= 2) {  // Q times gamma scale
                        const float f = j == 2 ? q0 : q1;
                        const float2 a = unbf2(w.x), b2 = unbf2(w.y), c = unbf2(w.z), d = unbf2(w.w);
                        w.x = h2(a.x * f, a.y * f); w.y = h2(b2.x * f, b2.y * f);
                        w.z = h2(c.x * f, c.y * f); w.w = h2(d.x * f, d.y * f);
                    } else {
                        const float2 a = unbf2(w.x), b2 = unbf2(w.y), c = unbf2(w.z), d = unbf2(w.w);
                        w.x = h2(a.x, a.y); w.y = h2(b2.x, b2.y); w.z = h2(c.x, c.y); w.w = h2(d.x, d.y);
                    }
                    base[ts + 256 * j] = w;
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_CONV0 + (m & 1)]);
            return true;
        };
        // -W^T of chunk m from TMEM (lane = key index i = j, columns = chunk
        // rows r; this thread: rows 32 hf .. + 31) into the MN-major fp16 B
        // tile of M3a, once M2w(m) has run; M3a(m - 1) has finished reading
        // the tile (DREADY(m - 1) was seen before every call)
        auto handoff_w = [&](int m) -> bool {
            if (!WAITW(B_M2W0 + (m & 1), (m >> 1) & 1)) return false;
            tc_fence_after();
            {
                uint32_t w[32];
                tmem_ld32(tmem + lane_base + T_W + 32 * hf, w);
                tmem_ld_wait();
                store_half_row_sw128(sm + OFF_WT, (uint32_t)j, reinterpret_cast<const float*>(w), hf);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_WREADY]);
            if (ws == 0 && lane == 0) GDN_TRACE_AT(13, m);
            return true;
        };
        TOut* o = static_cast<TOut*>(p.o);
        // conversions run two chunks ahead of the state: chunk n + 2 after the
        // output of chunk n (iterations n = -2, -1 only convert chunks 0, 1);
        // one call site keeps a single copy of the conversion code
        for (int n = -2; n < nc; ++n) {
            if (n >= 0) {
                if (!WAITW(B_GB_FULL + n % GB_SLOTS, (n / GB_SLOTS) & 1)) break;
                const float* gb = gb_slot(n);
                // Delta^T (fp32, TMEM) -> fp16 A operands: as is (for M4) and scaled
                // by Gamma_last,r (for M5); one TMEM load (a TMEM round trip costs
                // about 200 cycles while the tensor core is busy)
                if (!WAITW(B_DREADY, n & 1)) break;
                if (ws == 0 && lane == 0) GDN_TRACE_AT(10, n);
                tc_fence_after();
                {
                    // both halves loaded before the single wait
                    uint32_t dr0[16], dr1[16];
                    tmem_ld16(tmem + lane_base + T_DU + 32 * hf, dr0);
                    tmem_ld16(tmem + lane_base + T_DU + 32 * hf + 16, dr1);
                    tmem_ld_wait();
                    const float4* dec4 = reinterpret_cast<const float4*>(gb + GB_DEC + 32 * hf);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t* dr = hh ? dr1 : dr0;
                        uint32_t pk[8], pd[8];
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const float4 d4 = dec4[4 * hh + c4];
                            const float a0 = __uint_as_float(dr[4 * c4]), a1 = __uint_as_float(dr[4 * c4 + 1]);
                            const float a2 = __uint_as_float(dr[4 * c4 + 2]), a3 = __uint_as_float(dr[4 * c4 + 3]);
                            pk[2 * c4] = h2(a0, a1); pk[2 * c4 + 1] = h2(a2, a3);
                            pd[2 * c4] = h2(a0 * d4.x, a1 * d4.y); pd[2 * c4 + 1] = h2(a2 * d4.z, a3 * d4.w);
                        }
                        tmem_st8(tmem + lane_base + T_DTD + 16 * hf + 8 * hh, pd);
                        tmem_st8(tmem + lane_base + T_DT + 16 * hf + 8 * hh, pk);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_DELTA]);
            }
            // -W^T of chunk n + 1: handed over now, while M5(n) runs, if M2w(n + 1)
            // has already finished; otherwise after this chunk's state update
            // and output, so that a late prep does not hold those back
            bool w_pending = n + 1 >= 0 && n + 1 < nc;
            if (w_pending &&
                (n < 0 || __all_sync(0xffffffffu, mbar_test(&bars[B_M2W0 + ((n + 1) & 1)], ((n + 1) >> 1) & 1)))) {
                if (!handoff_w(n + 1)) break;
                w_pending = false;
            }
            if (n >= 0) {
                const float* gb = gb_slot(n);
                // state update S^T <- gamma_last S^T + Delta^T Kdec
                const float gC = gb[GB_GC];
                if (!WAITW(B_SREADY, n & 1)) break;
                if (ws == 0 && lane == 0) GDN_TRACE_AT(11, n);
                tc_fence_after();
                {
                    uint32_t acc0[32], acc1[32];
                    tmem_ld32(tmem + lane_base + T_SACC + 64 * hf, acc0);
                    tmem_ld32(tmem + lane_base + T_SACC + 64 * hf + 32, acc1);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 32; ++c) S[c] = fmaf(gC, S[c], __uint_as_float(acc0[c]));
#pragma unroll
                    for (int c = 0; c < 32; ++c) S[32 + c] = fmaf(gC, S[32 + c], __uint_as_float(acc1[c]));
                }
                if (npieces > 1 && n == nc0 - 1) {  // the first piece ends: the second one's initial state
                    finish_piece(pieces[0]);
                    load_initial(pieces[1]);
                }
                put_state_f16();
                tc_fence_before();
                __syncwarp();
                if (ws == 0 && lane == 0) GDN_TRACE_AT(12, n);
                if (lane == 0) {
                    mbar_arrive(&bars[B_STREADY]);
                    mbar_arrive(&bars[B_GB_EMPTY + n % GB_SLOTS]);
                }
                // output rows 32 hf .. 32 hf + 31 of this chunk
                if (!WAITW(B_OREADY, n & 1)) break;
                tc_fence_after();
                {
                    // o[t0 + nl C + r][h][j] for r < nv: one row per register, through a
                    // byte pointer stepped by the token stride
                    int nl;
                    const Piece& P = piece_of(n, nl);
                    const int nv = min(C, P.len - nl * C) - 32 * hf;  // valid rows of this half
                    // rows before token seg_a belong to the piece's prefix: not stored
                    const long long r0 = P.t0 + (long long)nl * C + 32 * hf;
                    const int nskip = P.seg_a > r0 ? (int)min(32LL, P.seg_a - r0) : 0;
                    char* orow = reinterpret_cast<char*>(o + ((size_t)r0 * p.h_v + P.h) * D + j);
                    const size_t ostep = (size_t)p.h_v * D * sizeof(TOut);
                    uint32_t ov[32];
                    tmem_ld32(tmem + lane_base + T_O + 32 * hf, ov);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars[B_OFREE]);
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        if (c < nv && c >= nskip) *reinterpret_cast<TOut*>(orow) = from_f32<TOut>(__uint_as_float(ov[c]));
                        orow += ostep;
                    }
                }
            }
            if (w_pending && !handoff_w(n + 1)) break;
            if (n + 2 < nc && !convert(n + 2)) break;
            if (n >= 0 && ws == 0 && lane == 0) GDN_TRACE_AT(14, n);
        }
        if (!*abort_flag) finish_piece(pieces[npieces - 1]);
    }

    // ---- teardown (also after an abort): the producer has drained its TMA
    //      loads; B_DONE completes when every MMA of both issuers is done;
    //      only then is TMEM freed
    __syncthreads();
    if (warp == 1) {
        mbar_wait(&bars[B_DONE], 0, nullptr, 10000u);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) set_device_error(2u);
    if (threadIdx.x == 0) GDN_TRACE_CTA(63);
}

}  // namespace tck

// ------------------------------------------------------------------ host side
// The driver's tensor-map encoder, looked up once (a function-local static
// initialised by a lambda: C++ makes the first initialisation thread-safe).
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

// The kernel is compiled for sm_103a only; it runs on compute capability 10.x.
inline bool tc_available() {
    int dev = 0, major = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
    return major == 10 && tensor_map_encoder() != nullptr;
}

// 3-D view [tokens][heads][128] of a bf16 tensor; box = 64 tokens x 1 head x 64
// elements (128 B rows, 128-byte swizzle).
inline bool make_head_map(CUtensorMap* m, const void* base, long long tokens, int heads) {
    cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)tokens};
    cuuint64_t strides[2] = {128 * 2, (cuuint64_t)heads * 128 * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    return tensor_map_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                                es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline gdn_status launch_tc(const TcArgs& a, bool out_bf16, cudaStream_t s) {
    CUtensorMap mq, mk, mv;
    if (!make_head_map(&mq, a.q, a.total, a.h_qk) || !make_head_map(&mk, a.k, a.total, a.h_qk) ||
        !make_head_map(&mv, a.v, a.total, a.h_v))
        return GDN_ERR_CUDA;
    const long long ctot = (long long)a.num_seqs * a.h_qk * ((a.eq_len + tck::C - 1) / tck::C);  // group chunks
    const long long blocks = a.bal_chunks > 0 ? (ctot + a.bal_chunks - 1) / a.bal_chunks * a.grp
                                              : (long long)a.num_seqs * a.h_v * a.nseg;
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    if (out_bf16) {
        auto kern = tck::chunk_tc_kernel<__nv_bfloat16>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tck::SMEM_BYTES) != cudaSuccess)
            return GDN_ERR_CUDA;
        kern<<<(unsigned)blocks, tck::NTHREADS, tck::SMEM_BYTES, s>>>(mq, mk, mv, a);
    } else {
        auto kern = tck::chunk_tc_kernel<float>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tck::SMEM_BYTES) != cudaSuccess)
            return GDN_ERR_CUDA;
        kern<<<(unsigned)blocks, tck::NTHREADS, tck::SMEM_BYTES, s>>>(mq, mk, mv, a);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace gdn
