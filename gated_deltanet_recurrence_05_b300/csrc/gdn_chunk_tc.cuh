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
//   W^T    = K^T Bw^T,  Bw = T diag(beta gamma)          (M2, 128x64x64)
//   U^T    = V^T Bu^T,  Bu = T diag(beta)                (M2, 128x64x64)
//   D^T    = U^T + S^T (-W)^T                            (M3a, 128x64x128)
//   O^T    = S^T (gamma scale Q)^T + D^T P^T             (M3b + M4)
//   Sacc   = D^T Kdec,  Kdec = diag(Gamma_last,.) K      (M5, 128x128x64)
//   S^T   <- gamma_last S^T + Sacc                       (fp32, registers)
// where D^T = Delta^T. Thread j of the state warps owns column j of S (TMEM
// lane j): its fp32 state lives in registers for the whole sequence; an fp16
// copy of S^T and of Delta^T is written to TMEM and read there as the A
// operand of the next products. Only exponentials of G_r - G_s with r >= s are
// formed, so no factor exceeds 1 for g <= 0.
//
// Operand precision: every product after X takes fp16 operands (10-bit
// mantissa) with fp32 accumulation; the bf16 inputs K, Q, V convert to fp16
// exactly (their magnitudes are far inside the fp16 range), so only the
// computed operands (S, Delta, T, W, P and the decay-scaled Q and K) are
// rounded, at 2^-11 instead of bf16's 2^-8. Decay-scaled values that fall
// below the fp16 range contribute less than 1e-7 of the largest terms. The
// path therefore assumes |v| and |S| stay well below 6e4 (the fp16 range).
//
// Warp roles (512 threads):
//   warp 0      TMA producer: K, Q (3-deep ring) and V (2-deep ring) tiles
//   warp 1      issues the state-dependent products M3a, M3b, M5, M4; owns TMEM
//   warp 2      issues the look-ahead products M1 (next chunk) and M2
//   warp 3      loads g, beta of upcoming chunks; cumulative decay and factors
//   warps 4-7   prep: A and P from X, T by blocked forward substitution, Bw/Bu,
//               -W^T, gamma scaling of Q, Kdec
//   warps 8-15  state: Delta^T and S^T hand-off, fp32 state update, output
// All waits are bounded (a timeout raises an abort flag, records
// GDN_DEVERR_TIMEOUT and every role unwinds); TMEM is always freed.
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
};

namespace tck {
constexpr int C = 64, D = 128;
constexpr int KQ_STAGES = 3, V_STAGES = 2, GB_SLOTS = 4;
constexpr int NTHREADS = 512;
// TMEM columns
constexpr uint32_t T_SACC = 0, T_DU = 128, T_O = 192, T_X = 256, T_W = 320, T_ST = 384, T_DT = 448;
constexpr uint32_t TMEM_COLS = 512;
// shared memory layout (byte offsets from a 1024-aligned base)
constexpr uint32_t KQ_BYTES = 32768;  // K kb0 | Q kb0 | K kb1 | Q kb1, 8 KB each (64 rows x 128 B)
constexpr uint32_t V_BYTES = 16384;   // V kb0 | V kb1
constexpr uint32_t OFF_KQ = 0;
constexpr uint32_t OFF_V = OFF_KQ + KQ_STAGES * KQ_BYTES;
constexpr uint32_t OFF_WT = OFF_V + V_STAGES * V_BYTES;  // -W^T, MN-major B: 128 rows (i) x 128 B (r)
constexpr uint32_t OFF_BW = OFF_WT + 16384;              // Bw, K-major B: 64 rows (r) x 128 B (s)
constexpr uint32_t OFF_BU = OFF_BW + 8192;
constexpr uint32_t OFF_P = OFF_BU + 8192;                // P x 2 buffers, K-major B
constexpr uint32_t LDA = 68;                             // fp32 row stride of A and T
constexpr uint32_t OFF_A = OFF_P + 16384;
constexpr uint32_t OFF_T = OFF_A + 64 * LDA * 4;
constexpr uint32_t OFF_GB = OFF_T + 64 * LDA * 4;
constexpr uint32_t GB_FLOATS = 6 * 64 + 4;               // G, gam, bet, bg, dec, qsc, gC
constexpr uint32_t GB_SLOT_BYTES = GB_FLOATS * 4;
constexpr uint32_t OFF_BAR = OFF_GB + GB_SLOTS * GB_SLOT_BYTES;
constexpr uint32_t NUM_BARS = 32;
constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;    // + alignment slack
static_assert(OFF_WT % 1024 == 0 && OFF_BW % 1024 == 0 && OFF_P % 1024 == 0, "tile alignment");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// barrier indices
enum {
    B_FULL_KQ = 0, B_EMPTY_KQ = 3, B_FULL_V = 6, B_EMPTY_V = 8, B_GB_FULL = 10, B_GB_EMPTY = 14,
    B_XREADY = 18, B_XFREE, B_BWU, B_M2DONE, B_WREADY, B_DREADY, B_DELTA, B_SREADY, B_STREADY,
    B_OREADY, B_OFREE, B_PFREE0, B_PFREE1, B_DONE
};
static_assert(B_DONE < (int)NUM_BARS, "barrier count");

// gb slot fields (float offsets)
constexpr int GB_G = 0, GB_GAM = 64, GB_BET = 128, GB_BG = 192, GB_DEC = 256, GB_QSC = 320, GB_GC = 384;

__device__ __forceinline__ uint32_t h2(float lo, float hi) { return tc::pack_f16x2(lo, hi); }
__device__ __forceinline__ float2 unbf2(uint32_t u) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(v);
}
__device__ __forceinline__ float2 unh2(uint32_t u) {
    __half2 v = *reinterpret_cast<__half2*>(&u);
    return __half22float2(v);
}
// One 128-byte tile row (64 values): bf16 in, fp16 out, times f, in place.
// Rows r..r+7 handled by neighbouring threads start at different 16-byte
// chunks (c ^ r), so a warp's accesses spread over all banks.
__device__ __forceinline__ void bf16_row_to_f16(uint8_t* row, uint32_t r, float f) {
    uint4* p = reinterpret_cast<uint4*>(row);
#pragma unroll
    for (int c0 = 0; c0 < 8; ++c0) {
        const uint32_t c = ((uint32_t)c0 ^ r) & 7u;
        uint4 u = p[c];
        float2 a = unbf2(u.x), b = unbf2(u.y), d = unbf2(u.z), e = unbf2(u.w);
        u.x = h2(a.x * f, a.y * f); u.y = h2(b.x * f, b.y * f);
        u.z = h2(d.x * f, d.y * f); u.w = h2(e.x * f, e.y * f);
        p[c] = u;
    }
}
// Chunks [c_lo, c_lo + n) (in swizzled visiting order) of one 128-byte row of
// fp16 values, times f, in place.
__device__ __forceinline__ void f16_row_scale(uint8_t* row, uint32_t r, float f, int c_lo, int n) {
    uint4* p = reinterpret_cast<uint4*>(row);
#pragma unroll
    for (int c0 = 0; c0 < 8; ++c0) {
        if (c0 < c_lo || c0 >= c_lo + n) continue;
        const uint32_t c = ((uint32_t)c0 ^ r) & 7u;
        uint4 u = p[c];
        float2 a = unh2(u.x), b = unh2(u.y), d = unh2(u.z), e = unh2(u.w);
        u.x = h2(a.x * f, a.y * f); u.y = h2(b.x * f, b.y * f);
        u.z = h2(d.x * f, d.y * f); u.w = h2(e.x * f, e.y * f);
        p[c] = u;
    }
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
        if (blockIdx.x == 0 && g_trace && (n) < 128) g_trace[(point) * 128 + (n)] = clock64(); \
    } while (0)
#else
#define GDN_TRACE_AT(point, n) \
    do {                       \
    } while (0)
#endif
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
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

template <typename TOut>
__global__ void __launch_bounds__(NTHREADS, 1)
chunk_tc_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV, TcArgs p) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + OFF_MISC);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + OFF_MISC + 4);

    // ---- unit of work: (sequence, value head)
    const int h = blockIdx.x % p.h_v;
    const int pos = blockIdx.x / p.h_v;
    int n_seq;
    if (!seq_of(p.order, pos, p.num_seqs, n_seq)) return;
    long long t0, t1;
    if (!seq_bounds(p.cu, n_seq, p.num_seqs, p.total, p.eq_len, t0, t1)) return;
    const int len = (int)(t1 - t0);
    const int nc = (len + C - 1) / C;
    const int hk = h / p.grp;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < KQ_STAGES; ++i) { mbar_init(&bars[B_FULL_KQ + i], 1); mbar_init(&bars[B_EMPTY_KQ + i], 1); }
        for (int i = 0; i < V_STAGES; ++i) { mbar_init(&bars[B_FULL_V + i], 1); mbar_init(&bars[B_EMPTY_V + i], 1); }
        for (int i = 0; i < GB_SLOTS; ++i) { mbar_init(&bars[B_GB_FULL + i], 1); mbar_init(&bars[B_GB_EMPTY + i], 12); }
        mbar_init(&bars[B_XREADY], 1); mbar_init(&bars[B_XFREE], 4); mbar_init(&bars[B_BWU], 4);
        mbar_init(&bars[B_M2DONE], 1); mbar_init(&bars[B_WREADY], 8); mbar_init(&bars[B_DREADY], 1);
        mbar_init(&bars[B_DELTA], 8); mbar_init(&bars[B_SREADY], 1); mbar_init(&bars[B_STREADY], 8);
        mbar_init(&bars[B_OREADY], 1); mbar_init(&bars[B_OFREE], 8); mbar_init(&bars[B_PFREE0], 1);
        mbar_init(&bars[B_PFREE1], 1); mbar_init(&bars[B_DONE], 2);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mapQ); tma_prefetch_desc(&mapK); tma_prefetch_desc(&mapV);
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto kq_tile = [&](int n) { return sm + OFF_KQ + (uint32_t)(n % KQ_STAGES) * KQ_BYTES; };
    auto v_tile = [&](int n) { return sm + OFF_V + (uint32_t)(n % V_STAGES) * V_BYTES; };
    auto gb_slot = [&](int n) { return reinterpret_cast<float*>(sm + OFF_GB + (uint32_t)(n % GB_SLOTS) * GB_SLOT_BYTES); };
    auto WAIT = [&](int b, uint32_t parity) { return mbar_wait(&bars[b], parity, abort_flag); };
    // warp-uniform wait (every lane polls; the warp proceeds only if all saw it)
    auto WAITW = [&](int b, uint32_t parity) { return __all_sync(0xffffffffu, WAIT(b, parity)) != 0; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued_kq = 0, issued_v = 0;
            for (int n = 0; n < nc && !*abort_flag; ++n) {
                const int t = (int)(t0 + (long long)n * C);
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
                mbar_wait(&bars[B_FULL_KQ + n % KQ_STAGES], (n / KQ_STAGES) & 1, nullptr, 200000000ull);
            for (int n = issued_v - 1; n >= 0 && n >= issued_v - V_STAGES; --n)
                mbar_wait(&bars[B_FULL_V + n % V_STAGES], (n / V_STAGES) & 1, nullptr, 200000000ull);
        }
    } else if (warp == 1) {
        // -------------------------------------------- state-dependent products
        if (lane == 0) {
            const uint32_t id_n64_mn = idesc_f16(128, 64, false, true);
            const uint32_t id_n64_k = idesc_f16(128, 64, false, false);
            const uint32_t id_n128_mn = idesc_f16(128, 128, false, true);
            const uint32_t wt = smem_u32(sm + OFF_WT);
            for (int n = 0; n < nc; ++n) {
                if (!WAIT(B_WREADY, n & 1) || !WAIT(B_STREADY, n & 1)) break;
                GDN_TRACE_AT(20, n);
                tc_fence_after();
                // M3a: D^T = U^T + S^T (-W)^T  (accumulates onto U^T written by M2)
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tmem + T_DU, tmem + T_ST + 8 * kk, sdesc_sw128(wt + kk * 2048, 16384, 1024), id_n64_mn, 1u);
                mma_commit(&bars[B_DREADY]);
                if (n >= 1 && !WAIT(B_OFREE, (n - 1) & 1)) break;
                tc_fence_after();
                // M3b: O^T = S^T (gamma scale Q)^T
                const uint32_t kq = smem_u32(kq_tile(n));
                for (int kk = 0; kk < 8; ++kk)
                    mma_bf16_ts(tmem + T_O, tmem + T_ST + 8 * kk,
                                sdesc_sw128(kq + 8192 + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024), id_n64_k,
                                kk > 0 ? 1u : 0u);
                if (!WAIT(B_DELTA, n & 1)) break;
                GDN_TRACE_AT(21, n);
                tc_fence_after();
                // M5: Sacc = D^T Kdec
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16_ts(tmem + T_SACC, tmem + T_DT + 8 * kk, sdesc_sw128(kq + kk * 2048, 16384, 1024),
                                id_n128_mn, kk > 0 ? 1u : 0u);
                mma_commit(&bars[B_SREADY]);
                // M4: O^T += D^T P^T
                const uint32_t pt = smem_u32(sm + OFF_P + (uint32_t)(n & 1) * 8192);
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
        if (lane == 0) {
            const uint32_t id_x = idesc_bf16(128, 64, false, false);  // raw bf16 K, Q
            const uint32_t id_wu = idesc_f16(128, 64, true, false);
            auto issue_m1 = [&](int n) {
                const uint32_t kq = smem_u32(kq_tile(n));
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + T_X, sdesc_sw128(kq + off, 16, 1024), sdesc_sw128(kq + off, 16, 1024), id_x,
                             kk > 0 ? 1u : 0u);
                }
                mma_commit(&bars[B_XREADY]);
            };
            auto issue_m2 = [&](int n) {
                const uint32_t kq = smem_u32(kq_tile(n)), vt = smem_u32(v_tile(n));
                const uint32_t bw = smem_u32(sm + OFF_BW), bu = smem_u32(sm + OFF_BU);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_W, sdesc_sw128(kq + kk * 2048, 16384, 1024), sdesc_sw128(bw + kk * 32, 16, 1024),
                             id_wu, kk > 0 ? 1u : 0u);
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(tmem + T_DU, sdesc_sw128(vt + kk * 2048, 8192, 1024), sdesc_sw128(bu + kk * 32, 16, 1024),
                             id_wu, kk > 0 ? 1u : 0u);
                mma_commit(&bars[B_M2DONE]);
                mma_commit(&bars[B_EMPTY_V + n % V_STAGES]);
            };
            // Issue whichever product is ready: M1(m1) once X of chunk m1-1 is
            // consumed and the stage has landed; M2(m2) once T of chunk m2 is
            // ready and the state warps released the U and W regions of chunk
            // m2-1. Polls back off with nanosleep so that this thread does not
            // take issue slots from the warps sharing its scheduler.
            if (nc > 0 && WAIT(B_FULL_KQ, 0)) {
                tc_fence_after();
                GDN_TRACE_AT(30, 0);
                issue_m1(0);
                int m1 = 1, m2 = 0;
                uint64_t t_last = globaltimer_ns();
                while (m2 < nc && !*abort_flag) {
                    bool progress = false;
                    if (m1 < nc && m1 <= m2 + 1 && mbar_test(&bars[B_FULL_KQ + m1 % KQ_STAGES], (m1 / KQ_STAGES) & 1) &&
                        mbar_test(&bars[B_XFREE], (m1 - 1) & 1)) {
                        tc_fence_after();
                        GDN_TRACE_AT(30, m1);
                        issue_m1(m1++);
                        progress = true;
                    }
                    if (mbar_test(&bars[B_BWU], m2 & 1) && mbar_test(&bars[B_FULL_V + m2 % V_STAGES], (m2 / V_STAGES) & 1) &&
                        (m2 == 0 || (mbar_test(&bars[B_WREADY], (m2 - 1) & 1) && mbar_test(&bars[B_DELTA], (m2 - 1) & 1)))) {
                        tc_fence_after();
                        GDN_TRACE_AT(31, m2);
                        issue_m2(m2++);
                        progress = true;
                    }
                    if (progress) {
                        t_last = globaltimer_ns();
                    } else {
                        __nanosleep(40);
                        if (globaltimer_ns() - t_last > 2000000000ull) *abort_flag = 1;
                    }
                }
            }
            mma_commit(&bars[B_DONE]);
        }
    } else if (warp == 3) {
        // ------------------------------------- g, beta -> decay factors per chunk
        for (int n = 0; n < nc; ++n) {
            const int slot = n % GB_SLOTS;
            if (n >= GB_SLOTS && !WAITW(B_GB_EMPTY + slot, ((n / GB_SLOTS) - 1) & 1)) break;
            float* gb = gb_slot(n);
            const long long t = t0 + (long long)n * C;
            const int L = min(C, len - n * C);
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
            if (lane == 0) mbar_arrive(&bars[B_GB_FULL + slot]);
            if (lane == 0) GDN_TRACE_AT(41, n);
        }
    } else if (warp < 8) {
        // ----------------------------------------------------------------- prep
        const int pt = threadIdx.x - 128;  // 0..127 = TMEM lane
        const int wq = warp - 4;           // lane quadrant
        float* Am = reinterpret_cast<float*>(sm + OFF_A);
        float* Tm = reinterpret_cast<float*>(sm + OFF_T);
        const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
        for (int n = 0; n < nc; ++n) {
            const float* gb = gb_slot(n);
            // the stage's TMA completion is observed here too: the prep threads
            // rescale Q and K in place with ordinary loads and stores
            bool ok = WAITW(B_GB_FULL + n % GB_SLOTS, (n / GB_SLOTS) & 1) &&
                      WAITW(B_FULL_KQ + n % KQ_STAGES, (n / KQ_STAGES) & 1) &&
                      WAITW(B_FULL_V + n % V_STAGES, (n / V_STAGES) & 1) && WAITW(B_XREADY, n & 1);
            if (ok && wq >= 2 && n >= 2) ok = WAITW(B_PFREE0 + (n & 1), ((n >> 1) - 1) & 1);
            if (named_sync_or(1, 128, !ok)) break;
            if (pt == 0) GDN_TRACE_AT(0, n);
            tc_fence_after();
            {
                uint32_t x[64];
                tmem_ld32(tmem + lane_base + T_X, *reinterpret_cast<uint32_t(*)[32]>(x));
                tmem_ld32(tmem + lane_base + T_X + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
                tmem_ld_wait();
                if (wq < 2) {  // rows of K K^T -> A (fp32)
                    const int r = pt;
                    const float Gr = gb[GB_G + r], br = gb[GB_BET + r];
                    float* arow = Am + r * LDA;
#pragma unroll
                    for (int s4 = 0; s4 < 64; s4 += 4) {
                        float4 a;
                        a.x = (s4 + 0 < r) ? br * ex2(Gr - gb[GB_G + s4 + 0]) * __uint_as_float(x[s4 + 0]) : 0.f;
                        a.y = (s4 + 1 < r) ? br * ex2(Gr - gb[GB_G + s4 + 1]) * __uint_as_float(x[s4 + 1]) : 0.f;
                        a.z = (s4 + 2 < r) ? br * ex2(Gr - gb[GB_G + s4 + 2]) * __uint_as_float(x[s4 + 2]) : 0.f;
                        a.w = (s4 + 3 < r) ? br * ex2(Gr - gb[GB_G + s4 + 3]) * __uint_as_float(x[s4 + 3]) : 0.f;
                        *reinterpret_cast<float4*>(arow + s4) = a;
                    }
                } else {  // rows of Q K^T -> P (bf16, decayed, causal, scaled)
                    const int r = pt - 64;
                    const float Gr = gb[GB_G + r];
                    const bool live = r < min(C, len - n * C);
                    float pv[64];
#pragma unroll
                    for (int s = 0; s < 64; ++s)
                        pv[s] = (live && s <= r) ? p.scale * ex2(Gr - gb[GB_G + s]) * __uint_as_float(x[s]) : 0.f;
                    store_row_sw128(sm + OFF_P + (uint32_t)(n & 1) * 8192, (uint32_t)r, pv);
                    fence_async_smem();
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_XFREE]);
            // ---- fp16 operands: K, V as they are, Q times gamma scale (M1 has
            //      consumed the bf16 K and Q of this chunk)
            {
                const int r = pt & 63, kb = pt >> 6;
                uint8_t* kq = kq_tile(n) + (uint32_t)kb * 16384 + (uint32_t)r * 128;
                bf16_row_to_f16(kq, r, 1.f);
                bf16_row_to_f16(kq + 8192, r, gb[GB_QSC + r]);
                bf16_row_to_f16(v_tile(n) + (uint32_t)kb * 8192 + (uint32_t)r * 128, r, 1.f);
            }
            if (pt == 0) GDN_TRACE_AT(1, n);
            named_sync(1, 128);
            // ---- T = (I + A)^{-1}: 16x16 diagonal blocks by substitution, then
            //      off-diagonal blocks level by level: T_ij = -T_ii sum_k A_ik T_kj
            if (pt < 64) {
                const int b = pt >> 4, c = pt & 15;
                float xs[16];
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) {
                    float acc = (rr == c) ? 1.f : 0.f;
                    const float* arow = Am + (16 * b + rr) * LDA + 16 * b;
#pragma unroll
                    for (int ss = 0; ss < rr; ++ss) acc = fmaf(-arow[ss], xs[ss], acc);
                    xs[rr] = acc;
                }
#pragma unroll
                for (int rr = 0; rr < 16; ++rr) Tm[(16 * b + rr) * LDA + 16 * b + c] = xs[rr];
            }
            named_sync(1, 128);
#pragma unroll
            for (int d = 1; d < 4; ++d) {
                const int nb = 4 - d;
                float y[6];
#pragma unroll
                for (int t = 0; t < 6; ++t) {
                    y[t] = 0.f;
                    if (t < 2 * nb) {
                        const int e = pt + 128 * t, j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
                        float acc = 0.f;
                        for (int kb = j; kb < i; ++kb) {
                            const float* arow = Am + (16 * i + r) * LDA + 16 * kb;
                            const float* tcol = Tm + (16 * kb) * LDA + 16 * j + c;
#pragma unroll
                            for (int m = 0; m < 16; ++m) acc = fmaf(arow[m], tcol[m * LDA], acc);
                        }
                        y[t] = acc;
                    }
                }
                named_sync(1, 128);
#pragma unroll
                for (int t = 0; t < 6; ++t)
                    if (t < 2 * nb) {
                        const int e = pt + 128 * t, j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
                        Tm[(16 * i + r) * LDA + 16 * j + c] = y[t];
                    }
                named_sync(1, 128);
#pragma unroll
                for (int t = 0; t < 6; ++t)
                    if (t < 2 * nb) {
                        const int e = pt + 128 * t, j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
                        const float* trow = Tm + (16 * i + r) * LDA + 16 * i;
                        const float* ycol = Tm + (16 * i) * LDA + 16 * j + c;
                        float acc = 0.f;
#pragma unroll
                        for (int m = 0; m < 16; ++m) acc = fmaf(trow[m], ycol[m * LDA], acc);
                        y[t] = -acc;
                    }
                named_sync(1, 128);
#pragma unroll
                for (int t = 0; t < 6; ++t)
                    if (t < 2 * nb) {
                        const int e = pt + 128 * t, j = e >> 8, r = (e >> 4) & 15, c = e & 15, i = j + d;
                        Tm[(16 * i + r) * LDA + 16 * j + c] = y[t];
                    }
                named_sync(1, 128);
            }
            if (pt == 0) GDN_TRACE_AT(5, n);
            // ---- Bw = T diag(beta gamma), Bu = T diag(beta) (fp16, K-major B
            //      tiles); the previous chunk's M2 must have read them
            ok = n < 1 || WAITW(B_M2DONE, (n - 1) & 1);
            if (named_sync_or(1, 128, !ok)) break;
            {
                const int r = pt & 63;
                const float* f = gb + ((pt < 64) ? GB_BG : GB_BET);
                const float* trow = Tm + r * LDA;
                float v[64];
#pragma unroll
                for (int s = 0; s < 64; ++s) v[s] = (s <= r) ? trow[s] * f[s] : 0.f;
                store_row_sw128(sm + ((pt < 64) ? OFF_BW : OFF_BU), (uint32_t)r, v);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[B_BWU]);
                mbar_arrive(&bars[B_GB_EMPTY + n % GB_SLOTS]);
            }
            if (pt == 0) GDN_TRACE_AT(2, n);
        }
    } else {
        // ---------------------------------------------------------------- state
        const int ws = warp - 8, q4 = ws & 3, hf = ws >> 2;
        const int j = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const size_t sbase = ((size_t)n_seq * p.h_v + h) * (size_t)(D * D);
        float S[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) S[c] = p.h0 ? p.h0[sbase + (size_t)(64 * hf + c) * D + j] : 0.f;
        auto put_state_f16 = [&]() {
            uint32_t pk[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) pk[c] = h2(S[2 * c], S[2 * c + 1]);
            tmem_st32(tmem + lane_base + T_ST + 32 * hf, pk);
            tmem_st_wait();
        };
        put_state_f16();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[B_STREADY]);
        TOut* o = static_cast<TOut*>(p.o);
        const int tid_s = ws * 32 + lane;  // 0..255
        // -W^T and Kdec of chunk m, once M2(m) has run: -W^T from TMEM (lane =
        // key index i, columns = chunk rows r) into the MN-major fp16 B tile;
        // K rows of the stage scaled by Gamma_last,r in place.
        auto produce_w = [&](int m) -> bool {
            if (!WAITW(B_GB_FULL + m % GB_SLOTS, (m / GB_SLOTS) & 1) || !WAITW(B_M2DONE, m & 1)) return false;
            tc_fence_after();
            {
                uint32_t w[32];
                tmem_ld32(tmem + lane_base + T_W + 32 * hf, w);
                tmem_ld_wait();
                float v[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) v[c] = -__uint_as_float(w[c]);
                store_half_row_sw128(sm + OFF_WT, (uint32_t)j, v, hf);
            }
            {
                const int r = tid_s & 63, kb = (tid_s >> 6) & 1, half = tid_s >> 7;
                f16_row_scale(kq_tile(m) + (uint32_t)kb * 16384 + (uint32_t)r * 128, (uint32_t)r,
                              gb_slot(m)[GB_DEC + r], 4 * half, 4);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_WREADY]);
            if (ws == 0 && lane == 0) GDN_TRACE_AT(13, m);
            return true;
        };
        bool alive = nc == 0 || produce_w(0);
        for (int n = 0; n < nc && alive; ++n) {
            // Delta^T (fp32, TMEM) -> fp16 A operand
            if (!WAITW(B_DREADY, n & 1)) break;
            if (ws == 0 && lane == 0) GDN_TRACE_AT(10, n);
            tc_fence_after();
            {
                uint32_t dr[32], pk[16];
                tmem_ld32(tmem + lane_base + T_DU + 32 * hf, dr);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) pk[c] = h2(__uint_as_float(dr[2 * c]), __uint_as_float(dr[2 * c + 1]));
                tmem_st16(tmem + lane_base + T_DT + 16 * hf, pk);
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[B_DELTA]);
            // next chunk's -W^T and Kdec while M5 of this chunk runs (M3a(n)
            // has finished reading -W^T(n): it completed before DREADY(n))
            if (n + 1 < nc && !produce_w(n + 1)) break;
            // state update S^T <- gamma_last S^T + Delta^T Kdec
            if (!WAITW(B_GB_FULL + n % GB_SLOTS, (n / GB_SLOTS) & 1)) break;
            const float gC = gb_slot(n)[GB_GC];
            if (!WAITW(B_SREADY, n & 1)) break;
            if (ws == 0 && lane == 0) GDN_TRACE_AT(11, n);
            tc_fence_after();
            {
                uint32_t acc[32];
                tmem_ld32(tmem + lane_base + T_SACC + 64 * hf, acc);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) S[c] = fmaf(gC, S[c], __uint_as_float(acc[c]));
                tmem_ld32(tmem + lane_base + T_SACC + 64 * hf + 32, acc);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) S[32 + c] = fmaf(gC, S[32 + c], __uint_as_float(acc[c]));
            }
            put_state_f16();
            tc_fence_before();
            __syncwarp();
            if (ws == 0 && lane == 0) GDN_TRACE_AT(12, n);
            if (lane == 0) {
                mbar_arrive(&bars[B_STREADY]);
                mbar_arrive(&bars[B_GB_EMPTY + n % GB_SLOTS]);
            }
            // output rows r = 32 hf .. 32 hf + 31 of this chunk
            if (!WAITW(B_OREADY, n & 1)) break;
            tc_fence_after();
            {
                uint32_t ov[32];
                tmem_ld32(tmem + lane_base + T_O + 32 * hf, ov);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[B_OFREE]);
                const int L = min(C, len - n * C);
                const long long tb = t0 + (long long)n * C + 32 * hf;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (32 * hf + c < L)
                        o[((size_t)(tb + c) * p.h_v + h) * D + j] = from_f32<TOut>(__uint_as_float(ov[c]));
            }
        }
        if (p.hT && !*abort_flag) {
#pragma unroll
            for (int c = 0; c < 64; ++c) p.hT[sbase + (size_t)(64 * hf + c) * D + j] = S[c];
        }
    }

    // ---- teardown: every product finished, then free TMEM
    __syncthreads();
    if (warp == 1) {
        mbar_wait(&bars[B_DONE], 0, nullptr, 200000000ull);
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort_flag) set_device_error(2u);
}

}  // namespace tck

// ------------------------------------------------------------------ host side
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
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
    const long long blocks = (long long)a.num_seqs * a.h_v;
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
