// C ABI of the GDN library: argument checks on the host, kernel dispatch.
// Declarations and the contract of every entry point: include/gdn.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>
#include <numeric>
#include <utility>
#include <vector>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_epilogue.cuh"
#include "gdn_prologue.cuh"
#include "gdn_decode.cuh"
#include "gdn_chunk_simt.cuh"
#include "gdn_chunk_tc.cuh"
#include "gdn_backward.cuh"
#include "gdn_kda.cuh"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
// Non-null and aligned to `a` bytes (16 for tensors read with 128-bit or TMA
// accesses, the element size for the rest).
bool ok_ptr(const void* p, uintptr_t a = 16) { return p != nullptr && aligned(p, a); }
bool ok_opt(const void* p, uintptr_t a = 16) { return p == nullptr || aligned(p, a); }
uintptr_t esize(int32_t dtype) { return dtype == GDN_BF16 ? 2 : 4; }
bool ok_dtype(int32_t d) { return d == GDN_F32 || d == GDN_BF16; }

// Query (once per device) the opt-in shared-memory limit and SM count.
struct DevInfo { int smem_optin = 0; int sms = 0; };
DevInfo dev_info() {
    int dev = 0;
    DevInfo di;
    if (cudaGetDevice(&dev) != cudaSuccess) return di;
    cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    return di;
}

template <typename TIn, typename TOut>
gdn_status launch_simt(const gdn::SimtArgs& a, size_t smem, cudaStream_t s) {
    auto kern = gdn::chunk_simt_kernel<TIn, TOut>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GDN_ERR_CUDA;
    const long long blocks = (long long)a.num_seqs * a.h_v * a.n_tiles;
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    kern<<<(unsigned)blocks, 256, smem, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// Epilogue over `rows` rows of d <= 1024 features (x, z may be different
// dtypes; y may alias x when TY == TX).
template <typename TX, typename TZ, typename TY>
gdn_status launch_gated_rmsnorm(const void* x, const void* z, const float* w, void* y, long long rows, int d,
                                float eps, cudaStream_t s) {
    if (rows == 0) return GDN_OK;
    const DevInfo di = dev_info();
    const long long want = (rows + 7) / 8;
    const long long cap = (long long)std::max(di.sms, 1) * 8;  // one resident wave, grid-strided
    const unsigned blocks = (unsigned)std::min(want, cap);
    auto X = static_cast<const TX*>(x);
    auto Z = static_cast<const TZ*>(z);
    auto Y = static_cast<TY*>(y);
    if (d == 128 && aligned(x, 16) && aligned(z, 16) && aligned(y, 16) && aligned(w, 16)) {
        auto kern = gdn::gated_rmsnorm_d128_kernel<TX, TZ, TY>;
        int per_sm = 0;  // one resident wave, grid-strided
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1)
            per_sm = 1;
        const long long groups = (rows + 3) / 4;  // 4 rows per warp, 8 warps per CTA
        const unsigned b128 = (unsigned)std::min((groups + 7) / 8, (long long)std::max(di.sms, 1) * per_sm);
        kern<<<b128, 256, 0, s>>>(X, Z, w, Y, rows, eps);
    } else if (d <= 128)
        gdn::gated_rmsnorm_kernel<TX, TZ, TY, 4><<<blocks, 256, 0, s>>>(X, Z, w, Y, rows, d, eps);
    else if (d <= 256)
        gdn::gated_rmsnorm_kernel<TX, TZ, TY, 8><<<blocks, 256, 0, s>>>(X, Z, w, Y, rows, d, eps);
    else if (d <= 512)
        gdn::gated_rmsnorm_kernel<TX, TZ, TY, 16><<<blocks, 256, 0, s>>>(X, Z, w, Y, rows, d, eps);
    else
        gdn::gated_rmsnorm_kernel<TX, TZ, TY, 32><<<blocks, 256, 0, s>>>(X, Z, w, Y, rows, d, eps);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// z == nullptr: plain decode; otherwise o goes through the gated RMSNorm
// epilogue (fused in the d = 128 kernel, a second launch elsewhere).
template <typename TIn, typename TOut>
gdn_status launch_decode(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, float* state, void* o, int N, int h_qk, int h_v,
                         int d_k, int d_v, float scale, cudaStream_t s,
                         const void* z = nullptr, const float* w = nullptr, float eps = 0.f) {
    const long long blocks = (long long)N * h_v;
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    const int grp = h_v / h_qk;
    if (d_k == 128 && d_v == 128) {
        if (z)
            gdn::decode_d128_kernel<TIn, TOut, true><<<(unsigned)blocks, 256, 0, s>>>(
                static_cast<const TIn*>(q), static_cast<const TIn*>(k), static_cast<const TIn*>(v), g, beta,
                state, static_cast<TOut*>(o), h_qk, h_v, grp, scale, static_cast<const TIn*>(z), w, eps);
        else
            gdn::decode_d128_kernel<TIn, TOut><<<(unsigned)blocks, 256, 0, s>>>(
                static_cast<const TIn*>(q), static_cast<const TIn*>(k), static_cast<const TIn*>(v), g, beta,
                state, static_cast<TOut*>(o), h_qk, h_v, grp, scale);
    } else {
        gdn::decode_generic_kernel<TIn, TOut><<<(unsigned)blocks, 128, 0, s>>>(
            static_cast<const TIn*>(q), static_cast<const TIn*>(k), static_cast<const TIn*>(v), g, beta,
            state, static_cast<TOut*>(o), h_qk, h_v, grp, d_k, d_v, scale);
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
        if (z) return launch_gated_rmsnorm<TOut, TIn, TOut>(o, z, w, o, blocks, d_v, eps, s);
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

// The TMA-fed filter (gdn::short_conv_tma_kernel) when the input is 16-byte
// aligned and whole 512-byte channel blocks cover the channels; false when
// the tensor map cannot be made (the caller then uses the register-tiled
// kernel).
template <typename T, int K>
bool launch_short_conv_tma(const void* x, const float* w, void* y, const int32_t* cu, const float* st_in,
                           float* st_out, int N, long long total, int C, int ng, float eps, cudaStream_t s,
                           gdn_status& st) {
    constexpr int V = 16 / (int)sizeof(T);
    if (C % (32 * V) != 0 || (ng != 0 && ng < V) || (reinterpret_cast<uintptr_t>(x) & 15u) != 0 || total <= 0 ||
        total >= (1LL << 31))
        return false;
    auto enc = gdn::tensor_map_encoder();
    if (enc == nullptr) return false;
    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)C, (cuuint64_t)total};
    cuuint64_t strides[1] = {(cuuint64_t)C * sizeof(T)};
    cuuint32_t box[2] = {(cuuint32_t)(32 * V), (cuuint32_t)(gdn::pro::TILE + K - 1)};
    cuuint32_t es[2] = {1, 1};
    if (enc(&map, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
            const_cast<void*>(x), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    auto kern = ng == 0 ? gdn::short_conv_tma_kernel<T, K, 0>
                        : ng == 128 ? gdn::short_conv_tma_kernel<T, K, 128> : gdn::short_conv_tma_kernel<T, K, -1>;
    const int smem = (int)gdn::pro::smem_bytes<K>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return false;
    const DevInfo di = dev_info();
    const long long ncb = C / (32 * V);
    const long long ntt = (total + gdn::pro::TILE - 1) / gdn::pro::TILE;
    // persistent: two CTAs per SM, a multiple of the channel blocks
    const long long per_cb = std::max(1LL, std::min(ntt, 2LL * std::max(di.sms, 1) / ncb));
    if (ncb * per_cb > 0x7fffffffLL) return false;
    const long long eq = cu ? 0 : total / N;
    kern<<<(unsigned)(ncb * per_cb), 256, smem, s>>>(map, static_cast<const T*>(x), w, static_cast<T*>(y), cu, st_in,
                                                     st_out, N, total, eq, C, ng, eps, 1u << 17);
    st = cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    return true;
}

template <typename T, int K>
gdn_status launch_short_conv(const void* x, const float* w, void* y, const int32_t* cu, const float* st_in,
                             float* st_out, int N, long long total, int C, int ng, float eps, cudaStream_t s) {
    const DevInfo di = dev_info();
    gdn_status tst = GDN_OK;
    if (launch_short_conv_tma<T, K>(x, w, y, cu, st_in, st_out, N, total, C, ng, eps, s, tst)) {
        if (tst != GDN_OK) return tst;
        if (st_out && (cu || total == 0) && K > 1) {  // empty sequences carry their state over
            const long long n = (long long)N * C * (K - 1);
            gdn::conv_state_carry_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(cu, st_in, st_out, N,
                                                                                      (long long)C * (K - 1));
        }
        return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
    }
    const long long runs = (total + 7) / 8;  // tiles of 8 tokens, one per warp
    // 8 channels per lane when the channels and the head size allow it
    const bool v8 = C % 256 == 0 && (ng == 0 || ng >= 8);
    const int cblocks = v8 ? C / 256 : (C + 127) / 128;
    if (runs > 0) {
        if (cblocks > 65535) return GDN_ERR_UNSUPPORTED;
        // the head size of q and k (128) and no norm (v) are compiled as constants
        auto kern = v8 ? (ng == 0 ? gdn::short_conv_kernel<T, K, 8, 0>
                                  : ng == 128 ? gdn::short_conv_kernel<T, K, 8, 128> : gdn::short_conv_kernel<T, K, 8, -1>)
                       : (ng == 0 ? gdn::short_conv_kernel<T, K, 4, 0>
                                  : ng == 128 ? gdn::short_conv_kernel<T, K, 4, 128> : gdn::short_conv_kernel<T, K, 4, -1>);
        int per_sm = 0;  // one resident wave over all channel blocks
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1)
            per_sm = 1;
        const long long cap = std::max(1LL, (long long)std::max(di.sms, 1) * per_sm / cblocks);
        const dim3 grid((unsigned)std::min((runs + 7) / 8, cap), (unsigned)cblocks);
        const long long eq = cu ? 0 : total / N;
        kern<<<grid, 256, 0, s>>>(static_cast<const T*>(x), w, static_cast<T*>(y), cu,
                                                           st_in, st_out, N, total, eq, C, ng, eps);
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    }
    if (st_out && (cu || total == 0) && K > 1) {  // empty sequences carry their state over
        const long long n = (long long)N * C * (K - 1);
        gdn::conv_state_carry_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(cu, st_in, st_out, N,
                                                                                  (long long)C * (K - 1));
    }
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T, int K>
gdn_status launch_short_conv_step(const void* x, const float* w, float* st, void* y, int N, int C, int ng,
                                  float eps, cudaStream_t s) {
    const DevInfo di = dev_info();
    const long long units = (long long)N * ((C + 127) / 128);
    const long long cap = (long long)std::max(di.sms, 1) * 64;
    const unsigned blocks = (unsigned)std::min((units + 7) / 8, cap);
    gdn::short_conv_step_kernel<T, K><<<blocks, 256, 0, s>>>(static_cast<const T*>(x), w, st, static_cast<T*>(y), N,
                                                              C, ng, eps);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename T>
gdn_status dispatch_conv(int K, const void* x, const float* w, void* y, const int32_t* cu, const float* st_in,
                         float* st_out, int N, long long total, int C, int ng, float eps, cudaStream_t s) {
    switch (K) {
        case 1: return launch_short_conv<T, 1>(x, w, y, cu, st_in, st_out, N, total, C, ng, eps, s);
        case 2: return launch_short_conv<T, 2>(x, w, y, cu, st_in, st_out, N, total, C, ng, eps, s);
        case 3: return launch_short_conv<T, 3>(x, w, y, cu, st_in, st_out, N, total, C, ng, eps, s);
        default: return launch_short_conv<T, 4>(x, w, y, cu, st_in, st_out, N, total, C, ng, eps, s);
    }
}

template <typename T>
gdn_status dispatch_conv_step(int K, const void* x, const float* w, float* st, void* y, int N, int C, int ng,
                              float eps, cudaStream_t s) {
    switch (K) {
        case 1: return launch_short_conv_step<T, 1>(x, w, st, y, N, C, ng, eps, s);
        case 2: return launch_short_conv_step<T, 2>(x, w, st, y, N, C, ng, eps, s);
        case 3: return launch_short_conv_step<T, 3>(x, w, st, y, N, C, ng, eps, s);
        default: return launch_short_conv_step<T, 4>(x, w, st, y, N, C, ng, eps, s);
    }
}

bool ok_norm_group(int ng, int C) {
    return ng == 0 || ((ng == 4 || ng == 8 || ng == 16 || ng == 32 || ng == 64 || ng == 128) && C % ng == 0);
}

// Workspace layout of gdn_chunk_bwd: checkpoints, then (grouped heads only)
// the per-value-head dq and dk parts, each part 256-byte aligned.
struct BwdLayout { long long nslots = 0; size_t ckpt = 0, part = 0, e = 0, qdq = 0, total = 0; };
BwdLayout bwd_layout(int32_t N, int64_t T, int32_t h_qk, int32_t h_v) {
    BwdLayout L;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    L.nslots = T / gdn::bwd::BLK + N + 1;
    L.ckpt = up((size_t)h_v * (size_t)L.nslots * gdn::bwd::SD * sizeof(float));
    L.part = h_v > h_qk ? up((size_t)T * h_v * gdn::bwd::D * sizeof(float)) : 0;
    L.e = up((size_t)T * h_v * gdn::bwd::D * sizeof(float));
    L.qdq = up((size_t)T * h_v * sizeof(float));
    L.total = L.ckpt + 2 * L.part + L.e + L.qdq;
    return L;
}

bool bwd_sizes_ok(int32_t N, int64_t T, int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v) {
    return N >= 0 && T >= 0 && h_qk > 0 && h_v > 0 && h_v % h_qk == 0 && d_k > 0 && d_v > 0;
}

template <typename TIn, typename TdO>
gdn_status launch_bwd(gdn::bwd::Args a, float* dq, float* dk, char* ws, const BwdLayout& L, cudaStream_t s) {
    const long long blocks = (long long)a.num_seqs * a.h_v;
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    const DevInfo di = dev_info();
    if (di.smem_optin < (int)gdn::bwd::SMEM_BYTES) return di.smem_optin <= 0 ? GDN_ERR_CUDA : GDN_ERR_UNSUPPORTED;
    auto kern = gdn::bwd::backward_kernel<TIn, TdO>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gdn::bwd::SMEM_BYTES) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    a.ckpt = reinterpret_cast<float*>(ws);
    a.nslots = L.nslots;
    float* dq_part = L.part ? reinterpret_cast<float*>(ws + L.ckpt) : dq;
    float* dk_part = L.part ? reinterpret_cast<float*>(ws + L.ckpt + L.part) : dk;
    a.dq = dq_part;
    a.dk = dk_part;
    a.e_ws = reinterpret_cast<float*>(ws + L.ckpt + 2 * L.part);
    a.qdq_ws = reinterpret_cast<float*>(ws + L.ckpt + 2 * L.part + L.e);
    kern<<<(unsigned)blocks, gdn::bwd::NT, gdn::bwd::SMEM_BYTES, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    if (L.part && a.total > 0) {
        const long long units = a.total * a.h_qk * (gdn::bwd::D / 4);
        const long long cap = (long long)std::max(di.sms, 1) * 8;
        const unsigned grid = (unsigned)std::min(cap, (units + 255) / 256);
        gdn::bwd::group_sum_kernel<<<grid, 256, 0, s>>>(dq_part, dk_part, dq, dk, units, a.h_qk, a.grp);
        if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    }
    return GDN_OK;
}

}  // namespace


namespace {

template <typename TIn, typename TOut>
gdn_status launch_kda_prefill(gdn::kda::Args a, cudaStream_t s) {
    const DevInfo di = dev_info();
    // fewer units than two per SM: split the units over several CTAs (not
    // when the final state overwrites the initial state: a later piece could
    // then finish before an earlier one has read it). Equal lengths: shares
    // of at least 256 tokens of the (sequence, q/k head) groups in order,
    // each taken by the group's value heads in neighbouring CTAs, so that
    // every slot gets the same work; otherwise sequence segments of at least
    // 512 tokens.
    a.nseg = 1;
    a.bal_tokens = 0;
    const long long units = (long long)a.num_seqs * a.h_v, slots = 2LL * std::max(di.sms, 1);
    long long blocks = units;
    if (units > 0 && units < slots && !(a.hT != nullptr && a.hT == a.h0)) {
        const long long gtot = (long long)a.num_seqs * a.h_qk * a.eq_len;  // eq_len = 0 with cu_seqlens
        const long long share_slots = std::max(1LL, slots / a.grp);
        const long long share = (gtot + share_slots - 1) / share_slots / gdn::kda::BLK * gdn::kda::BLK +
                                gdn::kda::BLK;  // rounded up to whole blocks
        if (a.cu == nullptr && a.eq_len > 0 && share >= 256 && share < a.eq_len) {
            a.bal_tokens = share;
            blocks = (gtot + share - 1) / share * a.grp;
        } else {
            const long long by_len = (long long)(a.total / a.num_seqs) / 512;
            a.nseg = (int)std::max(1LL, std::min(std::min(slots / units, by_len), 64LL));
            blocks = units * a.nseg;
        }
    }
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    if (di.smem_optin < (int)gdn::kda::SMEM_BYTES) return di.smem_optin <= 0 ? GDN_ERR_CUDA : GDN_ERR_UNSUPPORTED;
    auto kern = gdn::kda::kda_prefill_kernel<TIn, TOut>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gdn::kda::SMEM_BYTES) !=
        cudaSuccess)
        return GDN_ERR_CUDA;
    // the largest shared-memory carve-out, so that two CTAs fit on an SM
    if (cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return GDN_ERR_CUDA;
    kern<<<(unsigned)blocks, gdn::kda::NT, gdn::kda::SMEM_BYTES, s>>>(a);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

template <typename TIn, typename TOut>
gdn_status launch_kda_decode(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             float* state, void* o, int N, int h_qk, int h_v, float scale, cudaStream_t s) {
    const long long blocks = (long long)N * h_v;
    if (blocks > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    gdn::kda::kda_decode_d128_kernel<TIn, TOut><<<(unsigned)blocks, 256, 0, s>>>(
        static_cast<const TIn*>(q), static_cast<const TIn*>(k), static_cast<const TIn*>(v), g, beta, state,
        static_cast<TOut*>(o), h_qk, h_v, h_v / h_qk, scale);
    return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

}  // namespace

namespace {

// Host checks of gdn_chunk_bwd and gdn_chunk_bwd_static (everything except
// the scratch memory), in the order the header documents. GDN_OK with
// num_seqs == 0 means there is nothing to do.
gdn_status bwd_check(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     const float* initial_state, const int32_t* cu_seqlens, const int32_t* seq_order,
                     const void* d_o, const float* d_final_state, const float* dq, const float* dk,
                     const float* dv, const float* dg, const float* dbeta, const float* d_initial_state,
                     int32_t num_seqs, int64_t total_tokens, int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                     int32_t dtype_qkv, int32_t dtype_do) {
    if (!bwd_sizes_ok(num_seqs, total_tokens, h_qk, h_v, d_k, d_v)) return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype_qkv) || !ok_dtype(dtype_do)) return GDN_ERR_INVALID_ARG;
    if (d_k != gdn::bwd::D || d_v != gdn::bwd::D) return GDN_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && total_tokens % num_seqs != 0) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;  // cu_seqlens are int32
    if (total_tokens > 0 &&
        (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(g, 4) || !ok_ptr(beta, 4) || !ok_ptr(d_o) ||
         !ok_ptr(dq) || !ok_ptr(dk) || !ok_ptr(dv) || !ok_ptr(dg, 4) || !ok_ptr(dbeta, 4)))
        return GDN_ERR_INVALID_ARG;
    if (!ok_opt(initial_state) || !ok_opt(d_final_state) || !ok_opt(d_initial_state) || !ok_opt(cu_seqlens, 4) ||
        !ok_opt(seq_order, 4))
        return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

// Launch of the backward kernels on a checked problem and a scratch region of
// at least L.total bytes (256-byte aligned).
gdn_status bwd_launch(const void* q, const void* k, const void* v, const float* g, const float* beta,
                      const float* initial_state, const int32_t* cu_seqlens, const int32_t* seq_order,
                      const void* d_o, const float* d_final_state, float* dq, float* dk, float* dv, float* dg,
                      float* dbeta, float* d_initial_state, int32_t num_seqs, int64_t total_tokens, int32_t h_qk,
                      int32_t h_v, int32_t dtype_qkv, int32_t dtype_do, float scale, char* ws, const BwdLayout& L,
                      cudaStream_t s) {
    if (scale == 0.f) scale = 1.0f / sqrtf((float)gdn::bwd::D);
    gdn::bwd::Args a{};
    a.q = q; a.k = k; a.v = v; a.dout = d_o; a.g = g; a.beta = beta;
    a.h0 = initial_state; a.dht = d_final_state; a.cu = cu_seqlens; a.order = seq_order;
    a.dv = dv; a.dg = dg; a.dbeta = dbeta; a.dh0 = d_initial_state;
    a.total = total_tokens; a.eq_len = cu_seqlens ? 0 : total_tokens / num_seqs;
    a.num_seqs = num_seqs; a.h_qk = h_qk; a.h_v = h_v; a.grp = h_v / h_qk; a.scale = scale;
    const bool bq = dtype_qkv == GDN_BF16, bd = dtype_do == GDN_BF16;
    if (bq && bd) return launch_bwd<__nv_bfloat16, __nv_bfloat16>(a, dq, dk, ws, L, s);
    if (bq) return launch_bwd<__nv_bfloat16, float>(a, dq, dk, ws, L, s);
    if (bd) return launch_bwd<float, __nv_bfloat16>(a, dq, dk, ws, L, s);
    return launch_bwd<float, float>(a, dq, dk, ws, L, s);
}

}  // namespace

// Scratch of gdn_chunk_bwd_static: a fixed device array in this module, so
// that callers without an allocator can still take the gradient. Host code
// must not use the symbol's name as a pointer; the device address comes from
// cudaGetSymbolAddress, looked up with the device current.
static __device__ __align__(256) unsigned char g_bwd_static_scratch[GDN_BWD_STATIC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_static_scratch_mu;
struct ScratchSlot { unsigned long long ctx_id = 0; void* ptr = nullptr; };
ScratchSlot g_static_scratch[kMaxDevices];

// Unique id of the current CUDA context (0 if it cannot be read). A device
// reset destroys the primary context and a later call creates a new one with
// a new id, into which the module (and with it the array) may load at
// another address.
unsigned long long current_context_id() {
    static const auto fns = [] {
        std::pair<PFN_cuCtxGetCurrent_v4000, PFN_cuCtxGetId_v12000> f{nullptr, nullptr};
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.first = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            f.second = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
        return f;
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (fns.first && fns.second && fns.first(&ctx) == CUDA_SUCCESS && ctx && fns.second(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// Device address of the array on the current device: looked up once per
// device and context (the first call in a context does the lookup, with the
// device current; a reset device gets a fresh lookup).
gdn_status static_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    const unsigned long long id = current_context_id();  // 0 before the context exists
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    ScratchSlot& slot = g_static_scratch[dev];
    if (slot.ptr == nullptr || id == 0 || slot.ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_static_scratch) != cudaSuccess || p == nullptr) return GDN_ERR_CUDA;
        slot.ptr = p;
        slot.ctx_id = current_context_id();  // the lookup has made the context current
    }
    *out = slot.ptr;
    return GDN_OK;
}
}  // namespace

extern "C" {

const char* gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    }
    return "GDN_ERR_UNKNOWN";
}

int32_t gdn_version(void) { return 103; }

gdn_status gdn_plan_seq_order(const int32_t* cu, int32_t num_seqs, int32_t* order_out) {
    if (num_seqs < 0 || (num_seqs > 0 && (cu == nullptr || order_out == nullptr))) return GDN_ERR_INVALID_ARG;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu[n + 1] < cu[n]) return GDN_ERR_INVALID_ARG;
    std::vector<int32_t> idx(num_seqs);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
        return (cu[a + 1] - cu[a]) > (cu[b + 1] - cu[b]);
    });
    std::copy(idx.begin(), idx.end(), order_out);
    return GDN_OK;
}

gdn_status gdn_get_device_error(void* stream, uint32_t* code) {
    if (code == nullptr) return GDN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, gdn::g_device_error, sizeof v) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaMemcpyToSymbol(gdn::g_device_error, &zero, sizeof zero) != cudaSuccess) return GDN_ERR_CUDA;
    *code = v;
    return (v & GDN_DEVERR_TIMEOUT) ? GDN_ERR_TIMEOUT : GDN_OK;
}

gdn_status gdn_decode_step_gated(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, float* state, void* o, const void* gate,
                                 const float* norm_weight, float eps, int32_t num_seqs,
                                 int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                                 int32_t dtype_qkv, int32_t dtype_o, float scale, void* stream) {
    if (num_seqs < 0 || h_qk <= 0 || h_v <= 0 || h_v % h_qk != 0 || d_k <= 0 || d_v <= 0)
        return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype_qkv) || !ok_dtype(dtype_o)) return GDN_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return GDN_ERR_INVALID_ARG;
    if (d_k > 128 || d_v > 128) return GDN_ERR_UNSUPPORTED;
    if (num_seqs == 0) return GDN_OK;
    const uintptr_t ei = esize(dtype_qkv), eo = esize(dtype_o);
    if (!ok_ptr(q, ei) || !ok_ptr(k, ei) || !ok_ptr(v, ei) || !ok_ptr(g, 4) || !ok_ptr(beta, 4) ||
        !ok_ptr(state, 16) || !ok_ptr(o, eo) || !ok_opt(gate, ei) || !ok_opt(norm_weight, 4))
        return GDN_ERR_INVALID_ARG;
    if (gate == nullptr && norm_weight != nullptr) return GDN_ERR_INVALID_ARG;
    if (scale == 0.f) scale = 1.0f / sqrtf((float)d_k);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bf_in = dtype_qkv == GDN_BF16, bf_out = dtype_o == GDN_BF16;
    if (bf_in && bf_out)
        return launch_decode<__nv_bfloat16, __nv_bfloat16>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, d_k,
                                                           d_v, scale, s, gate, norm_weight, eps);
    if (bf_in)
        return launch_decode<__nv_bfloat16, float>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, d_k, d_v,
                                                   scale, s, gate, norm_weight, eps);
    if (bf_out)
        return launch_decode<float, __nv_bfloat16>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, d_k, d_v,
                                                   scale, s, gate, norm_weight, eps);
    return launch_decode<float, float>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, d_k, d_v, scale, s,
                                       gate, norm_weight, eps);
}

gdn_status gdn_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* state, void* o, int32_t num_seqs,
                           int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                           int32_t dtype_qkv, int32_t dtype_o, float scale, void* stream) {
    return gdn_decode_step_gated(q, k, v, g, beta, state, o, nullptr, nullptr, 0.f, num_seqs, h_qk, h_v, d_k,
                                 d_v, dtype_qkv, dtype_o, scale, stream);
}

gdn_status gdn_gated_rmsnorm(const void* x, const void* gate, const float* norm_weight, void* y, int64_t rows,
                             int32_t d, int32_t dtype_x, int32_t dtype_y, float eps, void* stream) {
    if (rows < 0 || d <= 0) return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype_x) || !ok_dtype(dtype_y)) return GDN_ERR_INVALID_ARG;
    if (!(eps >= 0.f) || !isfinite(eps)) return GDN_ERR_INVALID_ARG;
    if (d > 1024) return GDN_ERR_UNSUPPORTED;
    if (rows == 0) return GDN_OK;
    const uintptr_t ex = esize(dtype_x), ey = esize(dtype_y);
    if (!ok_ptr(x, ex) || !ok_ptr(gate, ex) || !ok_opt(norm_weight, 4) || !ok_ptr(y, ey))
        return GDN_ERR_INVALID_ARG;
    // in place only with equal element types (each row is read before it is written)
    if (y == x && dtype_x != dtype_y) return GDN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bx = dtype_x == GDN_BF16, by = dtype_y == GDN_BF16;
    if (bx && by)
        return launch_gated_rmsnorm<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(x, gate, norm_weight, y, rows, d,
                                                                                 eps, s);
    if (bx)
        return launch_gated_rmsnorm<__nv_bfloat16, __nv_bfloat16, float>(x, gate, norm_weight, y, rows, d, eps, s);
    if (by)
        return launch_gated_rmsnorm<float, float, __nv_bfloat16>(x, gate, norm_weight, y, rows, d, eps, s);
    return launch_gated_rmsnorm<float, float, float>(x, gate, norm_weight, y, rows, d, eps, s);
}

gdn_status gdn_short_conv(const void* x, const float* w, void* y, const int32_t* cu_seqlens,
                          const float* conv_state_in, float* conv_state_out, int32_t num_seqs,
                          int64_t total_tokens, int32_t channels, int32_t kernel_size, int32_t norm_group,
                          float eps, int32_t dtype, void* stream) {
    if (num_seqs < 0 || total_tokens < 0 || channels <= 0 || kernel_size < 1) return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype) || !(eps >= 0.f) || !isfinite(eps)) return GDN_ERR_INVALID_ARG;
    if (channels % 4 != 0 || !ok_norm_group(norm_group, channels)) return GDN_ERR_INVALID_ARG;
    if (kernel_size > 4) return GDN_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && total_tokens % num_seqs != 0) return GDN_ERR_INVALID_ARG;
    if (!ok_ptr(x) || !ok_ptr(w, 4) || !ok_ptr(y) || !ok_opt(cu_seqlens, 4) || !ok_opt(conv_state_in, 4) ||
        !ok_opt(conv_state_out, 4))
        return GDN_ERR_INVALID_ARG;
    if (y == x) return GDN_ERR_INVALID_ARG;  // the taps read neighbours: no in-place
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GDN_BF16)
        return dispatch_conv<__nv_bfloat16>(kernel_size, x, w, y, cu_seqlens, conv_state_in, conv_state_out, num_seqs,
                                            total_tokens, channels, norm_group, eps, s);
    return dispatch_conv<float>(kernel_size, x, w, y, cu_seqlens, conv_state_in, conv_state_out, num_seqs,
                                total_tokens, channels, norm_group, eps, s);
}

gdn_status gdn_short_conv_step(const void* x, const float* w, float* conv_state, void* y, int32_t num_seqs,
                               int32_t channels, int32_t kernel_size, int32_t norm_group, float eps, int32_t dtype,
                               void* stream) {
    if (num_seqs < 0 || channels <= 0 || kernel_size < 1) return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype) || !(eps >= 0.f) || !isfinite(eps)) return GDN_ERR_INVALID_ARG;
    if (channels % 4 != 0 || !ok_norm_group(norm_group, channels)) return GDN_ERR_INVALID_ARG;
    if (kernel_size > 4) return GDN_ERR_UNSUPPORTED;
    if (num_seqs == 0) return GDN_OK;
    if (!ok_ptr(x) || !ok_ptr(w, 4) || !ok_ptr(y) || (kernel_size > 1 && !ok_ptr(conv_state, 4)))
        return GDN_ERR_INVALID_ARG;
    if (y == x) return GDN_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GDN_BF16)
        return dispatch_conv_step<__nv_bfloat16>(kernel_size, x, w, conv_state, y, num_seqs, channels, norm_group, eps, s);
    return dispatch_conv_step<float>(kernel_size, x, w, conv_state, y, num_seqs, channels, norm_group, eps, s);
}

}  // extern "C"

namespace {

// gdn_chunk_fwd with an optional output epilogue (gate != nullptr), run as a
// second launch on o in place.
gdn_status chunk_fwd_impl(const void* q, const void* k, const void* v, const float* g, const float* beta,
                          const float* initial_state, const int32_t* cu_seqlens, const int32_t* seq_order, void* o,
                          float* final_state, int32_t num_seqs, int64_t total_tokens, int32_t h_qk, int32_t h_v,
                          int32_t d_k, int32_t d_v, int32_t dtype_qkv, int32_t dtype_o, float scale,
                          int32_t chunk_size, int32_t flags, const void* gate, const float* norm_weight, float eps,
                          void* stream) {
    if (num_seqs < 0 || total_tokens < 0 || h_qk <= 0 || h_v <= 0 || h_v % h_qk != 0 || d_k <= 0 || d_v <= 0)
        return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype_qkv) || !ok_dtype(dtype_o)) return GDN_ERR_INVALID_ARG;
    if (chunk_size != 0 && chunk_size != 16 && chunk_size != 32 && chunk_size != 64) return GDN_ERR_INVALID_ARG;
    if (flags & ~(GDN_FLAG_FORCE_SIMT | GDN_FLAG_TEST_WAIT_TIMEOUT | GDN_FLAG_NO_SPLIT | GDN_FLAG_BALANCE))
        return GDN_ERR_INVALID_ARG;
    if (gate && (!(eps >= 0.f) || !isfinite(eps))) return GDN_ERR_INVALID_ARG;
    if (d_k > 128 || d_v > 128) return GDN_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && total_tokens % num_seqs != 0) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0 && (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(g, 4) ||
                             !ok_ptr(beta, 4) || !ok_ptr(o, esize(dtype_o))))
        return GDN_ERR_INVALID_ARG;
    if (gate && total_tokens > 0 && (!ok_ptr(gate, 16) || !ok_opt(norm_weight, 16))) return GDN_ERR_INVALID_ARG;
    if (!ok_opt(initial_state) || !ok_opt(final_state) || !ok_opt(cu_seqlens, 4) || !ok_opt(seq_order, 4))
        return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;  // cu_seqlens are int32
    if (total_tokens == 0 && final_state == nullptr) return GDN_OK;
    if (scale == 0.f) scale = 1.0f / sqrtf((float)d_k);
    const int C = chunk_size == 0 ? 64 : chunk_size;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long eq_len = cu_seqlens ? 0 : total_tokens / num_seqs;

    const bool bf_in = dtype_qkv == GDN_BF16, bf_out = dtype_o == GDN_BF16;
    if (bf_in && d_k == 128 && d_v == 128 && total_tokens > 0 && !(flags & GDN_FLAG_FORCE_SIMT) &&
        gdn::tc_available()) {
        gdn::TcArgs a{};
        a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = initial_state;
        a.cu = cu_seqlens; a.order = seq_order; a.o = o; a.hT = final_state;
        a.num_seqs = num_seqs; a.total = total_tokens; a.eq_len = eq_len;
        a.h_qk = h_qk; a.h_v = h_v; a.grp = h_v / h_qk; a.scale = scale;
        const bool stall = (flags & GDN_FLAG_TEST_WAIT_TIMEOUT) != 0;
        a.max_polls = stall ? (1u << 12) : (1u << 17);
        a.withhold_chunk = stall ? 1 : -1;
        // Fewer (sequence, head) units than SMs: split the work of a unit over
        // several CTAs (the kernel starts a piece of a unit from a zero state
        // where the decay has made the earlier tokens' influence negligible,
        // else from the sequence start). Equal lengths with shares of at least
        // 32 chunks: the chunks of the (sequence, q/k head) groups are cut into
        // equal shares in order, each taken by the group's grp value heads in
        // grp neighbouring CTAs (they read the same q and k tiles at the same
        // time), so that all SMs share the work evenly (below 32 chunks a
        // piece's fixed costs, the prefix search at the start and the state
        // hand-over between two units, outweigh the balance). Otherwise
        // segments of at least 512 tokens, one CTA each, up to SMs / units
        // per sequence. Not when
        // the final state overwrites the initial state: a later piece could
        // then finish before an earlier one has read it.
        a.nseg = 1;
        a.bal_chunks = 0;
        if (!(flags & GDN_FLAG_NO_SPLIT) && !(final_state != nullptr && final_state == initial_state)) {
            const long long units = (long long)num_seqs * h_v, sms = std::max(dev_info().sms, 1);
            if (units < sms) {
                const long long nch = (eq_len + gdn::tck::C - 1) / gdn::tck::C, grp = h_v / h_qk;
                // shares of the (sequence, q/k head) groups' chunks; grp CTAs each
                const long long slots = std::max(1LL, sms / grp);
                const long long share = ((long long)num_seqs * h_qk * nch + slots - 1) / slots;
                const bool force = (flags & GDN_FLAG_BALANCE) != 0;
                const long long sh = force ? std::max(share, 3LL) : share;
                if (cu_seqlens == nullptr && (force || share >= 32) && sh < nch && sh <= 0x7fffffffLL) {
                    a.bal_chunks = (int)sh;
                } else {
                    const long long by_len = (long long)(total_tokens / num_seqs) / 512;
                    a.nseg = (int)std::max(1LL, std::min(std::min(sms / units, by_len), 64LL));
                }
            }
        }
        const gdn_status st = gdn::launch_tc(a, bf_out, s);
        if (st != GDN_OK || gate == nullptr) return st;
        // the epilogue as a second launch on o, in place (a fused output stage
        // measured slower: it lengthens the per-chunk chain of the state warps)
        const long long rows = total_tokens * h_v;
        if (bf_out) return launch_gated_rmsnorm<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(o, gate, norm_weight, o, rows, d_v, eps, s);
        return launch_gated_rmsnorm<float, __nv_bfloat16, float>(o, gate, norm_weight, o, rows, d_v, eps, s);
    }

    gdn::SimtArgs a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = initial_state;
    a.cu = cu_seqlens; a.order = seq_order; a.o = o; a.hT = final_state;
    a.num_seqs = num_seqs; a.total = total_tokens; a.eq_len = eq_len;
    a.h_qk = h_qk; a.h_v = h_v; a.d_k = d_k; a.d_v = d_v; a.grp = h_v / h_qk;
    a.C = C; a.dvt = d_v < 64 ? d_v : 64; a.n_tiles = (d_v + a.dvt - 1) / a.dvt; a.scale = scale;
    const size_t smem = gdn::simt_smem_floats(C, d_k, a.dvt) * sizeof(float);
    const DevInfo di = dev_info();
    if (di.smem_optin <= 0) return GDN_ERR_CUDA;
    if (smem > (size_t)di.smem_optin) return GDN_ERR_UNSUPPORTED;
    gdn_status st;
    if (bf_in && bf_out) st = launch_simt<__nv_bfloat16, __nv_bfloat16>(a, smem, s);
    else if (bf_in) st = launch_simt<__nv_bfloat16, float>(a, smem, s);
    else if (bf_out) st = launch_simt<float, __nv_bfloat16>(a, smem, s);
    else st = launch_simt<float, float>(a, smem, s);
    if (st != GDN_OK || gate == nullptr || total_tokens == 0) return st;
    // the epilogue as a second launch on o, in place (the gate has the dtype of q/k/v)
    const long long rows = total_tokens * h_v;
    if (bf_in && bf_out) return launch_gated_rmsnorm<__nv_bfloat16, __nv_bfloat16, __nv_bfloat16>(o, gate, norm_weight, o, rows, d_v, eps, s);
    if (bf_in) return launch_gated_rmsnorm<float, __nv_bfloat16, float>(o, gate, norm_weight, o, rows, d_v, eps, s);
    if (bf_out) return launch_gated_rmsnorm<__nv_bfloat16, float, __nv_bfloat16>(o, gate, norm_weight, o, rows, d_v, eps, s);
    return launch_gated_rmsnorm<float, float, float>(o, gate, norm_weight, o, rows, d_v, eps, s);
}

}  // namespace

extern "C" {

gdn_status gdn_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                         const int32_t* seq_order, void* o, float* final_state, int32_t num_seqs,
                         int64_t total_tokens, int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                         int32_t dtype_qkv, int32_t dtype_o, float scale, int32_t chunk_size,
                         int32_t flags, void* stream) {
    return chunk_fwd_impl(q, k, v, g, beta, initial_state, cu_seqlens, seq_order, o, final_state, num_seqs,
                          total_tokens, h_qk, h_v, d_k, d_v, dtype_qkv, dtype_o, scale, chunk_size, flags, nullptr,
                          nullptr, 0.f, stream);
}

gdn_status gdn_chunk_fwd_gated(const void* q, const void* k, const void* v, const float* g,
                               const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                               const int32_t* seq_order, void* o, const void* gate, const float* norm_weight,
                               float eps, float* final_state, int32_t num_seqs, int64_t total_tokens,
                               int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v, int32_t dtype_qkv,
                               int32_t dtype_o, float scale, int32_t chunk_size, int32_t flags, void* stream) {
    if (gate == nullptr) return GDN_ERR_INVALID_ARG;
    return chunk_fwd_impl(q, k, v, g, beta, initial_state, cu_seqlens, seq_order, o, final_state, num_seqs,
                          total_tokens, h_qk, h_v, d_k, d_v, dtype_qkv, dtype_o, scale, chunk_size, flags, gate,
                          norm_weight, eps, stream);
}

size_t gdn_chunk_fwd_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t h_qk, int32_t h_v,
                                    int32_t d_k, int32_t d_v, int32_t dtype_qkv) {
    (void)num_seqs; (void)total_tokens; (void)h_qk; (void)h_v; (void)d_k; (void)d_v; (void)dtype_qkv;
    return 0;  // both forward kernels keep every intermediate on chip
}

size_t gdn_chunk_bwd_workspace_size(int32_t num_seqs, int64_t total_tokens, int32_t h_qk, int32_t h_v,
                                    int32_t d_k, int32_t d_v) {
    if (!bwd_sizes_ok(num_seqs, total_tokens, h_qk, h_v, d_k, d_v) || total_tokens > 0x7fffffffLL) return 0;
    return bwd_layout(num_seqs, total_tokens, h_qk, h_v).total;
}

gdn_status gdn_chunk_bwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                         const float* initial_state, const int32_t* cu_seqlens, const int32_t* seq_order,
                         const void* d_o, const float* d_final_state, float* dq, float* dk, float* dv,
                         float* dg, float* dbeta, float* d_initial_state, int32_t num_seqs,
                         int64_t total_tokens, int32_t h_qk, int32_t h_v, int32_t d_k, int32_t d_v,
                         int32_t dtype_qkv, int32_t dtype_do, float scale, void* workspace,
                         size_t workspace_bytes, void* stream) {
    const gdn_status st = bwd_check(q, k, v, g, beta, initial_state, cu_seqlens, seq_order, d_o, d_final_state, dq,
                                    dk, dv, dg, dbeta, d_initial_state, num_seqs, total_tokens, h_qk, h_v, d_k, d_v,
                                    dtype_qkv, dtype_do);
    if (st != GDN_OK || num_seqs == 0) return st;
    const BwdLayout L = bwd_layout(num_seqs, total_tokens, h_qk, h_v);
    if (!ok_ptr(workspace, 256) || workspace_bytes < L.total) return GDN_ERR_INVALID_ARG;
    return bwd_launch(q, k, v, g, beta, initial_state, cu_seqlens, seq_order, d_o, d_final_state, dq, dk, dv, dg,
                      dbeta, d_initial_state, num_seqs, total_tokens, h_qk, h_v, dtype_qkv, dtype_do, scale,
                      static_cast<char*>(workspace), L, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_chunk_bwd_static(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* initial_state, const int32_t* cu_seqlens,
                                const int32_t* seq_order, const void* d_o, const float* d_final_state, float* dq,
                                float* dk, float* dv, float* dg, float* dbeta, float* d_initial_state,
                                int32_t num_seqs, int64_t total_tokens, int32_t h_qk, int32_t h_v, int32_t d_k,
                                int32_t d_v, int32_t dtype_qkv, int32_t dtype_do, float scale, void* stream) {
    // the same host checks as gdn_chunk_bwd, in the same order, then the size
    // limit of the array: nothing touches the device for a rejected call
    const gdn_status st = bwd_check(q, k, v, g, beta, initial_state, cu_seqlens, seq_order, d_o, d_final_state, dq,
                                    dk, dv, dg, dbeta, d_initial_state, num_seqs, total_tokens, h_qk, h_v, d_k, d_v,
                                    dtype_qkv, dtype_do);
    if (st != GDN_OK || num_seqs == 0) return st;
    const BwdLayout L = bwd_layout(num_seqs, total_tokens, h_qk, h_v);
    if (L.total > GDN_BWD_STATIC_SCRATCH_BYTES) return GDN_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const gdn_status sa = static_scratch_address(&scratch);
    if (sa != GDN_OK) return sa;
    return bwd_launch(q, k, v, g, beta, initial_state, cu_seqlens, seq_order, d_o, d_final_state, dq, dk, dv, dg,
                      dbeta, d_initial_state, num_seqs, total_tokens, h_qk, h_v, dtype_qkv, dtype_do, scale,
                      static_cast<char*>(scratch), L, static_cast<cudaStream_t>(stream));
}

gdn_status gdn_kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g, const float* beta,
                             const float* initial_state, const int32_t* cu_seqlens, const int32_t* seq_order,
                             void* o, float* final_state, int32_t num_seqs, int64_t total_tokens, int32_t h_qk,
                             int32_t h_v, int32_t d_k, int32_t d_v, int32_t dtype_qkv, int32_t dtype_o,
                             float scale, void* stream) {
    if (num_seqs < 0 || total_tokens < 0 || h_qk <= 0 || h_v <= 0 || h_v % h_qk != 0 || d_k <= 0 || d_v <= 0)
        return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype_qkv) || !ok_dtype(dtype_o)) return GDN_ERR_INVALID_ARG;
    if (d_k != gdn::kda::D || d_v != gdn::kda::D) return GDN_ERR_UNSUPPORTED;
    if (num_seqs == 0) return total_tokens == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (cu_seqlens == nullptr && total_tokens % num_seqs != 0) return GDN_ERR_INVALID_ARG;
    if (total_tokens > 0x7fffffffLL) return GDN_ERR_UNSUPPORTED;
    if (total_tokens > 0 && (!ok_ptr(q) || !ok_ptr(k) || !ok_ptr(v) || !ok_ptr(g) || !ok_ptr(beta, 4) ||
                             !ok_ptr(o, esize(dtype_o))))
        return GDN_ERR_INVALID_ARG;
    if (!ok_opt(initial_state) || !ok_opt(final_state) || !ok_opt(cu_seqlens, 4) || !ok_opt(seq_order, 4))
        return GDN_ERR_INVALID_ARG;
    if (total_tokens == 0 && final_state == nullptr) return GDN_OK;
    if (scale == 0.f) scale = 1.0f / sqrtf((float)d_k);
    gdn::kda::Args a{};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.h0 = initial_state; a.cu = cu_seqlens;
    a.order = seq_order; a.o = o; a.hT = final_state; a.total = total_tokens;
    a.eq_len = cu_seqlens ? 0 : total_tokens / num_seqs; a.num_seqs = num_seqs; a.h_qk = h_qk; a.h_v = h_v;
    a.grp = h_v / h_qk; a.scale = scale;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bi = dtype_qkv == GDN_BF16, bo = dtype_o == GDN_BF16;
    if (bi && bo) return launch_kda_prefill<__nv_bfloat16, __nv_bfloat16>(a, s);
    if (bi) return launch_kda_prefill<__nv_bfloat16, float>(a, s);
    if (bo) return launch_kda_prefill<float, __nv_bfloat16>(a, s);
    return launch_kda_prefill<float, float>(a, s);
}

gdn_status gdn_kda_decode_step(const void* q, const void* k, const void* v, const float* g, const float* beta,
                               float* state, void* o, int32_t num_seqs, int32_t h_qk, int32_t h_v, int32_t d_k,
                               int32_t d_v, int32_t dtype_qkv, int32_t dtype_o, float scale, void* stream) {
    if (num_seqs < 0 || h_qk <= 0 || h_v <= 0 || h_v % h_qk != 0 || d_k <= 0 || d_v <= 0)
        return GDN_ERR_INVALID_ARG;
    if (!ok_dtype(dtype_qkv) || !ok_dtype(dtype_o)) return GDN_ERR_INVALID_ARG;
    if (d_k != gdn::kda::D || d_v != gdn::kda::D) return GDN_ERR_UNSUPPORTED;
    if (num_seqs == 0) return GDN_OK;
    const uintptr_t ei = esize(dtype_qkv), eo = esize(dtype_o);
    // q and k are read 4 elements at a time
    if (!ok_ptr(q, 4 * ei) || !ok_ptr(k, 4 * ei) || !ok_ptr(v, ei) || !ok_ptr(g, 4) || !ok_ptr(beta, 4) ||
        !ok_ptr(state, 16) || !ok_ptr(o, eo))
        return GDN_ERR_INVALID_ARG;
    if (scale == 0.f) scale = 1.0f / sqrtf((float)d_k);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool bi = dtype_qkv == GDN_BF16, bo = dtype_o == GDN_BF16;
    if (bi && bo)
        return launch_kda_decode<__nv_bfloat16, __nv_bfloat16>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, scale, s);
    if (bi) return launch_kda_decode<__nv_bfloat16, float>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, scale, s);
    if (bo) return launch_kda_decode<float, __nv_bfloat16>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, scale, s);
    return launch_kda_decode<float, float>(q, k, v, g, beta, state, o, num_seqs, h_qk, h_v, scale, s);
}

#ifdef GDN_TRACE
// Instrumented builds only (not part of the ABI): device buffer of 64 x 128
// clock64 stamps that the prefill kernel's block 0 fills per role and chunk.
int gdn_debug_set_trace(unsigned long long* buf) {
    return cudaMemcpyToSymbol(gdn::tck::g_trace, &buf, sizeof buf) == cudaSuccess ? 0 : 3;
}
#endif

}  // extern "C"
