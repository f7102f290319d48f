// Output epilogue of a GDN layer: zero-centred RMSNorm of each row (one token
// of one value head, d features) times a sigmoid gate,
//     y = o / sqrt(mean_j o_j^2 + eps) * (1 + w) * sigmoid(z).
// The pages name the two pieces ("a sigmoid output gate, zero-centered
// RMSNorm", "Qwen3.8-Next design: hybrid attention, residuals and n-gram
// embeddings", transcript segment 14; the gate sigma(x W_g) (.) o in the
// component list of "Qwen3.8 attention gate"); the norm comes first and the
// gate multiplies its result, w is the zero-centred per-feature weight shared
// by all heads, and z (= x W_g) is the caller's.
//
// Standalone kernel (after the prefill, or on any [rows, d] tensor): one warp
// per row, one warp-shuffle reduction.
// It moves 3 values per feature (o and z in, y out) and is HBM-bound.
#pragma once

#include "gdn_common.cuh"

namespace gdn {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float sigmoid_f(float z) { return sigmoid_fast(z); }

// Rows r = blockIdx.x * 8 + warp (grid-strided); lane l owns features
// l + 32 m, m < NV (NV = the smallest of 4, 8, 16, 32 with 32 NV >= d).
template <typename TX, typename TZ, typename TY, int NV>
__global__ void __launch_bounds__(256)
gated_rmsnorm_kernel(const TX* x, const TZ* __restrict__ z, const float* __restrict__ w,
                     TY* y, long long rows, int d, float eps) {
    const int lane = threadIdx.x & 31;
    const float inv_d = 1.0f / (float)d;
    for (long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5); row < rows;
         row += (long long)gridDim.x * 8) {
        const TX* xr = x + row * d;
        const TZ* zr = z + row * d;
        // rows of up to 256 features stay in registers; longer ones are read
        // twice (the second read hits L1/L2)
        constexpr int NC = NV <= 8 ? NV : 1;
        float xv[NC];
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const int i = lane + 32 * m;
            const float xi = i < d ? to_f32(xr[i]) : 0.f;
            if (NV <= 8) xv[m < NC ? m : 0] = xi;
            ss = fmaf(xi, xi, ss);
        }
        const float rinv = rsqrtf(fmaf(warp_sum(ss), inv_d, eps));
        TY* yr = y + row * d;
#pragma unroll
        for (int m = 0; m < NV; ++m) {
            const int i = lane + 32 * m;
            if (i < d) {
                const float xi = NV <= 8 ? xv[m < NC ? m : 0] : to_f32(xr[i]);
                const float scale = w ? 1.0f + w[i] : 1.0f;
                yr[i] = from_f32<TY>(xi * rinv * scale * sigmoid_f(to_f32(zr[i])));
            }
        }
    }
}

// Four consecutive elements as fp32 (one 8- or 16-byte load).
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float4 load4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t*>(&a);
    u.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = u;
}
__device__ __forceinline__ void store4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// d = 128 with 16-byte aligned bases: lane l owns features 4l .. 4l + 3 of a
// row (one vector load of x and of z), and each warp keeps R = 4 rows in
// flight so that enough bytes are outstanding per SM to reach HBM bandwidth.
template <typename TX, typename TZ, typename TY>
__global__ void __launch_bounds__(256)
gated_rmsnorm_d128_kernel(const TX* x, const TZ* __restrict__ z, const float* __restrict__ w, TY* y,
                          long long rows, float eps) {
    constexpr int D = 128, R = 4;
    const int lane = threadIdx.x & 31;
    float4 ws = w ? *reinterpret_cast<const float4*>(w + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    ws.x += 1.0f; ws.y += 1.0f; ws.z += 1.0f; ws.w += 1.0f;  // zero-centred weight -> scale
    const long long warps = (long long)gridDim.x * 8;
    for (long long r0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * R; r0 < rows; r0 += warps * R) {
        float4 xv[R], zv[R];
        float ss[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const long long row = r0 + i < rows ? r0 + i : rows - 1;  // tail rows repeat the last row
            xv[i] = load4(x + row * D + 4 * lane);
            zv[i] = load4(z + row * D + 4 * lane);
        }
#pragma unroll
        for (int i = 0; i < R; ++i)
            ss[i] = xv[i].x * xv[i].x + xv[i].y * xv[i].y + xv[i].z * xv[i].z + xv[i].w * xv[i].w;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int i = 0; i < R; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if (r0 + i >= rows) break;
            const float rinv = rsqrtf(fmaf(ss[i], 1.0f / D, eps));
            float4 o;
            o.x = xv[i].x * (rinv * ws.x) * sigmoid_f(zv[i].x);
            o.y = xv[i].y * (rinv * ws.y) * sigmoid_f(zv[i].y);
            o.z = xv[i].z * (rinv * ws.z) * sigmoid_f(zv[i].z);
            o.w = xv[i].w * (rinv * ws.w) * sigmoid_f(zv[i].w);
            store4(y + (r0 + i) * D + 4 * lane, o);
        }
    }
}

}  // namespace gdn
