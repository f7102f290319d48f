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

// sigmoid(z) = 1 / (1 + 2^(-z log2 e)) on the special-function unit (PTX
// ex2.approx.ftz and rcp.approx.ftz, each within a few ulp): exactly 0 for
// z -> -inf (the reciprocal of +inf) and 1 for z -> +inf.
__device__ __forceinline__ float sigmoid_fast(float z) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-1.4426950408889634f * z));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return r;
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
// Raw 4-element vectors (kept packed until used: fewer registers, more rows
// in flight per SM).
template <typename T> struct Vec4;
template <> struct Vec4<__nv_bfloat16> { using type = uint2; };
template <> struct Vec4<float> { using type = float4; };
template <typename T>
__device__ __forceinline__ typename Vec4<T>::type load_raw4(const T* p) {
    return *reinterpret_cast<const typename Vec4<T>::type*>(p);
}
__device__ __forceinline__ float4 unpack4(uint2 u) {
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
__device__ __forceinline__ float4 unpack4(float4 f) { return f; }

// d = 128 with 16-byte aligned bases: lane l owns features 4l .. 4l + 3 of a
// row (one vector load of x and of z), and each warp keeps R = 4 rows in
// flight (raw vectors until used) so that enough bytes are outstanding per SM
// to reach HBM bandwidth.
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
        typename Vec4<TX>::type xr[R];
        typename Vec4<TZ>::type zr[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const long long row = r0 + i < rows ? r0 + i : rows - 1;  // tail rows repeat the last row
            xr[i] = load_raw4(x + row * D + 4 * lane);
            zr[i] = load_raw4(z + row * D + 4 * lane);
        }
        float ss[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const float4 v = unpack4(xr[i]);
            ss[i] = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
            for (int i = 0; i < R; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if (r0 + i >= rows) break;
            const float rinv = rsqrtf(fmaf(ss[i], 1.0f / D, eps));
            const float4 v = unpack4(xr[i]), g = unpack4(zr[i]);
            float4 o;
            o.x = v.x * (rinv * ws.x) * sigmoid_f(g.x);
            o.y = v.y * (rinv * ws.y) * sigmoid_f(g.y);
            o.z = v.z * (rinv * ws.z) * sigmoid_f(g.z);
            o.w = v.w * (rinv * ws.w) * sigmoid_f(g.w);
            store4(y + (r0 + i) * D + 4 * lane, o);
        }
    }
}

}  // namespace gdn
