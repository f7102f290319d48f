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
// Standalone kernels (after the prefill, or on any [rows, d] tensor): a
// half-warp per row of 128 (16-byte accesses), one warp per row otherwise.
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

// Eight consecutive elements as raw 32-bit words (one 16-byte load of bf16,
// two of fp32) and their fp32 values.
template <typename T> struct Raw8 { uint32_t u[4 * (int)sizeof(T) / 2]; };
template <typename T> __device__ __forceinline__ Raw8<T> load_raw8(const T* p) {
    Raw8<T> r;
#pragma unroll
    for (int i = 0; i < 2 * (int)sizeof(T); i += 4) {
        const uint4 a = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const uint32_t*>(p) + i));
        r.u[i] = a.x; r.u[i + 1] = a.y; r.u[i + 2] = a.z; r.u[i + 3] = a.w;
    }
    return r;
}
__device__ __forceinline__ float raw8_val(const Raw8<__nv_bfloat16>& r, int j) {
    return __uint_as_float((j & 1) ? (r.u[j >> 1] & 0xffff0000u) : (r.u[j >> 1] << 16));
}
__device__ __forceinline__ float raw8_val(const Raw8<float>& r, int j) { return __uint_as_float(r.u[j]); }
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float* v) {
    uint4 u;
    uint32_t* w = reinterpret_cast<uint32_t*>(&u);
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * h], v[2 * h + 1]);
        w[h] = *reinterpret_cast<uint32_t*>(&b);
    }
    __stcs(reinterpret_cast<uint4*>(p), u);
}
__device__ __forceinline__ void store8(float* p, const float* v) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[4], v[5], v[6], v[7]));
}

// d = 128 with 16-byte aligned bases: a half-warp per row, lane l owning
// features 8 (l % 16) .. + 7 (one 16-byte load of x and of z for bf16), the
// sum of squares reduced in four shuffles inside the half-warp. Each warp
// takes R row pairs per iteration and issues all their loads before any
// arithmetic, with streaming (evict-first) loads and stores: every byte is
// touched once.
template <typename TX, typename TZ, typename TY>
__global__ void __launch_bounds__(256)
gated_rmsnorm_d128_kernel(const TX* x, const TZ* __restrict__ z, const float* __restrict__ w, TY* y,
                          long long rows, float eps) {
    constexpr int D = 128, R = 2;
    const int lane = threadIdx.x & 31, hl = lane & 15, half = lane >> 4;
    float ws[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ws[j] = 1.0f + (w ? w[8 * hl + j] : 0.f);  // zero-centred weight -> scale
    const long long warps = (long long)gridDim.x * 8;
    for (long long r0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * (2 * R); r0 < rows;
         r0 += warps * (2 * R)) {
        Raw8<TX> xr[R];
        Raw8<TZ> zr[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            long long row = r0 + 2 * i + half;
            row = row < rows ? row : rows - 1;  // tail rows repeat the last row (not stored)
            xr[i] = load_raw8(x + row * D + 8 * hl);
            zr[i] = load_raw8(z + row * D + 8 * hl);
        }
        float ss[R];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float a = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) a = fmaf(raw8_val(xr[i], j), raw8_val(xr[i], j), a);
            ss[i] = a;
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
#pragma unroll
            for (int i = 0; i < R; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], off);
        }
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const long long row = r0 + 2 * i + half;
            const float rinv = rsqrtf(fmaf(ss[i], 1.0f / D, eps));
            float o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = raw8_val(xr[i], j) * (rinv * ws[j]) * sigmoid_f(raw8_val(zr[i], j));
            if (row < rows) store8(y + row * D + 8 * hl, o);
        }
    }
}

}  // namespace gdn
