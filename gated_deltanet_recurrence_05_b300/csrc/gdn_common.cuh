// Shared device helpers of the GDN library (one translation unit: gdn_lib.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Device error word (GDN_DEVERR_* bits), read and cleared by
// gdn_get_device_error(). One per device: each device that loads the library
// gets its own copy of this module variable.
__device__ unsigned int g_device_error;

__device__ __forceinline__ void set_device_error(unsigned int bits) {
    atomicOr(&g_device_error, bits);
}

// Element loads/stores for the two storage dtypes.
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Sequence bounds of sequence n: either from cu_seqlens or N equal lengths.
// Returns false (and records GDN_DEVERR_SEQLENS) if the entry is out of range.
__device__ __forceinline__ bool seq_bounds(const int32_t* cu, int n, int num_seqs,
                                           long long total, long long eq_len,
                                           long long& t0, long long& t1) {
    if (cu == nullptr) {
        t0 = (long long)n * eq_len;
        t1 = t0 + eq_len;
        return true;
    }
    t0 = cu[n];
    t1 = cu[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > total) {
        set_device_error(1u);
        return false;
    }
    return true;
}

// Resolve the scheduled position `pos` to a sequence index.
__device__ __forceinline__ bool seq_of(const int32_t* order, int pos, int num_seqs, int& n) {
    n = order ? order[pos] : pos;
    if (n < 0 || n >= num_seqs) {
        set_device_error(1u);
        return false;
    }
    return true;
}

}  // namespace gdn
