// Tensor-core (tcgen05/TMEM, TMA-fed) chunkwise prefill: placeholder until the
// kernel lands; the dispatcher falls back to the CUDA-core kernel.
#pragma once

#include "gdn_common.cuh"

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

inline bool tc_available() { return false; }
inline gdn_status launch_tc(const TcArgs&, bool, cudaStream_t) { return GDN_ERR_UNSUPPORTED; }

}  // namespace gdn
