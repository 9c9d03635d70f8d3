// attention_launch.cuh -- internal interface between the C ABI (gemm_f16.cu)
// and the attention-forward launch (attention.cu).
#pragma once

#include "gemm_launch.cuh"

namespace gemm_sm103 {

struct AttnLaunchArgs {
    const void *Q = nullptr, *K = nullptr, *V = nullptr;   // (batch, heads, seq, dim) fp16
    void *O = nullptr;
    int64_t batch = 0, heads = 0, seq = 0, dim = 0;
    float sm_scale = 1.0f;
    int causal = 0;
    DeviceInfo dev;
    cudaStream_t stream = nullptr;
    unsigned long long *status = nullptr;
    unsigned int *queue = nullptr;   // caller's work queue (two zero words), or null
};

// (batch * heads, seq, dim) fp16 tensor as a 3-D tensor map with boxes of
// 64 (dim) x 128 (seq) x 1 and 128-byte swizzle (defined in gemm_f16.cu).
int encode_bhsd(CUtensorMap *map, const void *ptr, uint64_t bh, uint64_t seq, uint64_t dim);

int launch_attention(const AttnLaunchArgs &a);

}  // namespace gemm_sm103
