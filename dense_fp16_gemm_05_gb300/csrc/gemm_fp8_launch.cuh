// gemm_fp8_launch.cuh -- internal interface between the C ABI (gemm_f16.cu) and the
// FP8 block-scaled GEMM launch (gemm_fp8.cu).
#pragma once

#include "gemm_launch.cuh"

namespace gemm_sm103 {

// Everything one FP8 launch needs, already validated by the C ABI.
struct Fp8LaunchArgs {
    const void *A = nullptr;     // (M,K) E4M3
    const float *SA = nullptr;   // (M, ceil(K/128))
    const void *W = nullptr;     // (N,K) E4M3
    const float *SW = nullptr;   // (ceil(N/128), ceil(K/128))
    void *C = nullptr;           // (M,N) fp16
    int64_t M = 0, N = 0, K = 0;
    int relu = 1;
    DeviceInfo dev;
    cudaStream_t stream = nullptr;
    unsigned long long *status = nullptr;
    uint64_t timeout_cycles = 0;   // 0: the normal budget
};

// Row-major one-byte-element matrix rows x cols, boxes of box_cols x box_rows
// with 128-byte swizzle (defined in gemm_f16.cu).
int encode_matrix_u8(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                     uint32_t box_rows);

int launch_fp8(const Fp8LaunchArgs &a);

// Everything one launch of the power-of-two-scale FP8 GEMM needs, already
// validated by the C ABI.
struct MxLaunchArgs {
    const void *A = nullptr;      // (M,K) E4M3
    const uint8_t *SA = nullptr;  // (M, ceil(K/128)) E8M0 exponents
    const void *W = nullptr;      // (N,K) E4M3
    const uint8_t *SW = nullptr;  // (ceil(N/128), ceil(K/128)) E8M0 exponents
    void *C = nullptr;            // (M,N) fp16
    int64_t M = 0, N = 0, K = 0;
    int relu = 1;
    DeviceInfo dev;
    cudaStream_t stream = nullptr;
    unsigned long long *status = nullptr;
    uint64_t timeout_cycles = 0;
};

int launch_mxfp8(const MxLaunchArgs &a);
int fp8_launch_info(int64_t M, int64_t N, const DeviceInfo &dev, int *grid_ctas, int *tiles);

}  // namespace gemm_sm103
