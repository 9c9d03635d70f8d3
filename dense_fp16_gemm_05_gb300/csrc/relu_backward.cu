// relu_backward.cu -- gradient of the fused ReLU epilogue: dZ = dC where C > 0,
// else +0, for the backward pass of C = ReLU(A @ B) (the pre-activation
// Z = A @ B is not stored; its sign is read from the stored output C).
//
// The backward pair of the autograd wrapper in "TileLang-MUSA operator
// development" (7yue.com, section 6) is dA = dC @ B^T and dB = A^T @ dC for the
// plain product; with the fused ReLU the incoming gradient is first masked by
// this kernel, then the same pair is applied to dZ.
//
// HBM-bound: per element 2 bytes of dC and 2 of C read, 2 bytes of dZ written.
// The test "C > 0" is made on the binary16 bit pattern: positive, nonzero and
// not NaN, i.e. 0x0001 <= bits <= 0x7C00 (+inf counts as positive).  Vector
// path: 16-byte loads and stores of 8 elements, grid-stride loop over a grid
// of a few CTAs per SM; any tail (or misaligned buffers) takes the scalar path.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_f16.h"
#include "gemm_launch.cuh"

namespace {

__device__ __forceinline__ uint32_t mask_pair(uint32_t c2, uint32_t g2)
{
    const uint32_t lo = c2 & 0xFFFFu, hi = c2 >> 16;
    const uint32_t keep_lo = (lo >= 1u && lo <= 0x7C00u) ? 0x0000FFFFu : 0u;
    const uint32_t keep_hi = (hi >= 1u && hi <= 0x7C00u) ? 0xFFFF0000u : 0u;
    return g2 & (keep_lo | keep_hi);
}

__global__ void __launch_bounds__(256) relu_backward_vec_kernel(const uint4 *__restrict__ dC,
                                                                const uint4 *__restrict__ C, uint4 *__restrict__ dZ,
                                                                int64_t n_vec)
{
    gemm_sm103::griddep_wait();   // dC and C may come from the kernel just before
    gemm_sm103::griddep_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
        const uint4 c = C[i];
        const uint4 g = dC[i];
        uint4 z;
        z.x = mask_pair(c.x, g.x);
        z.y = mask_pair(c.y, g.y);
        z.z = mask_pair(c.z, g.z);
        z.w = mask_pair(c.w, g.w);
        dZ[i] = z;
    }
}

__global__ void __launch_bounds__(256) relu_backward_scalar_kernel(const uint16_t *__restrict__ dC,
                                                                   const uint16_t *__restrict__ C,
                                                                   uint16_t *__restrict__ dZ, int64_t begin,
                                                                   int64_t n)
{
    gemm_sm103::griddep_wait();
    gemm_sm103::griddep_launch_dependents();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint32_t c = C[i];
        dZ[i] = (c >= 1u && c <= 0x7C00u) ? dC[i] : static_cast<uint16_t>(0);
    }
}

}  // namespace

namespace gemm_sm103 {

namespace {

// Launch as a programmatic dependent of the previous kernel on the stream
// (the kernels wait for it before touching memory).
template <class... Args>
int launch_pdl(void (*kern)(Args...), int64_t blocks, cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    lc.blockDim = dim3(256, 1, 1);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, kern, args...) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace

int relu_backward_launch(const void *dC, const void *C, void *dZ, int64_t n, int sm_count, cudaStream_t stream)
{
    const bool aligned = ((reinterpret_cast<uintptr_t>(dC) | reinterpret_cast<uintptr_t>(C) |
                           reinterpret_cast<uintptr_t>(dZ)) & 15u) == 0;
    const int64_t n_vec = aligned ? n / 8 : 0;
    const int64_t max_blocks = static_cast<int64_t>(sm_count) * 8;   // 8 CTAs of 256 threads per SM
    if (n_vec > 0) {
        int64_t blocks = (n_vec + 255) / 256;
        if (blocks > max_blocks) blocks = max_blocks;
        const int st = launch_pdl(relu_backward_vec_kernel, blocks, stream, static_cast<const uint4 *>(dC),
                                  static_cast<const uint4 *>(C), static_cast<uint4 *>(dZ), n_vec);
        if (st != GEMM_OK) return st;
    }
    const int64_t done = n_vec * 8;
    if (done < n) {
        int64_t blocks = (n - done + 255) / 256;
        if (blocks > max_blocks) blocks = max_blocks;
        const int st = launch_pdl(relu_backward_scalar_kernel, blocks, stream, static_cast<const uint16_t *>(dC),
                                  static_cast<const uint16_t *>(C), static_cast<uint16_t *>(dZ), done, n);
        if (st != GEMM_OK) return st;
    }
    return GEMM_OK;
}

}  // namespace gemm_sm103
