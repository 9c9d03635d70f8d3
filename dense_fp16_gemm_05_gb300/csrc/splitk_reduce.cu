// splitk_reduce.cu -- second step of a K-split GEMM: C = R(sum_s P_s) where P_s
// (s = 0 .. splits-1) are the fp32 partial products of K slice s that the GEMM
// kernel wrote to its workspace, R the optional ReLU (x > 0 ? x : +0), and the
// result is rounded once to fp16 (round to nearest even), as the one-pass
// epilogue does.  The slices are added in ascending order, so the result does
// not depend on which CTA finished first.
//
// HBM/L2-bound: per output element 4 bytes per slice read, 2 bytes written.
// 16-byte accesses (8 outputs per thread and iteration: two float4 per slice,
// one uint4 of fp16); M * N is a multiple of 8 (N is), so there is no tail.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <cstdint>

#include "gemm_f16.h"
#include "gemm_launch.cuh"

namespace {

template <bool kRelu>
__device__ __forceinline__ float reduce_out(float x)
{
    if constexpr (kRelu) return x > 0.0f ? x : 0.0f;   // -0, NaN and negatives give +0
    else return x;
}

template <bool kRelu>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float4 *__restrict__ ws, uint4 *__restrict__ C,
                                                            int64_t n_vec, int64_t slice_vec4, int splits)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
        float4 lo = ws[2 * i], hi = ws[2 * i + 1];
        for (int s = 1; s < splits; ++s) {
            const float4 a = ws[s * slice_vec4 + 2 * i];
            const float4 b = ws[s * slice_vec4 + 2 * i + 1];
            lo.x += a.x;
            lo.y += a.y;
            lo.z += a.z;
            lo.w += a.w;
            hi.x += b.x;
            hi.y += b.y;
            hi.z += b.z;
            hi.w += b.w;
        }
        const __half2 h0 = __floats2half2_rn(reduce_out<kRelu>(lo.x), reduce_out<kRelu>(lo.y));
        const __half2 h1 = __floats2half2_rn(reduce_out<kRelu>(lo.z), reduce_out<kRelu>(lo.w));
        const __half2 h2 = __floats2half2_rn(reduce_out<kRelu>(hi.x), reduce_out<kRelu>(hi.y));
        const __half2 h3 = __floats2half2_rn(reduce_out<kRelu>(hi.z), reduce_out<kRelu>(hi.w));
        uint4 o;
        o.x = *reinterpret_cast<const uint32_t *>(&h0);
        o.y = *reinterpret_cast<const uint32_t *>(&h1);
        o.z = *reinterpret_cast<const uint32_t *>(&h2);
        o.w = *reinterpret_cast<const uint32_t *>(&h3);
        C[i] = o;
    }
}

}  // namespace

namespace gemm_sm103 {

namespace {

// Scratch of gemm_f16_ex_noalloc (16 MiB per device): K-slice partials live
// here instead of in a stream-ordered allocation.  Nothing in it needs to
// start at zero: every element the reduction reads was written by the GEMM
// kernel of the same call.
constexpr size_t kNoallocScratchFloats = size_t{4} << 20;
static __device__ __align__(256) float g_noalloc_scratch[kNoallocScratchFloats];

std::atomic<float *> g_noalloc_ptr[kMaxDevices];

}  // namespace

int noalloc_scratch(int dev, float **ptr, size_t *bytes)
{
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    float *p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        // Once per device, outside any stream capture (the first call may
        // load the module's device data).
        void *sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_noalloc_scratch) != cudaSuccess || sym == nullptr) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        p = static_cast<float *>(sym);
        g_noalloc_ptr[dev].store(p, std::memory_order_release);
    }
    *ptr = p;
    *bytes = kNoallocScratchFloats * sizeof(float);
    return GEMM_OK;
}

int launch_splitk_reduce(const float *ws, void *C, int64_t M, int64_t N, int splits, int relu, int sm_count,
                         cudaStream_t stream)
{
    const int64_t elems = M * N;              // a multiple of 8
    const int64_t n_vec = elems / 8;
    if (n_vec == 0) return GEMM_OK;
    const int64_t want = (n_vec + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
    const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
    const float4 *w = reinterpret_cast<const float4 *>(ws);
    uint4 *c = static_cast<uint4 *>(C);
    if (relu) splitk_reduce_kernel<true><<<blocks, 256, 0, stream>>>(w, c, n_vec, elems / 4, splits);
    else splitk_reduce_kernel<false><<<blocks, 256, 0, stream>>>(w, c, n_vec, elems / 4, splits);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
    return GEMM_OK;
}

}  // namespace gemm_sm103
