// splitk_reduce.cu -- second step of a K-split GEMM: for every tile the GEMM
// kernel cut into K slices, C = R(sum_s P_s) over that tile, where P_s
// (s = 0 .. splits-1) are the fp32 partial products the slices wrote to the
// workspace (one SUPER_M x BN block per split tile and slice), R the optional
// ReLU (x > 0 ? x : +0), and the result is rounded once to fp16 (round to
// nearest even), as the one-pass epilogue does.  The slices are added in
// ascending order, so the result does not depend on which CTA finished first.
// Tiles are located with the GEMM's own rasterisation (tile_coords).
//
// HBM/L2-bound: per output element 4 bytes per slice read, 2 bytes written.
// 16-byte accesses (8 outputs per thread and iteration: two float4 per slice,
// one uint4 of fp16); N is a multiple of 8, so a group of 8 columns is wholly
// inside or outside C.
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
    else return __fadd_rn(x, 0.0f);                       // the cleared accumulator: -0 sums give +0
}

template <bool kRelu>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ ws, __half *__restrict__ C,
                                                            const gemm_sm103::GemmParams p, int super_m, int bn,
                                                            int64_t n_vec)
{
    // The partials come from the GEMM kernel just before this one on the
    // stream (launched as its programmatic dependent).
    gemm_sm103::griddep_wait();
    gemm_sm103::griddep_launch_dependents();
    const int64_t per_row = bn / 8;
    const int64_t per_tile = static_cast<int64_t>(super_m) * per_row;
    const int64_t tile_elems = static_cast<int64_t>(super_m) * bn;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
        const int64_t tr = i / per_tile;             // split tile, relative to ks_start
        const int64_t e = i - tr * per_tile;
        const int r = static_cast<int>(e / per_row);
        const int c = static_cast<int>(e - static_cast<int64_t>(r) * per_row) * 8;
        int mb, nb;
        gemm_sm103::tile_coords(p.ks_start + static_cast<int>(tr), p, mb, nb);
        const int64_t row = static_cast<int64_t>(mb) * super_m + r;
        const int64_t col = static_cast<int64_t>(nb) * bn + c;
        if (row >= p.M || col >= p.N) continue;
        const float *w = ws + tr * p.k_splits * tile_elems + static_cast<int64_t>(r) * bn + c;
        float4 lo = *reinterpret_cast<const float4 *>(w), hi = *reinterpret_cast<const float4 *>(w + 4);
        for (int sl = 1; sl < p.k_splits; ++sl) {
            const float4 a = *reinterpret_cast<const float4 *>(w + sl * tile_elems);
            const float4 b = *reinterpret_cast<const float4 *>(w + sl * tile_elems + 4);
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
        *reinterpret_cast<uint4 *>(C + row * p.N + col) = o;
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

int launch_splitk_reduce(const float *ws, void *C, const GemmParams &p, int super_m, int bn, int relu,
                         int sm_count, cudaStream_t stream)
{
    const int64_t split_tiles = static_cast<int64_t>(p.num_tiles) - p.ks_start;
    const int64_t n_vec = split_tiles * super_m * (bn / 8);
    if (n_vec <= 0) return GEMM_OK;
    const int64_t want = (n_vec + 255) / 256;
    const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;
    const unsigned blocks = static_cast<unsigned>(want < cap ? want : cap);
    __half *c = static_cast<__half *>(C);
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(blocks, 1, 1);
    lc.blockDim = dim3(256, 1, 1);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const cudaError_t e = relu ? cudaLaunchKernelEx(&lc, splitk_reduce_kernel<true>, ws, c, p, super_m, bn, n_vec)
                               : cudaLaunchKernelEx(&lc, splitk_reduce_kernel<false>, ws, c, p, super_m, bn, n_vec);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace gemm_sm103
