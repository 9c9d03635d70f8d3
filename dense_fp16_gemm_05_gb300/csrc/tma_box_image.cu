// tma_box_image.cu -- layout diagnostic: one operand box of a row-major fp16
// matrix loaded by TMA into shared memory exactly as the GEMM's producer loads
// its A and B tiles (the same tensor-map encoding: 128-byte swizzle, zero fill
// outside the matrix; the same cp.async.bulk.tensor load completing on an
// mbarrier), then the raw shared-memory image copied out to global memory.
//
// The GEMM's MMA descriptors assume the 128-byte swizzle atom: row r of a box
// (128 bytes = 64 fp16) sits at byte r * 128 of the tile, and its 16-byte
// piece j at piece position j ^ (r % 8) within that row.  "Writing
// High-Performance Kernels in TileLang, from GEMM to MLA" states that shared
// tiles are laid out to avoid bank conflicts, and the nxmr.cn A100 article
// (sections 3.3 and 6.2) warns that a shared-memory layout that disagrees with
// the copy engine's swizzle misplaces data by 16 bytes.  This kernel lets a
// test compare the image TMA actually writes with that formula, so a layout
// error is seen directly instead of only through wrong GEMM results.
//
// Not on the GEMM's path; one CTA of 128 threads per call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_f16.h"
#include "gemm_launch.cuh"

namespace {

using namespace gemm_sm103;

constexpr int kImageThreads = 128;

// Box of box_rows x 128 bytes at (x, y) of the map into 1024-byte-aligned
// shared memory, then bytes / 16 uint4 of the image to out.  The wait for the
// load is bounded (limit SM clocks); on expiry the status word records
// kSiteBoxImage and the image is not copied (the load is given the same bound
// to land before the CTA exits).
__global__ void __launch_bounds__(kImageThreads) tma_box_image_kernel(const __grid_constant__ CUtensorMap map,
                                                                      int32_t x, int32_t y, uint32_t bytes,
                                                                      uint4 *out, uint64_t limit,
                                                                      unsigned long long *status)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // a whole number of 1024-byte swizzle atoms
    const uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t bar = base + bytes;               // 8-byte aligned: bytes is a multiple of 128
    __shared__ int ok_flag;
    griddep_wait();
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        prefetch_tensormap(&map);
        mbar_arrive_expect_tx(bar, bytes);
        tma_load_2d(base, &map, bar, x, y);
        const long long t0 = clock64();
        int ok = 1;
        while (!mbar_try_wait(bar, 0)) {
            if (static_cast<uint64_t>(clock64() - t0) > limit) {
                atomicCAS(status, 0ull, kSiteBoxImage | (static_cast<unsigned long long>(blockIdx.x) << 8));
                ok = 0;
                // Give the copy the same bound to land before the CTA exits.
                const long long t1 = clock64();
                while (!mbar_try_wait(bar, 0) && static_cast<uint64_t>(clock64() - t1) <= limit) {
                }
                break;
            }
        }
        ok_flag = ok;
    }
    __syncthreads();
    griddep_launch_dependents();
    if (!ok_flag) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(base_ptr);
    for (uint32_t i = threadIdx.x; i < bytes / 16u; i += kImageThreads) out[i] = src[i];
}

}  // namespace

namespace gemm_sm103 {

int tma_box_image_launch(const void *X, int64_t rows, int64_t cols, int box_rows, int x, int y, void *out,
                         unsigned long long *status, cudaStream_t stream)
{
    CUtensorMap map;
    // The GEMM's own encoding: boxes 64 fp16 (128 bytes) wide, SW128, zero fill.
    const int st = encode_matrix(&map, X, static_cast<uint64_t>(rows), static_cast<uint64_t>(cols), 64,
                                 static_cast<uint32_t>(box_rows));
    if (st != GEMM_OK) return st;
    const uint32_t bytes = static_cast<uint32_t>(box_rows) * 128u;
    const size_t smem = 1024 + bytes + 8;
    auto kern = tma_box_image_kernel;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(1, 1, 1);
    lc.blockDim = dim3(kImageThreads, 1, 1);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, kern, map, static_cast<int32_t>(x), static_cast<int32_t>(y), bytes,
                           static_cast<uint4 *>(out), static_cast<uint64_t>(1ull << 31), status) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace gemm_sm103
