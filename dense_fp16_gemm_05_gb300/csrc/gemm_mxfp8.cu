// gemm_mxfp8.cu -- host-side launch of the FP8 GEMM with power-of-two block
// scales (gemm_mxfp8_kernel.cuh).  The C ABI entry, gemm_mxfp8_block_scaled in
// gemm_f16.cu, validates every argument and calls launch_mxfp8.
#include "gemm_fp8_launch.cuh"

#include "gemm_mxfp8_kernel.cuh"

namespace gemm_sm103 {

namespace {

// Per device and ReLU variant: the shared-memory attribute is set once and
// the number of co-resident CTA pairs cached (one CTA per SM).
template <bool kRelu>
struct MxPrepared {
    static std::atomic<int> slots[kMaxDevices];

    static int get(int dev, int sm_count)
    {
        int v = slots[dev].load(std::memory_order_acquire);
        if (v > 0) return v;
        auto kern = gemm_mxfp8_sm103a<kRelu>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, MxCfg::SMEM_BYTES) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        v = sm_count / 2;
        cudaLaunchConfig_t lc{};
        lc.blockDim = dim3(MxCfg::THREADS, 1, 1);
        lc.dynamicSmemBytes = MxCfg::SMEM_BYTES;
        lc.gridDim = dim3(2 * v, 1, 1);
        cudaLaunchAttribute attrs[1];
        attrs[0].id = cudaLaunchAttributeClusterDimension;
        attrs[0].val.clusterDim.x = 2;
        attrs[0].val.clusterDim.y = 1;
        attrs[0].val.clusterDim.z = 1;
        lc.attrs = attrs;
        lc.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &lc) == cudaSuccess && clusters > 0)
            v = clusters < v ? clusters : v;
        else
            cudaGetLastError();
        if (v > 0) slots[dev].store(v, std::memory_order_release);
        return v;
    }

    static void forget(int dev) { slots[dev].store(0, std::memory_order_release); }
};

template <bool kRelu>
std::atomic<int> MxPrepared<kRelu>::slots[kMaxDevices];

template <bool kRelu>
int launch_mx_variant(const MxLaunchArgs &a)
{
    CUtensorMap ta, tw, tc;
    int st;
    // A (M,K) and W (N,K): one-byte elements; per CTA and K block an A box of
    // 128 (K) x 128 rows and a W box of 128 (K) x 128 rows.
    if ((st = encode_matrix_u8(&ta, a.A, a.M, a.K, MxCfg::BK, MxCfg::BM)) != GEMM_OK) return st;
    if ((st = encode_matrix_u8(&tw, a.W, a.N, a.K, MxCfg::BK, MxCfg::BN_CTA)) != GEMM_OK) return st;
    if ((st = encode_matrix(&tc, a.C, a.M, a.N, MxCfg::EPI_COLS, 32)) != GEMM_OK) return st;

    MxParams p{};
    p.M = static_cast<int32_t>(a.M);
    p.N = static_cast<int32_t>(a.N);
    p.K = static_cast<int32_t>(a.K);
    p.num_m_blocks = static_cast<int32_t>((a.M + MxCfg::TILE_M - 1) / MxCfg::TILE_M);
    p.num_n_blocks = static_cast<int32_t>((a.N + MxCfg::BN - 1) / MxCfg::BN);
    p.num_k_blocks = static_cast<int32_t>((a.K + MxCfg::BK - 1) / MxCfg::BK);
    p.num_w_blocks = static_cast<int32_t>((a.N + MxCfg::SCALE_BLOCK - 1) / MxCfg::SCALE_BLOCK);
    const int64_t tiles = static_cast<int64_t>(p.num_m_blocks) * p.num_n_blocks;
    if (tiles > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    p.num_tiles = static_cast<int32_t>(tiles);
    p.group_m = 8;   // 2048-row panels, as the fp16 kernels
    p.timeout_cycles = a.timeout_cycles ? a.timeout_cycles : timeout_cycles_for(a.K);
    p.SA = a.SA;
    p.SW = a.SW;
    p.status = a.status;

    using Prep = MxPrepared<kRelu>;
    const int64_t slots = Prep::get(a.dev.device, a.dev.sm_count);
    if (slots <= 0) return GEMM_ERR_LAUNCH;
    const int64_t clusters = tiles < slots ? tiles : slots;
    auto kern = gemm_mxfp8_sm103a<kRelu>;
    cudaLaunchConfig_t lc{};
    lc.blockDim = dim3(MxCfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = MxCfg::SMEM_BYTES;
    lc.stream = a.stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 2;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // programmatic dependent launch
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attrs;
    lc.numAttrs = 2;
    lc.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
    if (cudaLaunchKernelEx(&lc, kern, ta, tw, tc, p) != cudaSuccess) {
        cudaGetLastError();
        Prep::forget(a.dev.device);
        if (Prep::get(a.dev.device, a.dev.sm_count) <= 0 || cudaLaunchKernelEx(&lc, kern, ta, tw, tc, p) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    }
    return GEMM_OK;
}

}  // namespace

int launch_mxfp8(const MxLaunchArgs &a)
{
    return a.relu ? launch_mx_variant<true>(a) : launch_mx_variant<false>(a);
}

}  // namespace gemm_sm103
