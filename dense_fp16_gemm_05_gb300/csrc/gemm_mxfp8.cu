// gemm_mxfp8.cu -- host-side launch of the FP8 GEMM with power-of-two block
// scales (gemm_mxfp8_kernel.cuh).  The C ABI entry, gemm_mxfp8_block_scaled in
// gemm_f16.cu, validates every argument and calls launch_mxfp8.
#include "gemm_fp8_launch.cuh"

#include "gemm_mxfp8_kernel.cuh"

namespace gemm_sm103 {

namespace {

// Per device and ReLU variant: the shared-memory attribute is set once (one
// CTA per SM, so the persistent grid is at most one CTA per SM).
template <bool kRelu>
struct MxPrepared {
    static std::atomic<int> ready[kMaxDevices];

    static bool get(int dev)
    {
        if (ready[dev].load(std::memory_order_acquire)) return true;
        if (cudaFuncSetAttribute(gemm_mxfp8_sm103a<kRelu>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 MxCfg::SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        ready[dev].store(1, std::memory_order_release);
        return true;
    }
};

template <bool kRelu>
std::atomic<int> MxPrepared<kRelu>::ready[kMaxDevices];

template <bool kRelu>
int launch_mx_variant(const MxLaunchArgs &a)
{
    CUtensorMap ta, tw, tc;
    int st;
    // A (M,K) and W (N,K): one-byte elements, boxes of 128 (K) x 128 and x 256 rows.
    if ((st = encode_matrix_u8(&ta, a.A, a.M, a.K, MxCfg::BK, MxCfg::BM)) != GEMM_OK) return st;
    if ((st = encode_matrix_u8(&tw, a.W, a.N, a.K, MxCfg::BK, MxCfg::BN)) != GEMM_OK) return st;
    if ((st = encode_matrix(&tc, a.C, a.M, a.N, MxCfg::EPI_COLS, 32)) != GEMM_OK) return st;

    MxParams p{};
    p.M = static_cast<int32_t>(a.M);
    p.N = static_cast<int32_t>(a.N);
    p.K = static_cast<int32_t>(a.K);
    p.num_m_blocks = static_cast<int32_t>((a.M + MxCfg::BM - 1) / MxCfg::BM);
    p.num_n_blocks = static_cast<int32_t>((a.N + MxCfg::BN - 1) / MxCfg::BN);
    p.num_k_blocks = static_cast<int32_t>((a.K + MxCfg::BK - 1) / MxCfg::BK);
    p.num_w_blocks = static_cast<int32_t>((a.N + MxCfg::SCALE_BLOCK - 1) / MxCfg::SCALE_BLOCK);
    const int64_t tiles = static_cast<int64_t>(p.num_m_blocks) * p.num_n_blocks;
    if (tiles > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    p.num_tiles = static_cast<int32_t>(tiles);
    p.group_m = 16;   // 2048-row panels, as the fp16 kernels
    p.timeout_cycles = a.timeout_cycles ? a.timeout_cycles : timeout_cycles_for(a.K);
    p.SA = a.SA;
    p.SW = a.SW;
    p.status = a.status;

    if (!MxPrepared<kRelu>::get(a.dev.device)) return GEMM_ERR_LAUNCH;
    const int64_t grid = tiles < a.dev.sm_count ? tiles : a.dev.sm_count;
    cudaLaunchConfig_t lc{};
    lc.blockDim = dim3(MxCfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = MxCfg::SMEM_BYTES;
    lc.stream = a.stream;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // programmatic dependent launch
    attrs[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attrs;
    lc.numAttrs = 1;
    lc.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    if (cudaLaunchKernelEx(&lc, gemm_mxfp8_sm103a<kRelu>, ta, tw, tc, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace

int launch_mxfp8(const MxLaunchArgs &a)
{
    return a.relu ? launch_mx_variant<true>(a) : launch_mx_variant<false>(a);
}

}  // namespace gemm_sm103
