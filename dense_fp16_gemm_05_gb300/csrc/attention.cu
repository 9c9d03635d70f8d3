// attention.cu -- host-side launch of the attention-forward kernel
// (attention_kernel.cuh).  The C ABI entry, attention_fwd_f16 in gemm_f16.cu,
// validates every argument and calls launch_attention.
#include "attention_launch.cuh"

#include <cmath>

#include "attention_kernel.cuh"

namespace gemm_sm103 {

namespace {

template <int kDim>
struct AttnPrepared {
    static std::atomic<int> ready[kMaxDevices];

    static bool get(int dev)
    {
        if (ready[dev].load(std::memory_order_acquire)) return true;
        if (cudaFuncSetAttribute(attention_fwd_sm103a<kDim>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 AttnCfg<kDim>::SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        ready[dev].store(1, std::memory_order_release);
        return true;
    }

    static void forget(int dev) { ready[dev].store(0, std::memory_order_release); }
};

template <int kDim>
std::atomic<int> AttnPrepared<kDim>::ready[kMaxDevices];

template <int kDim>
int launch_dim(const AttnLaunchArgs &a)
{
    using Cfg = AttnCfg<kDim>;
    const uint64_t bh = static_cast<uint64_t>(a.batch) * static_cast<uint64_t>(a.heads);
    CUtensorMap tq, tk, tv;
    int st;
    if ((st = encode_bhsd(&tq, a.Q, bh, a.seq, kDim)) != GEMM_OK) return st;
    if ((st = encode_bhsd(&tk, a.K, bh, a.seq, kDim)) != GEMM_OK) return st;
    if ((st = encode_bhsd(&tv, a.V, bh, a.seq, kDim)) != GEMM_OK) return st;
    AttnParams p{};
    p.batch = static_cast<int32_t>(a.batch);
    p.heads = static_cast<int32_t>(a.heads);
    p.seq = static_cast<int32_t>(a.seq);
    p.num_q_blocks = static_cast<int32_t>((a.seq + Cfg::BQ - 1) / Cfg::BQ);
    p.causal = a.causal;
    p.scale_log2 = static_cast<float>(static_cast<double>(a.sm_scale) * 1.4426950408889634);   // log2(e)
    p.timeout_cycles = timeout_cycles_for(a.seq * kDim);
    p.O = static_cast<__half *>(a.O);
    p.status = a.status;
    if (!AttnPrepared<kDim>::get(a.dev.device)) return GEMM_ERR_LAUNCH;
    // A persistent grid: one CTA per SM (the kernel's shared memory and TMEM
    // admit one).  With the work queue (causal only) each CTA starts with one
    // item and then takes tickets; otherwise each walks every G-th super-item
    // (with the causal mask two pairs of query blocks of one head and batch,
    // else one; see the kernel).
    const int64_t n_grp = (p.num_q_blocks + Cfg::TILES - 1) / Cfg::TILES;
    const bool use_queue = a.causal && a.queue != nullptr;
    p.queue = use_queue ? a.queue : nullptr;
    // Heads per group of the queue's order: about 32 MiB of K and V (16 heads
    // at seq 4096, dim 128), so that the groups in flight at once stay in L2.
    // Measured at 4 x 32 x 4096 x 128, causal: 16 MiB 1347 TFLOP/s, 32 MiB
    // 1373, 64 MiB 1357, 128 MiB 1320 (dim 64: 815 for all four).
    const int64_t kv_head_bytes = 2 * a.seq * kDim * 2;
    const int64_t chunk = (int64_t{32} << 20) / kv_head_bytes;
    p.chunk_heads = static_cast<int32_t>(chunk < 8 ? 8 : (chunk > 64 ? 64 : chunk));
    const int64_t units = use_queue ? n_grp * a.heads * a.batch : (a.causal ? (n_grp + 1) / 2 : n_grp) * a.heads * a.batch;
    const dim3 grid(static_cast<unsigned>(units < a.dev.sm_count ? units : a.dev.sm_count), 1, 1);
    cudaLaunchConfig_t lc{};
    lc.gridDim = grid;
    lc.blockDim = dim3(Cfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // programmatic dependent launch
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    if (cudaLaunchKernelEx(&lc, attention_fwd_sm103a<kDim>, tq, tk, tv, p) != cudaSuccess) {
        AttnPrepared<kDim>::forget(a.dev.device);
        return GEMM_ERR_LAUNCH;
    }
    return GEMM_OK;
}

}  // namespace

int launch_attention(const AttnLaunchArgs &a)
{
    return a.dim == 64 ? launch_dim<64>(a) : launch_dim<128>(a);
}

}  // namespace gemm_sm103
