// gemm_launch.cuh -- host-side launch machinery shared by the per-configuration
// translation units (gemm_cfg_*.cu) and the C ABI (gemm_f16.cu): the persistent
// schedule, the per-device preparation cache, tensor-map encoding and the
// templated launch of gemm_f16_relu_sm103a.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gemm_f16.h"
#include "gemm_kernel.cuh"

namespace gemm_sm103 {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int device = 0;
    int supported = 0;      // compute capability 10.3
    int sm_count = 0;
};

// Test-hook settings for a launch (all zero for normal calls).
struct LaunchHook {
    int producer_off = 0;          // producer issues nothing
    uint64_t timeout_cycles = 0;   // 0: the normal budget
};

// Everything one launch needs, already validated by the C ABI.
struct LaunchArgs {
    const void *A = nullptr;
    const void *B = nullptr;
    void *C = nullptr;
    int64_t M = 0, N = 0, K = 0;
    int relu = 1;
    int transa = 0;        // 1: A stored (K,M) row-major, op(A) = stored^T
    int transb = 0;        // 1: B stored (N,K) row-major, op(B) = stored^T
    DeviceInfo dev;
    cudaStream_t stream = nullptr;
    LaunchHook hook;
    unsigned long long *status = nullptr;   // device status word of this GPU
    bool allow_split = true;   // false: every work unit is a whole tile (no tail split)
    int k_splits = 1;          // > 1: split every tile's K loop into (up to) this many slices,
                               // fp32 partials in a stream-ordered workspace, then a reduction
    bool k_split_tail = false; // split only the tiles of a partly filled last wave in K
    int ck_request = 0;        // cluster K split configurations: 0 = the size rule, 1 = no split,
                               // 2 / 4 / 8 = that many CTAs per cluster (fewer if K is short)
    bool noalloc = false;      // never allocate: K-slice partials go to the library's fixed
                               // scratch (noalloc_scratch); a split that does not fit it is
                               // rejected before anything is launched
};

// Defined in gemm_f16.cu.
int encode_matrix(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows);
int group_m_override();

// For every tile from p.ks_start on: C = R(sum of its p.k_splits fp32 partial
// tiles in ws), fp16 (splitk_reduce.cu).
int launch_splitk_reduce(const float *ws, void *C, const GemmParams &p, int super_m, int bn, int relu,
                         int sm_count, cudaStream_t stream);

// Device address and size of the fixed K-slice scratch of gemm_f16_ex_noalloc
// on device `dev` (splitk_reduce.cu).
int noalloc_scratch(int dev, float **ptr, size_t *bytes);

// K slices for a requested split count: `per` K blocks each, `count` of them
// (count <= requested; every slice non-empty).  count == 1: no K split.
struct KSplit {
    int count = 1;
    int per = 0;
};

inline KSplit k_split_for(int64_t k_blocks, int requested);

// Which tiles a launch cuts into K slices, and into how many: with a requested
// count (k_req >= 2) every tile; with `tail` only the tiles of a partly filled
// last wave (as many slices as fill the slots once, at most 8, at least 8 K
// blocks each); otherwise none (ks_start = tiles).
struct KPlan {
    KSplit ks;
    int64_t ks_start = 0;
    int64_t units(int64_t tiles) const { return ks_start + (tiles - ks_start) * ks.count; }
    int64_t ws_floats(int64_t tiles, int64_t tile_m, int64_t tile_n) const
    {
        return ks.count > 1 ? (tiles - ks_start) * ks.count * tile_m * tile_n : 0;
    }
};

inline KPlan plan_k_split(int64_t tiles, int64_t slots, int64_t k_blocks, int k_req, bool tail)
{
    KPlan kp;
    kp.ks.count = 1;
    kp.ks.per = static_cast<int>(k_blocks);
    kp.ks_start = tiles;
    if (k_req > 1) {
        const KSplit ks = k_split_for(k_blocks, k_req);
        if (ks.count > 1) {
            kp.ks = ks;
            kp.ks_start = 0;
        }
    } else if (tail && slots > 0) {
        const int64_t full = (tiles / slots) * slots, rest = tiles - full;
        int64_t n = rest > 0 ? slots / rest : 0;
        if (n > 8) n = 8;
        if (n > k_blocks / 8) n = k_blocks / 8;
        if (n >= 2) {
            const KSplit ks = k_split_for(k_blocks, static_cast<int>(n));
            if (ks.count > 1) {
                kp.ks = ks;
                kp.ks_start = full;
            }
        }
    }
    return kp;
}

inline KSplit k_split_for(int64_t k_blocks, int requested)
{
    KSplit ks;
    ks.per = static_cast<int>(k_blocks);
    if (requested > 1 && k_blocks >= 2) {
        const int64_t per = (k_blocks + requested - 1) / requested;
        ks.per = static_cast<int>(per);
        ks.count = static_cast<int>((k_blocks + per - 1) / per);
    }
    return ks;
}

inline uint64_t timeout_cycles_for(int64_t K)
{
    // About a second of SM clocks plus a margin that grows with the K loop of
    // one tile; a legitimate wait is at most one tile's mainloop.
    return (1ull << 31) + 64ull * static_cast<uint64_t>(K);
}

// Per device and kernel instance, prepared once: the dynamic shared-memory
// attribute is set, and the number of CTAs (or CTA clusters) of this
// configuration that can be resident at once -- one per SM, or per group of
// SMs as the occupancy API reports for clusters -- is cached.  forget()
// drops the entry (after a failed launch, e.g. once the context was reset).
template <class Cfg, bool kRelu, bool kTA, bool kTB>
struct Prepared {
    static std::atomic<int> slots[kMaxDevices];   // 0: not prepared

    static int64_t get(int dev, int sm_count)
    {
        int v = slots[dev].load(std::memory_order_acquire);
        if (v > 0) return v;
        auto kern = gemm_f16_relu_sm103a<Cfg, kRelu, kTA, kTB>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        v = sm_count / Cfg::CLUSTER;
        if (Cfg::CLUSTER > 1) {
            cudaLaunchConfig_t lc{};
            lc.blockDim = dim3(Cfg::THREADS, 1, 1);
            lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
            lc.gridDim = dim3(Cfg::CLUSTER * v, 1, 1);
            cudaLaunchAttribute attrs[1];
            attrs[0].id = cudaLaunchAttributeClusterDimension;
            attrs[0].val.clusterDim.x = Cfg::CLUSTER;
            attrs[0].val.clusterDim.y = 1;
            attrs[0].val.clusterDim.z = 1;
            lc.attrs = attrs;
            lc.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, kern, &lc) == cudaSuccess && clusters > 0)
                v = clusters < v ? clusters : v;
            else
                cudaGetLastError();
        }
        if (v > 0) slots[dev].store(v, std::memory_order_release);
        return v;
    }

    static void forget(int dev) { slots[dev].store(0, std::memory_order_release); }
};

template <class Cfg, bool kRelu, bool kTA, bool kTB>
std::atomic<int> Prepared<Cfg, kRelu, kTA, kTB>::slots[kMaxDevices];

// Persistent schedule: full waves of work units, then the tiles of a partly
// filled last wave split along N into 2^shift units, with the shift that gives
// the shortest tail.
struct Schedule {
    int64_t tiles = 0, units = 0, split_start = 0, grid_units = 0;
    int shift = 0;
    double tail_cost = 0.0;   // modelled time of the last (partly filled) wave, in whole-tile times
};

template <class Cfg>
Schedule make_schedule(int64_t M, int64_t N, int64_t slots, bool allow_split)
{
    Schedule sc;
    sc.tiles = ((M + Cfg::SUPER_M - 1) / Cfg::SUPER_M) * ((N + Cfg::BN - 1) / Cfg::BN);
    sc.units = sc.tiles;
    sc.split_start = sc.tiles;
    if (slots <= 0) return sc;
    const int64_t full = (sc.tiles / slots) * slots;
    const int64_t rest = sc.tiles - full;
    // Tail time of split shift s: ceil(rest * 2^s / slots) / 2^s tile times,
    // times the cost of narrow units: a unit narrower than 256 columns (CTA
    // pair) or 128 (one CTA) reuses each operand byte for fewer MMAs and runs
    // narrower, slower MMAs; each halving below that width is charged 1.5x
    // (measured: 256 x 128 units of the 256 x 512 pair kernel ran a 4096^3
    // tail at a third of the whole tiles' rate per output).  Ties go to the
    // coarser split.
    constexpr int kFullReuseWidth = Cfg::CTA_GROUP == 2 ? 256 : 128;
    int shift = 0;
    double best = 1e30;
    for (int s = 0; allow_split && rest > 0 && s <= Cfg::MAX_SPLIT_LOG2; ++s) {
        const int64_t waves = ((rest << s) + slots - 1) / slots;
        double t = static_cast<double>(waves) / static_cast<double>(1 << s);
        for (int w = Cfg::BN >> s; w < kFullReuseWidth; w *= 2) t *= 1.5;
        if (t < best - 1e-9) {
            best = t;
            shift = s;
        }
    }
    sc.tail_cost = rest > 0 ? (allow_split ? best : 1.0) : 0.0;
    if (shift > 0) {
        sc.shift = shift;
        sc.split_start = full;
        sc.units = full + (rest << shift);
    }
    sc.grid_units = sc.units < slots ? sc.units : slots;
    return sc;
}

template <class Cfg, bool kRelu, bool kTA, bool kTB>
int launch_one(const LaunchArgs &a)
{
    CUtensorMap ta, tb, tc;
    int st;
    // A: (M,K) with boxes 64(K) x 128(M), or stored (K,M) with boxes 64(M) x 64(K).
    st = kTA ? encode_matrix(&ta, a.A, a.K, a.M, 64, 64) : encode_matrix(&ta, a.A, a.M, a.K, Cfg::BK, Cfg::BM);
    if (st != GEMM_OK) return st;
    // B: (K,N) with boxes 64(N) x 64(K), or stored (N,K) with boxes 64(K) x 64(N).
    st = kTB ? encode_matrix(&tb, a.B, a.N, a.K, Cfg::BK, Cfg::B_BOX_N)
             : encode_matrix(&tb, a.B, a.K, a.N, Cfg::B_BOX_N, Cfg::BK);
    if (st != GEMM_OK) return st;
    if ((st = encode_matrix(&tc, a.C, a.M, a.N, Cfg::EPI_COLS, 32)) != GEMM_OK) return st;

    GemmParams p{};
    p.M = static_cast<int32_t>(a.M);
    p.N = static_cast<int32_t>(a.N);
    p.K = static_cast<int32_t>(a.K);
    p.num_m_blocks = static_cast<int32_t>((a.M + Cfg::SUPER_M - 1) / Cfg::SUPER_M);
    p.num_n_blocks = static_cast<int32_t>((a.N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int32_t>((a.K + Cfg::BK - 1) / Cfg::BK);
    using Prep = Prepared<Cfg, kRelu, kTA, kTB>;
    const int64_t slots = Prep::get(a.dev.device, a.dev.sm_count);
    if (slots <= 0) return GEMM_ERR_LAUNCH;
    Schedule sc = make_schedule<Cfg>(a.M, a.N, slots, a.allow_split && a.k_splits <= 1 && !a.k_split_tail);
    KPlan kp = plan_k_split(sc.tiles, slots, p.num_k_blocks, a.k_splits, a.k_split_tail);
    float *ws = nullptr;
    const bool own_ws = !a.noalloc;
    if (kp.ks.count > 1) {
        // The workspace check is made on the plan this launch runs, before
        // anything is enqueued.
        const size_t need = static_cast<size_t>(kp.ws_floats(sc.tiles, Cfg::SUPER_M, Cfg::BN)) * sizeof(float);
        if (a.noalloc) {
            size_t have = 0;
            if (noalloc_scratch(a.dev.device, &ws, &have) != GEMM_OK) return GEMM_ERR_CUDA;
            if (need > have) return GEMM_ERR_INVALID_ARG;
        } else if (cudaMallocAsync(reinterpret_cast<void **>(&ws), need, a.stream) != cudaSuccess) {
            // Stream-ordered workspace: ordered with this call's kernels, private
            // to it, and legal inside a stream capture.  If it cannot be had, the
            // call runs without a K split.
            cudaGetLastError();
            ws = nullptr;
            kp = plan_k_split(sc.tiles, slots, p.num_k_blocks, 1, false);
            sc = make_schedule<Cfg>(a.M, a.N, slots, a.allow_split);
        }
    }
    if (kp.ks.count > 1) {
        // Whole tiles before ks_start, then each later tile as ks.count K slices.
        sc.units = kp.units(sc.tiles);
        sc.split_start = sc.tiles;
        sc.shift = 0;
        sc.grid_units = sc.units < slots ? sc.units : slots;
    }
    auto release_ws = [&]() {
        if (own_ws && ws != nullptr && cudaFreeAsync(ws, a.stream) != cudaSuccess) cudaGetLastError();
    };
    if (sc.units > INT32_MAX / 2) {
        release_ws();
        return GEMM_ERR_INVALID_ARG;
    }
    p.num_tiles = static_cast<int32_t>(sc.tiles);
    p.num_units = static_cast<int32_t>(sc.units);
    p.split_start = static_cast<int32_t>(sc.split_start);
    p.split_log2 = sc.shift;
    p.k_splits = kp.ks.count;
    p.k_per_split = kp.ks.per;
    p.ks_start = static_cast<int32_t>(kp.ks_start);
    p.ws = ws;
    // Rasterisation panels 2048 rows high whatever the tile height.
    p.group_m = group_m_override() ? group_m_override() : (Cfg::SUPER_M >= 2048 ? 1 : 2048 / Cfg::SUPER_M);
    p.timeout_cycles = a.hook.timeout_cycles ? a.hook.timeout_cycles : timeout_cycles_for(a.K);
    p.C = static_cast<__half *>(a.C);
    p.producer_off = a.hook.producer_off;
    p.status = a.status;

    auto kern = gemm_f16_relu_sm103a<Cfg, kRelu, kTA, kTB>;
    cudaLaunchConfig_t lc{};
    lc.blockDim = dim3(Cfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = a.stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = Cfg::CLUSTER;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    // Programmatic dependent launch: the kernel's set-up may overlap the end
    // of the previous kernel on the stream (the kernel waits for it before
    // touching memory).
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attrs;
    lc.numAttrs = 2;
    lc.gridDim = dim3(static_cast<unsigned>(sc.grid_units * Cfg::CLUSTER), 1, 1);
    if (cudaLaunchKernelEx(&lc, kern, ta, tb, tc, p) != cudaSuccess) {
        cudaGetLastError();
        // Prepare again (the attribute may have been lost) and retry once.
        Prep::forget(a.dev.device);
        if (Prep::get(a.dev.device, a.dev.sm_count) <= 0 || cudaLaunchKernelEx(&lc, kern, ta, tb, tc, p) != cudaSuccess) {
            cudaGetLastError();
            release_ws();
            return GEMM_ERR_LAUNCH;
        }
    }
    if (kp.ks.count > 1) {
        const int st2 = launch_splitk_reduce(ws, a.C, p, Cfg::SUPER_M, Cfg::BN, a.relu, a.dev.sm_count, a.stream);
        release_ws();
        if (st2 != GEMM_OK) return st2;
    }
    return GEMM_OK;
}

// ---------------------------------------------------------------- cluster K split

// Resident clusters of `size` CTAs (1, 2, 4, 8) of a cluster-K configuration,
// per device, prepared once like Prepared.
template <class Cfg, bool kRelu>
struct PreparedCK {
    static std::atomic<int> slots[kMaxDevices][4];   // index log2(size); 0: not prepared

    static int64_t get(int dev, int sm_count, int size)
    {
        const int li = size >= 8 ? 3 : size >= 4 ? 2 : size >= 2 ? 1 : 0;
        int v = slots[dev][li].load(std::memory_order_acquire);
        if (v > 0) return v;
        auto kern = gemm_f16_relu_sm103a<Cfg, kRelu, false, false>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
            cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        v = sm_count / size;
        cudaLaunchConfig_t lc{};
        lc.blockDim = dim3(Cfg::THREADS, 1, 1);
        lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
        lc.gridDim = dim3(static_cast<unsigned>(size * v), 1, 1);
        cudaLaunchAttribute attrs[1];
        attrs[0].id = cudaLaunchAttributeClusterDimension;
        attrs[0].val.clusterDim.x = static_cast<unsigned>(size);
        attrs[0].val.clusterDim.y = 1;
        attrs[0].val.clusterDim.z = 1;
        lc.attrs = attrs;
        lc.numAttrs = 1;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &lc) == cudaSuccess && clusters > 0)
            v = clusters < v ? clusters : v;
        else
            cudaGetLastError();
        if (v > 0) slots[dev][li].store(v, std::memory_order_release);
        return v;
    }

    static void forget(int dev)
    {
        for (int i = 0; i < 4; ++i) slots[dev][i].store(0, std::memory_order_release);
    }
};

template <class Cfg, bool kRelu>
std::atomic<int> PreparedCK<Cfg, kRelu>::slots[kMaxDevices][4];

// Cluster size and K blocks per CTA of a cluster K split.
struct CKPlan {
    int size = 1;           // CTAs per cluster = K slices per tile
    int per = 0;            // K blocks per CTA
    int64_t tiles = 0;      // output tiles (one per cluster at a time)
    int64_t slots = 0;      // resident clusters of `size` CTAs
};

// request: 0 = the size rule, 1 = no split, 2 / 4 / 8 = that size.  Every CTA
// of a cluster gets a non-empty slice: a size whose slices would leave one
// empty is halved.  The rule takes the largest size (up to 8) whose clusters
// hold every tile at once and leave each CTA at least two K blocks.
template <class Cfg>
CKPlan plan_cluster_k(int64_t M, int64_t N, int64_t K, int request, const DeviceInfo &dev)
{
    CKPlan pl;
    pl.tiles = ((M + Cfg::SUPER_M - 1) / Cfg::SUPER_M) * ((N + Cfg::BN - 1) / Cfg::BN);
    const int64_t kb = (K + Cfg::BK - 1) / Cfg::BK;
    auto fits = [&](int size) { return size == 1 || k_split_for(kb, size).count == size; };
    int size = 1;
    if (request == 0) {
        for (int c = 2; c <= Cfg::MAX_CLUSTER_K; c *= 2) {
            const int64_t slots = PreparedCK<Cfg, true>::get(dev.device, dev.sm_count, c);
            if (slots >= pl.tiles && kb >= 2 * c && fits(c)) size = c;
        }
    } else {
        size = request;
        while (size > 1 && !fits(size)) size /= 2;
    }
    pl.size = size;
    pl.per = size > 1 ? k_split_for(kb, size).per : static_cast<int>(kb);
    pl.slots = PreparedCK<Cfg, true>::get(dev.device, dev.sm_count, size);
    return pl;
}

template <class Cfg, bool kRelu>
int launch_one_ck(const LaunchArgs &a)
{
    static_assert(Cfg::CLUSTER_K, "cluster K split configuration");
    if (a.ck_request != 0 && a.ck_request != 1 && a.ck_request != 2 && a.ck_request != 4 && a.ck_request != 8)
        return GEMM_ERR_INVALID_ARG;
    CUtensorMap ta, tb, tc;
    int st;
    if ((st = encode_matrix(&ta, a.A, a.M, a.K, Cfg::BK, Cfg::BM)) != GEMM_OK) return st;
    if ((st = encode_matrix(&tb, a.B, a.K, a.N, Cfg::B_BOX_N, Cfg::BK)) != GEMM_OK) return st;
    if ((st = encode_matrix(&tc, a.C, a.M, a.N, Cfg::EPI_COLS, 32)) != GEMM_OK) return st;   // unused by the kernel
    const CKPlan pl = plan_cluster_k<Cfg>(a.M, a.N, a.K, a.ck_request, a.dev);
    if (pl.slots <= 0) return GEMM_ERR_LAUNCH;
    if (pl.tiles * pl.size > INT32_MAX / 2) return GEMM_ERR_INVALID_ARG;
    using Prep = PreparedCK<Cfg, kRelu>;
    if (Prep::get(a.dev.device, a.dev.sm_count, pl.size) <= 0) return GEMM_ERR_LAUNCH;

    GemmParams p{};
    p.M = static_cast<int32_t>(a.M);
    p.N = static_cast<int32_t>(a.N);
    p.K = static_cast<int32_t>(a.K);
    p.num_m_blocks = static_cast<int32_t>((a.M + Cfg::SUPER_M - 1) / Cfg::SUPER_M);
    p.num_n_blocks = static_cast<int32_t>((a.N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int32_t>((a.K + Cfg::BK - 1) / Cfg::BK);
    p.num_tiles = static_cast<int32_t>(pl.tiles);
    p.num_units = p.num_tiles;
    p.split_start = p.num_tiles;
    p.split_log2 = 0;
    p.k_splits = 1;
    p.k_per_split = p.num_k_blocks;
    p.ks_start = p.num_tiles;
    p.ws = nullptr;
    p.ck_per = pl.per;
    p.group_m = group_m_override() ? group_m_override() : 2048 / Cfg::SUPER_M;
    p.timeout_cycles = a.hook.timeout_cycles ? a.hook.timeout_cycles : timeout_cycles_for(a.K);
    p.C = static_cast<__half *>(a.C);
    p.producer_off = a.hook.producer_off;
    p.status = a.status;

    // One cluster per tile (not persistent): a CTA's operand ring holds its
    // reduction buffers once its tile is multiplied.
    const int64_t grid_units = pl.tiles;
    auto kern = gemm_f16_relu_sm103a<Cfg, kRelu, false, false>;
    cudaLaunchConfig_t lc{};
    lc.blockDim = dim3(Cfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = a.stream;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = static_cast<unsigned>(pl.size);
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attrs[1].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attrs;
    lc.numAttrs = 2;
    lc.gridDim = dim3(static_cast<unsigned>(grid_units * pl.size), 1, 1);
    if (cudaLaunchKernelEx(&lc, kern, ta, tb, tc, p) != cudaSuccess) {
        cudaGetLastError();
        Prep::forget(a.dev.device);
        PreparedCK<Cfg, true>::forget(a.dev.device);
        if (Prep::get(a.dev.device, a.dev.sm_count, pl.size) <= 0 || cudaLaunchKernelEx(&lc, kern, ta, tb, tc, p) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    }
    return GEMM_OK;
}

// Launch geometry of a cluster K split (no launch).
template <class Cfg>
int ck_launch_info(int64_t M, int64_t N, int64_t K, int request, const DeviceInfo &dev, int *grid_ctas,
                   int *cluster_size, int *tiles)
{
    const CKPlan pl = plan_cluster_k<Cfg>(M, N, K, request, dev);
    const int64_t ctas = pl.tiles * pl.size;   // one cluster per tile
    if (grid_ctas) *grid_ctas = static_cast<int>(ctas < INT32_MAX ? ctas : INT32_MAX);
    if (cluster_size) *cluster_size = pl.size;
    if (tiles) *tiles = static_cast<int>(pl.tiles < INT32_MAX ? pl.tiles : INT32_MAX);
    return GEMM_OK;
}

// Share of the GPU's SM time that computes in-range outputs (as
// config_wave_efficiency): a tile on a cluster of `size` CTAs takes 1/size of
// its whole K loop, and every SM of the device counts, also those that no
// cluster occupies.
template <class Cfg>
double ck_wave_efficiency(int64_t M, int64_t N, int64_t K, int request, const DeviceInfo &dev)
{
    if (M <= 0 || N <= 0 || dev.sm_count <= 0) return 0.0;
    const CKPlan pl = plan_cluster_k<Cfg>(M, N, K, request, dev);
    if (pl.slots <= 0) return 0.0;
    const double waves = static_cast<double>((pl.tiles + pl.slots - 1) / pl.slots);
    const double area = static_cast<double>(Cfg::SUPER_M) * static_cast<double>(Cfg::BN);
    return static_cast<double>(M) * static_cast<double>(N) * pl.size /
           (static_cast<double>(dev.sm_count) * waves * area);
}

// Dispatch over ReLU and the operand layouts this configuration supports.
template <class Cfg, bool kAllLayouts>
int launch_config(const LaunchArgs &a)
{
    const int layout = (a.transa ? 2 : 0) | (a.transb ? 1 : 0);
    if (!kAllLayouts && layout != 0) return GEMM_ERR_INVALID_ARG;
    if constexpr (kAllLayouts) {
        switch (layout | (a.relu ? 4 : 0)) {
            case 0: return launch_one<Cfg, false, false, false>(a);
            case 1: return launch_one<Cfg, false, false, true>(a);
            case 2: return launch_one<Cfg, false, true, false>(a);
            case 3: return launch_one<Cfg, false, true, true>(a);
            case 4: return launch_one<Cfg, true, false, false>(a);
            case 5: return launch_one<Cfg, true, false, true>(a);
            case 6: return launch_one<Cfg, true, true, false>(a);
            default: return launch_one<Cfg, true, true, true>(a);
        }
    } else {
        return a.relu ? launch_one<Cfg, true, false, false>(a) : launch_one<Cfg, false, false, false>(a);
    }
}

// Launch geometry of a configuration (no launch).
template <class Cfg>
int config_launch_info(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev, int *grid_ctas,
                       int *cluster_size, int *tiles)
{
    const Schedule sc =
        make_schedule<Cfg>(M, N, Prepared<Cfg, true, false, false>::get(dev.device, dev.sm_count), allow_split);
    if (tiles) *tiles = static_cast<int>(sc.tiles < INT32_MAX ? sc.tiles : INT32_MAX);
    if (cluster_size) *cluster_size = Cfg::CLUSTER;
    if (grid_ctas) *grid_ctas = static_cast<int>(sc.grid_units * Cfg::CLUSTER);
    return GEMM_OK;
}

// Share of the persistent grid's slot time that computes in-range outputs:
// M*N over (slots x the busiest slot's time x tile area), where the time is
// counted in whole-tile units (a unit split 2^s ways takes 2^-s of a tile).
// Scales a throughput measured at one shape to another shape for the same
// configuration; 0 when the configuration cannot be launched.
template <class Cfg>
double config_wave_efficiency(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev)
{
    const int64_t slots = Prepared<Cfg, true, false, false>::get(dev.device, dev.sm_count);
    if (slots <= 0 || M <= 0 || N <= 0) return 0.0;
    const Schedule sc = make_schedule<Cfg>(M, N, slots, allow_split);
    // full waves of whole tiles, then the modelled tail (narrow units charged)
    const double t = static_cast<double>(sc.tiles / slots) + sc.tail_cost;
    const double area = static_cast<double>(Cfg::SUPER_M) * static_cast<double>(Cfg::BN);
    return static_cast<double>(M) * static_cast<double>(N) / (static_cast<double>(slots) * t * area);
}

// One pair of entry points per configuration, each defined in its own
// translation unit (gemm_cfg_<id>.cu) so that they compile in parallel.
#define GEMM_DECLARE_CONFIG(ID)                                                                              \
    int launch_config_##ID(const LaunchArgs &a);                                                             \
    int launch_info_config_##ID(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev, int *grid_ctas, \
                                int *cluster_size, int *tiles);                                               \
    double wave_eff_config_##ID(int64_t M, int64_t N, bool allow_split, const DeviceInfo &dev);
GEMM_DECLARE_CONFIG(1)
GEMM_DECLARE_CONFIG(2)
GEMM_DECLARE_CONFIG(3)
GEMM_DECLARE_CONFIG(4)
GEMM_DECLARE_CONFIG(5)
GEMM_DECLARE_CONFIG(6)
#undef GEMM_DECLARE_CONFIG
// The cluster K split configuration (6) also answers with its cluster size.
int ck_launch_info_config_6(int64_t M, int64_t N, int64_t K, int request, const DeviceInfo &dev, int *grid_ctas,
                            int *cluster_size, int *tiles);
double ck_wave_eff_config_6(int64_t M, int64_t N, int64_t K, int request, const DeviceInfo &dev);

// The configurations, by id (1-based).
using Cfg1x256 = GemmCfg<1, 256, 4>;
using Cfg1x128 = GemmCfg<1, 128, 6>;
using Cfg2x256 = GemmCfg<2, 256, 6>;
using Cfg2x256d = GemmCfg<2, 256, 7, /*stage C in smem*/ false>;
using Cfg2x512 = GemmCfg<2, 512, 4>;
using Cfg1x128ck = GemmCfg<1, 128, 6, /*stage C in smem*/ false, /*cluster K split*/ true>;

}  // namespace gemm_sm103
