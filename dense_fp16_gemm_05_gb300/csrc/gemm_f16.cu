// gemm_f16.cu -- host side of the GB300 fp16 GEMM + ReLU library: argument
// checks, TMA tensor-map encoding, configuration choice, launch, and the
// extern "C" entry points declared in include/gemm_f16.h.
//
// Nothing here computes the product on the host; every element of C is
// written by the sm_103a kernel in gemm_kernel.cuh (or, for K == 0, by one
// cudaMemsetAsync of +0, the value of the empty sum).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <atomic>
#include <mutex>

#include "gemm_f16.h"
#include "gemm_kernel.cuh"

using namespace gemm_sm103;

namespace {

// ---------------------------------------------------------------- configurations

struct ConfigInfo {
    const char *name;
    int tile_m;       // rows of C per tile (all CTAs of the tile together)
    int tile_n;       // columns of C per tile
};

// id 1..kNumConfigs; index 0 is "auto".
using Cfg1x256 = GemmCfg<1, 256, 4>;
using Cfg1x128 = GemmCfg<1, 128, 6>;
using Cfg2x256 = GemmCfg<2, 256, 6>;
using Cfg2x256d = GemmCfg<2, 256, 7, /*stage C in smem*/ false>;
using Cfg2x512 = GemmCfg<2, 512, 4>;
using Cfg4x256mc = GemmCfg<2, 256, 6, /*stage C in smem*/ true, /*pairs sharing B*/ 2>;

constexpr ConfigInfo kConfigs[] = {
    {"auto", 0, 0},
    {"1sm_128x256_s4", Cfg1x256::SUPER_M, Cfg1x256::BN},
    {"1sm_128x128_s6", Cfg1x128::SUPER_M, Cfg1x128::BN},
    {"2sm_256x256_s6", Cfg2x256::SUPER_M, Cfg2x256::BN},
    {"2sm_256x256_s7_direct", Cfg2x256d::SUPER_M, Cfg2x256d::BN},
    {"2sm_256x512_s4", Cfg2x512::SUPER_M, Cfg2x512::BN},
    {"4sm_512x256_mc_s6", Cfg4x256mc::SUPER_M, Cfg4x256mc::BN},
};
constexpr int kNumConfigs = static_cast<int>(sizeof(kConfigs) / sizeof(kConfigs[0])) - 1;

// ---------------------------------------------------------------- driver entry points

struct DriverFns {
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    PFN_cuMemGetAddressRange_v3020 range = nullptr;
    bool ok = false;
};

const DriverFns &driver()
{
    static DriverFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
        void *f1 = nullptr, *f2 = nullptr;
        cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f1, 12000, cudaEnableDefault, &q1);
        cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f2, 3020, cudaEnableDefault, &q2);
        if (e1 == cudaSuccess && q1 == cudaDriverEntryPointSuccess && f1 && e2 == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess && f2) {
            fns.encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f1);
            fns.range = reinterpret_cast<PFN_cuMemGetAddressRange_v3020>(f2);
            fns.ok = true;
        }
    });
    return fns;
}

// ---------------------------------------------------------------- per-device facts

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    int device = 0;
    int supported = 0;      // compute capability 10.3
    int sm_count = 0;
};

// Filled once per device; read without locking afterwards.
std::atomic<int> g_device_state[kMaxDevices];   // 0 unknown, 1 supported, 2 unsupported
int g_device_sms[kMaxDevices];

int current_device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    int state = g_device_state[dev].load(std::memory_order_acquire);
    if (state == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        g_device_sms[dev] = sms;
        state = (major == 10 && minor == 3) ? 1 : 2;
        g_device_state[dev].store(state, std::memory_order_release);
    }
    out->device = dev;
    out->sm_count = g_device_sms[dev];
    out->supported = state == 1;
    return state == 1 ? GEMM_OK : GEMM_ERR_UNSUPPORTED_DEVICE;
}

// ---------------------------------------------------------------- argument checks

// A device buffer of `bytes` bytes starting at p: device (or managed) memory of
// the current device, entirely inside one allocation.
int check_device_buffer(const void *p, uint64_t bytes, int dev)
{
    if (p == nullptr) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return GEMM_ERR_ALIGNMENT;
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_INVALID_ARG;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged) return GEMM_ERR_INVALID_ARG;
    if (attr.type == cudaMemoryTypeDevice && attr.device != dev) return GEMM_ERR_INVALID_ARG;
    const DriverFns &fns = driver();
    if (!fns.ok) return GEMM_ERR_CUDA;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (fns.range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return GEMM_ERR_INVALID_ARG;
    const uint64_t off = static_cast<uint64_t>(reinterpret_cast<CUdeviceptr>(p) - base);
    if (off > size || bytes > size - off) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

bool ranges_overlap(const void *a, uint64_t abytes, const void *b, uint64_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

int check_sizes(int64_t M, int64_t N, int64_t K, int relu)
{
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_ARG;
    if (relu != 0 && relu != 1) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

// ---------------------------------------------------------------- tensor maps

// Row-major fp16 matrix rows x cols (leading dimension cols), boxes of
// box_cols x box_rows with 128-byte swizzle; out-of-range loads read zero.
int encode_matrix(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                  uint32_t box_rows)
{
    const DriverFns &fns = driver();
    if (!fns.ok) return GEMM_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fns.encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// ---------------------------------------------------------------- launch

uint64_t timeout_cycles_for(int64_t K)
{
    // About a second of SM clocks plus a margin that grows with the K loop of
    // one tile; a legitimate wait is at most one tile's mainloop.
    return (1ull << 31) + 64ull * static_cast<uint64_t>(K);
}

int pick_config(int64_t M, int64_t N, int64_t K, int sm_count)
{
    (void)K;
    const int64_t pairs = sm_count / 2;
    const int64_t tiles_256x512 = ((M + 255) / 256) * ((N + 511) / 512);
    // Many 256x512 tiles (about 13 or more waves): the wide pair tile needs the
    // fewest operand bytes per flop; its single accumulator costs little
    // when tiles are long and the tail is a small share.
    if (tiles_256x512 >= 13 * pairs) return 5;
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    // Enough 256x256 tiles to keep every SM pair busy: the CTA-pair kernel.
    if (pair_tiles >= pairs) return 3;
    const int64_t tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
    if (tiles256 >= sm_count / 2) return 1;
    // Few tiles: narrower tiles put more SMs to work.
    return 2;
}

int group_m_override()
{
    static int v = [] {
        const char *e = std::getenv("GEMM_F16_GROUP_M");
        const int x = e ? std::atoi(e) : 0;
        return x > 0 && x <= 4096 ? x : 0;
    }();
    return v;
}

// Per device and kernel instance, prepared once: the dynamic shared-memory
// attribute is set, and the number of CTAs (or CTA clusters) of this
// configuration that can be resident at once -- one per SM, or per group of
// SMs as the occupancy API reports for clusters -- is cached.  forget()
// drops the entry (after a failed launch, e.g. once the context was reset).
template <class Cfg, bool kRelu>
struct Prepared {
    static std::atomic<int> slots[kMaxDevices];   // 0: not prepared

    static int64_t get(int dev, int sm_count)
    {
        int v = slots[dev].load(std::memory_order_acquire);
        if (v > 0) return v;
        auto kern = gemm_f16_relu_sm103a<Cfg, kRelu>;
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

template <class Cfg, bool kRelu>
std::atomic<int> Prepared<Cfg, kRelu>::slots[kMaxDevices];

// Persistent schedule: full waves of tiles, then the tiles of a partly filled
// last wave split along N into 2^shift units while the split units still fit
// in one wave (the tail then costs 1/2^shift of a tile time).
struct Schedule {
    int64_t tiles = 0, units = 0, split_start = 0, grid_units = 0;
    int shift = 0;
};

template <class Cfg>
Schedule make_schedule(int64_t M, int64_t N, int64_t slots)
{
    Schedule sc;
    sc.tiles = ((M + Cfg::SUPER_M - 1) / Cfg::SUPER_M) * ((N + Cfg::BN - 1) / Cfg::BN);
    sc.units = sc.tiles;
    sc.split_start = sc.tiles;
    if (slots <= 0) return sc;
    const int64_t full = (sc.tiles / slots) * slots;
    const int64_t rest = sc.tiles - full;
    // Split shift with the shortest tail: ceil(rest * 2^s / slots) / 2^s tile
    // times (ties go to the coarser split).
    int shift = 0;
    double best = 1e30;
    for (int s = 0; rest > 0 && s <= Cfg::MAX_SPLIT_LOG2; ++s) {
        const int64_t waves = ((rest << s) + slots - 1) / slots;
        const double t = static_cast<double>(waves) / static_cast<double>(1 << s);
        if (t < best - 1e-9) {
            best = t;
            shift = s;
        }
    }
    if (shift > 0) {
        sc.shift = shift;
        sc.split_start = full;
        sc.units = full + (rest << shift);
    }
    sc.grid_units = sc.units < slots ? sc.units : slots;
    return sc;
}

template <class Cfg>
int fill_launch_info(int64_t M, int64_t N, const DeviceInfo &dev, int *grid_ctas, int *cluster_size, int *tiles)
{
    const Schedule sc = make_schedule<Cfg>(M, N, Prepared<Cfg, true>::get(dev.device, dev.sm_count));
    if (tiles) *tiles = static_cast<int>(sc.tiles < INT32_MAX ? sc.tiles : INT32_MAX);
    if (cluster_size) *cluster_size = Cfg::CLUSTER;
    if (grid_ctas) *grid_ctas = static_cast<int>(sc.grid_units * Cfg::CLUSTER);
    return GEMM_OK;
}

// Test-hook settings for a launch (all zero for normal calls).
struct LaunchHook {
    int producer_off = 0;          // producer issues nothing
    uint64_t timeout_cycles = 0;   // 0: the normal budget
};

template <class Cfg, bool kRelu>
int launch(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, const DeviceInfo &dev,
           cudaStream_t stream, const LaunchHook &hook = LaunchHook())
{
    CUtensorMap ta, tb, tc;
    int st;
    if ((st = encode_matrix(&ta, A, M, K, Cfg::BK, Cfg::BM)) != GEMM_OK) return st;
    if ((st = encode_matrix(&tb, B, K, N, Cfg::B_BOX_N, Cfg::BK)) != GEMM_OK) return st;
    if ((st = encode_matrix(&tc, C, M, N, Cfg::EPI_COLS, 32)) != GEMM_OK) return st;

    GemmParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.num_m_blocks = static_cast<int32_t>((M + Cfg::SUPER_M - 1) / Cfg::SUPER_M);
    p.num_n_blocks = static_cast<int32_t>((N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int32_t>((K + Cfg::BK - 1) / Cfg::BK);
    const int64_t slots = Prepared<Cfg, kRelu>::get(dev.device, dev.sm_count);
    if (slots <= 0) return GEMM_ERR_LAUNCH;
    const Schedule sc = make_schedule<Cfg>(M, N, slots);
    if (sc.units > INT32_MAX / 2) return GEMM_ERR_INVALID_ARG;
    p.num_tiles = static_cast<int32_t>(sc.tiles);
    p.num_units = static_cast<int32_t>(sc.units);
    p.split_start = static_cast<int32_t>(sc.split_start);
    p.split_log2 = sc.shift;
    // Rasterisation panels 2048 rows high whatever the tile height.
    p.group_m = group_m_override() ? group_m_override() : (Cfg::SUPER_M >= 2048 ? 1 : 2048 / Cfg::SUPER_M);
    p.timeout_cycles = hook.timeout_cycles ? hook.timeout_cycles : timeout_cycles_for(K);
    p.C = static_cast<__half *>(C);
    p.producer_off = hook.producer_off;

    auto kern = gemm_f16_relu_sm103a<Cfg, kRelu>;
    cudaLaunchConfig_t lc{};
    lc.blockDim = dim3(Cfg::THREADS, 1, 1);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = stream;
    cudaLaunchAttribute attrs[1];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = Cfg::CLUSTER;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    lc.attrs = attrs;
    lc.numAttrs = 1;

    lc.gridDim = dim3(static_cast<unsigned>(sc.grid_units * Cfg::CLUSTER), 1, 1);
    if (cudaLaunchKernelEx(&lc, kern, ta, tb, tc, p) != cudaSuccess) {
        cudaGetLastError();
        // Prepare again (the attribute may have been lost) and retry once.
        Prepared<Cfg, kRelu>::forget(dev.device);
        if (Prepared<Cfg, kRelu>::get(dev.device, dev.sm_count) <= 0 ||
            cudaLaunchKernelEx(&lc, kern, ta, tb, tc, p) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_LAUNCH;
        }
    }
    return GEMM_OK;
}

template <class Cfg>
int launch_cfg(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int relu,
               const DeviceInfo &dev, cudaStream_t stream, const LaunchHook &hook = LaunchHook())
{
    return relu ? launch<Cfg, true>(A, B, C, M, N, K, dev, stream, hook)
                : launch<Cfg, false>(A, B, C, M, N, K, dev, stream, hook);
}

thread_local uint64_t t_last_timeout_record = 0;

}  // namespace

// ==================================================================== C ABI

namespace {

int run_gemm(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int relu, int config,
             void *stream, const LaunchHook &hook)
{
    int st = check_sizes(M, N, K, relu);
    if (st != GEMM_OK) return st;
    if (config < 0 || config > kNumConfigs) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;

    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t c_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(N) * 2u;
    if ((st = check_device_buffer(C, c_bytes, dev.device)) != GEMM_OK) return st;

    if (K == 0) {
        // Empty sum: every output is R(+0) = +0.
        if (cudaMemsetAsync(C, 0, c_bytes, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    if ((N % 8) != 0 || (K % 8) != 0) return GEMM_ERR_ALIGNMENT;
    const uint64_t a_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(K) * 2u;
    const uint64_t b_bytes = static_cast<uint64_t>(K) * static_cast<uint64_t>(N) * 2u;
    if ((st = check_device_buffer(A, a_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(B, b_bytes, dev.device)) != GEMM_OK) return st;
    if (ranges_overlap(C, c_bytes, A, a_bytes) || ranges_overlap(C, c_bytes, B, b_bytes))
        return GEMM_ERR_INVALID_ARG;

    const int cfg = config == 0 ? pick_config(M, N, K, dev.sm_count) : config;
    switch (cfg) {
        case 1: return launch_cfg<Cfg1x256>(A, B, C, M, N, K, relu, dev, s, hook);
        case 2: return launch_cfg<Cfg1x128>(A, B, C, M, N, K, relu, dev, s, hook);
        case 3: return launch_cfg<Cfg2x256>(A, B, C, M, N, K, relu, dev, s, hook);
        case 4: return launch_cfg<Cfg2x256d>(A, B, C, M, N, K, relu, dev, s, hook);
        case 5: return launch_cfg<Cfg2x512>(A, B, C, M, N, K, relu, dev, s, hook);
        case 6: return launch_cfg<Cfg4x256mc>(A, B, C, M, N, K, relu, dev, s, hook);
        default: return GEMM_ERR_INVALID_ARG;
    }
}

}  // namespace

extern "C" int gemm_f16_ex(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int relu,
                           int config, void *stream)
{
    return run_gemm(A, B, C, M, N, K, relu, config, stream, LaunchHook());
}

extern "C" int gemm_f16_selftest_timeout(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                                         int config, uint64_t timeout_cycles, void *stream)
{
    if (K == 0 || M == 0 || N == 0) return GEMM_ERR_INVALID_ARG;   // nothing would be launched
    if (timeout_cycles < (1ull << 16) || timeout_cycles > (1ull << 32)) return GEMM_ERR_INVALID_ARG;
    LaunchHook hook;
    hook.producer_off = 1;
    hook.timeout_cycles = timeout_cycles;
    return run_gemm(A, B, C, M, N, K, 1, config, stream, hook);
}

extern "C" int gemm_f16(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int relu,
                        void *stream)
{
    return gemm_f16_ex(A, B, C, M, N, K, relu, 0, stream);
}

extern "C" int gemm_f16_num_configs(void) { return kNumConfigs; }

extern "C" const char *gemm_f16_config_name(int config)
{
    if (config < 0 || config > kNumConfigs) return nullptr;
    return kConfigs[config].name;
}

extern "C" int gemm_f16_auto_config(int64_t M, int64_t N, int64_t K)
{
    int st = check_sizes(M, N, K, 0);
    if (st != GEMM_OK) return st;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    return pick_config(M, N, K, dev.sm_count);
}

extern "C" int gemm_f16_launch_info(int64_t M, int64_t N, int64_t K, int config, int *grid_ctas,
                                    int *cluster_size, int *tiles)
{
    int st = check_sizes(M, N, K, 0);
    if (st != GEMM_OK) return st;
    if (config < 0 || config > kNumConfigs) return GEMM_ERR_INVALID_ARG;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    const int cfg = config == 0 ? pick_config(M, N, K, dev.sm_count) : config;
    switch (cfg) {
        case 1: return fill_launch_info<Cfg1x256>(M, N, dev, grid_ctas, cluster_size, tiles);
        case 2: return fill_launch_info<Cfg1x128>(M, N, dev, grid_ctas, cluster_size, tiles);
        case 3: return fill_launch_info<Cfg2x256>(M, N, dev, grid_ctas, cluster_size, tiles);
        case 4: return fill_launch_info<Cfg2x256d>(M, N, dev, grid_ctas, cluster_size, tiles);
        case 5: return fill_launch_info<Cfg2x512>(M, N, dev, grid_ctas, cluster_size, tiles);
        case 6: return fill_launch_info<Cfg4x256mc>(M, N, dev, grid_ctas, cluster_size, tiles);
        default: return GEMM_ERR_INVALID_ARG;
    }
}

extern "C" int gemm_f16_from_host(const void *A_host, const void *B_host, void *C_host, void *A_dev, void *B_dev,
                                  void *C_dev, int64_t M, int64_t N, int64_t K, int relu, void *stream)
{
    int st = check_sizes(M, N, K, relu);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C_host == nullptr || (K > 0 && (A_host == nullptr || B_host == nullptr))) return GEMM_ERR_INVALID_ARG;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t a_bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * 2u;
    const size_t b_bytes = static_cast<size_t>(K) * static_cast<size_t>(N) * 2u;
    const size_t c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * 2u;
    if (K > 0) {
        // Validate the device side before any copy is enqueued.
        DeviceInfo dev;
        if ((st = current_device_info(&dev)) != GEMM_OK) return st;
        if ((N % 8) != 0 || (K % 8) != 0) return GEMM_ERR_ALIGNMENT;
        if ((st = check_device_buffer(A_dev, a_bytes, dev.device)) != GEMM_OK) return st;
        if ((st = check_device_buffer(B_dev, b_bytes, dev.device)) != GEMM_OK) return st;
        if ((st = check_device_buffer(C_dev, c_bytes, dev.device)) != GEMM_OK) return st;
        if (cudaMemcpyAsync(A_dev, A_host, a_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(B_dev, B_host, b_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
    }
    if ((st = gemm_f16(A_dev, B_dev, C_dev, M, N, K, relu, stream)) != GEMM_OK) return st;
    if (cudaMemcpyAsync(C_host, C_dev, c_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

extern "C" int gemm_f16_check(void *stream)
{
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    unsigned long long v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_f16_status, sizeof(v)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (v != 0) {
        t_last_timeout_record = v;
        const unsigned long long zero = 0;
        if (cudaMemcpyToSymbol(g_gemm_f16_status, &zero, sizeof(zero)) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}

extern "C" uint64_t gemm_f16_last_timeout_record(void) { return t_last_timeout_record; }

extern "C" const char *gemm_f16_strerror(int status)
{
    switch (status) {
        case GEMM_OK: return "success";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_ALIGNMENT: return "misaligned pointer, or N or K not a multiple of 8";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (GB300)";
        case GEMM_ERR_LAUNCH: return "kernel launch failed";
        case GEMM_ERR_TIMEOUT: return "a kernel wait exceeded its limit; the output is incomplete";
        case GEMM_ERR_CUDA: return "CUDA runtime or driver call failed";
        default: return "unknown status";
    }
}

extern "C" int gemm_f16_version(void) { return GEMM_F16_VERSION; }
