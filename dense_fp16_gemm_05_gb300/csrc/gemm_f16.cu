// gemm_f16.cu -- host side of the GB300 fp16 GEMM + ReLU library: argument
// checks, TMA tensor-map encoding, configuration choice, the device status
// word, and the extern "C" entry points declared in include/gemm_f16.h.  The
// kernel instances themselves are launched from gemm_cfg_<id>.cu.
//
// Nothing here computes the product on the host; every element of C is
// written by the sm_103a kernel in gemm_kernel.cuh (or, for K == 0, by one
// cudaMemsetAsync of +0, the value of the empty sum).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "gemm_f16.h"
#include "attention_launch.cuh"
#include "gemm_fp8_launch.cuh"
#include "gemm_launch.cuh"

using namespace gemm_sm103;

// Device status word of each GPU: 0 = fine; otherwise the first timeout record
// written by a kernel (wait site | block << 8).  Kernels get its address.
__device__ unsigned long long g_gemm_f16_status;

namespace {

// Reason for the last rejected call on this thread (static strings only).
thread_local const char *t_last_detail = "";

constexpr int kMaxFromHostPanels = 8;   // row panels of gemm_f16_from_host

int reject(int status, const char *why)
{
    t_last_detail = why;
    return status;
}

// ---------------------------------------------------------------- configurations

struct ConfigInfo {
    const char *name;
    int tile_m;       // rows of C per work unit (all CTAs of the unit together)
    int tile_n;       // columns of C per work unit
    int all_layouts;  // 1: NN, NT, TN and TT operand layouts; 0: NN only
};

// id 1..kNumConfigs; index 0 is "auto".
constexpr ConfigInfo kConfigs[] = {
    {"auto", 0, 0, 1},
    {"1sm_128x256_s4", Cfg1x256::SUPER_M, Cfg1x256::BN, 1},
    {"1sm_128x128_s6", Cfg1x128::SUPER_M, Cfg1x128::BN, 1},
    {"2sm_256x256_s6", Cfg2x256::SUPER_M, Cfg2x256::BN, 1},
    {"2sm_256x256_s7_direct", Cfg2x256d::SUPER_M, Cfg2x256d::BN, 0},
    {"2sm_256x512_s4", Cfg2x512::SUPER_M, Cfg2x512::BN, 1},
    {"1sm_128x128_ck_s6", Cfg1x128ck::SUPER_M, Cfg1x128ck::BN, 0},
};
// The configuration whose K split runs across a cluster (no workspace).
constexpr int kClusterKConfig = 6;
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

// Filled once per device; read without locking afterwards.
std::atomic<int> g_device_state[kMaxDevices];   // 0 unknown, 1 supported, 2 unsupported
int g_device_sms[kMaxDevices];
std::atomic<unsigned long long *> g_status_addr[kMaxDevices];

int current_device_info(DeviceInfo *out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    // Driver-level calls (cuMemGetAddressRange) need the device's primary
    // context current on this thread; a thread whose first CUDA work is this
    // call (e.g. the autograd engine's backward thread) has none yet.
    // cudaSetDevice initialises the primary context and makes it current.
    thread_local int t_bound_device = -1;
    if (t_bound_device != dev) {
        if (cudaSetDevice(dev) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        t_bound_device = dev;
    }
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

// Device address of this GPU's status word (cached per device).
unsigned long long *status_word(int dev)
{
    unsigned long long *p = g_status_addr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void *q = nullptr;
    if (cudaGetSymbolAddress(&q, g_gemm_f16_status) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    p = static_cast<unsigned long long *>(q);
    g_status_addr[dev].store(p, std::memory_order_release);
    return p;
}

// ---------------------------------------------------------------- argument checks

// A device buffer of `bytes` bytes starting at p: device (or managed) memory of
// device `dev`, entirely inside one allocation.
int check_device_buffer(const void *p, uint64_t bytes, int dev, uintptr_t align = 16)
{
    if (p == nullptr) return reject(GEMM_ERR_INVALID_ARG, "a buffer pointer is NULL");
    if ((reinterpret_cast<uintptr_t>(p) & (align - 1)) != 0)
        return reject(GEMM_ERR_ALIGNMENT, "a buffer pointer is not aligned (16 bytes for GEMM operands)");
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return reject(GEMM_ERR_INVALID_ARG, "cudaPointerGetAttributes failed on a buffer pointer");
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return reject(GEMM_ERR_INVALID_ARG, "a buffer is not device or managed memory");
    if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
        return reject(GEMM_ERR_INVALID_ARG, "a buffer lives on another device than the current one");
    const DriverFns &fns = driver();
    if (!fns.ok) return reject(GEMM_ERR_CUDA, "driver entry points unavailable");
    CUdeviceptr base = 0;
    size_t size = 0;
    if (fns.range(&base, &size, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS)
        return reject(GEMM_ERR_INVALID_ARG, "cuMemGetAddressRange does not know a buffer pointer");
    const uint64_t off = static_cast<uint64_t>(reinterpret_cast<CUdeviceptr>(p) - base);
    if (off > size || bytes > size - off)
        return reject(GEMM_ERR_INVALID_ARG, "a buffer is smaller than its matrix (runs past its allocation)");
    return GEMM_OK;
}

bool ranges_overlap(const void *a, uint64_t abytes, const void *b, uint64_t bbytes)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bbytes && b0 < a0 + abytes;
}

int check_sizes(int64_t M, int64_t N, int64_t K, int relu)
{
    if (M < 0 || N < 0 || K < 0) return reject(GEMM_ERR_INVALID_ARG, "a size is negative");
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return reject(GEMM_ERR_INVALID_ARG, "a size exceeds INT32_MAX");
    if (relu != 0 && relu != 1) return reject(GEMM_ERR_INVALID_ARG, "relu is not 0 or 1");
    return GEMM_OK;
}

}  // namespace

namespace gemm_sm103 {

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

// Row-major one-byte-element matrix (E4M3 codes) rows x cols, leading
// dimension cols bytes, boxes of box_cols x box_rows with 128-byte swizzle.
int encode_matrix_u8(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t cols, uint32_t box_cols,
                     uint32_t box_rows)
{
    const DriverFns &fns = driver();
    if (!fns.ok) return GEMM_ERR_CUDA;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fns.encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// (batch * heads, seq, dim) fp16 tensor, dims innermost first: dim, seq,
// batch * heads; boxes of 64 x 128 x 1 with 128-byte swizzle.  A box never
// crosses into another head's rows: rows past seq read as zero.
int encode_bhsd(CUtensorMap *map, const void *ptr, uint64_t bh, uint64_t seq, uint64_t dim)
{
    const DriverFns &fns = driver();
    if (!fns.ok) return GEMM_ERR_CUDA;
    cuuint64_t dims[3] = {dim, seq, bh};
    cuuint64_t strides[2] = {dim * 2, seq * dim * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fns.encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// Optional rasterisation panel height (in work units) for tuning sweeps.
int group_m_override()
{
    static int v = [] {
        const char *e = std::getenv("GEMM_F16_GROUP_M");
        const int x = e ? std::atoi(e) : 0;
        return x > 0 && x <= 4096 ? x : 0;
    }();
    return v;
}

}  // namespace gemm_sm103

namespace {

// ---------------------------------------------------------------- configuration choice

int pick_config(int64_t M, int64_t N, int64_t K, int sm_count)
{
    const int64_t pairs = sm_count / 2;
    const int64_t tiles_256x512 = ((M + 255) / 256) * ((N + 511) / 512);
    // At least one full wave of 256x512 pair tiles and a long K loop: the wide
    // tile needs the fewest operand bytes per flop.  Its tail is left whole:
    // a split tail runs 256-column MMAs on half the operand reuse.
    if (tiles_256x512 >= pairs && K >= 2048) return 5 | GEMM_F16_NO_SPLIT;
    const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
    // Enough 256x256 tiles to keep every SM pair busy: the CTA-pair kernel.
    if (pair_tiles >= pairs) return 3;
    const int64_t tiles256 = ((M + 127) / 128) * ((N + 255) / 256);
    if (tiles256 >= sm_count / 2) return 1;
    // Few tiles: narrower tiles put more SMs to work.
    return 2;
}

// ---------------------------------------------------------------- tuned selection

#if __has_include("gemm_f16_tuned.inc")
#include "gemm_f16_tuned.inc"
#define GEMM_F16_HAVE_TUNED 1
#else
#define GEMM_F16_HAVE_TUNED 0
#endif

int config_info(int cfg, int64_t M, int64_t N, bool split, const DeviceInfo &dev, int *grid_ctas, int *cluster_size,
                int *tiles)
{
    switch (cfg) {
        case 1: return launch_info_config_1(M, N, split, dev, grid_ctas, cluster_size, tiles);
        case 2: return launch_info_config_2(M, N, split, dev, grid_ctas, cluster_size, tiles);
        case 3: return launch_info_config_3(M, N, split, dev, grid_ctas, cluster_size, tiles);
        case 4: return launch_info_config_4(M, N, split, dev, grid_ctas, cluster_size, tiles);
        case 5: return launch_info_config_5(M, N, split, dev, grid_ctas, cluster_size, tiles);
        case 6: return launch_info_config_6(M, N, split, dev, grid_ctas, cluster_size, tiles);
        default: return GEMM_ERR_INVALID_ARG;
    }
}

// Resident CTAs (or clusters) of configuration `cfg` on this device: the grid
// of a problem large enough to fill every slot.
int64_t config_slots(int cfg, const DeviceInfo &dev)
{
    int grid = 0, cluster = 1, tiles = 0;
    if (config_info(cfg, int64_t{1} << 16, int64_t{1} << 16, false, dev, &grid, &cluster, &tiles) != GEMM_OK ||
        cluster <= 0)
        return 0;
    return grid / cluster;
}

// The slice count of GEMM_F16_KSPLIT_AUTO for configuration `cfg` (1: none):
// if its tiles are fewer than its CTA slots, as many slices as fill the slots
// once, at least 16 K blocks each, at most 16.
int rule_k_splits(int cfg, int64_t M, int64_t N, int64_t K, const DeviceInfo &dev)
{
    int grid = 0, cluster = 1, tiles = 0;
    if (config_info(cfg, M, N, false, dev, &grid, &cluster, &tiles) != GEMM_OK || cluster <= 0) return 1;
    const int64_t slots = config_slots(cfg, dev);
    const int64_t k_blocks = (K + 63) / 64;
    if (tiles <= 0 || tiles >= slots) return 1;
    int64_t n = slots / tiles;
    if (n > k_blocks / 16) n = k_blocks / 16;
    if (n > 16) n = 16;
    return n >= 2 ? static_cast<int>(n) : 1;
}

double wave_eff(int id, int64_t M, int64_t N, bool split, const DeviceInfo &dev)
{
    switch (id) {
        case 1: return wave_eff_config_1(M, N, split, dev);
        case 2: return wave_eff_config_2(M, N, split, dev);
        case 3: return wave_eff_config_3(M, N, split, dev);
        case 4: return wave_eff_config_4(M, N, split, dev);
        case 5: return wave_eff_config_5(M, N, split, dev);
        case 6: return wave_eff_config_6(M, N, split, dev);
        default: return 0.0;
    }
}

// Cluster size request of a config word for the cluster K split configuration:
// GEMM_F16_KSPLIT(n) asks for n CTAs per cluster, GEMM_F16_NO_KSPLIT for one,
// anything else for the size rule (0).
int ck_request_of(int word)
{
    const int n = (word & GEMM_F16_KSPLIT_MASK) >> GEMM_F16_KSPLIT_SHIFT;
    if (n >= 2) return n;
    if (word & GEMM_F16_NO_KSPLIT) return 1;
    return 0;
}

// The automatic choice.  The offline sweep (tune.py) measured every candidate
// (configuration x tail policy, and the cluster K split's sizes) on a grid of
// shapes.  None of the candidates allocates memory: a workspace K split is
// taken only on an explicit request (gemm_f16_ex with the K-split bits).  For a problem, take the
// nearest measured shape in log2 space (K weighted by half: it changes the
// per-tile work but not the wave count), scale each candidate's measured
// throughput by its wave efficiency here over its wave efficiency there, and
// take the best.  `any_layout`: only configurations with transposed-layout
// kernels qualify.  Without a table, the size rule above.
int select_config(int64_t M, int64_t N, int64_t K, bool any_layout, const DeviceInfo &dev)
{
#if GEMM_F16_HAVE_TUNED
    // The last choices are kept per thread (callers often repeat a few shapes).
    struct Last {
        int64_t M = -1, N = -1, K = -1;
        int device = -1, any_layout = -1, choice = 0;
    };
    constexpr int kCached = 64;
    thread_local Last cache[kCached];
    thread_local int next_slot = 0;
    for (const Last &c : cache)
        if (c.M == M && c.N == N && c.K == K && c.device == dev.device && c.any_layout == (any_layout ? 1 : 0))
            return c.choice;
    const double lm = std::log2(static_cast<double>(M > 0 ? M : 1));
    const double ln = std::log2(static_cast<double>(N > 0 ? N : 1));
    const double lk = std::log2(static_cast<double>(K > 0 ? K : 1));
    int row = 0;
    double best_d = 1e300;
    for (int r = 0; r < GEMM_F16_TUNED_ROWS; ++r) {
        const TunedRow &t = kTunedRows[r];
        const double d = std::fabs(lm - std::log2(static_cast<double>(t.M))) +
                         std::fabs(ln - std::log2(static_cast<double>(t.N))) +
                         0.5 * std::fabs(lk - std::log2(static_cast<double>(t.K)));
        if (d < best_d) {
            best_d = d;
            row = r;
        }
    }
    const TunedRow &t = kTunedRows[row];
    int choice = 0;
    double best = 0.0;
    for (int i = 0; i < GEMM_F16_TUNED_CANDIDATES; ++i) {
        const int c = kTunedCandidates[i];
        const int id = c & GEMM_F16_CONFIG_ID_MASK;
        if (id < 1 || id > kNumConfigs || (any_layout && !kConfigs[id].all_layouts)) continue;
        const bool split = (c & GEMM_F16_NO_SPLIT) == 0;
        const bool ck = id == kClusterKConfig;
        // The automatic choice allocates nothing: no workspace K split.
        if (!ck && (c & (GEMM_F16_KSPLIT_AUTO | GEMM_F16_KSPLIT_TAIL | GEMM_F16_KSPLIT_MASK)) != 0) continue;
        const double here = ck ? ck_wave_eff_config_6(M, N, K, ck_request_of(c), dev) : wave_eff(id, M, N, split, dev);
        const double there =
            ck ? ck_wave_eff_config_6(t.M, t.N, t.K, ck_request_of(c), dev) : wave_eff(id, t.M, t.N, split, dev);
        if (here <= 0.0 || there <= 0.0) continue;
        // (ratio first: exactly 1 on a measured shape, so ties keep table order)
        const double predicted = static_cast<double>(t.tflops[i]) * (here / there);
        if (predicted > best) {
            best = predicted;
            choice = c;
        }
    }
    if (choice != 0) {
        cache[next_slot] = Last{M, N, K, dev.device, any_layout ? 1 : 0, choice};
        next_slot = (next_slot + 1) % kCached;
        return choice;
    }
#endif
    (void)any_layout;
    return pick_config(M, N, K, dev.sm_count);
}

// K-split requests of a config word (parse_config's *k_request).
constexpr int kKsplitNever = -1;   // GEMM_F16_NO_KSPLIT (0: no K-split bit set)
constexpr int kKsplitRule = -2;    // GEMM_F16_KSPLIT_AUTO
constexpr int kKsplitTail = -3;    // GEMM_F16_KSPLIT_TAIL
                                   // n >= 2: GEMM_F16_KSPLIT(n)

// Splits a config argument into the configuration id and its flag bits;
// false for an unknown id or flag or contradictory K-split bits.
bool parse_config(int config, int *id, bool *allow_split, int *k_request = nullptr)
{
    constexpr int kKnown = GEMM_F16_CONFIG_ID_MASK | GEMM_F16_NO_SPLIT | GEMM_F16_NO_KSPLIT | GEMM_F16_KSPLIT_AUTO |
                           GEMM_F16_KSPLIT_TAIL | GEMM_F16_KSPLIT_MASK;
    if (config < 0 || (config & ~kKnown) != 0) return false;
    const int n = (config & GEMM_F16_KSPLIT_MASK) >> GEMM_F16_KSPLIT_SHIFT;
    const bool never = (config & GEMM_F16_NO_KSPLIT) != 0;
    const bool rule = (config & GEMM_F16_KSPLIT_AUTO) != 0;
    const bool tail = (config & GEMM_F16_KSPLIT_TAIL) != 0;
    if (n == 1 || n > 16 ||
        static_cast<int>(never) + static_cast<int>(rule) + static_cast<int>(tail) + static_cast<int>(n != 0) > 1)
        return false;
    *id = config & GEMM_F16_CONFIG_ID_MASK;
    *allow_split = (config & GEMM_F16_NO_SPLIT) == 0;
    if (k_request) *k_request = never ? kKsplitNever : rule ? kKsplitRule : tail ? kKsplitTail : n;
    return *id <= kNumConfigs;
}

// Workspace slice count for a parsed request on configuration `cfg` (the
// automatic choice never asks for one).
int k_splits_for(int k_request, int cfg, int64_t M, int64_t N, int64_t K, const DeviceInfo &dev)
{
    if (k_request >= 2) return k_request;
    if (k_request == kKsplitRule) return rule_k_splits(cfg, M, N, K, dev);
    return 1;
}

// ---------------------------------------------------------------- launch path

int run_gemm(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int transa, int transb,
             int relu, int config, void *stream, const LaunchHook &hook, bool noalloc = false)
{
    int st = check_sizes(M, N, K, relu);
    if (st != GEMM_OK) return st;
    if ((transa != 0 && transa != 1) || (transb != 0 && transb != 1))
        return reject(GEMM_ERR_INVALID_ARG, "transa / transb is not 0 or 1");
    int id = 0, k_request = 0;
    bool allow_split = true;
    if (!parse_config(config, &id, &allow_split, &k_request))
        return reject(GEMM_ERR_INVALID_ARG, "unknown configuration id or flag");
    if ((transa || transb) && !kConfigs[id].all_layouts)
        return reject(GEMM_ERR_INVALID_ARG, "this configuration has no transposed-layout kernels");
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
    // Row pitches of the stored matrices must be multiples of 16 bytes.
    const int64_t lda = transa ? M : K, ldb = transb ? K : N;
    if ((lda % 8) != 0 || (ldb % 8) != 0 || (N % 8) != 0)
        return reject(GEMM_ERR_ALIGNMENT, "a row pitch (leading dimension) is not a multiple of 8 elements");
    const uint64_t a_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(K) * 2u;
    const uint64_t b_bytes = static_cast<uint64_t>(K) * static_cast<uint64_t>(N) * 2u;
    if ((st = check_device_buffer(A, a_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(B, b_bytes, dev.device)) != GEMM_OK) return st;
    if (ranges_overlap(C, c_bytes, A, a_bytes) || ranges_overlap(C, c_bytes, B, b_bytes))
        return reject(GEMM_ERR_INVALID_ARG, "C overlaps A or B");

    LaunchArgs a;
    a.A = A;
    a.B = B;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.relu = relu;
    a.transa = transa;
    a.transb = transb;
    a.dev = dev;
    a.stream = s;
    a.hook = hook;
    a.status = status_word(dev.device);
    if (a.status == nullptr) return GEMM_ERR_CUDA;

    int cfg = id, picked = 0;
    if (id == 0) {
        picked = select_config(M, N, K, transa || transb, dev);
        cfg = picked & GEMM_F16_CONFIG_ID_MASK;
        a.allow_split = allow_split && (picked & GEMM_F16_NO_SPLIT) == 0;
    } else {
        a.allow_split = allow_split;
    }
    if (cfg == kClusterKConfig) {
        // The K split runs across the cluster: its size from the config word
        // (or from the automatic choice's word), no workspace.
        if (k_request == kKsplitTail)
            return reject(GEMM_ERR_INVALID_ARG, "the cluster K split configuration has no tail split");
        a.ck_request = id == 0 ? ck_request_of(picked)
                       : k_request >= 2 ? k_request
                       : k_request == kKsplitNever ? 1 : 0;
        if (a.ck_request != 0 && a.ck_request != 1 && a.ck_request != 2 && a.ck_request != 4 && a.ck_request != 8)
            return reject(GEMM_ERR_INVALID_ARG, "a cluster K split takes 2, 4 or 8 CTAs per cluster");
        a.k_splits = 1;
        a.k_split_tail = false;
    } else {
        a.k_splits = k_splits_for(k_request, cfg, M, N, K, dev);
        a.k_split_tail = k_request == kKsplitTail;
    }
    if (hook.producer_off) {
        // the timeout self-test never writes C
        a.k_splits = 1;
        a.k_split_tail = false;
    }
    // K-slice partials of a noalloc call go to the library's fixed scratch;
    // the launch rejects a split that does not fit before it enqueues anything.
    a.noalloc = noalloc;
    switch (cfg) {
        case 1: st = launch_config_1(a); break;
        case 2: st = launch_config_2(a); break;
        case 3: st = launch_config_3(a); break;
        case 4: st = launch_config_4(a); break;
        case 5: st = launch_config_5(a); break;
        case 6: st = launch_config_6(a); break;
        default: return GEMM_ERR_INVALID_ARG;
    }
    if (st == GEMM_ERR_INVALID_ARG)
        return reject(st, noalloc ? "the K-slice partials exceed the 16 MiB scratch of gemm_f16_ex_noalloc"
                                  : "the problem has too many work units");
    return st;
}

thread_local uint64_t t_last_timeout_record = 0;

}  // namespace

// ==================================================================== C ABI

extern "C" int gemm_f16_tx(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int transa,
                           int transb, int relu, int config, void *stream)
{
    return run_gemm(A, B, C, M, N, K, transa, transb, relu, config, stream, LaunchHook());
}

extern "C" int gemm_f16_ex(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int relu,
                           int config, void *stream)
{
    return run_gemm(A, B, C, M, N, K, 0, 0, relu, config, stream, LaunchHook());
}

extern "C" int gemm_f16_ex_noalloc(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int relu,
                                   int config, void *stream)
{
    return run_gemm(A, B, C, M, N, K, 0, 0, relu, config, stream, LaunchHook{}, true);
}

extern "C" int gemm_f16(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K, int relu,
                        void *stream)
{
    return run_gemm(A, B, C, M, N, K, 0, 0, relu, 0, stream, LaunchHook());
}

extern "C" int gemm_f16_selftest_timeout(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                                         int config, uint64_t timeout_cycles, void *stream)
{
    if (K == 0 || M == 0 || N == 0) return reject(GEMM_ERR_INVALID_ARG, "an empty problem launches no kernel");
    if (timeout_cycles < (1ull << 16) || timeout_cycles > (1ull << 32))
        return reject(GEMM_ERR_INVALID_ARG, "timeout_cycles outside 2^16 .. 2^32");
    LaunchHook hook;
    hook.producer_off = 1;
    hook.timeout_cycles = timeout_cycles;
    return run_gemm(A, B, C, M, N, K, 0, 0, 1, config, stream, hook);
}

namespace gemm_sm103 {
int tma_box_image_launch(const void *X, int64_t rows, int64_t cols, int box_rows, int x, int y, void *out,
                         unsigned long long *status, cudaStream_t stream);
}

extern "C" int gemm_f16_tma_box_image(const void *X, int64_t rows, int64_t cols, int64_t box_rows, int64_t x,
                                      int64_t y, void *out, void *stream)
{
    if (rows < 1 || cols < 1 || rows > INT32_MAX || cols > INT32_MAX)
        return reject(GEMM_ERR_INVALID_ARG, "rows and cols must be 1 .. INT32_MAX");
    if (box_rows < 1 || box_rows > 256) return reject(GEMM_ERR_INVALID_ARG, "box_rows must be 1 .. 256");
    if (x < INT32_MIN || x > INT32_MAX || y < INT32_MIN || y > INT32_MAX)
        return reject(GEMM_ERR_INVALID_ARG, "a box coordinate is outside the 32-bit range");
    if ((cols % 8) != 0) return reject(GEMM_ERR_ALIGNMENT, "cols (the row pitch) is not a multiple of 8 elements");
    if ((x % 8) != 0)
        return reject(GEMM_ERR_ALIGNMENT, "x is not a multiple of 8 elements (a box starts on a 16-byte boundary)");
    DeviceInfo dev;
    int st = current_device_info(&dev);
    if (st != GEMM_OK) return st;
    const uint64_t x_bytes = static_cast<uint64_t>(rows) * static_cast<uint64_t>(cols) * 2u;
    const uint64_t out_bytes = static_cast<uint64_t>(box_rows) * 128u;
    if ((st = check_device_buffer(X, x_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(out, out_bytes, dev.device)) != GEMM_OK) return st;
    if (ranges_overlap(out, out_bytes, X, x_bytes)) return reject(GEMM_ERR_INVALID_ARG, "out overlaps X");
    unsigned long long *status = status_word(dev.device);
    if (status == nullptr) return GEMM_ERR_CUDA;
    return tma_box_image_launch(X, rows, cols, static_cast<int>(box_rows), static_cast<int>(x), static_cast<int>(y),
                                out, status, static_cast<cudaStream_t>(stream));
}

namespace gemm_sm103 {
int relu_backward_launch(const void *dC, const void *C, void *dZ, int64_t n, int sm_count, cudaStream_t stream);
}

extern "C" int gemm_f16_relu_backward(const void *dC, const void *C, void *dZ, int64_t n, void *stream)
{
    if (n < 0) return reject(GEMM_ERR_INVALID_ARG, "n is negative");
    if (n == 0) return GEMM_OK;
    DeviceInfo dev;
    int st = current_device_info(&dev);
    if (st != GEMM_OK) return st;
    const uint64_t bytes = static_cast<uint64_t>(n) * 2u;
    if ((st = check_device_buffer(dC, bytes, dev.device, 2)) != GEMM_OK) return st;
    if ((st = check_device_buffer(C, bytes, dev.device, 2)) != GEMM_OK) return st;
    if ((st = check_device_buffer(dZ, bytes, dev.device, 2)) != GEMM_OK) return st;
    // In place over dC (or C) is fine element by element; a partial overlap is not.
    if ((dZ != dC && ranges_overlap(dZ, bytes, dC, bytes)) || (dZ != C && ranges_overlap(dZ, bytes, C, bytes)))
        return reject(GEMM_ERR_INVALID_ARG, "dZ partly overlaps dC or C");
    return relu_backward_launch(dC, C, dZ, n, dev.sm_count, static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_fp8_block_scaled(const void *A, const float *SA, const void *W, const float *SW, void *C,
                                     int64_t M, int64_t N, int64_t K, int relu, void *stream)
{
    int st = check_sizes(M, N, K, relu);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t c_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(N) * 2u;
    if ((st = check_device_buffer(C, c_bytes, dev.device)) != GEMM_OK) return st;
    if (K == 0) {
        // Empty sum in every block: every output is R(+0) = +0.
        if (cudaMemsetAsync(C, 0, c_bytes, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    if ((K % 16) != 0)
        return reject(GEMM_ERR_ALIGNMENT, "K is not a multiple of 16 (the E4M3 row pitch of A and W is K bytes)");
    if ((N % 8) != 0) return reject(GEMM_ERR_ALIGNMENT, "N is not a multiple of 8 (the fp16 row pitch of C)");
    const uint64_t KB = static_cast<uint64_t>((K + 127) / 128), NB = static_cast<uint64_t>((N + 127) / 128);
    const uint64_t a_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(K);
    const uint64_t w_bytes = static_cast<uint64_t>(N) * static_cast<uint64_t>(K);
    const uint64_t sa_bytes = static_cast<uint64_t>(M) * KB * 4u, sw_bytes = NB * KB * 4u;
    if ((st = check_device_buffer(A, a_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(W, w_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(SA, sa_bytes, dev.device, 4)) != GEMM_OK) return st;
    if ((st = check_device_buffer(SW, sw_bytes, dev.device, 4)) != GEMM_OK) return st;
    if (ranges_overlap(C, c_bytes, A, a_bytes) || ranges_overlap(C, c_bytes, W, w_bytes) ||
        ranges_overlap(C, c_bytes, SA, sa_bytes) || ranges_overlap(C, c_bytes, SW, sw_bytes))
        return reject(GEMM_ERR_INVALID_ARG, "C overlaps an input");
    Fp8LaunchArgs a;
    a.A = A;
    a.SA = SA;
    a.W = W;
    a.SW = SW;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.relu = relu;
    a.dev = dev;
    a.stream = s;
    a.status = status_word(dev.device);
    if (a.status == nullptr) return GEMM_ERR_CUDA;
    return launch_fp8(a);
}

extern "C" int gemm_mxfp8_block_scaled(const void *A, const uint8_t *SA, const void *W, const uint8_t *SW, void *C,
                                       int64_t M, int64_t N, int64_t K, int relu, void *stream)
{
    int st = check_sizes(M, N, K, relu);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t c_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(N) * 2u;
    if ((st = check_device_buffer(C, c_bytes, dev.device)) != GEMM_OK) return st;
    if (K == 0) {
        // Empty sum in every block: every output is R(+0) = +0.
        if (cudaMemsetAsync(C, 0, c_bytes, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    if ((K % 16) != 0)
        return reject(GEMM_ERR_ALIGNMENT, "K is not a multiple of 16 (the E4M3 row pitch of A and W is K bytes)");
    if ((N % 8) != 0) return reject(GEMM_ERR_ALIGNMENT, "N is not a multiple of 8 (the fp16 row pitch of C)");
    const uint64_t KB = static_cast<uint64_t>((K + 127) / 128), NB = static_cast<uint64_t>((N + 127) / 128);
    const uint64_t a_bytes = static_cast<uint64_t>(M) * static_cast<uint64_t>(K);
    const uint64_t w_bytes = static_cast<uint64_t>(N) * static_cast<uint64_t>(K);
    const uint64_t sa_bytes = static_cast<uint64_t>(M) * KB, sw_bytes = NB * KB;
    if ((st = check_device_buffer(A, a_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(W, w_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(SA, sa_bytes, dev.device, 1)) != GEMM_OK) return st;
    if ((st = check_device_buffer(SW, sw_bytes, dev.device, 1)) != GEMM_OK) return st;
    if (ranges_overlap(C, c_bytes, A, a_bytes) || ranges_overlap(C, c_bytes, W, w_bytes) ||
        ranges_overlap(C, c_bytes, SA, sa_bytes) || ranges_overlap(C, c_bytes, SW, sw_bytes))
        return reject(GEMM_ERR_INVALID_ARG, "C overlaps an input");
    MxLaunchArgs a;
    a.A = A;
    a.SA = SA;
    a.W = W;
    a.SW = SW;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.relu = relu;
    a.dev = dev;
    a.stream = s;
    a.status = status_word(dev.device);
    if (a.status == nullptr) return GEMM_ERR_CUDA;
    return launch_mxfp8(a);
}

extern "C" int gemm_fp8_launch_info(int64_t M, int64_t N, int64_t K, int *grid_ctas, int *tiles)
{
    int st = check_sizes(M, N, K, 0);
    if (st != GEMM_OK) return st;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    return fp8_launch_info(M, N, dev, grid_ctas, tiles);
}

extern "C" int attention_fwd_f16(const void *Q, const void *K, const void *V, void *O, int64_t batch,
                                 int64_t heads, int64_t seq, int64_t dim, float sm_scale, int causal, void *stream)
{
    return attention_fwd_f16_queue(Q, K, V, O, batch, heads, seq, dim, sm_scale, causal, nullptr, stream);
}

extern "C" int attention_fwd_f16_queue(const void *Q, const void *K, const void *V, void *O, int64_t batch,
                                       int64_t heads, int64_t seq, int64_t dim, float sm_scale, int causal,
                                       unsigned int *queue, void *stream)
{
    if (batch < 0 || heads < 0 || seq < 0) return reject(GEMM_ERR_INVALID_ARG, "a size is negative");
    if (dim != 64 && dim != 128) return reject(GEMM_ERR_INVALID_ARG, "dim is not 64 or 128");
    if (causal != 0 && causal != 1) return reject(GEMM_ERR_INVALID_ARG, "causal is not 0 or 1");
    if (!std::isfinite(sm_scale)) return reject(GEMM_ERR_INVALID_ARG, "sm_scale is not finite");
    if (batch > 65535 || heads > 65535 || seq > INT32_MAX)
        return reject(GEMM_ERR_INVALID_ARG, "batch or heads above 65535, or seq above INT32_MAX");
    if (batch == 0 || heads == 0 || seq == 0) return GEMM_OK;
    DeviceInfo dev;
    int st = current_device_info(&dev);
    if (st != GEMM_OK) return st;
    const uint64_t bytes = static_cast<uint64_t>(batch) * static_cast<uint64_t>(heads) * static_cast<uint64_t>(seq) *
                           static_cast<uint64_t>(dim) * 2u;
    if ((st = check_device_buffer(Q, bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(K, bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(V, bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(O, bytes, dev.device)) != GEMM_OK) return st;
    if (ranges_overlap(O, bytes, Q, bytes) || ranges_overlap(O, bytes, K, bytes) || ranges_overlap(O, bytes, V, bytes))
        return reject(GEMM_ERR_INVALID_ARG, "O overlaps Q, K or V");
    if (causal && queue != nullptr) {
        const uint64_t qb = 2 * sizeof(unsigned int);
        if ((st = check_device_buffer(queue, qb, dev.device, 4)) != GEMM_OK) return st;
        if (ranges_overlap(queue, qb, O, bytes) || ranges_overlap(queue, qb, Q, bytes) ||
            ranges_overlap(queue, qb, K, bytes) || ranges_overlap(queue, qb, V, bytes))
            return reject(GEMM_ERR_INVALID_ARG, "queue overlaps Q, K, V or O");
    }
    AttnLaunchArgs a;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.O = O;
    a.batch = batch;
    a.heads = heads;
    a.seq = seq;
    a.dim = dim;
    a.sm_scale = sm_scale;
    a.causal = causal;
    a.dev = dev;
    a.stream = static_cast<cudaStream_t>(stream);
    a.status = status_word(dev.device);
    if (a.status == nullptr) return GEMM_ERR_CUDA;
    a.queue = causal ? queue : nullptr;
    return launch_attention(a);
}

extern "C" int gemm_f16_num_configs(void) { return kNumConfigs; }

extern "C" const char *gemm_f16_config_name(int config)
{
    int id = 0;
    bool allow_split = true;
    if (!parse_config(config, &id, &allow_split)) return nullptr;
    return kConfigs[id].name;
}

extern "C" int gemm_f16_config_layouts(int config)
{
    int id = 0;
    bool allow_split = true;
    if (!parse_config(config, &id, &allow_split))
        return reject(GEMM_ERR_INVALID_ARG, "unknown configuration id or flag");
    return kConfigs[id].all_layouts ? 0xF : 0x1;
}

extern "C" int gemm_f16_config_cluster_k(int config)
{
    int id = 0;
    bool allow_split = true;
    if (!parse_config(config, &id, &allow_split))
        return reject(GEMM_ERR_INVALID_ARG, "unknown configuration id or flag");
    return id == kClusterKConfig ? 1 : 0;
}

extern "C" int gemm_f16_auto_config(int64_t M, int64_t N, int64_t K)
{
    int st = check_sizes(M, N, K, 0);
    if (st != GEMM_OK) return st;
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    const int picked = select_config(M, N, K, false, dev);
    const int cfg = picked & GEMM_F16_CONFIG_ID_MASK;
    if (cfg == kClusterKConfig) {
        // The cluster size resolved for this problem.
        int cluster = 1;
        ck_launch_info_config_6(M, N, K, ck_request_of(picked), dev, nullptr, &cluster, nullptr);
        return cfg | (cluster >= 2 ? GEMM_F16_KSPLIT(cluster) : GEMM_F16_NO_KSPLIT);
    }
    return picked;
}

extern "C" int gemm_f16_launch_info(int64_t M, int64_t N, int64_t K, int config, int *grid_ctas,
                                    int *cluster_size, int *tiles)
{
    int st = check_sizes(M, N, K, 0);
    if (st != GEMM_OK) return st;
    int id = 0, k_request = 0;
    bool split = true;
    if (!parse_config(config, &id, &split, &k_request))
        return reject(GEMM_ERR_INVALID_ARG, "unknown configuration id or flag");
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    int cfg = id, picked = 0;
    if (id == 0) {
        picked = select_config(M, N, K, false, dev);
        cfg = picked & GEMM_F16_CONFIG_ID_MASK;
        split = split && (picked & GEMM_F16_NO_SPLIT) == 0;
    }
    if (cfg == kClusterKConfig) {
        const int request = id == 0 ? ck_request_of(picked)
                            : k_request >= 2 ? k_request
                            : k_request == kKsplitNever ? 1 : 0;
        return ck_launch_info_config_6(M, N, K, request, dev, grid_ctas, cluster_size, tiles);
    }
    const int k_req = k_splits_for(k_request, cfg, M, N, K, dev);
    const bool tail = k_request == kKsplitTail;
    int grid = 0, cluster = 1, n_tiles = 0;
    if ((st = config_info(cfg, M, N, split && k_req <= 1 && !tail, dev, &grid, &cluster, &n_tiles)) != GEMM_OK)
        return st;
    const int64_t slots = config_slots(cfg, dev);
    const KPlan kp = plan_k_split(n_tiles, slots, (K + 63) / 64, k_req, tail);
    if (kp.ks.count > 1) {
        // Whole tiles, then K slices, on at most one CTA (cluster) per slot.
        const int64_t units = kp.units(n_tiles);
        grid = static_cast<int>((units < slots ? units : slots) * cluster);
    }
    if (grid_ctas) *grid_ctas = grid;
    if (cluster_size) *cluster_size = cluster;
    if (tiles) *tiles = n_tiles;
    return GEMM_OK;
}

namespace {

// Per device: the two streams the host-buffer entry point moves data on
// (uploads, downloads), created by its first call on that device.
struct CopyStreams {
    cudaStream_t in = nullptr, out = nullptr;
    int status = GEMM_ERR_CUDA;
};
CopyStreams g_copy_streams[kMaxDevices];
std::once_flag g_copy_once[kMaxDevices];

int copy_streams(int dev, CopyStreams **out)
{
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::call_once(g_copy_once[dev], [dev]() {
        CopyStreams &c = g_copy_streams[dev];
        if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) == cudaSuccess) {
            c.status = GEMM_OK;
        } else {
            cudaGetLastError();
        }
    });
    *out = &g_copy_streams[dev];
    return g_copy_streams[dev].status;
}

// Events of one call, destroyed once enqueued (they are released when the
// work they mark completes).
struct EventSet {
    cudaEvent_t ev[2 * kMaxFromHostPanels + 2] = {};
    int n = 0;
    bool make(int count)
    {
        for (n = 0; n < count; ++n) {
            if (cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming) != cudaSuccess) {
                cudaGetLastError();
                return false;
            }
        }
        return true;
    }
    ~EventSet()
    {
        for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
    }
};

}  // namespace

extern "C" int gemm_f16_from_host(const void *A_host, const void *B_host, void *C_host, void *A_dev, void *B_dev,
                                  void *C_dev, int64_t M, int64_t N, int64_t K, int relu, void *stream)
{
    int st = check_sizes(M, N, K, relu);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    if (C_host == nullptr || (K > 0 && (A_host == nullptr || B_host == nullptr)))
        return reject(GEMM_ERR_INVALID_ARG, "a host buffer pointer is NULL");
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t a_bytes = static_cast<size_t>(M) * static_cast<size_t>(K) * 2u;
    const size_t b_bytes = static_cast<size_t>(K) * static_cast<size_t>(N) * 2u;
    const size_t c_bytes = static_cast<size_t>(M) * static_cast<size_t>(N) * 2u;
    if (K == 0) {
        if ((st = gemm_f16(A_dev, B_dev, C_dev, M, N, K, relu, stream)) != GEMM_OK) return st;
        if (cudaMemcpyAsync(C_host, C_dev, c_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    // Validate the device side before anything is enqueued.
    DeviceInfo dev;
    if ((st = current_device_info(&dev)) != GEMM_OK) return st;
    if ((N % 8) != 0 || (K % 8) != 0)
        return reject(GEMM_ERR_ALIGNMENT, "a row pitch (leading dimension) is not a multiple of 8 elements");
    if ((st = check_device_buffer(A_dev, a_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(B_dev, b_bytes, dev.device)) != GEMM_OK) return st;
    if ((st = check_device_buffer(C_dev, c_bytes, dev.device)) != GEMM_OK) return st;
    if (ranges_overlap(C_dev, c_bytes, A_dev, a_bytes) || ranges_overlap(C_dev, c_bytes, B_dev, b_bytes))
        return reject(GEMM_ERR_INVALID_ARG, "C overlaps A or B");
    CopyStreams *cs = nullptr;
    if ((st = copy_streams(dev.device, &cs)) != GEMM_OK) return st;

    // Row panels of A and C (multiples of 256 rows, at least 1024 each, at
    // most kMaxFromHostPanels): B goes up first, then panel i of A; the GEMM
    // of panel i runs on `stream` once its rows are up; panel i of C comes
    // down while later panels are uploaded and computed.
    int64_t panels = M / 1024;
    if (panels < 1) panels = 1;
    if (panels > kMaxFromHostPanels) panels = kMaxFromHostPanels;
    const int64_t rows = ((M + panels - 1) / panels + 255) / 256 * 256;
    panels = (M + rows - 1) / rows;
    const int np = static_cast<int>(panels);
    EventSet evs;
    if (!evs.make(2 * np + 2)) return GEMM_ERR_CUDA;
    cudaEvent_t e_start = evs.ev[0], e_done = evs.ev[1];
    auto ea = [&](int i) { return evs.ev[2 + i]; };        // panel i of A is up
    auto ec = [&](int i) { return evs.ev[2 + np + i]; };   // panel i of C is computed
    auto fail = []() {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    };
    // The copy streams start after everything already enqueued on `stream`
    // (which may still use A_dev, B_dev or C_dev).
    if (cudaEventRecord(e_start, s) != cudaSuccess || cudaStreamWaitEvent(cs->in, e_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(cs->out, e_start, 0) != cudaSuccess)
        return fail();
    if (cudaMemcpyAsync(B_dev, B_host, b_bytes, cudaMemcpyHostToDevice, cs->in) != cudaSuccess) return fail();
    for (int i = 0; i < np; ++i) {
        const int64_t r0 = i * rows, mi = (M - r0 < rows) ? M - r0 : rows;
        const size_t off = static_cast<size_t>(r0) * static_cast<size_t>(K) * 2u;
        if (cudaMemcpyAsync(static_cast<char *>(A_dev) + off, static_cast<const char *>(A_host) + off,
                            static_cast<size_t>(mi) * static_cast<size_t>(K) * 2u, cudaMemcpyHostToDevice,
                            cs->in) != cudaSuccess ||
            cudaEventRecord(ea(i), cs->in) != cudaSuccess)
            return fail();
    }
    for (int i = 0; i < np; ++i) {
        const int64_t r0 = i * rows, mi = (M - r0 < rows) ? M - r0 : rows;
        if (cudaStreamWaitEvent(s, ea(i), 0) != cudaSuccess) return fail();
        st = gemm_f16(static_cast<const char *>(A_dev) + static_cast<size_t>(r0) * static_cast<size_t>(K) * 2u,
                      B_dev, static_cast<char *>(C_dev) + static_cast<size_t>(r0) * static_cast<size_t>(N) * 2u, mi,
                      N, K, relu, stream);
        if (st != GEMM_OK) return st;
        if (cudaEventRecord(ec(i), s) != cudaSuccess || cudaStreamWaitEvent(cs->out, ec(i), 0) != cudaSuccess)
            return fail();
        const size_t off = static_cast<size_t>(r0) * static_cast<size_t>(N) * 2u;
        if (cudaMemcpyAsync(static_cast<char *>(C_host) + off, static_cast<const char *>(C_dev) + off,
                            static_cast<size_t>(mi) * static_cast<size_t>(N) * 2u, cudaMemcpyDeviceToHost,
                            cs->out) != cudaSuccess)
            return fail();
    }
    // `stream` covers the downloads: synchronising it is enough to read C_host.
    if (cudaEventRecord(e_done, cs->out) != cudaSuccess || cudaStreamWaitEvent(s, e_done, 0) != cudaSuccess)
        return fail();
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

extern "C" const char *gemm_f16_last_error_detail(void) { return t_last_detail; }

extern "C" const char *gemm_f16_strerror(int status)
{
    switch (status) {
        case GEMM_OK: return "success";
        case GEMM_ERR_INVALID_ARG: return "invalid argument";
        case GEMM_ERR_ALIGNMENT: return "misaligned pointer, or a row pitch not a multiple of 8 elements";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (GB300)";
        case GEMM_ERR_LAUNCH: return "kernel launch failed";
        case GEMM_ERR_TIMEOUT: return "a kernel wait exceeded its limit; the output is incomplete";
        case GEMM_ERR_CUDA: return "CUDA runtime or driver call failed";
        default: return "unknown status";
    }
}

extern "C" int gemm_f16_version(void) { return GEMM_F16_VERSION; }
