// gemm_kernel.cuh -- persistent, warp-specialised fp16 GEMM + fused ReLU for
// sm_103a (GB300): TMA -> 128B-swizzled shared-memory ring -> tcgen05.mma with
// the fp32 accumulator in tensor memory -> ReLU / fp16 cast -> TMA store.
//
// The method is the tiled GEMM of "Writing High-Performance Kernels in
// TileLang, from GEMM to MLA" (atlascloud.ai), section "Let's write a GEMM":
// shared-memory tiles of A and B, a software-pipelined K loop with several
// stages in flight, a tile-level MMA into a float accumulator that is cleared
// per output tile, ReLU on the accumulator, one cast on write-back, and an L2
// rasterisation swizzle of the tile order.  Here each of those steps is a
// Blackwell mechanism:
//   * tile copies        -> TMA boxes with 128-byte swizzle (bank-conflict free
//                            for both the copy and the MMA read)
//   * K pipeline         -> a ring of STAGES shared-memory slots guarded by
//                            "full" (TMA bytes landed) and "empty" (MMA done)
//                            mbarriers
//   * tile MMA           -> tcgen05.mma.kind::f16 issued by one thread,
//                            accumulating in TMEM; the first MMA of a tile runs
//                            with accumulate = 0 (the accumulator clear)
//   * ReLU + cast + copy -> 4 epilogue warps: tcgen05.ld -> max(x,0) -> cvt.rn
//                            f16x2 -> swizzled smem -> TMA store
//   * L2 swizzle         -> grouped rasterisation in a persistent tile loop
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of i+1.
//
// CTA-pair mode (CTA_GROUP == 2, a cluster of two CTAs on two SMs): one
// tcgen05.mma.cta_group::2 computes a 256 x BN tile.  Each CTA loads its own
// 128 rows of A and its own BN/2 columns of B into its own shared memory; the
// pair's tensor cores read both halves, and each CTA's TMEM receives its 128
// rows of the accumulator.  Only the even CTA (the leader) issues MMAs: both
// CTAs' loads complete on the leader's "full" barrier, the leader's commits
// arrive on both CTAs' "empty" and "tmem full" barriers, and both CTAs'
// epilogue warps arrive on the leader's "tmem empty" barrier.
//
// Ragged edges: TMA loads fill out-of-range elements with zeros, so partial
// tiles in M, N and K contribute nothing; TMA stores do not write outside C.
//
// Every mbarrier wait is bounded (clock64 budget).  On expiry the waiting
// thread records the site in a device status word, raises the abort flag of
// its CTA (and of the peer CTA in pair mode), and every role leaves its loop;
// the producer then waits (bounded) for its own loads in flight, the MMA thread
// for its own MMAs, the epilogue for its own stores, and the TMEM is freed
// before the CTA exits.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "sm103_ptx.cuh"

namespace gemm_sm103 {

// Problem description passed by value to the kernel.
// Work units: tiles in rasterised order, except that the tiles of a last,
// partly filled wave may be split along N into 2^split_log2 narrower units
// (so that the tail costs a fraction of a tile time instead of a whole one).
struct GemmParams {
    int32_t M, N, K;
    int32_t num_m_blocks;   // ceil(M / tile rows)
    int32_t num_n_blocks;   // ceil(N / tile cols)
    int32_t num_k_blocks;   // ceil(K / BK)
    int32_t num_tiles;      // num_m_blocks * num_n_blocks
    int32_t group_m;        // rasterisation panel height, in tiles
    int32_t num_units;      // split_start + (num_tiles - split_start) << split_log2
    int32_t split_start;    // first split tile (== num_tiles: no split)
    int32_t split_log2;     // each tile from split_start on is 2^split_log2 units
    int32_t k_splits;       // > 1: tiles from ks_start on are cut into k_splits K slices: unit
                            // ks_start + (t - ks_start) * k_splits + s is slice s of tile t (K blocks
                            // [s * k_per_split, +k_per_split) clipped at num_k_blocks), and its
                            // epilogue writes the fp32 partial to ws instead of C
    int32_t k_per_split;    // K blocks per slice
    int32_t ks_start;       // first tile cut into slices (0: every tile; num_tiles: none)
    float *ws;              // per split tile and slice, a SUPER_M x BN fp32 row-major partial:
                            // ws[((t - ks_start) * k_splits + s) * SUPER_M * BN + r * BN + c]
    int32_t ck_per;         // cluster K split (configurations with CLUSTER_K): K blocks per CTA of
                            // the cluster; CTA r of a cluster runs blocks [r * ck_per, +ck_per)
    uint64_t timeout_cycles;
    __half *C;              // output base (used by the direct-store epilogues)
    int32_t producer_off;   // test hook: 1 = the producer issues nothing, so the
                            // MMA thread's first wait runs out (see gemm_f16_selftest_timeout)
    unsigned long long *status;   // device status word of this GPU (first timeout record)
};

// Where a bounded wait expired (bits 0-7 of the status word).
enum WaitSite : uint32_t {
    kSiteProducerEmpty = 1,
    kSiteMmaTmemEmpty = 2,
    kSiteMmaFull = 3,
    kSiteEpilogueTmemFull = 4,
    kSiteDrainLoads = 5,
    kSiteDrainMma = 6,
    kSiteBoxImage = 7,   // the layout diagnostic's wait for its one box (tma_box_image.cu)
    kSiteClusterPartial = 8,   // cluster K split: waiting for the cluster's partial tiles (or their reads)
};

constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// Tile shapes and shared-memory budget of one kernel configuration.
//   kCtaGroup  1: one CTA per tile; 2: a CTA pair per tile (cta_group::2)
//   kBN        columns of C per tile; tiles wider than 256 (the largest MMA N)
//              issue BN/256 MMAs per K step into adjacent TMEM columns
//   kStages    depth of the shared-memory K ring
//   kEpiSmem   true: stage C tiles in shared memory and store them with TMA;
//              false: store C from registers (frees shared memory for a deeper ring)
//   kClusterK  cluster K split (single-CTA tiles only): the launch forms clusters
//              of S = 1, 2, 4 or 8 CTAs (a run-time cluster size); all CTAs of a
//              cluster compute the same output tile, CTA r over the r-th slice of
//              its K blocks.  Each CTA writes its fp32 partial tile to its own
//              shared memory; then CTA r adds the S partials of rows
//              [r * 128/S, (r+1) * 128/S) in rank order, reading the other CTAs'
//              shared memory through the cluster (distributed shared memory),
//              applies R and stores fp16 C.  No global workspace, no second
//              kernel; the result is the same sum as the workspace K split with
//              the same slices.
// Every CTA loads its operand boxes from global memory itself (no load is
// shared across a cluster by multicast).
template <int kCtaGroup, int kBN, int kStages, bool kEpiSmem = true, bool kClusterK = false>
struct GemmCfg {
    static constexpr int CTA_GROUP = kCtaGroup;
    static constexpr int CLUSTER = CTA_GROUP;         // CTAs per cluster (the pair, or one CTA);
                                                      // with CLUSTER_K the cluster size is a launch choice
    static constexpr bool CLUSTER_K = kClusterK;
    static constexpr int MAX_CLUSTER_K = 8;           // largest cluster of a cluster K split
    static constexpr bool EPI_SMEM = kEpiSmem;
    static constexpr int BM = 128;                    // rows of C per CTA = TMEM lanes
    static constexpr int TILE_M = BM * CTA_GROUP;     // rows of C per MMA tile (the MMA's M)
    static constexpr int SUPER_M = TILE_M;            // rows of C per work unit (one per cluster)
    static constexpr int BN = kBN;
    static constexpr int UMMA_N = BN < 256 ? BN : 256;   // N of one MMA instruction
    static constexpr int N_MMAS = BN / UMMA_N;        // MMAs per K step
    static constexpr int BN_CTA = BN / CTA_GROUP;     // columns of B each CTA loads
    static constexpr int BK = 64;                     // 64 fp16 = 128 bytes = one swizzle row
    static constexpr int UMMA_K = 16;                 // K of one tcgen05.mma.kind::f16
    static constexpr int STAGES = kStages;
    static constexpr int THREADS = 192;               // producer, MMA, 4 epilogue warps
    static constexpr int B_BOX_N = 64;                // N extent of one B box (128 bytes)
    static constexpr int B_BOXES = BN_CTA / B_BOX_N;
    static constexpr int A_STAGE_BYTES = BM * BK * 2;
    static constexpr int B_BOX_BYTES = B_BOX_N * BK * 2;
    static constexpr int B_STAGE_BYTES = B_BOXES * B_BOX_BYTES;
    static constexpr int STAGE_TX_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;   // loaded per CTA per stage
    static constexpr int ACC_COLS = BN;               // fp32 TMEM columns of one accumulator
    static constexpr int ACC_STAGES = 2 * BN <= 512 ? 2 : 1;   // double-buffer when TMEM allows
    static constexpr int TMEM_COLS = ACC_STAGES * ACC_COLS;
    static constexpr int EPI_COLS = 64;               // columns per epilogue chunk (128 bytes of fp16)
    static constexpr int C_BUF_BYTES = 32 * EPI_COLS * 2;
    static constexpr int SMEM_A_OFF = 0;
    static constexpr int SMEM_B_OFF = SMEM_A_OFF + STAGES * A_STAGE_BYTES;
    static constexpr int SMEM_C_OFF = SMEM_B_OFF + STAGES * B_STAGE_BYTES;
    // Cluster K split: once a CTA's single tile is multiplied, its operand ring
    // holds its fp32 partial tile (BM rows of BN floats) and a receive buffer
    // of the same size for the other CTAs' row blocks; the 16-byte piece j of
    // tile row r is stored at piece j ^ (r % 8) of the row.
    static constexpr int PART_BYTES = kClusterK ? 2 * BM * BN * 4 : 0;
    static constexpr int SMEM_CTL_OFF = SMEM_C_OFF + (kEpiSmem ? 4 * 2 * C_BUF_BYTES : 0);
    // Narrowest split unit: one B box per CTA per MMA.
    static constexpr int MAX_SPLIT_LOG2 = ilog2(BN / (B_BOX_N * CTA_GROUP));
    static constexpr int SMEM_CTL_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 /* alignment slack */ + SMEM_CTL_OFF + SMEM_CTL_BYTES;
    static constexpr uint32_t IDESC = idesc_f16_f32(TILE_M, UMMA_N, /*A MN-major*/ false, /*B MN-major*/ true);

    static_assert(CTA_GROUP == 1 || CTA_GROUP == 2, "one CTA or a CTA pair");
    static_assert(BN % (B_BOX_N * CTA_GROUP) == 0 && BN <= 512, "whole B boxes per CTA; at most 512 TMEM columns");
    static_assert(UMMA_N % 16 == 0 && UMMA_N <= 256, "UMMA N: multiple of 16 up to 256");
    static_assert(TMEM_COLS == 128 || TMEM_COLS == 256 || TMEM_COLS == 512, "TMEM allocation is a power of 2");
    static_assert((2 * STAGES + 8) * 8 <= SMEM_CTL_BYTES, "control block");
    static_assert(!kClusterK || (kCtaGroup == 1 && !kEpiSmem), "cluster K split: single-CTA tiles, direct stores");
    static_assert(PART_BYTES <= STAGES * (A_STAGE_BYTES + B_STAGE_BYTES), "cluster K buffers fit in the ring");
    static_assert(SMEM_BYTES <= 232448, "shared memory per block on sm_103");
};

// Abort flag of this CTA.  In a cluster, raising it also raises the flag (at
// the same shared-memory offset) of every other CTA of the cluster.
struct AbortFlag {
    volatile int *local;
    unsigned long long *status;   // device status word
    uint32_t addr;          // shared::cta address of the flag
    uint32_t cluster;       // CTAs in the cluster
    uint32_t rank;          // this CTA's rank in the cluster

    __device__ __forceinline__ bool raised() const { return *local != 0; }
    __device__ __forceinline__ void raise(uint32_t site) const
    {
        *local = 1;
        for (uint32_t i = 0; i < cluster; ++i)
            if (i != rank) st_shared_cluster_u32(mapa_shared(addr, i), 1u);
        atomicCAS(status, 0ull,
                  static_cast<unsigned long long>(site) | (static_cast<unsigned long long>(blockIdx.x) << 8));
    }
};

// Bounded wait on an mbarrier phase.  Fast path: one probe.  Slow path: probe
// until the phase completes, the abort flag is raised, or the clock64 budget
// is spent (then record the site and raise the abort flag).  The probe is the
// default (CTA-scope) form also for barriers another CTA arrives on: TMA bytes
// become visible through the barrier's transaction count, and TMEM hand-offs
// are ordered by the tcgen05 fences around the waits.
// kSleepNs > 0 adds a short sleep to each slow-path probe (fewer issue slots
// spent on polling).  The fp16 GEMM's waits do not use it: a 256 ns sleep in
// the epilogue's wait for a finished accumulator delayed the hand-back of TMEM
// to the next tile and measured 1.6 % slower (the try_wait probe already
// suspends the thread for a while when the phase is not complete).  Roles that
// run far ahead of the MMAs (the scale writers of the E8M0 FP8 kernel) use it.
template <int kSleepNs = 0>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const AbortFlag &abort, uint64_t limit,
                                           uint32_t site)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if constexpr (kSleepNs > 0) __nanosleep(kSleepNs);
        if (mbar_try_wait(bar, parity)) return true;
        if (abort.raised()) return false;
        if (static_cast<uint64_t>(clock64() - t0) > limit) {
            abort.raise(site);
            return false;
        }
    }
}

// Bounded wait used while tearing down after an abort: ignores the abort flag.
__device__ __forceinline__ bool wait_phase_drain(uint32_t bar, uint32_t parity, uint64_t limit, uint32_t site,
                                                 unsigned long long *status)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (static_cast<uint64_t>(clock64() - t0) > limit) {
            atomicCAS(status, 0ull,
                      static_cast<unsigned long long>(site) | (static_cast<unsigned long long>(blockIdx.x) << 8));
            return false;
        }
    }
    return true;
}

// Grouped rasterisation: tiles are visited in panels of group_m tile rows; inside
// a panel the row index runs fastest, so tiles that run at the same time share
// the same few A row-panels and B column-panels in L2.
__device__ __forceinline__ void tile_coords(int t, const GemmParams &p, int &mb, int &nb)
{
    const int per_group = p.group_m * p.num_n_blocks;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.num_m_blocks - first_m, p.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % rows;
    nb = r / rows;
}

// K blocks [kb0, kb1) of work unit u, and its K slice (-1: a whole tile, no
// K split).
__device__ __forceinline__ void unit_k_range(int u, const GemmParams &p, int &kb0, int &kb1, int &slice)
{
    slice = -1;
    kb0 = 0;
    kb1 = p.num_k_blocks;
    if (p.k_splits > 1 && u >= p.ks_start) {
        slice = (u - p.ks_start) % p.k_splits;
        kb0 = slice * p.k_per_split;
        kb1 = min(p.num_k_blocks, kb0 + p.k_per_split);
    }
}

// Tile of work unit u under a K split (units of one split tile are adjacent).
__device__ __forceinline__ int unit_tile_k(int u, const GemmParams &p)
{
    return (p.k_splits > 1 && u >= p.ks_start) ? p.ks_start + (u - p.ks_start) / p.k_splits : u;
}

// Work unit u -> tile row block mb, first output column col0 of the unit, and
// the split shift (the unit is BN >> shift columns wide).  With a K split
// there is no N split (split_start = num_tiles).
template <int kBN>
__device__ __forceinline__ void unit_coords(int u, const GemmParams &p, int &mb, int &col0, int &shift)
{
    if (p.k_splits > 1) u = unit_tile_k(u, p);
    int t = u, sub = 0;
    shift = 0;
    if (u >= p.split_start) {
        shift = p.split_log2;
        const int d = u - p.split_start;
        t = p.split_start + (d >> shift);
        sub = d & ((1 << shift) - 1);
    }
    int nb;
    tile_coords(t, p, mb, nb);
    col0 = nb * kBN + sub * (kBN >> shift);
}

__device__ __forceinline__ void st_global_v4(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// R(x) of the epilogue.  Without ReLU the value is x + (+0): the pages' tile
// GEMM clears its accumulator to +0 before adding the products, and
// +0 + (-0) = +0, so a sum whose terms are all -0 is +0 (the MMA's first
// product with accumulate = 0 does not add that +0 itself).  No other value
// changes.
__device__ __forceinline__ float4 ld_shared_f32x4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

template <bool kRelu>
__device__ __forceinline__ float epilogue_value(uint32_t bits)
{
    const float x = __uint_as_float(bits);
    if constexpr (kRelu) return x > 0.0f ? x : 0.0f;  // -0, NaN and negatives give +0
    else return __fadd_rn(x, 0.0f);
}

template <bool kRelu>
__device__ __forceinline__ uint32_t pack_f16x2(uint32_t lo_bits, uint32_t hi_bits)
{
    const __half2 h = __floats2half2_rn(epilogue_value<kRelu>(lo_bits), epilogue_value<kRelu>(hi_bits));
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Cluster K split: receive slot of sender s at the owner of rank o (senders
// in rank order, the owner itself skipped).
__device__ __forceinline__ int ck_slot(int s, int o) { return s < o ? s : s - 1; }

// Cluster K split, stage 2: the owner (rank `crank` of a cluster of S) adds
// its R = 128 / S tile rows over the S senders in rank order, applies R(x),
// rounds to fp16 and stores them.  Thread t (0..127) takes owned row t % R and
// the (t / R)-th of S column segments (BN / S columns).  Sender s's rows are in
// this CTA's partial tile (s == crank) or in receive slot ck_slot(s, crank);
// tile row r's 16-byte piece j is at piece j ^ (r % 8) of its 4 * BN-byte row.
template <int S, bool kRelu, int BN>
__device__ __forceinline__ void ck_reduce_rows(const GemmParams &p, uint32_t part, uint32_t recv, int crank, int mb,
                                               int col0, int t)
{
    constexpr int R = 128 / S;
    constexpr int kRowBytes = BN * 4;
    constexpr int SEG = BN / S;               // columns of this thread
    constexpr int PIECES = SEG / 4;           // fp32 16-byte pieces of this thread
    static_assert(PIECES % 2 == 0, "whole 16-byte fp16 outputs");
    const int rr = t % R;
    const int seg = t / R;
    const int trow = crank * R + rr;
    const uint32_t sw = static_cast<uint32_t>(trow & 7);
    uint32_t src_row[S];
#pragma unroll
    for (int s = 0; s < S; ++s)
        src_row[s] = s == crank ? part + static_cast<uint32_t>(trow * kRowBytes)
                                : recv + static_cast<uint32_t>((ck_slot(s, crank) * R + rr) * kRowBytes);
    const int row = mb * 128 + trow;
    const int cbase = col0 + seg * SEG;
    if (row >= p.M) return;
    __half *crow = p.C + static_cast<int64_t>(row) * p.N + cbase;
#pragma unroll
    for (int j = 0; j < PIECES; j += 2) {
        const uint32_t pc = static_cast<uint32_t>(seg * PIECES + j);
        const uint32_t off_lo = (pc ^ sw) << 4, off_hi = ((pc + 1u) ^ sw) << 4;
        float4 lo = ld_shared_f32x4(src_row[0] + off_lo), hi = ld_shared_f32x4(src_row[0] + off_hi);
#pragma unroll
        for (int s = 1; s < S; ++s) {
            const float4 a = ld_shared_f32x4(src_row[s] + off_lo);
            const float4 d = ld_shared_f32x4(src_row[s] + off_hi);
            lo.x += a.x;
            lo.y += a.y;
            lo.z += a.z;
            lo.w += a.w;
            hi.x += d.x;
            hi.y += d.y;
            hi.z += d.z;
            hi.w += d.w;
        }
        if (cbase + 4 * j < p.N)
            st_global_v4(crow + 4 * j, pack_f16x2<kRelu>(__float_as_uint(lo.x), __float_as_uint(lo.y)),
                         pack_f16x2<kRelu>(__float_as_uint(lo.z), __float_as_uint(lo.w)),
                         pack_f16x2<kRelu>(__float_as_uint(hi.x), __float_as_uint(hi.y)),
                         pack_f16x2<kRelu>(__float_as_uint(hi.z), __float_as_uint(hi.w)));
    }
}

// Operand layouts (the transpose_A / transpose_B of the pages' tile GEMM):
//   kTA = false: A stored (M,K) row-major (K-major);  true: stored (K,M) row-major,
//                op(A) = stored^T (M-major; TMA boxes 64(M) x 64(K), two per stage).
//   kTB = false: B stored (K,N) row-major (N-major);  true: stored (N,K) row-major,
//                op(B) = stored^T (K-major; TMA boxes 64(K) x 64(N rows)).
// Shared-memory offsets of every box are the same in all four layouts; only the
// tensor-map orientation, the box coordinates and the descriptor type change.
template <class Cfg, bool kRelu, bool kTA = false, bool kTB = false>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    gemm_f16_relu_sm103a(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                         const __grid_constant__ CUtensorMap tmap_c, const GemmParams p)
{
    constexpr bool kPair = Cfg::CTA_GROUP == 2;
    // Instruction descriptor with this kernel's operand majors (bit 15: A MN-major,
    // bit 16: B MN-major).
    // One accumulator of two 256-column N halves (the 256 x 512 pair tile): the
    // epilogue hands the halves back separately, so the next unit's MMAs start
    // on half 0 while half 1 is still being read.
    constexpr bool kHalfRelease = Cfg::ACC_STAGES == 1 && Cfg::N_MMAS == 2;
    constexpr uint32_t kIdesc = (Cfg::IDESC & ~((1u << 15) | (1u << 16))) | (kTA ? (1u << 15) : 0u) |
                                (kTB ? 0u : (1u << 16));

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // SW128 atoms need 1024-byte alignment
    uint8_t *base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base + Cfg::SMEM_A_OFF;
    const uint32_t sB = base + Cfg::SMEM_B_OFF;
    const uint32_t sC = base + Cfg::SMEM_C_OFF;
    const uint32_t ctl = base + Cfg::SMEM_CTL_OFF;
    auto full_bar = [&](int s) { return ctl + 8u * s; };
    auto empty_bar = [&](int s) { return ctl + 8u * (Cfg::STAGES + s); };
    auto tfull_bar = [&](int b) { return ctl + 8u * (2 * Cfg::STAGES + b); };
    auto tempty_bar = [&](int b) { return ctl + 8u * (2 * Cfg::STAGES + 2 + b); };
    const uint32_t drain_bar = ctl + 8u * (2 * Cfg::STAGES + 4);
    const uint32_t tmem_slot = ctl + 8u * (2 * Cfg::STAGES + 5);
    // Cluster K split: this CTA's receive buffer holds the other CTAs' row
    // blocks of the tile (rfull: one arrival with the expected bytes, then the
    // senders' bulk copies) / every CTA of the cluster has finished its MMAs,
    // so its operand ring may receive (rready: one arrival per CTA).
    const uint32_t rfull_bar = ctl + 8u * (2 * Cfg::STAGES + 6);
    const uint32_t rready_bar = ctl + 8u * (2 * Cfg::STAGES + 7);
    const uint32_t abort_addr = tmem_slot + 4;
    volatile uint32_t *tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t *>(base_ptr + Cfg::SMEM_CTL_OFF + 8 * (2 * Cfg::STAGES + 5));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTAs in the cluster: the pair, one, or (cluster K split) the launch's choice
    const uint32_t ncl = Cfg::CLUSTER_K ? cluster_nctarank() : static_cast<uint32_t>(Cfg::CLUSTER);
    const uint32_t crank = (Cfg::CLUSTER > 1 || Cfg::CLUSTER_K) ? cluster_ctarank() : 0u;   // rank in the cluster
    const uint32_t rank = kPair ? (crank & 1u) : 0u;                    // rank in the pair; 0 = leader
    const uint32_t leader_rank = 0u;                                      // cluster rank of the pair's leader
    const bool leader = rank == 0;
    const int cluster_id = static_cast<int>(blockIdx.x / ncl);
    const int num_clusters = static_cast<int>(gridDim.x / ncl);
    const uint16_t pair_mask = 0x3u;   // both CTAs of the pair

    AbortFlag abort;
    abort.local = reinterpret_cast<volatile int *>(tmem_slot_ptr + 1);
    abort.status = p.status;
    abort.addr = abort_addr;
    abort.cluster = ncl;
    abort.rank = crank;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(full_bar(s), Cfg::CTA_GROUP);   // each CTA of the pair: arrive.expect_tx
            mbar_init(empty_bar(s), 1);               // one MMA commit (by the pair leader)
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);                       // commit after a tile's last MMA
            mbar_init(tempty_bar(b), 4 * Cfg::CTA_GROUP);     // one arrive per epilogue warp
        }
        mbar_init(drain_bar, 1);
        if constexpr (Cfg::CLUSTER_K) {
            mbar_init(rfull_bar, 1);
            mbar_init(rready_bar, ncl);
        }
        *abort.local = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_b);
        prefetch_tensormap(&tmap_c);
    }
    if (warp == 1) {
        tmem_alloc<Cfg::CTA_GROUP>(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish<Cfg::CTA_GROUP>();
    }
    tc_fence_before_sync();
    __syncthreads();
    if (ncl > 1) {
        // Every CTA's barriers are initialised and its TMEM allocated before
        // any CTA of the cluster signals another.
        cluster_arrive();
        cluster_wait();
    }
    tc_fence_after_sync();
    // The set-up above touches no global memory of this call, so it may run
    // while the previous kernel of the stream finishes.  Each role waits for
    // that kernel's results (griddep_wait) just before its own first global
    // access: the producer before its first load, the epilogue before its
    // first store; the MMA thread touches only shared and tensor memory.  The
    // next kernel may be scheduled on SMs this grid leaves free (it waits the
    // same way).
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot_ptr;
    const uint64_t limit = p.timeout_cycles;
    bool aborted = false;
    // K blocks [kb0, kb1) this CTA runs for unit u (and the workspace slice).
    auto k_range = [&](int u, int &kb0, int &kb1, int &slice) {
        unit_k_range(u, p, kb0, kb1, slice);
        if constexpr (Cfg::CLUSTER_K) {
            kb0 = static_cast<int>(crank) * p.ck_per;
            kb1 = min(p.num_k_blocks, kb0 + p.ck_per);
        }
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            // The pair leader's full barrier 0 (its full[s] is 8 * s bytes further).
            const uint32_t full_base = (kPair && !leader) ? mapa_shared(full_bar(0), leader_rank) : full_bar(0);
            (void)full_base;
            bool dep_waited = false;
            for (int u = cluster_id; ok && p.producer_off == 0 && u < p.num_units; u += num_clusters) {
                int mb, col0, shift, kb0, kb1, slice;
                unit_coords<Cfg::BN>(u, p, mb, col0, shift);
                k_range(u, kb0, kb1, slice);
                const int m0 = mb * Cfg::SUPER_M + static_cast<int>(rank) * Cfg::BM;
                // Unit width W = BN >> shift, issued as W / umma_n MMAs of N = umma_n.
                // For MMA h, this CTA supplies umma_n / CTA_GROUP columns (bpm boxes),
                // starting at tile column h * umma_n + rank * umma_n / CTA_GROUP.
                const int width = Cfg::BN >> shift;
                const int umma_n = width < Cfg::UMMA_N ? width : Cfg::UMMA_N;
                const int bpm = umma_n / (Cfg::CTA_GROUP * Cfg::B_BOX_N);   // 1, 2 or 4
                const int bpm_log2 = __ffs(bpm) - 1;
                const int boxes = Cfg::B_BOXES >> shift;
                const int n_cta = col0 + static_cast<int>(rank) * (umma_n / Cfg::CTA_GROUP);
                const uint32_t tx = Cfg::A_STAGE_BYTES + boxes * Cfg::B_BOX_BYTES;
                // Everything that is fixed for the unit is computed here, once: the
                // per-stage path below is only the arrive and the TMA issues (a
                // slot's refill waits behind it).
                int bxs[Cfg::B_BOXES];
#pragma unroll
                for (int j = 0; j < Cfg::B_BOXES; ++j)
                    bxs[j] = n_cta + (j >> bpm_log2) * umma_n + (j & (bpm - 1)) * Cfg::B_BOX_N;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort, limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (!dep_waited) {
                        griddep_wait();   // the operands may come from the previous kernel
                        dep_waited = true;
                    }
                    const int k0 = kb * Cfg::BK;
                    const uint32_t a_dst = sA + s * Cfg::A_STAGE_BYTES;
                    const uint32_t b_dst = sB + s * Cfg::B_STAGE_BYTES;
                    if constexpr (!kPair) {
                        const uint32_t fb = full_bar(s);
                        mbar_arrive_expect_tx(fb, tx);
                        if constexpr (!kTA) {
                            tma_load_2d(a_dst, &tmap_a, fb, k0, m0);
                        } else {
                            tma_load_2d(a_dst, &tmap_a, fb, m0, k0);
                            tma_load_2d(a_dst + Cfg::A_STAGE_BYTES / 2, &tmap_a, fb, m0 + 64, k0);
                        }
#pragma unroll
                        for (int j = 0; j < Cfg::B_BOXES; ++j) {
                            if (j < boxes) {
                                if constexpr (!kTB) tma_load_2d(b_dst + j * Cfg::B_BOX_BYTES, &tmap_b, fb, bxs[j], k0);
                                else tma_load_2d(b_dst + j * Cfg::B_BOX_BYTES, &tmap_b, fb, k0, bxs[j]);
                            }
                        }
                    } else {
                        // The bytes landing in both CTAs of a pair are counted on the
                        // pair leader's barrier; each CTA announces its own bytes.
                        const uint32_t fb = full_base + 8u * s;
                        if (leader) mbar_arrive_expect_tx(fb, tx);
                        else mbar_arrive_expect_tx_cluster(fb, tx);
                        if constexpr (!kTA) {
                            tma_load_2d_pair(a_dst, &tmap_a, fb, k0, m0);
                        } else {
                            tma_load_2d_pair(a_dst, &tmap_a, fb, m0, k0);
                            tma_load_2d_pair(a_dst + Cfg::A_STAGE_BYTES / 2, &tmap_a, fb, m0 + 64, k0);
                        }
#pragma unroll
                        for (int j = 0; j < Cfg::B_BOXES; ++j) {
                            if (j < boxes) {
                                const int bx = kTB ? k0 : bxs[j], by = kTB ? bxs[j] : k0;
                                tma_load_2d_pair(b_dst + j * Cfg::B_BOX_BYTES, &tmap_b, fb, bx, by);
                            }
                        }
                    }
                    issued_mask |= 1u << s;
                    issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                    if (++s == Cfg::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                aborted = true;
                if (leader) {
                    // Let the loads in flight land before the CTA exits.
                    for (int i = 0; i < Cfg::STAGES; ++i)
                        if (issued_mask & (1u << i))
                            wait_phase_drain(full_bar(i), (issued_parity >> i) & 1u, limit, kSiteDrainLoads, p.status);
                } else {
                    // This CTA's loads complete on the leader's barrier, which it
                    // cannot probe: give them a bounded time (~1e6 cycles) to land.
                    const long long t0 = clock64();
                    while (clock64() - t0 < 1000000) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA)
        if (lane == 0 && leader) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true, issued_any = false;
            // Stage-0 descriptors; every other operand address is a constant offset.
            // K-major operand: 8-row groups 1024 B apart (SBO); a K step of 16
            // elements is 32 B inside the 128-byte swizzle row.  MN-major operand:
            // 64-element boxes B_BOX_BYTES apart (LBO), 8-row K groups 1024 B
            // apart (SBO); a K step of 16 rows is 16 * 128 B.
            const uint64_t a_desc0 = kTA ? smem_desc_sw128(sA, Cfg::B_BOX_BYTES, 1024) : smem_desc_sw128(sA, 16, 1024);
            const uint64_t b_desc0 = kTB ? smem_desc_sw128(sB, 16, 1024) : smem_desc_sw128(sB, Cfg::B_BOX_BYTES, 1024);
            constexpr uint32_t kAStep = kTA ? Cfg::UMMA_K * 128 : Cfg::UMMA_K * 2;   // bytes per K step
            constexpr uint32_t kBStep = kTB ? Cfg::UMMA_K * 2 : Cfg::UMMA_K * 128;
            for (int u = cluster_id; ok && u < p.num_units; u += num_clusters, ++it) {
                const int b = it % Cfg::ACC_STAGES;
                const uint32_t acc_ph = (it / Cfg::ACC_STAGES) & 1;
                const int shift = (p.k_splits <= 1 && u >= p.split_start) ? p.split_log2 : 0;
                int kb0, kb1, slice;
                k_range(u, kb0, kb1, slice);
                const int width = Cfg::BN >> shift;
                const int umma_n = width < Cfg::UMMA_N ? width : Cfg::UMMA_N;
                const int n_mmas = width / umma_n;
                const uint32_t bpm_bytes = static_cast<uint32_t>(umma_n / (Cfg::CTA_GROUP * Cfg::B_BOX_N)) *
                                           Cfg::B_BOX_BYTES;
                // The MMA's N field (bits 17-22, N >> 3) for this unit's width.
                const uint32_t idesc =
                    (kIdesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(umma_n >> 3) << 17);
                const uint32_t d_tmem = tmem_base + b * Cfg::ACC_COLS;
                // The MMAs of K block kb (ring slot st), N halves [h_lo, h_hi).
                auto issue = [&](int kb, int st, int h_lo, int h_hi) {
                    // Descriptors of this stage: the start-address field (bits 0-13)
                    // holds address >> 4, so advancing an operand by n bytes adds
                    // n >> 4 (no carry out of the field: shared addresses < 2^18).
                    const uint64_t a_st = a_desc0 + static_cast<uint64_t>((st * Cfg::A_STAGE_BYTES) >> 4);
                    const uint64_t b_st = b_desc0 + static_cast<uint64_t>((st * Cfg::B_STAGE_BYTES) >> 4);
                    const uint32_t acc0 = kb != kb0 ? 1u : 0u;
#pragma unroll
                    for (int ks = 0; ks < Cfg::BK / Cfg::UMMA_K; ++ks) {
                        const uint64_t a_desc = a_st + static_cast<uint64_t>((ks * kAStep) >> 4);
#pragma unroll
                        for (int h = 0; h < Cfg::N_MMAS; ++h) {
                            if (h < h_lo) continue;
                            if (h >= h_hi || h >= n_mmas) break;
                            // MMA h starts at its own B boxes.
                            const uint64_t b_desc = b_st + static_cast<uint64_t>((h * bpm_bytes + ks * kBStep) >> 4);
                            mma_f16_ss<Cfg::CTA_GROUP>(d_tmem + h * umma_n, a_desc, b_desc, idesc,
                                                       ks != 0 ? 1u : acc0);
                        }
                    }
                };
                // Frees slot st once the MMAs issued so far have read it, in both CTAs
                // of the pair.
                auto release = [&](int st) {
                    if constexpr (kPair) mma_commit_pair_mc(empty_bar(st), pair_mask);
                    else mma_commit(empty_bar(st));
                };
                int kb = kb0;
                if (kHalfRelease && n_mmas == 2) {
                    // One accumulator of two N halves: the epilogue of the previous
                    // unit hands each half back as soon as it has read it.  Start
                    // on half 0 with the K blocks already in the ring, then run
                    // half 1 over the same slots once it is free.
                    if (!wait_phase(tempty_bar(0), acc_ph ^ 1u, abort, limit, kSiteMmaTmemEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int npre = min(Cfg::STAGES, kb1 - kb0);
                    int pre_slot[Cfg::STAGES];
                    for (int i = 0; i < npre; ++i) {
                        if (!wait_phase(full_bar(s), ph, abort, limit, kSiteMmaFull)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        pre_slot[i] = s;
                        issue(kb0 + i, s, 0, 1);
                        issued_any = true;
                        if (++s == Cfg::STAGES) {
                            s = 0;
                            ph ^= 1u;
                        }
                    }
                    if (!ok) break;
                    if (!wait_phase(tempty_bar(1), acc_ph ^ 1u, abort, limit, kSiteMmaTmemEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    for (int i = 0; i < npre; ++i) {
                        issue(kb0 + i, pre_slot[i], 1, 2);
                        release(pre_slot[i]);
                    }
                    kb = kb0 + npre;
                } else {
                    if (!wait_phase(tempty_bar(b), acc_ph ^ 1u, abort, limit, kSiteMmaTmemEmpty) ||
                        (kHalfRelease && !wait_phase(tempty_bar(1), acc_ph ^ 1u, abort, limit, kSiteMmaTmemEmpty))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                }
                for (; kb < kb1; ++kb) {
                    if (!wait_phase(full_bar(s), ph, abort, limit, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    issue(kb, s, 0, Cfg::N_MMAS);
                    release(s);
                    issued_any = true;
                    if (++s == Cfg::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                // Accumulator b complete (in both CTAs' TMEM).
                if constexpr (kPair) mma_commit_pair_mc(tfull_bar(b), pair_mask);
                else mma_commit(tfull_bar(b));
            }
            if (!ok) {
                aborted = true;
                if (issued_any) {
                    // Wait for this thread's MMAs before the TMEM is freed.
                    if constexpr (kPair) mma_commit_pair_mc(drain_bar, static_cast<uint16_t>(1u << crank));
                    else mma_commit(drain_bar);
                    wait_phase_drain(drain_bar, 0, limit, kSiteDrainMma, p.status);
                }
            }
        }
        __syncwarp();
    } else if constexpr (Cfg::CLUSTER_K) {
        // ------------------------------------------------------------ epilogue, cluster K split (warps 2..5)
        // One tile per cluster.  CTA o owns rows [o * R, (o+1) * R) of the tile
        // (R = 128 / ncl).  Once this CTA's MMAs are done, its operand ring is
        // free and holds two buffers: the fp32 partial tile and a receive buffer
        // for the other CTAs' row blocks of the owned rows.  Stage 1: the four
        // warps write the accumulator (TMEM lane = tile row) into the partial
        // buffer; one thread copies each other owner its R rows (one bulk
        // shared-memory copy per owner into the owner's receive buffer, slot of
        // this sender, counted on the owner's rfull barrier) once every owner
        // has said its ring is free (rready).  Stage 2, once the other ncl - 1
        // blocks have arrived: the owner adds each of its rows over the senders
        // in rank order (its own rows from its partial buffer), applies R,
        // rounds to fp16 and stores C.
        const int q = warp & 3;
        const int ew = warp - 2;
        const bool lead = ew == 0 && lane == 0;   // issues the copies and the cluster signals
        constexpr uint32_t kEpiBarrier = 1;       // named barrier of the 128 epilogue threads
        constexpr int kRowBytes = Cfg::BN * 4;
        const int rows_per_cta = Cfg::BM / static_cast<int>(ncl);
        const uint32_t block_bytes = static_cast<uint32_t>(rows_per_cta * kRowBytes);
        const int row_t = q * 32 + lane;          // tile row = TMEM lane of this thread
        const uint32_t part = sA;                                   // over the operand ring
        const uint32_t recv = sA + static_cast<uint32_t>(Cfg::BM * kRowBytes);
        const uint32_t my_row = part + static_cast<uint32_t>(row_t * kRowBytes);
        const uint32_t rsw = static_cast<uint32_t>(row_t & 7);
        auto slot = [](int s, int o) { return ck_slot(s, o); };
        const int u = cluster_id;   // the launch gives every cluster exactly one tile
        if (u < p.num_units) {
            int mb, col0_unit, shift, kb0, kb1, slice;
            unit_coords<Cfg::BN>(u, p, mb, col0_unit, shift);
            k_range(u, kb0, kb1, slice);
            int ok = 1;
            if (lane == 0) ok = wait_phase(tfull_bar(0), 0, abort, limit, kSiteEpilogueTmemFull) ? 1 : 0;
            if (lead && ok && ncl > 1) {
                // This CTA's MMAs have read their last operands: its ring may
                // take the other CTAs' row blocks.
                mbar_arrive_expect_tx(rfull_bar, (ncl - 1) * block_bytes);
                for (uint32_t cta = 0; cta < ncl; ++cta) mbar_arrive_cluster(mapa_shared(rready_bar, cta));
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            // one decision for the four warps: each reaches every later barrier, or none
            if (named_barrier_and(kEpiBarrier, 128, ok != 0)) {
                griddep_wait();   // before this warp's first store of C
                tc_fence_after_sync();
                const uint32_t acc_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
                for (int c = 0; c < Cfg::BN / 64; ++c) {
                    uint32_t r[64];
                    if (kb1 > kb0) {
                        tmem_load_32x32b_x64(acc_addr + c * 64, r);
                    } else {
#pragma unroll
                        for (int j = 0; j < 64; ++j) r[j] = 0u;   // an empty K slice adds +0
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t piece = static_cast<uint32_t>(c * 16 + j);
                        st_shared_v4(my_row + ((piece ^ rsw) << 4), r[4 * j], r[4 * j + 1], r[4 * j + 2],
                                     r[4 * j + 3]);
                    }
                }
                // All TMEM reads of this warp are done.
                tc_fence_before_sync();
                fence_proxy_async_smem();   // the partial rows are read by the bulk copies
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(0));
                named_barrier_sync(kEpiBarrier, 128);
                if (lead && ncl > 1) {
                    if (wait_phase(rready_bar, 0, abort, limit, kSiteClusterPartial)) {
                        for (int o = 0; o < static_cast<int>(ncl); ++o) {
                            if (o == static_cast<int>(crank)) continue;
                            const uint32_t dst =
                                recv + static_cast<uint32_t>(slot(static_cast<int>(crank), o)) * block_bytes;
                            bulk_copy_to_cluster(mapa_shared(dst, o), part + static_cast<uint32_t>(o) * block_bytes,
                                                 block_bytes, mapa_shared(rfull_bar, o));
                        }
                        bulk_commit_group();
                    }
                }
                if (ncl > 1) {
                    if (lane == 0) ok = wait_phase(rfull_bar, 0, abort, limit, kSiteClusterPartial) ? 1 : 0;
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                }
                if (ok) {
                    switch (ncl) {
                        case 1: ck_reduce_rows<1, kRelu, Cfg::BN>(p, part, recv, static_cast<int>(crank), mb, col0_unit, ew * 32 + lane); break;
                        case 2: ck_reduce_rows<2, kRelu, Cfg::BN>(p, part, recv, static_cast<int>(crank), mb, col0_unit, ew * 32 + lane); break;
                        case 4: ck_reduce_rows<4, kRelu, Cfg::BN>(p, part, recv, static_cast<int>(crank), mb, col0_unit, ew * 32 + lane); break;
                        default: ck_reduce_rows<8, kRelu, Cfg::BN>(p, part, recv, static_cast<int>(crank), mb, col0_unit, ew * 32 + lane); break;
                    }
                }
                if (!ok) aborted = true;
            } else {
                aborted = true;
            }
        }
        if (lead) bulk_wait_group<0>();   // this CTA's copies have completed before it exits
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int ew = warp - 2;        // owner of smem staging buffers
        const int q = warp & 3;         // TMEM lane quarter this warp may access
        const uint32_t row_off = static_cast<uint32_t>(lane) * 128u;
        const uint32_t sw = static_cast<uint32_t>(lane & 7);
        const uint32_t tempty_leader0 = kPair && !leader ? mapa_shared(tempty_bar(0), leader_rank) : tempty_bar(0);
        int it = 0;
        uint32_t chunk = 0;
        for (int u = cluster_id; u < p.num_units; u += num_clusters, ++it) {
            int mb, col0_unit, shift, kb0, kb1, slice;
            unit_coords<Cfg::BN>(u, p, mb, col0_unit, shift);
            k_range(u, kb0, kb1, slice);
            const int chunks = (Cfg::BN >> shift) / Cfg::EPI_COLS;
            const int b = it % Cfg::ACC_STAGES;
            const uint32_t acc_ph = (it / Cfg::ACC_STAGES) & 1;
            int ok = 1;
            if (lane == 0)
                ok = wait_phase(tfull_bar(b), acc_ph, abort, limit, kSiteEpilogueTmemFull) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                aborted = true;
                break;
            }
            if (it == 0) griddep_wait();   // before this warp's first store of C (or of partials)
            tc_fence_after_sync();
            const int row0 = mb * Cfg::SUPER_M + static_cast<int>(rank) * Cfg::BM + q * 32;
            const uint32_t acc_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + b * Cfg::ACC_COLS;
            // Chunk c (64 columns) of the accumulator: hand back TMEM when this
            // warp's reads of it are complete, then convert and store it.
            auto chunk_out = [&](const uint32_t (&r)[64], int c) {
                if constexpr (kHalfRelease) {
                    // One accumulator in two N halves of 256 columns (chunks 0-3
                    // and 4-7): hand each back once this warp has read it (both at
                    // the last chunk of a narrower unit).
                    const int half0_last = chunks < 4 ? chunks - 1 : 3;
                    if (c == half0_last || c == chunks - 1) {
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            for (int h = (c == half0_last ? 0 : 1); h <= (c == chunks - 1 ? 1 : 0); ++h) {
                                if (kPair && !leader) mbar_arrive_cluster(tempty_leader0 + 8u * h);
                                else mbar_arrive(tempty_bar(h));
                            }
                        }
                    }
                } else if (c == chunks - 1) {
                    // All TMEM reads of accumulator b by this warp are done.
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (kPair && !leader) mbar_arrive_cluster(tempty_leader0 + 8u * b);
                        else mbar_arrive(tempty_bar(b));
                    }
                }
                const int col0 = col0_unit + c * Cfg::EPI_COLS;
                if (slice >= 0) {
                    // K slice: this row's 64 fp32 partial sums, as they are, into the
                    // slice's tile in the workspace (16-byte pieces; N is a multiple
                    // of 8, so every piece is wholly in or out; rows and columns
                    // outside C are not written, nor read by the reduction).
                    const int row = row0 + lane;
                    if (row < p.M) {
                        const int t = unit_tile_k(u, p);
                        const int64_t tile_base =
                            (static_cast<int64_t>(t - p.ks_start) * p.k_splits + slice) *
                            static_cast<int64_t>(Cfg::SUPER_M * Cfg::BN);
                        float *wrow = p.ws + tile_base + static_cast<int64_t>(row - mb * Cfg::SUPER_M) * Cfg::BN +
                                      (col0 - (col0_unit - (col0_unit % Cfg::BN)));
#pragma unroll
                        for (int j = 0; j < Cfg::EPI_COLS / 4; ++j) {
                            if (col0 + 4 * j < p.N)
                                st_global_v4(wrow + 4 * j, r[4 * j + 0], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                        }
                    }
                } else if constexpr (Cfg::EPI_SMEM) {
                    const bool in_range = row0 < p.M && col0 < p.N;
                    const uint32_t cbuf = sC + (ew * 2 + (chunk & 1u)) * Cfg::C_BUF_BYTES;
                    ++chunk;
                    if (lane == 0) bulk_wait_group_read<1>();   // the store that used cbuf has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t w0 = pack_f16x2<kRelu>(r[8 * j + 0], r[8 * j + 1]);
                        const uint32_t w1 = pack_f16x2<kRelu>(r[8 * j + 2], r[8 * j + 3]);
                        const uint32_t w2 = pack_f16x2<kRelu>(r[8 * j + 4], r[8 * j + 5]);
                        const uint32_t w3 = pack_f16x2<kRelu>(r[8 * j + 6], r[8 * j + 7]);
                        // 16-byte chunk j of this row goes to chunk j ^ (row % 8): the
                        // layout a SWIZZLE_128B tensor-map store expects.
                        st_shared_v4(cbuf + row_off + ((static_cast<uint32_t>(j) ^ sw) << 4), w0, w1, w2, w3);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (in_range) tma_store_2d(&tmap_c, cbuf, col0, row0);
                        // One group per chunk, empty or not, so that "at most one group
                        // pending" above always means the other buffer's store.
                        bulk_commit_group();
                    }
                } else {
                    // Each thread owns one row: 64 fp16 = 128 contiguous bytes.  N is
                    // a multiple of 8, so every 16-byte piece is wholly in or out.
                    const int row = row0 + lane;
                    if (row < p.M) {
                        __half *crow = p.C + static_cast<int64_t>(row) * p.N + col0;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (col0 + 8 * j < p.N)
                                st_global_v4(crow + 8 * j, pack_f16x2<kRelu>(r[8 * j + 0], r[8 * j + 1]),
                                             pack_f16x2<kRelu>(r[8 * j + 2], r[8 * j + 3]),
                                             pack_f16x2<kRelu>(r[8 * j + 4], r[8 * j + 5]),
                                             pack_f16x2<kRelu>(r[8 * j + 6], r[8 * j + 7]));
                        }
                    }
                }
            };
            // Double-buffered: the TMEM load of chunk c + 1 runs while chunk c
            // is converted and stored.
            uint32_t ra[64], rb[64];
            tmem_load_32x32b_x64_async(acc_addr, ra);
#pragma unroll 1
            for (int c = 0; c < chunks; c += 2) {
                tmem_wait_ld_x64(ra);
                if (c + 1 < chunks) tmem_load_32x32b_x64_async(acc_addr + (c + 1) * Cfg::EPI_COLS, rb);
                chunk_out(ra, c);
                if (c + 1 < chunks) {
                    tmem_wait_ld_x64(rb);
                    if (c + 2 < chunks) tmem_load_32x32b_x64_async(acc_addr + (c + 2) * Cfg::EPI_COLS, ra);
                    chunk_out(rb, c + 1);
                }
            }
        }
        if constexpr (Cfg::EPI_SMEM) {
            if (lane == 0) bulk_wait_group<0>();
        }
    }
    (void)aborted;
    (void)sC;

    tc_fence_before_sync();
    __syncthreads();
    if (ncl > 1) {
        // No CTA of the cluster exits while another may still signal its
        // barriers or read or write its shared memory.
        cluster_arrive();
        cluster_wait();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<Cfg::CTA_GROUP>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_sm103
