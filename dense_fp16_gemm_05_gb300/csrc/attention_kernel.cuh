// attention_kernel.cuh -- attention forward for sm_103a (the FlashAttention
// loop of the TileLang-MUSA lesson, 7yue.com, section 5, and of "Writing
// High-Performance Kernels in TileLang, from GEMM to MLA", MLA section):
//
//   O[b,h,i,:] = sum_j softmax_j(sm_scale * Q[b,h,i,:] . K[b,h,j,:]) V[b,h,j,:]
//
// over keys j < seq (j <= i when causal); Q, K, V, O (batch, heads, seq, dim)
// row-major fp16, dim 64 or 128.  Per query block of 128 rows the keys are
// streamed in blocks of 128 with a running row maximum and row sum, so the
// score matrix is never stored.
//
// A persistent grid (one CTA per SM) walks the work items (pair of query
// blocks, head, batch) head by head, causal items paired heaviest with
// lightest so that each CTA's share has the same work, or from a work queue
// (see static_item and queue_item below);
// per item two query tiles of 128 rows share every K/V block.
// The next item's Q is loaded once the current item's last score MMAs are
// complete and its first score MMAs follow the current item's last products
// in the tensor core's stream, so an item's start overlaps the previous
// item's last softmax and output stores.  384 threads in three warpgroups (two of
// softmax warps, one of control warps), launched at 168 registers a thread
// (three warps share each SM sub-partition's register file); the control
// warpgroup then hands registers to the softmax warpgroups (setmaxnreg: 104
// and 200), so the 128 scores a softmax thread holds stay in registers and
// nothing spills:
//   warps 0..7         softmax (below)
//   warp 8, one lane   TMA: the two Q tiles once (3-D tensor maps: rows of
//                      another head are never read, rows past seq read as
//                      zero), then K and V blocks through rings of KV_STAGES
//                      slots, each loaded once for both tiles
//   warp 9, one lane   MMA issuer (and TMEM owner): per tile t,
//                      S^t_j = Q^t K_j^T (both from shared memory) into the
//                      tile's 128-column TMEM score buffer and
//                      O^t += P^t_j V_j into its TMEM output accumulator.  The
//                      stream alternates tiles (O^0 += P^0_j V_j, S^0_{j+1},
//                      O^1 += P^1_j V_j, S^1_{j+1}), so the tensor core works
//                      on one tile while the other tile's softmax runs
//   warps 10, 11       idle (they complete the control warpgroup)
//   warps 0..7         softmax, four warps per tile, one thread per query row
//                      (TMEM lane) and all 128 keys of a block: masked
//                      scores, row maximum, p = 2^(s*c - m) with
//                      c = sm_scale * log2(e), row sum, P in fp16 written back
//                      into TMEM over the scores it came from (the MMA reads
//                      it there as its A operand, so P costs no shared-memory
//                      traffic); at the end each thread writes its row O / l
// The reference maximum m only moves when a block's maximum exceeds it by more
// than 8 (in log2 units); then O (in TMEM) and l are multiplied by 2^(m_old -
// m_new).  Otherwise p <= 2^8 is used as is: every weight is relative to the
// same m, so the normalised result is the same, and fp16 holds p exactly as
// well (relative precision does not depend on magnitude).
// Every wait is bounded; on expiry the site is recorded in the device status
// word and all roles leave.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "gemm_kernel.cuh"

namespace gemm_sm103 {

// ---------------------------------------------------------------- PTX

// 3-D tiled load of one box into this CTA's shared memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int32_t x, int32_t y,
                                            int32_t z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// 32 consecutive fp32 TMEM columns of the warp's 32 lanes: load (and wait),
// and store (and wait).
__device__ __forceinline__ void attn_tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void attn_tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 32 consecutive 32-bit TMEM columns of the warp's 32 lanes: load without
// waiting (the registers are valid after attn_tmem_wait_ld).
__device__ __forceinline__ void attn_tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void attn_tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit TMEM columns of the warp's 32 lanes: store without
// waiting (complete after attn_tmem_wait_st).
__device__ __forceinline__ void attn_tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void attn_tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x on the special-function unit (approximate, about 2 ulp of fp32;
// 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (two lanes of arithmetic per instruction, each rounded
// to nearest as the scalar form): (d0, d1) = (a0, a1) * b + c, and
// (d0, d1) += (a0, a1).
__device__ __forceinline__ void fma2_bcast(float &d0, float &d1, float a0, float a1, float b, float c)
{
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %4};\n\t"
        "mov.b64 rc, {%5, %5};\n\t"
        "fma.rn.f32x2 ra, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1)
{
    asm("{\n\t.reg .b64 ra, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "add.rn.f32x2 rc, rc, ra;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a0), "f"(a1));
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Per-warpgroup register budget (every warp of the warpgroup executes it).
template <int kRegs>
__device__ __forceinline__ void setmaxnreg_inc()
{
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <int kRegs>
__device__ __forceinline__ void setmaxnreg_dec()
{
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// D[tmem] (+)= A[tmem] * B[smem], fp16 inputs, fp32 accumulator: the A
// operand is read from tensor memory (one row per lane, K packed two fp16 per
// 32-bit column).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ---------------------------------------------------------------- configuration

template <int kDim>
struct AttnCfg {
    static constexpr int TILES = 2;               // query tiles per CTA, sharing every K/V block
    static constexpr int BQ = 128;                // query rows per tile (TMEM lanes)
    static constexpr int BKV = 128;               // keys per block
    static constexpr int TILE_WARPS = 4;          // softmax warps per tile: one per TMEM lane quarter
    static constexpr int SOFTMAX_WARPS = TILES * TILE_WARPS;   // warps 0 .. 7
    static constexpr int TMA_WARP = SOFTMAX_WARPS;              // 8
    static constexpr int MMA_WARP = SOFTMAX_WARPS + 1;          // 9
    static constexpr int THREADS = 32 * (SOFTMAX_WARPS + 4);    // a whole control warpgroup
    static constexpr int LAUNCH_REGS = 168;   // 65536 / 384, rounded down to a multiple of 8
    static constexpr int CONTROL_REGS = 104;  // below this the MMA issuer's loop spills
    static constexpr int SOFTMAX_REGS = 200;
    static constexpr int ATOMS = kDim / 64;       // 128-byte swizzle atoms along dim
    static constexpr int TILE_BYTES = 128 * kDim * 2;   // Q, K or V tile of 128 rows
    static constexpr int ATOM_BYTES = 128 * 128;        // 128 rows x 128 bytes
    // K and V ring depth: dim 128, what shared memory holds; dim 64, measured
    // (2, 3, 4 and 6 slots: 923, 925, 911 and 906 TFLOP/s at 4 x 64 x 4096).
    static constexpr int KV_STAGES = kDim == 64 ? 3 : 2;
    static constexpr int SMEM_Q_OFF = 0;                   // TILES query tiles
    static constexpr int SMEM_K_OFF = SMEM_Q_OFF + TILES * TILE_BYTES;
    static constexpr int SMEM_V_OFF = SMEM_K_OFF + KV_STAGES * TILE_BYTES;
    static constexpr int SMEM_CTL_OFF = SMEM_V_OFF + KV_STAGES * TILE_BYTES;
    static constexpr int SMEM_CTL_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + SMEM_CTL_OFF + SMEM_CTL_BYTES;
    static constexpr int TMEM_S_COL = 0;          // per tile one 128-column score buffer; P (fp16
                                                  // pairs) overwrites the first 64 of it
    static constexpr int TMEM_O_COL = TILES * BKV;   // per tile a 128-column output accumulator
    static constexpr int TMEM_COLS = 512;
    static constexpr uint32_t IDESC_S = idesc_f16_f32(BQ, BKV, false, false);   // Q K-major, K K-major
    static constexpr uint32_t IDESC_O = idesc_f16_f32(BQ, kDim, false, true);   // P K-major, V MN-major

    static_assert(kDim == 64 || kDim == 128, "head dimension 64 or 128");
    static_assert(SOFTMAX_WARPS == 8 && THREADS == 384, "two softmax warpgroups and one control warpgroup");
    // setmaxnreg can only hand out what the launch reserved: the new budgets
    // must sum to no more than THREADS x LAUNCH_REGS.
    static_assert(32 * SOFTMAX_WARPS * SOFTMAX_REGS + 128 * CONTROL_REGS <= THREADS * LAUNCH_REGS,
                  "register budgets exceed the launch's");
    static_assert(TMEM_O_COL + TILES * 128 <= TMEM_COLS, "TMEM columns");
    static_assert(SMEM_BYTES <= 232448, "shared memory per block on sm_103");
    static_assert((14 + 4 * KV_STAGES) * 8 <= SMEM_CTL_BYTES, "control block");
};

struct AttnParams {
    int32_t batch, heads, seq;
    int32_t num_q_blocks;    // ceil(seq / 128)
    int32_t causal;
    float scale_log2;        // sm_scale * log2(e)
    uint64_t timeout_cycles;
    __half *O;
    unsigned long long *status;
    // Causal only, may be null: {next ticket, CTAs done}, zero at launch and
    // left zero at exit; with it the CTAs take work items from a shared
    // queue (heaviest first within groups of chunk_heads heads) instead of
    // the fixed assignment.
    unsigned int *queue;
    int32_t chunk_heads;
};

template <int kDim>
__global__ void __launch_bounds__(AttnCfg<kDim>::THREADS, 1)
    attention_fwd_sm103a(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const AttnParams p)
{
    using Cfg = AttnCfg<kDim>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t sQ = base + Cfg::SMEM_Q_OFF;
    const uint32_t sK = base + Cfg::SMEM_K_OFF;
    const uint32_t sV = base + Cfg::SMEM_V_OFF;
    const uint32_t ctl = base + Cfg::SMEM_CTL_OFF;
    // Barriers (8 bytes each): q_full; k_full, k_empty, v_full, v_empty
    // [KV_STAGES] (the K and V rings); per tile s_full, p_full, o_ready;
    // drain; q_empty; then the TMEM address slot and the abort flag;
    // item_full[2]; the item ring[2] (query-block pair and head-batch index
    // of the CTA's item k in entry k % 2, written by the producer before it
    // arrives on item_full[k % 2]).  Their phases run over all items of the
    // CTA: the K/V ring by the CTA's running count of key blocks, s_full /
    // p_full by each tile's running count of blocks, q_full / q_empty /
    // item_full / o_ready by the item count.  The producer publishes item
    // k + 2 only after item k + 1's score MMAs are complete (q_empty), when
    // both tiles' softmax warps are past reading entry k.
    //
    // Order of the MMA stream: S^0_0, S^1_0, then per block j and tile t:
    // O^t += P^t_j V_j, S^t_{j+1}.  Tile t's score buffer is rewritten by
    // S^t_{j+1} only after O^t += P^t_j V_j (issued before it) read P^t_j, and
    // S^t_j completes after O^t += P^t_{j-1} V_{j-1}: when the softmax sees
    // the scores of block j, tile t's output holds blocks 0 .. j-1 exactly.
    constexpr int S = Cfg::KV_STAGES;
    const uint32_t q_full = ctl;
    auto k_full = [&](int i) { return ctl + 8u * (1 + i); };
    auto k_empty = [&](int i) { return ctl + 8u * (1 + S + i); };
    auto v_full = [&](int i) { return ctl + 8u * (1 + 2 * S + i); };
    auto v_empty = [&](int i) { return ctl + 8u * (1 + 3 * S + i); };
    auto s_full = [&](int t) { return ctl + 8u * (1 + 4 * S + t); };
    auto p_full = [&](int t) { return ctl + 8u * (3 + 4 * S + t); };
    auto o_ready = [&](int t) { return ctl + 8u * (5 + 4 * S + t); };
    const uint32_t drain = ctl + 8u * (7 + 4 * S);
    const uint32_t q_empty = ctl + 8u * (8 + 4 * S);   // the item's score MMAs (readers of Q) are complete
    const uint32_t tmem_slot = ctl + 8u * (9 + 4 * S);
    const uint32_t abort_addr = tmem_slot + 4;
    volatile uint32_t *tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t *>(base_ptr + Cfg::SMEM_CTL_OFF + 8 * (9 + 4 * S));
    auto item_full = [&](int i) { return ctl + 8u * (10 + 4 * S + i); };
    volatile int *ring = reinterpret_cast<volatile int *>(base_ptr + Cfg::SMEM_CTL_OFF + 8 * (12 + 4 * S));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work items: an item is a pair of query blocks grp (tile t covers query
    // block 2 * grp + t) of one head-batch index bh.
    //
    // Fixed assignment: with the causal mask the items are grouped two by two
    // into super-items of one head, the heaviest pair with the lightest, the
    // next heaviest with the next lightest, ..., so that every super-item has
    // the same number of key blocks; without it every item has the same work
    // and a super-item is one item.  Super-items are numbered head by head,
    // and CTA c takes super-items c, c + G, ... (G CTAs): at any time the CTAs
    // work on a few heads at once, whose K and V the L2 then serves to all of
    // them.  static_item(k) decodes this CTA's k-th item: 1 = an item, 0 =
    // none at this k (the middle pair of an odd count), -1 = no more.
    //
    // Work queue (causal, p.queue given): items are numbered in groups of
    // chunk_heads heads, heaviest pairs first within a group, so that the
    // light items come last in each group and the CTAs finish together; CTA c
    // starts with item c and then takes item G + the next ticket.
    const int n_grp = (p.num_q_blocks + Cfg::TILES - 1) / Cfg::TILES;
    const int hb_count = p.batch * p.heads;
    const bool use_queue = p.causal && p.queue != nullptr;
    const int num_items = n_grp * hb_count;
    const int sup_shift = p.causal ? 1 : 0;   // log2 of the items per super-item
    const int n_sub = p.causal ? (n_grp + 1) / 2 : n_grp;
    const int num_super = n_sub * hb_count;
    const int first = static_cast<int>(blockIdx.x), stride = static_cast<int>(gridDim.x);
    const int kv_blocks_all = (p.seq + Cfg::BKV - 1) / Cfg::BKV;
    auto static_item = [&](int k, int &grp, int &bh) -> int {
        const int sup = first + (k >> sup_shift) * stride;
        if (sup >= num_super) return -1;
        bh = sup / n_sub;
        const int kp = sup - bh * n_sub;
        if (!p.causal) {
            grp = kp;
            return 1;
        }
        grp = (k & 1) ? kp : n_grp - 1 - kp;
        if ((k & 1) && grp == n_grp - 1 - kp) return 0;
        return 1;
    };
    auto queue_item = [&](int w, int &grp, int &bh) {
        const int per_chunk = p.chunk_heads * n_grp;
        const int c = w / per_chunk;
        const int h0 = c * p.chunk_heads;
        const int ych = min(p.chunk_heads, hb_count - h0);
        const int r = w - c * per_chunk;
        grp = n_grp - 1 - r / ych;
        bh = h0 + (r - (r / ych) * ych);
    };
    // Key blocks of each tile (tile 1 never needs fewer than tile 0; both >= 1).
    auto tile_blocks = [&](int grp, int &nb0, int &nb1) {
        nb0 = p.causal ? min(2 * grp + 1, kv_blocks_all) : kv_blocks_all;
        nb1 = p.causal ? min(2 * grp + 2, kv_blocks_all) : kv_blocks_all;
    };

    AbortFlag abort;
    abort.local = reinterpret_cast<volatile int *>(tmem_slot_ptr + 1);
    abort.status = p.status;
    abort.addr = abort_addr;
    abort.cluster = 1;
    abort.rank = 0;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < S; ++i) {
            mbar_init(k_full(i), 1);
            mbar_init(k_empty(i), 1);
            mbar_init(v_full(i), 1);
            mbar_init(v_empty(i), 1);
        }
        for (int t = 0; t < Cfg::TILES; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), Cfg::TILE_WARPS);
            mbar_init(o_ready(t), 1);
        }
        mbar_init(drain, 1);
        mbar_init(q_empty, 1);
        mbar_init(item_full(0), 1);
        mbar_init(item_full(1), 1);
        *abort.local = 0;
        fence_mbar_init();
    }
    if (warp == Cfg::TMA_WARP && lane == 0) {
        prefetch_tensormap(&tmap_q);
        prefetch_tensormap(&tmap_k);
        prefetch_tensormap(&tmap_v);
    }
    if (warp == Cfg::MMA_WARP) {
        tmem_alloc<1>(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // Set-up above may overlap the previous kernel of the stream; nothing
    // below runs before its results are visible (programmatic dependent launch).
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot_ptr;
    const uint64_t limit = p.timeout_cycles;
    // Each role sets its warpgroup's register budget first thing in its own
    // branch (the compiler allocates each branch's registers within it).

    if (warp == Cfg::TMA_WARP) {
        // ------------------------------------------------------------ TMA producer
        setmaxnreg_dec<Cfg::CONTROL_REGS>();
        if (lane == 0) {
            bool ok = true;
            int kvc = 0;   // key blocks loaded by this CTA so far (the K/V rings' position)
            int ks = 0;    // position in the fixed assignment
            for (int it = 0; ok; ++it) {
                int grp = -1, bh = 0;
                if (use_queue) {
                    const int w = it == 0 ? first : stride + static_cast<int>(atomicAdd(p.queue, 1u));
                    if (w < num_items) queue_item(w, grp, bh);
                } else {
                    int have;
                    while ((have = static_item(ks++, grp, bh)) == 0) {
                    }
                    if (have < 0) grp = -1;
                }
                // Item it - 1's score MMAs, the readers of Q, are complete (and
                // every consumer is past ring entry it - 2).
                if (it > 0 && !wait_phase(q_empty, (it - 1) & 1u, abort, limit, kSiteProducerEmpty)) {
                    ok = false;
                    break;
                }
                ring[2 * (it & 1)] = grp;   // grp < 0: no more items
                ring[2 * (it & 1) + 1] = bh;
                mbar_arrive(item_full(it & 1));
                if (grp < 0) break;
                int nb0, nb1;
                tile_blocks(grp, nb0, nb1);
                mbar_arrive_expect_tx(q_full, Cfg::TILES * Cfg::TILE_BYTES);
                for (int t = 0; t < Cfg::TILES; ++t) {
#pragma unroll
                    for (int a = 0; a < Cfg::ATOMS; ++a)
                        tma_load_3d(sQ + t * Cfg::TILE_BYTES + a * Cfg::ATOM_BYTES, &tmap_q, q_full, a * 64,
                                    (2 * grp + t) * Cfg::BQ, bh);
                }
                for (int j = 0; j < nb1; ++j, ++kvc) {
                    const int slot = kvc % S;
                    const uint32_t ph = (kvc / S) & 1u;
                    if (!wait_phase(k_empty(slot), ph ^ 1u, abort, limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(k_full(slot), Cfg::TILE_BYTES);
#pragma unroll
                    for (int a = 0; a < Cfg::ATOMS; ++a)
                        tma_load_3d(sK + slot * Cfg::TILE_BYTES + a * Cfg::ATOM_BYTES, &tmap_k, k_full(slot),
                                    a * 64, j * Cfg::BKV, bh);
                    if (!wait_phase(v_empty(slot), ph ^ 1u, abort, limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(v_full(slot), Cfg::TILE_BYTES);
#pragma unroll
                    for (int a = 0; a < Cfg::ATOMS; ++a)
                        tma_load_3d(sV + slot * Cfg::TILE_BYTES + a * Cfg::ATOM_BYTES, &tmap_v, v_full(slot),
                                    a * 64, j * Cfg::BKV, bh);
                }
            }
            if (use_queue) {
                // Every CTA stops taking tickets before it counts itself done;
                // the last one to count leaves the queue zero for the next launch.
                if (atomicAdd(p.queue + 1, 1u) == gridDim.x - 1u) {
                    atomicExch(p.queue, 0u);
                    atomicExch(p.queue + 1, 0u);
                }
            }
            if (!ok) {
                // Let every load this thread issued land before the CTA exits
                // (each ring slot holds at most one load in flight).
                const long long t0 = clock64();
                while (clock64() - t0 < 1000000) {
                }
            }
        }
        __syncwarp();
    } else if (warp == Cfg::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuer
        setmaxnreg_dec<Cfg::CONTROL_REGS>();
        if (lane == 0) {
            bool ok = true;
            bool issued_any = false;
            int kvb = 0;          // key blocks of this CTA's earlier items (the K/V rings' position)
            int bc[2] = {0, 0};   // each tile's blocks in this CTA's earlier items
            const uint64_t q_desc0 = smem_desc_sw128(sQ, 16, 1024);
            const uint64_t k_desc0 = smem_desc_sw128(sK, 16, 1024);
            const uint64_t v_desc0 = smem_desc_sw128(sV, Cfg::ATOM_BYTES, 1024);
            // K step t of 16 elements along dim (K-major tiles of 128 rows):
            // atom t/4, +32 B per step inside it.
            auto dim_step = [](int t) -> uint64_t {
                return static_cast<uint64_t>(((t >> 2) * Cfg::ATOM_BYTES + (t & 3) * 32) >> 4);
            };
            // S^t_j = Q^t K_j^T into tile t's score buffer; the second user of
            // a K slot (tile 1) releases it.  Tile 1 waits for the K block only
            // when tile 0 does not use it (tile 0, issued before, has seen it
            // arrive, and the slot is not refilled before tile 1 releases it).
            auto issue_s = [&](int t, int j, bool seen) -> bool {
                const int ks = (kvb + j) % S;
                if (!seen && !wait_phase(k_full(ks), ((kvb + j) / S) & 1u, abort, limit, kSiteMmaFull)) return false;
                const uint32_t s_tmem = tmem_base + Cfg::TMEM_S_COL + t * Cfg::BKV;
                const uint64_t q_desc = q_desc0 + static_cast<uint64_t>((t * Cfg::TILE_BYTES) >> 4);
                const uint64_t k_desc = k_desc0 + static_cast<uint64_t>((ks * Cfg::TILE_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < kDim / 16; ++k)
                    mma_f16_ss<1>(s_tmem, q_desc + dim_step(k), k_desc + dim_step(k), Cfg::IDESC_S,
                                  k > 0 ? 1u : 0u);
                if (t == 1) mma_commit(k_empty(ks));
                mma_commit(s_full(t));
                issued_any = true;
                return true;
            };
            // O^t += P^t_j V_j (P in TMEM, over the scores it came from); the
            // second user of a V slot (tile 1) releases it (the V block waited
            // for as the K block above).  o_ready(t) is signalled after the
            // tile's last product of the item only (last).
            auto issue_pv = [&](int t, int j, bool seen, bool last) -> bool {
                const int vs = (kvb + j) % S;
                if ((!seen && !wait_phase(v_full(vs), ((kvb + j) / S) & 1u, abort, limit, kSiteMmaFull)) ||
                    !wait_phase(p_full(t), (bc[t] + j) & 1u, abort, limit, kSiteMmaTmemEmpty))
                    return false;
                tc_fence_after_sync();
                const uint32_t p_tmem = tmem_base + Cfg::TMEM_S_COL + t * Cfg::BKV;
                const uint32_t o_tmem = tmem_base + Cfg::TMEM_O_COL + t * 128;
                const uint64_t v_desc = v_desc0 + static_cast<uint64_t>((vs * Cfg::TILE_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < Cfg::BKV / 16; ++k) {
                    // P (A, in TMEM): 16 keys = 8 columns per step; V (B,
                    // MN-major along dim): 16 key rows = +2 KB per step.
                    const uint64_t vb = v_desc + static_cast<uint64_t>((k * 16 * 128) >> 4);
                    mma_f16_ts(o_tmem, p_tmem + k * 8, vb, Cfg::IDESC_O, (j > 0 || k > 0) ? 1u : 0u);
                }
                if (t == 1) mma_commit(v_empty(vs));
                if (last) mma_commit(o_ready(t));
                return true;
            };
            for (int it = 0; ok; ++it) {
                if (!wait_phase(item_full(it & 1), (it >> 1) & 1u, abort, limit, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                const int grp = ring[2 * (it & 1)];
                if (grp < 0) break;
                int nb0, nb1;
                tile_blocks(grp, nb0, nb1);
                // This item's Q is in shared memory.  Its first score MMAs follow
                // the previous item's last products in the stream: tile t's
                // score buffer holds that item's last P until then, and each
                // tile's output is overwritten (accumulate = 0 at block 0) only
                // once the softmax warps, done with the previous item's output,
                // have handed over this item's first P.
                if (!wait_phase(q_full, it & 1u, abort, limit, kSiteMmaFull)) {
                    ok = false;
                    break;
                }
                ok = issue_s(0, 0, false) && issue_s(1, 0, true);
                // The item's last score MMA is S^1_{nb1-1}; once it completes, Q
                // may be overwritten with the next item's.
                if (ok && nb1 == 1) mma_commit(q_empty);
                for (int j = 0; ok && j < nb1; ++j) {
                    if (j < nb0) {
                        if (!issue_pv(0, j, false, j + 1 == nb0) || (j + 1 < nb0 && !issue_s(0, j + 1, false))) {
                            ok = false;
                            break;
                        }
                    }
                    if (!issue_pv(1, j, j < nb0, j + 1 == nb1) || (j + 1 < nb1 && !issue_s(1, j + 1, j + 1 < nb0))) {
                        ok = false;
                        break;
                    }
                    if (j + 2 == nb1) mma_commit(q_empty);
                }
                kvb += nb1;
                bc[0] += nb0;
                bc[1] += nb1;
            }
            if (!ok) {
                if (issued_any) {
                    // Wait for this thread's MMAs before the TMEM is freed.
                    mma_commit(drain);
                    wait_phase_drain(drain, 0, limit, kSiteDrainMma, p.status);
                }
            }
        }
        __syncwarp();
    } else if (warp < Cfg::SOFTMAX_WARPS) {
        // ------------------------------------------------------------ softmax (warps 0..7)
        setmaxnreg_inc<Cfg::SOFTMAX_REGS>();
        // One thread per query row (TMEM lane) and all 128 keys of a block.
        const int t = warp / Cfg::TILE_WARPS;        // query tile
        const int q = warp & 3;                      // TMEM lane quarter
        const int row_local = q * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t s_base = tmem_base + lane_addr + Cfg::TMEM_S_COL + t * Cfg::BKV;
        const uint32_t o_addr = tmem_base + lane_addr + Cfg::TMEM_O_COL + t * 128;
        constexpr int NK = Cfg::BKV;   // keys per block
        bool ok = true;
        int bc = 0;   // this tile's blocks in the CTA's earlier items (the barriers' phases)
        for (int it = 0; ok; ++it) {
            const bool got_item = wait_phase(item_full(it & 1), (it >> 1) & 1u, abort, limit, kSiteEpilogueTmemFull);
            if (!__all_sync(0xffffffffu, got_item)) {
                ok = false;
                break;
            }
            const int grp = ring[2 * (it & 1)];
            const int bh = ring[2 * (it & 1) + 1];
            if (grp < 0) break;
            int nb0, nb1;
            tile_blocks(grp, nb0, nb1);
            const int row = (2 * grp + t) * Cfg::BQ + row_local;
            const int nblk = t == 0 ? nb0 : nb1;
            float m_ref = -INFINITY;       // reference maximum (log2 units, scaled scores)
            float l = 0.0f;                // row sum of weights relative to m_ref
            for (int j = 0; j < nblk; ++j) {
                const bool got = wait_phase(s_full(t), (bc + j) & 1u, abort, limit, kSiteEpilogueTmemFull);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // The row's 128 raw scores of block j; the scale (positive) is
                // applied inside the exponent's argument.
                float x[NK];
                {
                    uint32_t r[4][32];
    #pragma unroll
                    for (int c = 0; c < 4; ++c) attn_tmem_ld32_nowait(s_base + c * 32, r[c]);
                    attn_tmem_wait_ld();
    #pragma unroll
                    for (int c = 0; c < 4; ++c)
    #pragma unroll
                        for (int i = 0; i < 32; ++i) x[c * 32 + i] = __uint_as_float(r[c][i]);
                }
                const int key0 = j * Cfg::BKV;
                const int last_key = p.causal ? min(row, p.seq - 1) : p.seq - 1;
                if (key0 + NK - 1 > last_key) {
    #pragma unroll
                    for (int i = 0; i < NK; ++i)
                        if (key0 + i > last_key) x[i] = -INFINITY;
                }
                // Maximum as eight independent chains of three-input maxima.
                float m8[8];
    #pragma unroll
                for (int k = 0; k < 8; ++k) {
                    m8[k] = max3(x[16 * k], x[16 * k + 1], x[16 * k + 2]);
    #pragma unroll
                    for (int i = 3; i < 15; i += 2) m8[k] = max3(m8[k], x[16 * k + i], x[16 * k + i + 1]);
                    m8[k] = fmaxf(m8[k], x[16 * k + 15]);
                }
                const float mx = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])) *
                                 p.scale_log2;
                // Move the reference only when the block's maximum exceeds it by
                // more than 8 (weights then stay <= 2^8).
                float alpha = 1.0f;
                if (mx > m_ref + 8.0f) {
                    alpha = ex2_approx(m_ref - mx);   // 0 on the first block (m_ref = -inf)
                    l *= alpha;
                    m_ref = mx;
                }
                const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.0f);
                // P (fp16 pairs) into TMEM over the scores of this block: keys
                // 32c .. 32c+31 are columns 16c .. 16c+15 of the buffer, scores
                // this thread has already read into registers.
                float lsum0 = 0.0f, lsum1 = 0.0f;
                const float neg_m = -m_ref;
    #pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pw[16];
    #pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float a0, a1;   // s * c - m for the pair, one packed instruction
                        fma2_bcast(a0, a1, x[32 * c + 2 * i], x[32 * c + 2 * i + 1], p.scale_log2, neg_m);
                        const float p0 = ex2_approx(a0);
                        const float p1 = ex2_approx(a1);
                        add2(lsum0, lsum1, p0, p1);
                        const __half2 v = __floats2half2_rn(p0, p1);
                        pw[i] = *reinterpret_cast<const uint32_t *>(&v);
                    }
                    attn_tmem_st16_nowait(s_base + c * 16, pw);
                }
                l += lsum0 + lsum1;
                if (rescale) {
                    // The output holds exactly blocks 0 .. j-1 (see the MMA order
                    // above): rescale the row's dim columns.
    #pragma unroll
                    for (int c = 0; c < kDim / 32; ++c) {
                        uint32_t r[32];
                        attn_tmem_ld32(o_addr + c * 32, r);
    #pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                        attn_tmem_st32(o_addr + c * 32, r);
                    }
                }
                attn_tmem_wait_st();
                tc_fence_before_sync();   // P (and a rescaled O) in TMEM before the MMA is told
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(t));
            }
            if (ok) {
                // The MMAs of the tile's last block (one phase per item: signalled
                // after the tile's last product; those before completed before it).
                const bool got_o = wait_phase(o_ready(t), it & 1u, abort, limit, kSiteEpilogueTmemFull);
                if (!__all_sync(0xffffffffu, got_o)) {
                    ok = false;
                } else {
                    tc_fence_after_sync();
                    const float inv_l = 1.0f / l;
                    __half *orow = p.O + (static_cast<int64_t>(bh) * p.seq + row) * kDim;
    #pragma unroll
                    for (int c = 0; c < kDim / 32; ++c) {
                        uint32_t r[32];
                        attn_tmem_ld32(o_addr + c * 32, r);
                        if (row < p.seq) {
    #pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                uint32_t wv[4];
    #pragma unroll
                                for (int h = 0; h < 4; ++h) {
                                    const __half2 hv = __floats2half2_rn(__uint_as_float(r[8 * v + 2 * h]) * inv_l,
                                                                         __uint_as_float(r[8 * v + 2 * h + 1]) * inv_l);
                                    wv[h] = *reinterpret_cast<const uint32_t *>(&hv);
                                }
                                st_global_v4(orow + c * 32 + v * 8, wv[0], wv[1], wv[2], wv[3]);
                            }
                        }
                    }
                }
            }
            bc += nblk;
        }
    }

    else {
        // ------------------------------------------------------------ idle (warps 10, 11)
        setmaxnreg_dec<Cfg::CONTROL_REGS>();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == Cfg::MMA_WARP) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_sm103
