// gemm_mxfp8_kernel.cuh -- FP8 (E4M3) block-scaled GEMM with power-of-two
// block scales applied inside the tensor core, for sm_103a:
//
//   C[i,j] = R( sum_b 2^(SA[i,b] - 127) * 2^(SW[j/128, b] - 127) * sum_{k in block b} A[i,k] W[j,k] )
//
// The operation of gemm_fp8_kernel.cuh (the FP8 block-scaled linear layer of
// the TileLang-MUSA lesson, 7yue.com, section 8.2, blocks of 128) with every
// scale a power of two, given as its E8M0 exponent byte (value 2^(byte-127)):
// SA (M, KB) per row of A and 128-element K block, SW (ceil(N/128), KB) per
// 128 x 128 block of W, KB = ceil(K/128).  A power-of-two scale is exactly
// what tcgen05.mma.kind::mxf8f6f4.block_scale multiplies each 32-element
// product group by, so no partial sum leaves the tensor core: the MMAs of all
// K blocks accumulate into one fp32 accumulator in TMEM, as in the fp16
// kernel, and the promotion work of the fp32-scale kernel disappears.
//
// Scale factors in TMEM: the MMA reads one 32-bit word per row of A (at the
// row's lane) and per group of 32 columns of B, and takes the byte that the
// instruction descriptor's scale ids select.  Four consecutive K blocks share
// one word (byte i = K block 4g + i), so one store serves four blocks and the
// MMAs of block kb select byte kb % 4; a TMEM slot holds four such words (16
// K blocks per hand-off between the scale writers and the MMA issuer; one word
// per slot measured 1.5 % slower).  Every K block of 128 is four MMAs of
// K = 32 with the same scales.  The scale of A row m is stored in every
// column of its lane's A range, so whichever column the MMA reads for a row
// it finds the row's word.  For the B scales, each CTA of the pair supplies
// the words for the accumulator rows in its own TMEM, for all N = 256
// columns of the MMA: column group n / 32 at column sfb + n / 32, the same
// word in every lane.  Columns [0, 128) of the tile lie in W block 2 nb and
// [128, 256) in block 2 nb + 1, so both CTAs write block 2 nb's word into
// columns 0..3 of the B range and block 2 nb + 1's into 4..7.  (Established
// on this GPU by decoding which exponent each output element received, with
// A, W and the scales chosen so that every element names its byte.)
//
// Roles per CTA (320 threads, one CTA per SM, a cluster = one CTA pair, a
// persistent grid over 256 x 256 output tiles in grouped raster order; each
// CTA holds 128 rows of the tile's accumulator, 256 TMEM columns):
//   warp 0, one lane   TMA producer: an A box 128 (K) x 128 rows and a W box
//                      128 (K) x 128 rows per K block (each CTA supplies 128
//                      of the tile's 256 columns), completing on the pair
//                      leader's "full" barrier
//   warp 1, one lane   (leader CTA only) MMA issuer, tcgen05.mma.cta_group::2
//                      M = 256, N = 256; warp 1 also allocates the 512 TMEM
//                      columns (the accumulator and a ring of scale slots)
//   warps 2..5         epilogue: reads the whole accumulator out of TMEM
//                      (double-buffered loads, ReLU, fp16, into a swizzled
//                      staging tile in shared memory) and hands TMEM back
//                      before the TMA stores, so the next tile's MMAs wait
//                      only for the reads
//   warps 6..9         scale writers: per 16 K blocks, read the scale bytes
//                      and store the packed words into a TMEM slot
// Ragged edges: TMA zero-fills operand elements outside A or W; rows and
// columns outside C are not stored.  Every wait is bounded; on expiry the
// site is recorded in the device status word and all roles leave.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "gemm_kernel.cuh"

namespace gemm_sm103 {

// ---------------------------------------------------------------- PTX

// D[tmem] (+)= (A[smem] x scale_A) * (B[smem] x scale_B), E4M3 operands,
// E8M0 scales from TMEM (one per row of A and per column of B for the
// instruction's K = 32), fp32 accumulator, CTA pair (M = 256).
__device__ __forceinline__ void mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Stores one 32-bit column of the warp's 32 TMEM lanes (one value per thread).
__device__ __forceinline__ void tmem_store_x1(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

// Stores eight consecutive 32-bit columns of the warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_store_x8(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3,
                                              uint32_t v4, uint32_t v5, uint32_t v6, uint32_t v7)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(v0), "r"(v1), "r"(v2), "r"(v3), "r"(v4), "r"(v5), "r"(v6), "r"(v7)
                 : "memory");
}

// Waits until this thread's TMEM stores are complete.
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Instruction descriptor for tcgen05.mma.kind::mxf8f6f4.block_scale: E4M3 A and
// B (format 0 in bits 7-9 and 10-12), both K-major (bits 15, 16 = 0), N >> 3
// (17-22), E8M0 scale type (bit 23), M >> 4 (24-28), scale ids 0 (bits 4-5 for
// B, 29-30 for A).
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(int M, int N)
{
    return (static_cast<uint32_t>(N >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(M >> 4) << 24);
}

// The descriptor with both scale ids set to `id` (byte `id` of the scale words).
__device__ __forceinline__ uint32_t idesc_with_sf_id(uint32_t idesc, uint32_t id)
{
    return idesc | (id << 4) | (id << 29);
}

// Stores four consecutive 32-bit columns of the warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_store_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
                 "r"(v2), "r"(v3)
                 : "memory");
}

// ---------------------------------------------------------------- configuration

struct MxCfg {
    static constexpr int BM = 128;             // rows of C per CTA (TMEM lanes)
    static constexpr int TILE_M = 256;         // rows per pair tile (the MMA's M)
    static constexpr int BN = 256;             // columns of C per tile (the MMA's N)
    static constexpr int BN_CTA = BN / 2;      // rows of W each CTA loads
    static constexpr int BK = 128;             // E4M3 elements per K block = one 128-byte swizzle row
    static constexpr int SCALE_BLOCK = 128;
    static constexpr int UMMA_K = 32;
    static constexpr int SF_PACK = 4;          // K blocks per scale word (one byte each)
    static constexpr int STAGES = 5;           // operand ring
    static constexpr int SF_WORDS = 4;         // scale words per TMEM slot (SF_PACK K blocks each)
    static constexpr int SF_KB = SF_PACK * SF_WORDS;   // K blocks per slot (one hand-off)
    static constexpr int SF_SLOTS = SF_WORDS == 4 ? 4 : 8;   // scale slots in TMEM
    static constexpr int SF_BATCH = 4;         // scale words a writer loads ahead, per batch
    static constexpr int THREADS = 320;
    static constexpr int A_STAGE_BYTES = BM * BK;       // 16 KiB
    static constexpr int W_STAGE_BYTES = BN_CTA * BK;   // 16 KiB
    static constexpr int STAGE_TX_BYTES = A_STAGE_BYTES + W_STAGE_BYTES;
    static constexpr int ACC_COLS = BN;                 // one accumulator
    static constexpr int SF_COL0 = ACC_COLS;            // first scale slot
    // Slot layout: A word w in columns 4w .. 4w+3, B words w from column
    // SFB_COL + 8w (8 columns each); slots start on multiples of 16 columns.
    static constexpr int SFB_COL = SF_WORDS == 1 ? 8 : 4 * SF_WORDS;
    static constexpr int SF_SLOT_COLS = SF_WORDS == 1 ? 16 : (SF_WORDS == 2 ? 32 : 64);
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_COLS = 64;
    static constexpr int EPI_CHUNKS = BN / EPI_COLS;    // 4
    static constexpr int C_BUF_BYTES = 32 * EPI_COLS * 2;   // one warp's 32 rows of one chunk
    static constexpr int SMEM_A_OFF = 0;
    static constexpr int SMEM_W_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int SMEM_C_OFF = SMEM_W_OFF + STAGES * W_STAGE_BYTES;
    static constexpr int SMEM_CTL_OFF = SMEM_C_OFF + 4 * EPI_CHUNKS * C_BUF_BYTES;   // the whole tile staged
    static constexpr int SMEM_CTL_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + SMEM_CTL_OFF + SMEM_CTL_BYTES;
    static constexpr uint32_t IDESC = idesc_mxf8_e4m3(TILE_M, BN);

    static_assert(BK == SCALE_BLOCK && 2 * SCALE_BLOCK == BN, "one scale per K block and W block");
    static_assert(SF_COL0 + SF_SLOTS * SF_SLOT_COLS <= TMEM_COLS, "TMEM columns");
    static_assert(SFB_COL + 8 * SF_WORDS <= SF_SLOT_COLS && SF_BATCH % SF_WORDS == 0, "scale slot layout");
    static_assert((2 * STAGES + 2 * SF_SLOTS + 4) * 8 + 8 <= SMEM_CTL_BYTES, "control block");
    static_assert(SMEM_BYTES <= 232448, "shared memory per block on sm_103");
};

struct MxParams {
    int32_t M, N, K;
    int32_t num_m_blocks;   // ceil(M / 256)
    int32_t num_n_blocks;   // ceil(N / 256)
    int32_t num_k_blocks;   // ceil(K / 128) = KB, the columns of SA and SW
    int32_t num_w_blocks;   // ceil(N / 128), the rows of SW
    int32_t num_tiles;
    int32_t group_m;        // rasterisation panel height, in tiles
    uint64_t timeout_cycles;
    const uint8_t *SA;      // (M, KB) E8M0
    const uint8_t *SW;      // (num_w_blocks, KB) E8M0
    unsigned long long *status;
};

__device__ __forceinline__ void mx_tile_coords(int t, const MxParams &p, int &mb, int &nb)
{
    const int per_group = p.group_m * p.num_n_blocks;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.num_m_blocks - first_m, p.group_m);
    const int r = t - g * per_group;
    mb = first_m + r % rows;
    nb = r / rows;
}

template <bool kRelu>
__global__ void __launch_bounds__(MxCfg::THREADS, 1)
    gemm_mxfp8_sm103a(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                      const __grid_constant__ CUtensorMap tmap_c, const MxParams p)
{
    using Cfg = MxCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // SW128 atoms need 1024-byte alignment
    uint8_t *base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base + Cfg::SMEM_A_OFF;
    const uint32_t sW = base + Cfg::SMEM_W_OFF;
    const uint32_t sC = base + Cfg::SMEM_C_OFF;
    const uint32_t ctl = base + Cfg::SMEM_CTL_OFF;
    constexpr int S = Cfg::STAGES, SF = Cfg::SF_SLOTS, P = Cfg::SF_PACK;
    auto full_bar = [&](int s) { return ctl + 8u * s; };
    auto empty_bar = [&](int s) { return ctl + 8u * (S + s); };
    auto sfull_bar = [&](int j) { return ctl + 8u * (2 * S + j); };
    auto sempty_bar = [&](int j) { return ctl + 8u * (2 * S + SF + j); };
    const uint32_t tfull_bar = ctl + 8u * (2 * S + 2 * SF);
    const uint32_t tempty_bar = ctl + 8u * (2 * S + 2 * SF + 1);
    const uint32_t drain_bar = ctl + 8u * (2 * S + 2 * SF + 2);
    const uint32_t tmem_slot = ctl + 8u * (2 * S + 2 * SF + 3);
    const uint32_t abort_addr = tmem_slot + 4;
    volatile uint32_t *tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t *>(base_ptr + Cfg::SMEM_CTL_OFF + 8 * (2 * S + 2 * SF + 3));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();   // 0: the pair leader, which issues the MMAs
    const bool leader = rank == 0;
    constexpr uint16_t kPairMask = 0x3u;

    AbortFlag abort;
    abort.local = reinterpret_cast<volatile int *>(tmem_slot_ptr + 1);
    abort.status = p.status;
    abort.addr = abort_addr;
    abort.cluster = 2;
    abort.rank = rank;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 2);    // each CTA's arrive.expect_tx (used on the leader)
            mbar_init(empty_bar(s), 1);   // one MMA commit, sent to both CTAs
        }
        for (int j = 0; j < SF; ++j) {
            mbar_init(sfull_bar(j), 8);   // one arrive per scale-writer warp of both CTAs
            mbar_init(sempty_bar(j), 1);  // one MMA commit, sent to both CTAs
        }
        mbar_init(tfull_bar, 1);          // one MMA commit, sent to both CTAs
        mbar_init(tempty_bar, 8);         // one arrive per epilogue warp of both CTAs
        mbar_init(drain_bar, 1);
        *abort.local = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_w);
        prefetch_tensormap(&tmap_c);
    }
    if (warp == 1) {
        tmem_alloc<2>(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish<2>();
    }
    tc_fence_before_sync();
    __syncthreads();
    // Both CTAs' barriers are initialised and their TMEM allocated before
    // either signals the other.
    cluster_arrive();
    cluster_wait();
    tc_fence_after_sync();
    // The set-up above may overlap the previous kernel of the stream; each
    // role waits for it (griddep_wait) before its first global access.
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot_ptr;
    const uint64_t limit = p.timeout_cycles;
    const int KB = p.num_k_blocks;
    const int first = static_cast<int>(blockIdx.x >> 1), stride = static_cast<int>(gridDim.x >> 1);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true, dep_waited = false;
            const uint32_t full_base = leader ? full_bar(0) : mapa_shared(full_bar(0), 0);
            for (int t = first; ok && t < p.num_tiles; t += stride) {
                int mb, nb;
                mx_tile_coords(t, p, mb, nb);
                const int m0 = mb * Cfg::TILE_M + static_cast<int>(rank) * Cfg::BM;
                const int n0 = nb * Cfg::BN + static_cast<int>(rank) * Cfg::BN_CTA;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort, limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (!dep_waited) {
                        griddep_wait();
                        dep_waited = true;
                    }
                    // Both CTAs' bytes are counted on the leader's barrier; each
                    // announces its own.
                    const uint32_t fb = full_base + 8u * s;
                    if (leader) mbar_arrive_expect_tx(fb, Cfg::STAGE_TX_BYTES);
                    else mbar_arrive_expect_tx_cluster(fb, Cfg::STAGE_TX_BYTES);
                    const int k0 = kb * Cfg::BK;
                    tma_load_2d_pair(sA + s * Cfg::A_STAGE_BYTES, &tmap_a, fb, k0, m0);
                    tma_load_2d_pair(sW + s * Cfg::W_STAGE_BYTES, &tmap_w, fb, k0, n0);
                    issued_mask |= 1u << s;
                    issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    // Let the loads in flight land before the CTA exits.
                    for (int i = 0; i < S; ++i)
                        if (issued_mask & (1u << i))
                            wait_phase_drain(full_bar(i), (issued_parity >> i) & 1u, limit, kSiteDrainLoads,
                                             p.status);
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
            int s = 0, j = 0;
            uint32_t ph = 0, sph = 0, acc_it = 0;
            bool ok = true, issued_any = false;
            // K-major SW128 operands: 8-row groups 1024 B apart; a K step of 32
            // one-byte elements is +32 B inside the swizzle row.
            const uint64_t a_desc0 = smem_desc_sw128(sA, 16, 1024);
            const uint64_t w_desc0 = smem_desc_sw128(sW, 16, 1024);
            for (int t = first; ok && t < p.num_tiles; t += stride, ++acc_it) {
                // The previous tile's accumulator has been read by both CTAs.
                if (!wait_phase(tempty_bar, (acc_it & 1u) ^ 1u, abort, limit, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                for (int kb = 0; kb < KB; ++kb) {
                    const int in_slot = kb % Cfg::SF_KB;
                    const int word = in_slot / P, in_word = in_slot % P;
                    if (in_slot == 0) {
                        // The next scale slot (this and the next P - 1 K blocks).
                        if (!wait_phase(sfull_bar(j), sph, abort, limit, kSiteMmaFull)) {
                            ok = false;
                            break;
                        }
                    }
                    if (!wait_phase(full_bar(s), ph, abort, limit, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t a_st = a_desc0 + static_cast<uint64_t>((s * Cfg::A_STAGE_BYTES) >> 4);
                    const uint64_t w_st = w_desc0 + static_cast<uint64_t>((s * Cfg::W_STAGE_BYTES) >> 4);
                    const uint32_t sf = tmem_base + Cfg::SF_COL0 + static_cast<uint32_t>(j * Cfg::SF_SLOT_COLS);
                    const uint32_t sfa = sf + static_cast<uint32_t>(4 * word);
                    const uint32_t sfb = sf + static_cast<uint32_t>(Cfg::SFB_COL + 8 * word);
                    const uint32_t idesc = idesc_with_sf_id(Cfg::IDESC, static_cast<uint32_t>(in_word));
#pragma unroll
                    for (int ks = 0; ks < Cfg::BK / Cfg::UMMA_K; ++ks) {
                        const uint64_t step = static_cast<uint64_t>((ks * Cfg::UMMA_K) >> 4);
                        mma_mxf8_pair(tmem_base, a_st + step, w_st + step, idesc, sfa, sfb,
                                      (kb != 0 || ks != 0) ? 1u : 0u);
                    }
                    issued_any = true;
                    // Operand slot s is free in both CTAs once these MMAs have read it.
                    mma_commit_pair_mc(empty_bar(s), kPairMask);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (in_slot == Cfg::SF_KB - 1 || kb == KB - 1) {
                        mma_commit_pair_mc(sempty_bar(j), kPairMask);
                        if (++j == SF) {
                            j = 0;
                            sph ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                mma_commit_pair_mc(tfull_bar, kPairMask);   // the tile's accumulator is complete in both CTAs
            }
            if (!ok && issued_any) {
                // Wait for this thread's MMAs before the TMEM is freed.
                mma_commit_pair_mc(drain_bar, static_cast<uint16_t>(1u << rank));
                wait_phase_drain(drain_bar, 0, limit, kSiteDrainMma, p.status);
            }
        }
        __syncwarp();
    } else if (warp < 6) {
        // ------------------------------------------------------------ epilogue (warps 2..5)
        const int ew = warp - 2;       // owner of smem staging buffers
        const int q = warp & 3;        // TMEM lane quarter this warp may access
        const uint32_t row_off = static_cast<uint32_t>(lane) * 128u;
        const uint32_t sw = static_cast<uint32_t>(lane & 7);
        const uint32_t tempty_leader = leader ? tempty_bar : mapa_shared(tempty_bar, 0);
        const uint32_t cbuf0 = sC + static_cast<uint32_t>(ew * Cfg::EPI_CHUNKS * Cfg::C_BUF_BYTES);
        // Chunk c of this warp's 32 rows, 64 fp32 columns -> ReLU -> fp16 into
        // its staging buffer (16-byte piece jj of a row at piece jj ^ (row % 8):
        // the layout a SWIZZLE_128B tensor-map store expects).
        auto stage = [&](const uint32_t (&r)[64], int c) {
            const uint32_t cbuf = cbuf0 + static_cast<uint32_t>(c * Cfg::C_BUF_BYTES);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const uint32_t w0 = pack_f16x2<kRelu>(r[8 * jj + 0], r[8 * jj + 1]);
                const uint32_t w1 = pack_f16x2<kRelu>(r[8 * jj + 2], r[8 * jj + 3]);
                const uint32_t w2 = pack_f16x2<kRelu>(r[8 * jj + 4], r[8 * jj + 5]);
                const uint32_t w3 = pack_f16x2<kRelu>(r[8 * jj + 6], r[8 * jj + 7]);
                st_shared_v4(cbuf + row_off + ((static_cast<uint32_t>(jj) ^ sw) << 4), w0, w1, w2, w3);
            }
        };
        uint32_t acc_it = 0;
        for (int t = first; t < p.num_tiles; t += stride, ++acc_it) {
            int mb, nb;
            mx_tile_coords(t, p, mb, nb);
            int ok = 1;
            if (lane == 0) {
                ok = wait_phase(tfull_bar, acc_it & 1u, abort, limit, kSiteEpilogueTmemFull) ? 1 : 0;
                // The previous tile's stores have read the staging buffers.
                bulk_wait_group_read<0>();
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (acc_it == 0) griddep_wait();   // before this warp's first store of C
            tc_fence_after_sync();
            const int row0 = mb * Cfg::TILE_M + static_cast<int>(rank) * Cfg::BM + q * 32;
            const uint32_t acc_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            // Double-buffered reads of the four chunks; TMEM goes back to the
            // MMA issuer as soon as the last read has completed.
            uint32_t ra[64], rb[64];
            tmem_load_32x32b_x64_async(acc_addr, ra);
            tmem_wait_ld_x64(ra);
            tmem_load_32x32b_x64_async(acc_addr + 1 * Cfg::EPI_COLS, rb);
            stage(ra, 0);
            tmem_wait_ld_x64(rb);
            tmem_load_32x32b_x64_async(acc_addr + 2 * Cfg::EPI_COLS, ra);
            stage(rb, 1);
            tmem_wait_ld_x64(ra);
            tmem_load_32x32b_x64_async(acc_addr + 3 * Cfg::EPI_COLS, rb);
            stage(ra, 2);
            tmem_wait_ld_x64(rb);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(tempty_bar);
                else mbar_arrive_cluster(tempty_leader);
            }
            stage(rb, 3);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                if (row0 < p.M) {
#pragma unroll 1
                    for (int c = 0; c < Cfg::EPI_CHUNKS; ++c) {
                        const int col0 = nb * Cfg::BN + c * Cfg::EPI_COLS;
                        if (col0 < p.N)
                            tma_store_2d(&tmap_c, cbuf0 + static_cast<uint32_t>(c * Cfg::C_BUF_BYTES), col0, row0);
                    }
                }
                bulk_commit_group();
            }
        }
        if (lane == 0) bulk_wait_group<0>();
    } else {
        // ------------------------------------------------------------ scale writers (warps 6..9)
        // Per slot (SF_WORDS words of P K blocks), in each CTA of the pair: for
        // word w, this warp's 32 rows of A scale words (row m at lane m) into
        // columns 4w .. 4w+3 of the slot, and the W block scale words into
        // columns SFB_COL + 8w .. SFB_COL + 8w + 7 (block 2 nb in the first
        // four, block 2 nb + 1 in the next four), the same word in every lane.
        const int q = warp & 3;
        const uint32_t sfull0 = leader ? sfull_bar(0) : mapa_shared(sfull_bar(0), 0);
        int j = 0;
        uint32_t sph = 0;
        griddep_wait();   // the scales may come from the previous kernel
        for (int t = first; t < p.num_tiles; t += stride) {
            int mb, nb;
            mx_tile_coords(t, p, mb, nb);
            const int row = mb * Cfg::TILE_M + static_cast<int>(rank) * Cfg::BM + q * 32 + lane;
            const int wb = nb * (Cfg::BN / Cfg::SCALE_BLOCK);
            const bool w0_in = wb < p.num_w_blocks, w1_in = wb + 1 < p.num_w_blocks;
            const uint8_t *sa = p.SA + static_cast<int64_t>(row < p.M ? row : 0) * KB;
            const uint8_t *sw0 = p.SW + static_cast<int64_t>(w0_in ? wb : 0) * KB;
            const uint8_t *sw1 = p.SW + static_cast<int64_t>(w1_in ? wb + 1 : 0) * KB;
            int ok = 1;
            // Byte i of each word: K block 4 g + i.  Rows or W blocks outside
            // the problem multiply zero operands: 2^0.  The bytes of the next
            // batch of words are loaded while this batch is stored, so a
            // load's latency (about one word's worth of MMAs at this size) is
            // never waited for.
            constexpr int D = Cfg::SF_BATCH;
            auto load_batch = [&](int kg0, uint32_t (&wa)[D], uint32_t (&w0)[D], uint32_t (&w1)[D]) {
#pragma unroll
                for (int g = 0; g < D; ++g) {
                    wa[g] = w0[g] = w1[g] = 0;
#pragma unroll
                    for (int i = 0; i < P; ++i) {
                        const int kb = kg0 + g * P + i;
                        const uint32_t ea = (kb < KB && row < p.M) ? __ldg(sa + kb) : 127u;
                        const uint32_t e0 = (kb < KB && w0_in) ? __ldg(sw0 + kb) : 127u;
                        const uint32_t e1 = (kb < KB && w1_in) ? __ldg(sw1 + kb) : 127u;
                        wa[g] |= ea << (8 * i);
                        w0[g] |= e0 << (8 * i);
                        w1[g] |= e1 << (8 * i);
                    }
                }
            };
            uint32_t ca[D], c0[D], c1[D];
            load_batch(0, ca, c0, c1);
            for (int kg0 = 0; ok && kg0 < KB; kg0 += D * P) {
                uint32_t na[D], n0[D], n1[D];
                load_batch(kg0 + D * P, na, n0, n1);
#pragma unroll
                for (int sl = 0; sl < D / Cfg::SF_WORDS; ++sl) {
                    if (kg0 + sl * Cfg::SF_KB >= KB) break;
                    // The writers run up to SF_SLOTS words ahead of the MMAs: their
                    // waits sleep between probes, leaving issue slots and barrier
                    // traffic to the roles on the critical path (measured 1.5 %
                    // faster than polling without a pause).
                    if (lane == 0)
                        ok = wait_phase<1000>(sempty_bar(j), sph ^ 1u, abort, limit, kSiteMmaTmemEmpty) ? 1 : 0;
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t slot = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + Cfg::SF_COL0 +
                                          static_cast<uint32_t>(j * Cfg::SF_SLOT_COLS);
#pragma unroll
                    for (int w = 0; w < Cfg::SF_WORDS; ++w) {
                        const int g = sl * Cfg::SF_WORDS + w;
                        tmem_store_x4(slot + static_cast<uint32_t>(4 * w), ca[g], ca[g], ca[g], ca[g]);
                        tmem_store_x8(slot + static_cast<uint32_t>(Cfg::SFB_COL + 8 * w), c0[g], c0[g], c0[g], c0[g],
                                      c1[g], c1[g], c1[g], c1[g]);
                    }
                    tmem_wait_st();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) {
                        if (leader) mbar_arrive(sfull_bar(j));
                        else mbar_arrive_cluster(sfull0 + 8u * static_cast<uint32_t>(j));
                    }
                    if (++j == SF) {
                        j = 0;
                        sph ^= 1u;
                    }
                }
#pragma unroll
                for (int g = 0; g < D; ++g) {
                    ca[g] = na[g];
                    c0[g] = n0[g];
                    c1[g] = n1[g];
                }
            }
            if (!ok) break;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // Neither CTA exits while the other may still signal its barriers or its
    // MMAs may still use this CTA's shared or tensor memory.
    cluster_arrive();
    cluster_wait();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_sm103
