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
// Layout of the scale factors in TMEM (established with a layout probe of
// the instruction on this GPU): the scale of A row m is read from lane m,
// column sfa + m / 32; the scale of B column n (of one MMA's N) from lane
// 32 * q + n % 32, column sfb + n / 32, by the lanes of quarter q, so it is
// written to all four lane quarters; byte 0 of the 32-bit word (scale id 0).
// Every K block of 128 is four MMAs of K = 32 that share one scale, so each
// word repeats its byte.
//
// Roles per CTA (320 threads, one CTA per SM, persistent grid over 128 x 256
// output tiles in grouped raster order; the tile's accumulator is 256 TMEM
// columns, computed as two N = 128 halves):
//   warp 0, one lane   TMA producer: A box 128 (K) x 128 rows, W box 128 (K)
//                      x 256 rows per stage
//   warp 1, one lane   MMA issuer; allocates the 512 TMEM columns (the
//                      accumulator and a ring of scale-factor slots)
//   warps 2..5         epilogue: TMEM -> ReLU -> fp16 -> swizzled smem -> TMA
//                      store, handing each half of the accumulator back as soon
//                      as it is read (the next tile's MMAs start on half 0)
//   warps 6..9         scale writers: per K block, read the block's scale
//                      bytes and store them into a TMEM slot (tcgen05.st)
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
// instruction's K = 32), fp32 accumulator, one CTA.
__device__ __forceinline__ void mma_mxf8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
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

// ---------------------------------------------------------------- configuration

struct MxCfg {
    static constexpr int BM = 128;             // rows of C per tile (TMEM lanes)
    static constexpr int BN = 256;             // columns of C per tile
    static constexpr int HALF_N = 128;         // columns per MMA (one half of the accumulator)
    static constexpr int BK = 128;             // E4M3 elements per K block = one 128-byte swizzle row
    static constexpr int SCALE_BLOCK = 128;
    static constexpr int UMMA_K = 32;
    static constexpr int STAGES = 4;           // operand ring
    static constexpr int SF_STAGES = 8;        // scale-factor slots in TMEM (>= STAGES: a slot is
                                               // held as long as its operands)
    static constexpr int THREADS = 320;
    static constexpr int A_STAGE_BYTES = BM * BK;     // 16 KiB
    static constexpr int W_STAGE_BYTES = BN * BK;     // 32 KiB
    static constexpr int STAGE_TX_BYTES = A_STAGE_BYTES + W_STAGE_BYTES;
    static constexpr int ACC_COLS = BN;               // one accumulator of two halves
    static constexpr int SF_COL0 = ACC_COLS;          // first scale-factor slot
    static constexpr int SF_SLOT_COLS = 16;           // A: 4 columns, B: 8 columns (2 halves x 4)
    static constexpr int TMEM_COLS = 512;
    static constexpr int EPI_COLS = 64;
    static constexpr int C_BUF_BYTES = 32 * EPI_COLS * 2;
    static constexpr int SMEM_A_OFF = 0;
    static constexpr int SMEM_W_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int SMEM_C_OFF = SMEM_W_OFF + STAGES * W_STAGE_BYTES;
    static constexpr int SMEM_CTL_OFF = SMEM_C_OFF + 4 * 2 * C_BUF_BYTES;
    static constexpr int SMEM_CTL_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + SMEM_CTL_OFF + SMEM_CTL_BYTES;
    static constexpr uint32_t IDESC = idesc_mxf8_e4m3(BM, HALF_N);

    static_assert(BK == SCALE_BLOCK && 2 * HALF_N == BN && HALF_N == SCALE_BLOCK, "one scale per K block and half");
    static_assert(SF_STAGES >= STAGES, "a scale slot lives as long as its operand slot");
    static_assert(SF_COL0 + SF_STAGES * SF_SLOT_COLS <= TMEM_COLS, "TMEM columns");
    static_assert((2 * STAGES + 2 * SF_STAGES + 5) * 8 <= SMEM_CTL_BYTES, "control block");
    static_assert(SMEM_BYTES <= 232448, "shared memory per block on sm_103");
};

struct MxParams {
    int32_t M, N, K;
    int32_t num_m_blocks;   // ceil(M / 128)
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
    constexpr int S = Cfg::STAGES, SF = Cfg::SF_STAGES;
    auto full_bar = [&](int s) { return ctl + 8u * s; };
    auto empty_bar = [&](int s) { return ctl + 8u * (S + s); };
    auto sfull_bar = [&](int j) { return ctl + 8u * (2 * S + j); };
    auto sempty_bar = [&](int j) { return ctl + 8u * (2 * S + SF + j); };
    const uint32_t tfull_bar = ctl + 8u * (2 * S + 2 * SF);
    auto tempty_bar = [&](int h) { return ctl + 8u * (2 * S + 2 * SF + 1 + h); };
    const uint32_t drain_bar = ctl + 8u * (2 * S + 2 * SF + 3);
    const uint32_t tmem_slot = ctl + 8u * (2 * S + 2 * SF + 4);
    const uint32_t abort_addr = tmem_slot + 4;
    volatile uint32_t *tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t *>(base_ptr + Cfg::SMEM_CTL_OFF + 8 * (2 * S + 2 * SF + 4));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    AbortFlag abort;
    abort.local = reinterpret_cast<volatile int *>(tmem_slot_ptr + 1);
    abort.status = p.status;
    abort.addr = abort_addr;
    abort.cluster = 1;
    abort.rank = 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);    // the producer's arrive.expect_tx
            mbar_init(empty_bar(s), 1);   // one MMA commit
        }
        for (int j = 0; j < SF; ++j) {
            mbar_init(sfull_bar(j), 4);   // one arrive per scale-writer warp
            mbar_init(sempty_bar(j), 1);  // one MMA commit
        }
        mbar_init(tfull_bar, 1);
        for (int h = 0; h < 2; ++h) mbar_init(tempty_bar(h), 4);   // one arrive per epilogue warp
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
        tmem_alloc<1>(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish<1>();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // The set-up above may overlap the previous kernel of the stream; each
    // role waits for it (griddep_wait) before its first global access.
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot_ptr;
    const uint64_t limit = p.timeout_cycles;
    const int KB = p.num_k_blocks;
    const int first = static_cast<int>(blockIdx.x), stride = static_cast<int>(gridDim.x);

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true, dep_waited = false;
            for (int t = first; ok && t < p.num_tiles; t += stride) {
                int mb, nb;
                mx_tile_coords(t, p, mb, nb);
                const int m0 = mb * Cfg::BM, n0 = nb * Cfg::BN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort, limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    if (!dep_waited) {
                        griddep_wait();
                        dep_waited = true;
                    }
                    const uint32_t fb = full_bar(s);
                    mbar_arrive_expect_tx(fb, Cfg::STAGE_TX_BYTES);
                    const int k0 = kb * Cfg::BK;
                    tma_load_2d(sA + s * Cfg::A_STAGE_BYTES, &tmap_a, fb, k0, m0);
                    tma_load_2d(sW + s * Cfg::W_STAGE_BYTES, &tmap_w, fb, k0, n0);
                    issued_mask |= 1u << s;
                    issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let the loads in flight land before the CTA exits.
                for (int i = 0; i < S; ++i)
                    if (issued_mask & (1u << i))
                        wait_phase_drain(full_bar(i), (issued_parity >> i) & 1u, limit, kSiteDrainLoads, p.status);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int s = 0, j = 0;
            uint32_t ph = 0, sph = 0, acc_it = 0;
            bool ok = true, issued_any = false;
            // K-major SW128 operands: 8-row groups 1024 B apart; a K step of 32
            // one-byte elements is +32 B inside the swizzle row; W half h starts
            // 128 rows (16 KiB) further.
            const uint64_t a_desc0 = smem_desc_sw128(sA, 16, 1024);
            const uint64_t w_desc0 = smem_desc_sw128(sW, 16, 1024);
            auto issue = [&](int st, int slot, int h_lo, int h_hi, bool first_block) {
                const uint64_t a_st = a_desc0 + static_cast<uint64_t>((st * Cfg::A_STAGE_BYTES) >> 4);
                const uint64_t w_st = w_desc0 + static_cast<uint64_t>((st * Cfg::W_STAGE_BYTES) >> 4);
                const uint32_t sf = tmem_base + Cfg::SF_COL0 + static_cast<uint32_t>(slot * Cfg::SF_SLOT_COLS);
#pragma unroll
                for (int ks = 0; ks < Cfg::BK / Cfg::UMMA_K; ++ks) {
                    const uint64_t step = static_cast<uint64_t>((ks * Cfg::UMMA_K) >> 4);
                    for (int h = h_lo; h < h_hi; ++h) {
                        const uint64_t w_h = w_st + static_cast<uint64_t>((h * Cfg::HALF_N * 128) >> 4);
                        mma_mxf8_ss(tmem_base + static_cast<uint32_t>(h * Cfg::HALF_N), a_st + step, w_h + step,
                                    Cfg::IDESC, sf, sf + 4u + static_cast<uint32_t>(4 * h),
                                    (ks != 0 || !first_block) ? 1u : 0u);
                    }
                }
            };
            auto release = [&](int st, int slot) {
                mma_commit(empty_bar(st));
                mma_commit(sempty_bar(slot));
            };
            auto wait_block = [&](int st, uint32_t sph_, int slot, uint32_t ph_) {
                return wait_phase(full_bar(st), ph_, abort, limit, kSiteMmaFull) &&
                       wait_phase(sfull_bar(slot), sph_, abort, limit, kSiteMmaFull);
            };
            auto advance = [&]() {
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++j == SF) {
                    j = 0;
                    sph ^= 1u;
                }
            };
            for (int t = first; ok && t < p.num_tiles; t += stride, ++acc_it) {
                const uint32_t acc_ph = acc_it & 1u;
                // Half 0 as soon as the previous tile's epilogue has read it: the
                // first ring-full of K blocks on half 0, then the same blocks on
                // half 1 once it is free too (same per-column order of sums).
                if (!wait_phase(tempty_bar(0), acc_ph ^ 1u, abort, limit, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int npre = KB < S ? KB : S;
                int pre_s[S], pre_j[S];
                for (int i = 0; i < npre; ++i) {
                    if (!wait_block(s, sph, j, ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    pre_s[i] = s;
                    pre_j[i] = j;
                    issue(s, j, 0, 1, i == 0);
                    issued_any = true;
                    advance();
                }
                if (!ok) break;
                if (!wait_phase(tempty_bar(1), acc_ph ^ 1u, abort, limit, kSiteMmaTmemEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                for (int i = 0; i < npre; ++i) {
                    issue(pre_s[i], pre_j[i], 1, 2, i == 0);
                    release(pre_s[i], pre_j[i]);
                }
                for (int kb = npre; kb < KB; ++kb) {
                    if (!wait_block(s, sph, j, ph)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    issue(s, j, 0, 2, false);
                    release(s, j);
                    advance();
                }
                if (!ok) break;
                mma_commit(tfull_bar);   // the tile's accumulator is complete
            }
            if (!ok && issued_any) {
                // Wait for this thread's MMAs before the TMEM is freed.
                mma_commit(drain_bar);
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
        constexpr int kChunks = Cfg::BN / Cfg::EPI_COLS;   // 4: chunks 0-1 are half 0, 2-3 half 1
        uint32_t chunk = 0, acc_it = 0;
        for (int t = first; t < p.num_tiles; t += stride, ++acc_it) {
            int mb, nb;
            mx_tile_coords(t, p, mb, nb);
            int ok = 1;
            if (lane == 0) ok = wait_phase(tfull_bar, acc_it & 1u, abort, limit, kSiteEpilogueTmemFull) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (acc_it == 0) griddep_wait();   // before this warp's first store of C
            tc_fence_after_sync();
            const int row0 = mb * Cfg::BM + q * 32;
            const uint32_t acc_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c) {
                uint32_t r[64];
                tmem_load_32x32b_x64(acc_addr + c * Cfg::EPI_COLS, r);
                if (c == 1 || c == 3) {
                    // This warp has read half c / 2 of the accumulator.
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(c / 2));
                }
                const int col0 = nb * Cfg::BN + c * Cfg::EPI_COLS;
                const bool in_range = row0 < p.M && col0 < p.N;
                const uint32_t cbuf = sC + (ew * 2 + (chunk & 1u)) * Cfg::C_BUF_BYTES;
                ++chunk;
                if (lane == 0) bulk_wait_group_read<1>();   // the store that used cbuf has read it
                __syncwarp();
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const uint32_t w0 = pack_f16x2<kRelu>(r[8 * jj + 0], r[8 * jj + 1]);
                    const uint32_t w1 = pack_f16x2<kRelu>(r[8 * jj + 2], r[8 * jj + 3]);
                    const uint32_t w2 = pack_f16x2<kRelu>(r[8 * jj + 4], r[8 * jj + 5]);
                    const uint32_t w3 = pack_f16x2<kRelu>(r[8 * jj + 6], r[8 * jj + 7]);
                    // 16-byte piece jj of this row goes to piece jj ^ (row % 8): the
                    // layout a SWIZZLE_128B tensor-map store expects.
                    st_shared_v4(cbuf + row_off + ((static_cast<uint32_t>(jj) ^ sw) << 4), w0, w1, w2, w3);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (in_range) tma_store_2d(&tmap_c, cbuf, col0, row0);
                    bulk_commit_group();   // one group per chunk, empty or not
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();
    } else {
        // ------------------------------------------------------------ scale writers (warps 6..9)
        // Per K block: this warp's 32 rows of A scales into column q of the
        // slot (row m at lane m, column m / 32) and the two W block scales of
        // the tile's column halves into columns 4..11 (four columns per half,
        // the same word in every lane).
        const int q = warp & 3;
        int j = 0;
        uint32_t sph = 0;
        bool dep_waited = false;
        for (int t = first; t < p.num_tiles; t += stride) {
            int mb, nb;
            mx_tile_coords(t, p, mb, nb);
            const int row = mb * Cfg::BM + q * 32 + lane;
            const int wb = nb * (Cfg::BN / Cfg::SCALE_BLOCK);
            const uint8_t *sa = p.SA + static_cast<int64_t>(row < p.M ? row : 0) * KB;
            const uint8_t *sw0 = p.SW + static_cast<int64_t>(wb < p.num_w_blocks ? wb : 0) * KB;
            const uint8_t *sw1 = p.SW + static_cast<int64_t>(wb + 1 < p.num_w_blocks ? wb + 1 : 0) * KB;
            int ok = 1;
            for (int kb = 0; kb < KB; ++kb) {
                if (lane == 0) ok = wait_phase(sempty_bar(j), sph ^ 1u, abort, limit, kSiteMmaTmemEmpty) ? 1 : 0;
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (!dep_waited) {
                    griddep_wait();   // the scales may come from the previous kernel
                    dep_waited = true;
                }
                tc_fence_after_sync();
                // Rows or W blocks outside the problem multiply zero operands: 2^0.
                const uint32_t ea = row < p.M ? __ldg(sa + kb) : 127u;
                const uint32_t e0 = wb < p.num_w_blocks ? __ldg(sw0 + kb) : 127u;
                const uint32_t e1 = wb + 1 < p.num_w_blocks ? __ldg(sw1 + kb) : 127u;
                const uint32_t slot = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + Cfg::SF_COL0 +
                                      static_cast<uint32_t>(j * Cfg::SF_SLOT_COLS);
                const uint32_t wa = ea * 0x01010101u, w0 = e0 * 0x01010101u, w1 = e1 * 0x01010101u;
                tmem_store_x1(slot + static_cast<uint32_t>(q), wa);
                tmem_store_x8(slot + 4u, w0, w0, w0, w0, w1, w1, w1, w1);
                tmem_wait_st();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfull_bar(j));
                if (++j == SF) {
                    j = 0;
                    sph ^= 1u;
                }
            }
            if (!ok) break;
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<1>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_sm103
