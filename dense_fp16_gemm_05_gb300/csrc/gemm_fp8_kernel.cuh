// gemm_fp8_kernel.cuh -- FP8 (E4M3) block-scaled GEMM for sm_103a:
//
//   C[i,j] = R( sum_b SA[i,b] * SW[j/128, b] * sum_{k in block b} A[i,k] W[j,k] )
//
// A (M,K) and W (N,K) are row-major E4M3 (the weight kept out-features x
// in-features, as a linear layer stores it: C = A @ W^T), SA (M, KB) holds one
// fp32 scale per row of A per 128 K elements, SW (NB, KB) one per 128 x 128
// block of W, KB = ceil(K/128), NB = ceil(N/128); C (M,N) is fp16 and R is the
// optional ReLU.  This is the plainest reading of the FP8 block-scaled linear
// layer of the TileLang-MUSA lesson (7yue.com, section 8.2:
// fp8_block_scaled_linear(x, w_fp8, scale_w, block=128)) with the per-block
// scaling the nxmr.cn TileLang article (section 7) names.
//
// The scales change from one 128-element K block to the next, so they cannot
// ride inside one MMA accumulation.  The mainloop is the CTA-pair loop of the
// fp16 kernel on 8-bit operands (one 128-byte swizzle row = one K block = 4
// tcgen05.mma.kind::f8f6f4 of K = 32); each K block's MMAs write a fresh
// partial P_b into one of two TMEM buffers, and eight "promotion" warps per
// CTA read P_b, multiply by SA[i,b] * SW[j/128,b] and add it into an fp32
// accumulator held in registers (one output row per thread, 128 columns per
// warp; 16-column TMEM loads kept two in flight, packed fp32 FMAs).  While
// they promote P_b the MMAs of block b+1 fill the other buffer.
// After a tile's last block the promotion warps apply ReLU, round to fp16 and
// store their row segment directly (16-byte stores).
//
// Roles per CTA (320 threads, one CTA per SM, a cluster = one CTA pair, a
// persistent grid over 256 x 256 output tiles in grouped raster order):
//   warp 0, one lane   TMA producer: A box 128(K) x 128(rows) and W box
//                      128(K) x 128(rows) per stage, completing on the pair
//                      leader's "full" barrier
//   warp 1, one lane   (leader CTA only) MMA issuer; also allocates the
//                      512 TMEM columns (two 256-column partial buffers)
//   warps 2..9         promotion + epilogue; warp w reads TMEM lanes
//                      32*(w%4) .. +31 and columns 128*((w-2)/4) .. +127
// Ragged edges: TMA zero-fills operand elements outside A or W (they add
// nothing), the scales of a partial last block apply to what it holds, and
// rows or columns outside C are not stored.  Every wait is bounded; on expiry
// the site is recorded in the device status word and all roles leave.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "gemm_kernel.cuh"

namespace gemm_sm103 {

// ---------------------------------------------------------------- PTX

// D[tmem] (+)= A[smem] * B[smem] for 8-bit floating-point operands (formats
// named in the instruction descriptor), fp32 accumulator, CTA pair; one
// instruction covers K = 32 elements (32 bytes of each operand row).
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Starts a load of 16 consecutive fp32 columns of the warp's 32 TMEM lanes
// (one lane per thread).  The registers are valid only after tmem_wait_ld.
__device__ __forceinline__ void tmem_load_x16_async(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Waits for every TMEM load this thread started.  The registers of the load
// in flight are in/out operands, so that no read of them is placed before
// the wait and they stay in place until it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15])
                 :
                 : "memory");
}

// d0 = fma(a, b0, d0), d1 = fma(a, b1, d1): two fp32 fused multiply-adds,
// each rounded once to nearest (the packed form of two fmaf calls).
__device__ __forceinline__ void fma2_rn(float &d0, float &d1, float a, uint32_t b0, uint32_t b1)
{
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %2};\n\t"
        "mov.b64 rb, {%3, %4};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "f"(a), "r"(b0), "r"(b1));
}

// Instruction descriptor for tcgen05.mma.kind::f8f6f4 with E4M3 A and B
// (format code 0 in bits 7-9 and 10-12), an fp32 accumulator (bits 4-5 = 1),
// both operands K-major (bits 15, 16 = 0), N >> 3 (17-22), M >> 4 (24-28).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N)
{
    return (1u << 4) | (0u << 7) | (0u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- configuration

struct Fp8Cfg {
    static constexpr int BM = 128;            // rows of C per CTA (TMEM lanes)
    static constexpr int TILE_M = 256;        // rows per pair tile (the MMA's M)
    static constexpr int BN = 256;            // columns per tile (the MMA's N)
    static constexpr int BN_CTA = 128;        // rows of W each CTA loads
    static constexpr int BK = 128;            // E4M3 elements per K block = one 128-byte swizzle row
    static constexpr int SCALE_BLOCK = 128;   // the scale granularity of the method
    static constexpr int UMMA_K = 32;
    static constexpr int STAGES = 6;
    static constexpr int PROMO_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * PROMO_WARPS;
    static constexpr int A_STAGE_BYTES = BM * BK;          // 16 KiB
    static constexpr int W_STAGE_BYTES = BN_CTA * BK;      // 16 KiB
    static constexpr int STAGE_TX_BYTES = A_STAGE_BYTES + W_STAGE_BYTES;
    static constexpr int P_COLS = BN;                       // one partial buffer
    static constexpr int TMEM_COLS = 2 * P_COLS;            // two partial buffers
    static constexpr int SMEM_A_OFF = 0;
    static constexpr int SMEM_W_OFF = STAGES * A_STAGE_BYTES;
    static constexpr int SMEM_CTL_OFF = SMEM_W_OFF + STAGES * W_STAGE_BYTES;
    static constexpr int SMEM_CTL_BYTES = 256;
    static constexpr int SMEM_BYTES = 1024 + SMEM_CTL_OFF + SMEM_CTL_BYTES;
    static constexpr uint32_t IDESC = idesc_e4m3_f32(TILE_M, BN);

    static_assert(BK == SCALE_BLOCK, "one K block per scale block");
    static_assert(2 * BN_CTA == BN && BN_CTA == SCALE_BLOCK, "each CTA's W half is one scale block of N");
    static_assert(TMEM_COLS == 512, "TMEM allocation");
    static_assert((2 * STAGES + 5) * 8 + 8 <= SMEM_CTL_BYTES, "control block");
    static_assert(SMEM_BYTES <= 232448, "shared memory per block on sm_103");
};

struct Fp8Params {
    int32_t M, N, K;
    int32_t num_m_blocks;   // ceil(M / 256)
    int32_t num_n_blocks;   // ceil(N / 256)
    int32_t num_k_blocks;   // ceil(K / 128) = KB, the columns of SA and SW
    int32_t num_tiles;
    int32_t group_m;        // rasterisation panel height, in tiles
    uint64_t timeout_cycles;
    __half *C;
    const float *SA;        // (M, num_k_blocks)
    const float *SW;        // (ceil(N/128), num_k_blocks)
    unsigned long long *status;
};

__device__ __forceinline__ void fp8_tile_coords(int t, const Fp8Params &p, int &mb, int &nb)
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
__global__ void __launch_bounds__(Fp8Cfg::THREADS, 1)
    gemm_fp8_block_scaled_sm103a(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_w,
                                 const Fp8Params p)
{
    using Cfg = Fp8Cfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // SW128 atoms need 1024-byte alignment
    uint8_t *base_ptr = smem_raw + (base - raw);

    const uint32_t sA = base + Cfg::SMEM_A_OFF;
    const uint32_t sW = base + Cfg::SMEM_W_OFF;
    const uint32_t ctl = base + Cfg::SMEM_CTL_OFF;
    auto full_bar = [&](int s) { return ctl + 8u * s; };
    auto empty_bar = [&](int s) { return ctl + 8u * (Cfg::STAGES + s); };
    auto pfull_bar = [&](int b) { return ctl + 8u * (2 * Cfg::STAGES + b); };
    auto pempty_bar = [&](int b) { return ctl + 8u * (2 * Cfg::STAGES + 2 + b); };
    const uint32_t drain_bar = ctl + 8u * (2 * Cfg::STAGES + 4);
    const uint32_t tmem_slot = ctl + 8u * (2 * Cfg::STAGES + 5);
    const uint32_t abort_addr = tmem_slot + 4;
    volatile uint32_t *tmem_slot_ptr =
        reinterpret_cast<volatile uint32_t *>(base_ptr + Cfg::SMEM_CTL_OFF + 8 * (2 * Cfg::STAGES + 5));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank() & 1u;   // 0 = pair leader
    const bool leader = rank == 0;
    const int cluster_id = static_cast<int>(blockIdx.x) / 2;
    const int num_clusters = static_cast<int>(gridDim.x) / 2;
    constexpr uint16_t kPairMask = 0x3;

    AbortFlag abort;
    abort.local = reinterpret_cast<volatile int *>(tmem_slot_ptr + 1);
    abort.status = p.status;
    abort.addr = abort_addr;
    abort.cluster = 2;
    abort.rank = rank;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(full_bar(s), 2);    // each CTA of the pair: arrive.expect_tx
            mbar_init(empty_bar(s), 1);   // one MMA commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(pfull_bar(b), 1);                          // commit after a K block's MMAs
            mbar_init(pempty_bar(b), 2 * Cfg::PROMO_WARPS);     // every promotion warp of the pair
        }
        mbar_init(drain_bar, 1);
        *abort.local = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmap_a);
        prefetch_tensormap(&tmap_w);
    }
    if (warp == 1) {
        tmem_alloc<2>(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish<2>();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_arrive();
    cluster_wait();
    tc_fence_after_sync();
    // Set-up above may overlap the previous kernel of the stream; nothing
    // below runs before its results are visible (programmatic dependent launch).
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = *tmem_slot_ptr;
    const uint64_t limit = p.timeout_cycles;
    const int KB = p.num_k_blocks;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            const uint32_t full_base = leader ? full_bar(0) : mapa_shared(full_bar(0), 0);
            for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
                int mb, nb;
                fp8_tile_coords(t, p, mb, nb);
                const int m0 = mb * Cfg::TILE_M + static_cast<int>(rank) * Cfg::BM;
                const int n0 = nb * Cfg::BN + static_cast<int>(rank) * Cfg::BN_CTA;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort, limit, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_base + 8u * s;
                    if (leader) mbar_arrive_expect_tx(fb, Cfg::STAGE_TX_BYTES);
                    else mbar_arrive_expect_tx_cluster(fb, Cfg::STAGE_TX_BYTES);
                    const int k0 = kb * Cfg::BK;
                    tma_load_2d_pair(sA + s * Cfg::A_STAGE_BYTES, &tmap_a, fb, k0, m0);
                    tma_load_2d_pair(sW + s * Cfg::W_STAGE_BYTES, &tmap_w, fb, k0, n0);
                    issued_mask |= 1u << s;
                    issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
                    if (++s == Cfg::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                if (leader) {
                    for (int i = 0; i < Cfg::STAGES; ++i)
                        if (issued_mask & (1u << i))
                            wait_phase_drain(full_bar(i), (issued_parity >> i) & 1u, limit, kSiteDrainLoads, p.status);
                } else {
                    // This CTA's loads complete on the leader's barrier: give them
                    // a bounded time (~1e6 cycles) to land.
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
            uint32_t pidx = 0;      // K blocks issued so far (selects the partial buffer)
            bool ok = true, issued_any = false;
            const uint64_t a_desc0 = smem_desc_sw128(sA, 16, 1024);
            const uint64_t w_desc0 = smem_desc_sw128(sW, 16, 1024);
            for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
                for (int kb = 0; kb < KB; ++kb) {
                    const uint32_t pb = pidx & 1u;
                    const uint32_t pph = (pidx >> 1) & 1u;
                    if (!wait_phase(pempty_bar(pb), pph ^ 1u, abort, limit, kSiteMmaTmemEmpty) ||
                        !wait_phase(full_bar(s), ph, abort, limit, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t a_st = a_desc0 + static_cast<uint64_t>((s * Cfg::A_STAGE_BYTES) >> 4);
                    const uint64_t w_st = w_desc0 + static_cast<uint64_t>((s * Cfg::W_STAGE_BYTES) >> 4);
                    const uint32_t d = tmem_base + pb * Cfg::P_COLS;
#pragma unroll
                    for (int ks = 0; ks < Cfg::BK / Cfg::UMMA_K; ++ks) {
                        // K step of 32 one-byte elements = +32 bytes inside the swizzle row.
                        const uint64_t step = static_cast<uint64_t>((ks * Cfg::UMMA_K) >> 4);
                        mma_f8f6f4_pair(d, a_st + step, w_st + step, Cfg::IDESC, ks != 0 ? 1u : 0u);
                    }
                    mma_commit_pair_mc(empty_bar(s), kPairMask);   // the slot is free in both CTAs
                    mma_commit_pair_mc(pfull_bar(pb), kPairMask);  // P_b is ready in both CTAs
                    issued_any = true;
                    ++pidx;
                    if (++s == Cfg::STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok && issued_any) {
                mma_commit_pair_mc(drain_bar, static_cast<uint16_t>(1u << rank));
                wait_phase_drain(drain_bar, 0, limit, kSiteDrainMma, p.status);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ promotion + epilogue (warps 2..9)
        const int q = warp & 3;                  // TMEM lane quarter this warp may read
        const int half = (warp - 2) >> 2;        // column half of the tile (0 or 1)
        const uint32_t pempty_leader0 = leader ? pempty_bar(0) : mapa_shared(pempty_bar(0), 0);
        uint32_t pidx = 0;
        bool ok = true;
        for (int t = cluster_id; ok && t < p.num_tiles; t += num_clusters) {
            int mb, nb;
            fp8_tile_coords(t, p, mb, nb);
            const int row = mb * Cfg::TILE_M + static_cast<int>(rank) * Cfg::BM + q * 32 + lane;
            const int col0 = nb * Cfg::BN + half * Cfg::SCALE_BLOCK;
            const bool row_ok = row < p.M;
            const bool cols_ok = col0 < p.N;
            const float *sa = p.SA + static_cast<int64_t>(row_ok ? row : 0) * KB;
            const float *sw = p.SW + static_cast<int64_t>(cols_ok ? col0 / Cfg::SCALE_BLOCK : 0) * KB;
            float acc[Cfg::SCALE_BLOCK];
#pragma unroll
            for (int c = 0; c < Cfg::SCALE_BLOCK; ++c) acc[c] = 0.0f;
            // Scales of blocks kb and kb + 1 in registers; block kb + 2's are
            // fetched while block kb is promoted (two blocks of latency cover).
            float s_a = row_ok ? __ldg(sa) : 0.0f;
            float s_w = cols_ok ? __ldg(sw) : 0.0f;
            float s_a1 = (row_ok && KB > 1) ? __ldg(sa + 1) : 0.0f;
            float s_w1 = (cols_ok && KB > 1) ? __ldg(sw + 1) : 0.0f;
            for (int kb = 0; kb < KB; ++kb) {
                const uint32_t pb = pidx & 1u;
                const uint32_t pph = (pidx >> 1) & 1u;
                // Every lane probes the barrier itself (no broadcast from one
                // lane); a vote keeps the outcome warp-uniform, as the
                // warp-collective TMEM loads below require.
                const bool got = wait_phase(pfull_bar(pb), pph, abort, limit, kSiteEpilogueTmemFull);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const float scale = s_a * s_w;
                s_a = s_a1;
                s_w = s_w1;
                if (kb + 2 < KB) {
                    s_a1 = row_ok ? __ldg(sa + kb + 2) : 0.0f;
                    s_w1 = cols_ok ? __ldg(sw + kb + 2) : 0.0f;
                }
                const uint32_t taddr =
                    tmem_base + (static_cast<uint32_t>(q * 32) << 16) + pb * Cfg::P_COLS + half * Cfg::SCALE_BLOCK;
                // 16-column pieces, two in flight: the load of piece c+1 runs
                // while piece c is multiplied in.
                constexpr int kPieces = Cfg::SCALE_BLOCK / 16;
                uint32_t r0[16], r1[16];
                tmem_load_x16_async(taddr, r0);
                tmem_wait_ld(r0);
#pragma unroll
                for (int c = 0; c < kPieces; c += 2) {
                    tmem_load_x16_async(taddr + (c + 1) * 16, r1);
#pragma unroll
                    for (int i = 0; i < 16; i += 2) fma2_rn(acc[c * 16 + i], acc[c * 16 + i + 1], scale, r0[i], r0[i + 1]);
                    tmem_wait_ld(r1);
                    if (c + 2 < kPieces) {
                        tmem_load_x16_async(taddr + (c + 2) * 16, r0);
                    } else {
                        // The last piece is in registers: this warp's reads of
                        // P_b are complete, hand the buffer back.
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if (leader) mbar_arrive(pempty_bar(pb));
                            else mbar_arrive_cluster(pempty_leader0 + 8u * pb);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 16; i += 2)
                        fma2_rn(acc[(c + 1) * 16 + i], acc[(c + 1) * 16 + i + 1], scale, r1[i], r1[i + 1]);
                    if (c + 2 < kPieces) tmem_wait_ld(r0);
                }
                ++pidx;
            }
            if (!ok) break;
            // ReLU, fp16 rounding, and 16-byte stores of this thread's row segment.
            if (row_ok && cols_ok) {
                __half *crow = p.C + static_cast<int64_t>(row) * p.N + col0;
#pragma unroll
                for (int j = 0; j < Cfg::SCALE_BLOCK / 8; ++j) {
                    if (col0 + 8 * j < p.N) {
                        uint32_t w[4];
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            float lo = acc[8 * j + 2 * h], hi = acc[8 * j + 2 * h + 1];
                            if constexpr (kRelu) {
                                lo = lo > 0.0f ? lo : 0.0f;
                                hi = hi > 0.0f ? hi : 0.0f;
                            }
                            const __half2 v = __floats2half2_rn(lo, hi);
                            w[h] = *reinterpret_cast<const uint32_t *>(&v);
                        }
                        st_global_v4(crow + 8 * j, w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    // No CTA of the pair exits while the other may still signal its barriers
    // or read its shared memory.
    cluster_arrive();
    cluster_wait();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem_base, Cfg::TMEM_COLS);
    }
}

}  // namespace gemm_sm103
