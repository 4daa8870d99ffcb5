// gemm2sm.cuh -- the block-scaled NVFP4 GEMM on CTA pairs (tcgen05
// cta_group::2): one MMA instruction computes a 256 x 256 x 64 product on
// the tensor cores of two SMs.
//
// Same product and numerics as gemm.cuh (NVIDIA blog "NVFP4 Trains with
// Precision of 16-Bit and Speed and Efficiency of 4-Bit", Figure 1 and
// recipe bullets 1-2): D = alpha * sum_k (qa sa)(qb sb), FP32 accumulation.
//
// Why pairs: a single-CTA 128 x 256 tile must stream A (128 rows) and all of
// B (256 rows) through each SM's shared memory.  With a CTA pair each SM
// holds its own 128 rows of A and only half of B (128 rows); the MMA reads
// the peer's half across the pair.  Shared-memory fill per SM per k block
// drops from 54 KB to 38 KB for the same FLOPs.
//
// Cluster of 2 CTAs (rank 0 = leader).  Per CTA:
//  * warp 0   : TMA producer for its own A tile (rows of its m tile), its
//               half of the B tile, its A scales and both halves of B's
//               scales (each SM needs all of B's scales in its own TMEM).
//  * warps 6-9: scale-factor warps: shared memory -> own TMEM slot
//               (tcgen05.st) as soon as the stage's scale tiles land, then,
//               once the CTA's A/B tiles landed too, arrive on the LEADER's
//               scale barrier.
//  * warp 1   : (leader only) issues tcgen05.mma.cta_group::2 M=256 N=256
//               K=64, 4 per stage; tcgen05.commit multicasts the stage
//               release to both CTAs' empty barriers and the tile's end to
//               both CTAs' accumulator barriers.
//  * warps 2-5, 10-13: epilogue of the CTA's own 128 accumulator rows, two
//               warps per TMEM lane quarter (accumulator columns 0-127 and
//               128-255); they release the accumulator on the LEADER's barrier.
// TMEM (each CTA, allocated collectively): [0, 256) accumulator, [256, 496)
// scale slots of the 5-stage ring.  Every wait is bounded as in gemm.cuh.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include "gemm.cuh"
#include "ptx.cuh"
#include "status.cuh"

namespace nvfp4 {
namespace gemm2 {

using gemm::Args;
using gemm::BK;
using gemm::BN;
constexpr int HALF = 128;                               // rows of A and of B per CTA
constexpr int A_BYTES = HALF * BK / 2;                  // 16 KB
constexpr int B_BYTES = HALF * BK / 2;                  // 16 KB
// Scale-factor format of a stage: NVFP4 (E4M3, one scale per 16 elements,
// a 512-byte scale tile per 64 k) or MXFP4 (E8M0, one per 32, a tile per
// 128 k).  Each stage holds A's tiles and both 128-row halves of B's.
template <bool MX>
struct Fmt {
    static constexpr int SF_TILES = BK / (MX ? 128 : 64);     // scale tiles per stage and 128 rows
    static constexpr int SFA_BYTES = SF_TILES * 512;
    static constexpr int SFB_BYTES = 2 * SF_TILES * 512;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int SF_COLS = 3 * SF_TILES * 4;             // TMEM columns of a stage's scales
    static_assert(STAGE_BYTES % 1024 == 0, "stage buffers must stay 1024-byte aligned");
};
constexpr int STAGES = 5;
// epilogue staging: per epilogue warp one 32-row x 64-column BF16 block
// (4 KB, 128-byte swizzle)
constexpr int EPI_WARPS = 8;
constexpr int EPI_BLOCK = 32 * 64 * 2;
constexpr int EPI_BYTES = EPI_WARPS * EPI_BLOCK;
// warps: 0 TMA producer, 1 MMA issuer, 2-5 and 10-13 epilogue, 6-9 scale factors
constexpr int THREADS = 14 * 32;
constexpr int TMEM_COLS = gemm::TMEM_COLS;
constexpr int TMEM_SF_BASE = gemm::TMEM_SF_BASE;
__host__ __device__ constexpr int smem_bytes_for(bool tma_epi, bool mx = false) {
    return STAGES * (mx ? Fmt<true>::STAGE_BYTES : Fmt<false>::STAGE_BYTES) + (tma_epi ? EPI_BYTES : 0) +
           gemm::BAR_BYTES + 1024;
}
static_assert(smem_bytes_for(true) <= gemm::SMEM_LIMIT, "shared memory budget");
static_assert(TMEM_SF_BASE + STAGES * Fmt<false>::SF_COLS <= TMEM_COLS, "TMEM budget");

// Instruction descriptor for M = 256 (a CTA pair), N = 256, E2M1 A and B,
// K-major: kind::mxf4nvf4 with UE4M3 scales, or (mx) kind::mxf4 with UE8M0
// scales (bit 23) and the scale-factor ids of A (bits 29-30) and B (bits 4-5).
__host__ __device__ constexpr uint32_t make_idesc(bool mx = false, uint32_t sf_id = 0) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24) |
           (mx ? (1u << 23) | (sf_id << 29) | (sf_id << 4) : 0u);
}

// Unit u -> (M unit, N block).  The walk keeps the smaller operand resident
// in L2: M fastest when A is the smaller one (every A tile is revisited for
// each N block while B streams), N fastest otherwise.
__device__ __forceinline__ int unit_m(int u, int m_units, const Args& a) {
    return a.n_fastest ? u / a.n_tiles : u % m_units;
}
__device__ __forceinline__ int unit_n(int u, int m_units, const Args& a) {
    return a.n_fastest ? u % a.n_tiles : u / m_units;
}

template <bool TMA_EPI, bool MX>
__global__ void __launch_bounds__(THREADS, 1)
k_gemm_nvfp4_2sm(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                 const __grid_constant__ CUtensorMap tma_d, const __grid_constant__ CUtensorMap tma_sfa,
                 const __grid_constant__ CUtensorMap tma_sfb, const Args args) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    {
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        const uint32_t pad = (uint32_t)(smem - smem_raw);
        if (pad + (uint32_t)(smem_bytes_for(TMA_EPI, MX) - 1024) > dyn) {
            if (threadIdx.x == 0) record_device_error(NVFP4_DEV_LAUNCH);
            return;
        }
    }
    using F = Fmt<MX>;
    uint8_t* epi_stage = smem + STAGES * F::STAGE_BYTES;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(epi_stage + (TMA_EPI ? EPI_BYTES : 0));
    uint64_t* sf_full = full_bar + STAGES;         // the stage's scale tiles landed
    uint64_t* sf_bar = sf_full + STAGES;           // leader: scales of both CTAs in TMEM
    uint64_t* empty_bar = sf_bar + STAGES;         // stage consumed by the pair MMA
    uint64_t* acc_full = empty_bar + STAGES;
    uint64_t* acc_empty = acc_full + 1;            // leader: both epilogues drained TMEM
    uint64_t* drain_bar = acc_empty + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t leader = lane == 0 ? 1u : 0u;
    const int rank = (int)(cluster_ctarank() & 1u);
    const int m_units = args.m_tiles / 2;
    const int num_units = m_units * args.n_tiles;
    const int unit0 = (int)blockIdx.x / 2, unit_step = (int)gridDim.x / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&sf_full[s], 1);
            mbar_init(&sf_bar[s], 8);              // 4 scale warps x 2 CTAs
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 2 * EPI_WARPS);       // 8 epilogue warps x 2 CTAs
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        tma_prefetch_desc(&tma_a);
        tma_prefetch_desc(&tma_b);
        tma_prefetch_desc(&tma_sfa);
        tma_prefetch_desc(&tma_sfb);
        if (TMA_EPI) tma_prefetch_desc(&tma_d);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_holder, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                            // both CTAs' barriers exist
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const uint32_t sf_bar_leader = mapa_shared(smem_addr(sf_bar), 0);
    const uint32_t acc_empty_leader = mapa_shared(smem_addr(acc_empty), 0);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        int stage = 0;
        uint32_t phase = 0;
        uint32_t fills[STAGES] = {};
        bool ok = true;
        for (int u = unit0; u < num_units && ok; u += unit_step) {
            const int m_blk = unit_m(u, m_units, args) * 2 + rank, n_blk = unit_n(u, m_units, args);
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    uint8_t* sa = smem + stage * F::STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    uint8_t* ssfa = sb + B_BYTES;
                    uint8_t* ssfb = ssfa + F::SFA_BYTES;
                    // scale tiles first (3D tensor loads of A's 4 tiles and both of
                    // B's 128-row halves, zero-filled beyond the buffer) on their
                    // own barrier, so the scale warps overlap them with A and B
                    mbar_arrive_expect_tx(&sf_full[stage], F::SFA_BYTES + F::SFB_BYTES);
                    tma_load_3d(ssfa, &tma_sfa, &sf_full[stage], 0, kb * F::SF_TILES, m_blk);
                    tma_load_3d(ssfb, &tma_sfb, &sf_full[stage], 0, kb * F::SF_TILES, n_blk * 2);
                    mbar_arrive_expect_tx(&full_bar[stage], A_BYTES + B_BYTES);
                    tma_load_2d(sa, &tma_a, &full_bar[stage], kb * (BK / 2), m_blk * HALF);
                    tma_load_2d(sb, &tma_b, &full_bar[stage], kb * (BK / 2), n_blk * BN + rank * HALF);
                }
                __syncwarp();
                fills[stage] += 1;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!ok) {
            for (int s = 0; s < STAGES; ++s)
                if (fills[s]) {
                    mbar_wait_bounded(&sf_full[s], (fills[s] - 1) & 1u, nullptr);
                    mbar_wait_bounded(&full_bar[s], (fills[s] - 1) & 1u, nullptr);
                }
        } else {
            // the pair MMA has finished reading every stage of this CTA
            for (int s = 0; s < STAGES; ++s)
                if (fills[s]) mbar_wait_bounded(&empty_bar[s], (fills[s] - 1) & 1u, abort_flag);
        }
    } else if (warp >= 6 && warp < 10) {
        // --------------------------------------------- scale-factor warps --
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = unit0; u < num_units && ok; u += unit_step) {
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&sf_full[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t ssfa = smem_addr(smem + stage * F::STAGE_BYTES + A_BYTES + B_BYTES);
                const uint32_t ssfb = ssfa + F::SFA_BYTES;
                // TMEM slot of the stage: A's tiles in columns [0, 4T), B's in
                // [4T, 12T): tile kt, row group g of A at 4kt + g, of B half h at
                // 4T + 8kt + 4h + g (T = scale tiles per stage)
                constexpr int T = F::SF_TILES;
                uint32_t r[F::SF_COLS];
#pragma unroll
                for (int kt = 0; kt < T; ++kt) {
                    const uint4 a = lds128(ssfa + kt * 512 + lane * 16);
                    r[kt * 4 + 0] = a.x; r[kt * 4 + 1] = a.y; r[kt * 4 + 2] = a.z; r[kt * 4 + 3] = a.w;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 b = lds128(ssfb + h * (T * 512) + kt * 512 + lane * 16);
                        const int c = 4 * T + kt * 8 + h * 4;
                        r[c + 0] = b.x; r[c + 1] = b.y; r[c + 2] = b.z; r[c + 3] = b.w;
                    }
                }
                const uint32_t t = tmem_base + lane_base + TMEM_SF_BASE + stage * F::SF_COLS;
                tmem_st_32x32b_x16(t, r);
                if constexpr (MX) {
                    tmem_st_32x32b_x8(t + 16, r + 16);
                } else {
                    tmem_st_32x32b_x16(t + 16, r + 16);
                    tmem_st_32x32b_x16(t + 32, r + 32);
                }
                tmem_st_wait();
                tc_fence_before();
                // this CTA's A and B tiles of the stage must be in place too:
                // the leader's MMA reads both CTAs' shared memory
                if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                if (leader) mbar_arrive_cluster(sf_bar_leader + stage * 8);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------ MMA issuer (leader CTA) ----
        if (rank == 0) {
            constexpr int T = F::SF_TILES;
            constexpr int KS_PER_TILE = (BK / 64) / T;     // MMAs sharing one scale word
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            bool issued = false;
            int local = 0;
            for (int u = unit0; u < num_units && ok; u += unit_step, ++local) {
                if (!mbar_wait_bounded(acc_empty, ((uint32_t)local & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < args.k_blocks; ++kb) {
                    if (!mbar_wait_bounded(&sf_bar[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(smem + stage * F::STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const uint32_t t_sf = tmem_base + TMEM_SF_BASE + stage * F::SF_COLS;
                    const int nks = min(BK / 64, args.k_steps - kb * (BK / 64));
#pragma unroll
                    for (int ks = 0; ks < BK / 64; ++ks) {
                        const uint64_t adesc = smem_desc(sa + ks * 32, 16, 1024, 2);
                        const uint64_t bdesc = smem_desc(sb + ks * 32, 16, 1024, 2);
                        const int kt = ks / KS_PER_TILE;
                        const uint32_t pr = leader & (ks < nks ? 1u : 0u), acc = (kb | ks) != 0 ? 1u : 0u;
                        if (MX) {
                            // byte pair (ks % 2) * 2 of the tile's scale words
                            constexpr uint32_t id0 = make_idesc(true, 0), id1 = make_idesc(true, 2);
                            tc_mma_mxf4_pair_if(pr, tmem_base, adesc, bdesc, (ks % KS_PER_TILE) ? id1 : id0,
                                                t_sf + kt * 4, t_sf + 4 * T + kt * 8, acc);
                        } else {
                            tc_mma_nvf4_pair_if(pr, tmem_base, adesc, bdesc, make_idesc(), t_sf + kt * 4,
                                                t_sf + 4 * T + kt * 8, acc);
                        }
                    }
                    issued = true;
                    tc_commit_pair_mc_if(leader, &empty_bar[stage], (uint16_t)0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_mc_if(leader, acc_full, (uint16_t)0x3);
            }
            if (!ok && issued) {
                tc_commit_pair_mc_if(leader, drain_bar, (uint16_t)0x1);
                mbar_wait_bounded(drain_bar, 0, nullptr);
            }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------- epilogue ----
        // Each epilogue warp drains 32 accumulator rows (its TMEM lane
        // quarter) x 128 columns (its half), 16 columns per TMEM load with the
        // next load in flight, and releases the accumulator as soon as its
        // last column has been read.  Columns 0-63 of the half stream out
        // through the warp's 4 KB staging block before the release, columns
        // 64-127 are held in registers and follow it.
        const int quarter = warp & 3;
        const int col0 = warp >= 10 ? BN / 2 : 0;
        const int ew = warp < 6 ? warp - 2 : warp - 6;
        // MXFP4 has no tensor scales: D is the plain sum of the scaled products
        const gemm::Alpha alpha = MX ? gemm::Alpha{1.0f, 1.0f} : gemm::make_alpha(*args.gs_a, *args.gs_b);
        const uint32_t stg = smem_addr(epi_stage) + (uint32_t)ew * EPI_BLOCK;
        const uint64_t out_policy = l2_policy_evict_first();   // D is written once
        int local = 0;
        for (int u = unit0; u < num_units; u += unit_step, ++local) {
            if (!mbar_wait_bounded(acc_full, (uint32_t)local & 1u, abort_flag)) break;
            tc_fence_after();
            const int m_blk = unit_m(u, m_units, args) * 2 + rank, n_blk = unit_n(u, m_units, args);
            const int64_t row = (int64_t)m_blk * HALF + quarter * 32 + lane;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col0;
            if (TMA_EPI) {
                const int y = m_blk * HALF + quarter * 32;
                uint32_t packed[32];
                uint32_t acc[2][16];
                tmem_ld_32x32b_x16(t_row, acc[0]);
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
                    tmem_ld_wait16(acc[c & 1]);
                    if (c + 1 < BN / 32) tmem_ld_32x32b_x16(t_row + (c + 1) * 16, acc[(c + 1) & 1]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float2 r = alpha.apply2(__uint_as_float(acc[c & 1][2 * j]),
                                                      __uint_as_float(acc[c & 1][2 * j + 1]));
                        __nv_bfloat162 hv = __floats2bfloat162_rn(r.x, r.y);
                        packed[(c & 3) * 8 + j] = *reinterpret_cast<uint32_t*>(&hv);
                    }
                    if (c == 3 || c == BN / 32 - 1) {
                        if (c == BN / 32 - 1) {             // accumulator fully read
                            tc_fence_before();
                            __syncwarp();
                            if (leader) mbar_arrive_cluster(acc_empty_leader);
                        }
                        if (leader) bulk_wait_read_all();   // the block's last store has read it
                        __syncwarp();
                        const uint32_t rowp = stg + (uint32_t)lane * 128;
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const uint32_t unit = (uint32_t)q ^ (uint32_t)(lane & 7);
                            sts128(rowp + unit * 16, packed[q * 4], packed[q * 4 + 1], packed[q * 4 + 2],
                                   packed[q * 4 + 3]);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (leader) {
                            const int x = n_blk * BN + col0 + (c == 3 ? 0 : 64);
                            if (x < args.N && y < args.M)
                                tma_store_2d_hint(&tma_d, epi_stage + ew * EPI_BLOCK, x, y, out_policy);
                            bulk_commit_group();
                        }
                    }
                }
            } else {
                uint32_t acc[32];
                for (int c = 0; c < BN / 64; ++c) {
                    tmem_ld_32x32b_x32(t_row + c * 32, acc);
                    tmem_ld_wait();
                    if (c == BN / 64 - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (leader) mbar_arrive_cluster(acc_empty_leader);
                    }
                    const int64_t cc = (int64_t)n_blk * BN + col0 + c * 32;
                    if (cc < args.N) gemm::store_chunk(args, row, cc, acc, alpha);
                }
            }
        }
        if (TMA_EPI && leader) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                            // the pair finishes together
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

}  // namespace gemm2
}  // namespace nvfp4
