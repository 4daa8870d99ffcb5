// gemm.cuh -- block-scaled NVFP4 GEMM on the 5th-generation tensor cores.
//
//   D[m, n] = alpha * sum_k (qa[m,k] * sa[m,k/16]) * (qb[n,k] * sb[n,k/16])
//
// with E2M1 codes qa/qb, E4M3 block scales sa/sb (one per 16 elements along
// k), FP32 accumulation in tensor memory and alpha = 1 / (S_A * S_B) applied
// in the epilogue (FP32 or BF16 output).  Source: NVIDIA blog "NVFP4 Trains
// with Precision of 16-Bit and Speed and Efficiency of 4-Bit", Figure 1 (GEMMs
// of the linear layers dominate) and recipe bullets 1-2 (16-element blocks
// with E4M3 scales, natively supported by Blackwell tensor cores).
//
// Design (sm_103a, one CTA per SM, persistent over 128 x 256 output tiles,
// 10 warps; every role runs as a converged warp and the single-thread
// tcgen05 / TMA operations are predicated on one lane):
//  * warp 0   : TMA producer.  Per 256-wide k block it loads the A tile
//               (128 rows x 128 B, 128-byte swizzle), the B tile (256 rows x
//               128 B) and the matching 512-byte scale tiles (3D tensor loads
//               over the scale buffer) into a 3- or 4-stage ring.
//  * warps 6-9: scale-factor warps, one per TMEM lane quarter.  They copy a
//               stage's E4M3 scales from shared memory to its TMEM slot with
//               tcgen05.st, replicating each 32-row scale tile into all four
//               lane quarters (the layout the block-scaled MMA reads).
//  * warp 1   : allocates TMEM and issues 4 MMAs per stage
//               (tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X,
//               M = 128, N = 256, K = 64), releasing the stage with
//               tcgen05.commit.  Nothing else runs on this thread, so the MMA
//               issue rate stays above the tensor core's.
//  * warps 2-5: epilogue.  Each warp drains its 32-lane quarter of the
//               128 x 256 FP32 accumulator with tcgen05.ld, scales by alpha,
//               converts and stores.  The accumulator is released after the
//               last TMEM read, before the last stores.
// TMEM: columns [0, 256) accumulator; [256, 448) the per-stage scale slots
// (16 columns of A scales + 32 of B scales per stage).
// Every mbarrier wait is bounded (2 s); on expiry the kernel records
// NVFP4_DEV_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include "guard.cuh"
#include "ptx.cuh"
#include "status.cuh"

namespace nvfp4 {
namespace gemm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 256;                       // k elements per stage (128 bytes of codes)
constexpr int A_BYTES = BM * BK / 2;          // 16 KB
constexpr int B_BYTES = BN * BK / 2;          // 32 KB
constexpr int SFA_BYTES = (BM / 128) * (BK / 64) * 512;   // 2 KB
constexpr int SFB_BYTES = (BN / 128) * (BK / 64) * 512;   // 4 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
// BF16 output: 3 stages + a 64 KB staging tile for the TMA-store epilogue
// (16 KB per epilogue warp); FP32 output: 4 stages, direct stores.
constexpr int EPI_WARP_BYTES = 32 * BN * 2;
constexpr int EPI_BYTES = 4 * EPI_WARP_BYTES;
constexpr int BAR_BYTES = 256;
__host__ __device__ constexpr int stages_for(bool tma_epi) { return tma_epi ? 3 : 4; }
__host__ __device__ constexpr int smem_bytes_for(bool tma_epi) {
    return stages_for(tma_epi) * STAGE_BYTES + (tma_epi ? EPI_BYTES : 0) + BAR_BYTES + 1024;
}
constexpr int SMEM_LIMIT = 232448;    // 227 KB opt-in maximum per CTA
constexpr int THREADS = 320;
constexpr int TMEM_COLS = 512;
constexpr int TMEM_SF_BASE = 256;
constexpr int SF_COLS_PER_STAGE = 48;
static_assert(STAGE_BYTES % 1024 == 0, "stage buffers must stay 1024-byte aligned");
static_assert(TMEM_SF_BASE + 4 * SF_COLS_PER_STAGE <= TMEM_COLS, "TMEM budget");
static_assert(smem_bytes_for(false) <= SMEM_LIMIT, "shared memory budget");
static_assert(smem_bytes_for(true) - 1024 <= SMEM_LIMIT, "shared memory budget");

struct Args {
    const uint8_t* sfa;        // swizzled scales of A (rows padded to 128)
    const uint8_t* sfb;
    const float* gs_a;         // S_enc of A and B (device)
    const float* gs_b;
    void* d;
    int64_t ldd;
    int d_bf16;
    int M, N, K;
    int m_tiles, n_tiles;
    int k_blocks;              // ceil(K / BK)
    int k_steps;               // ceil(K / 64): MMAs along k
    int sf_col_tiles;          // ceil(K / 64): 512-byte scale tiles per 128-row group
    int b_row_tiles;           // ceil(N / 128)
    int n_fastest;             // tile walk: 1 = N blocks fastest (B stays in L2), 0 = M fastest
};

// Instruction descriptor of kind::mxf4nvf4: dense, A and B E2M1 (format 1),
// both K-major, UE4M3 scales, scale-factor ids 0, N >> 3 at bit 17,
// M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc() {
    return (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

// alpha = 1 / (S_A * S_B), carried as m * p: m an FP32 number in the normal
// range and p a power of two.  1/(S_A S_B) spans about 2^-256 .. 2^233 (each
// S_enc lies in [2688 / bf16 max, FLT_MAX]), far beyond FP32's normal range;
// rounding it to one FP32 number would leave a subnormal alpha with fewer
// than 24 significant bits (or zero) when both operands have a tiny amax.
// D = fp32(fp32(acc * m) * p): with p = 1 (the usual case) this is
// fp32(acc * fp32(alpha)); otherwise the second product is exact unless its
// result is itself outside the normal range.
struct Alpha {
    float m, p;
    __device__ __forceinline__ float apply(float acc) const { return __fmul_rn(__fmul_rn(acc, m), p); }
    // two accumulators at once on packed two-lane FP32 (per lane the same
    // IEEE products as apply); the second product only when p != 1
    __device__ __forceinline__ float2 apply2(float a0, float a1) const {
        float2 r = __fmul2_rn(make_float2(a0, a1), make_float2(m, m));
        if (p != 1.0f) r = __fmul2_rn(r, make_float2(p, p));
        return r;
    }
};

__device__ __forceinline__ Alpha make_alpha(float s_a, float s_b) {
    const double a = 1.0 / ((double)s_a * (double)s_b);
    if (a < 0x1p-126) return Alpha{(float)(a * 0x1p80), 0x1p-80f};
    if (a > 0x1p127) return Alpha{(float)fmin(a * 0x1p-80, 0x1.fffffep127), 0x1p80f};
    return Alpha{(float)a, 1.0f};
}

__device__ __forceinline__ void store_chunk(const Args& a, int64_t row, int64_t col0,
                                            const uint32_t* acc, Alpha alpha) {
    if (row >= a.M) return;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = alpha.apply(__uint_as_float(acc[j]));
    const bool full = col0 + 32 <= a.N;
    if (a.d_bf16) {
        uint16_t* dst = reinterpret_cast<uint16_t*>(a.d) + row * a.ldd + col0;
        if (!NVFP4_GUARD(a.d, stored_extent(a.M, a.N, a.ldd, 2), dst, 2 * (uint32_t)min64(32, a.N - col0),
                         kGuardGemmD)) {
        } else if (full) {
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
                p[j] = *reinterpret_cast<uint32_t*>(&h);
            }
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int j = 0; j < 4; ++j) d4[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
        } else {
            for (int j = 0; j < 32; ++j)
                if (col0 + j < a.N) {
                    __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
                    dst[j] = *reinterpret_cast<uint16_t*>(&h);
                }
        }
    } else {
        float* dst = reinterpret_cast<float*>(a.d) + row * a.ldd + col0;
        if (!NVFP4_GUARD(a.d, stored_extent(a.M, a.N, a.ldd, 4), dst, 4 * (uint32_t)min64(32, a.N - col0),
                         kGuardGemmD)) {
        } else if (full) {
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int j = 0; j < 8; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        } else {
            for (int j = 0; j < 32; ++j)
                if (col0 + j < a.N) dst[j] = v[j];
        }
    }
}

// BF16 epilogue through shared memory: a warp's 32 rows x 256 columns in
// four 64-column blocks, each 32 rows x 128 bytes in the 128-byte swizzle
// (16-byte unit u of row r at unit u ^ (r % 8)), stored by TMA.
__device__ __forceinline__ void stage_bf16_chunk(uint32_t stg, int c, int lane, const uint32_t* acc,
                                                 Alpha alpha) {
    uint32_t p[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float2 r = alpha.apply2(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
        __nv_bfloat162 h = __floats2bfloat162_rn(r.x, r.y);
        p[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    const uint32_t blk = stg + (uint32_t)(c >> 1) * (32 * 128) + (uint32_t)lane * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t unit = (uint32_t)((c & 1) * 4 + q) ^ (uint32_t)(lane & 7);
        sts128(blk + unit * 16, p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
    }
}

template <bool TMA_EPI>
__global__ void __launch_bounds__(THREADS, 1)
k_gemm_nvfp4(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
             const __grid_constant__ CUtensorMap tma_d, const __grid_constant__ CUtensorMap tma_sfa,
             const __grid_constant__ CUtensorMap tma_sfb, const Args args) {
    constexpr int STAGES = stages_for(TMA_EPI);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    {
        // the 1024-byte aligned layout must fit the dynamic allocation
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        const uint32_t pad = (uint32_t)(smem - smem_raw);
        if (pad + (uint32_t)(smem_bytes_for(TMA_EPI) - 1024) > dyn) {
            if (threadIdx.x == 0) record_device_error(NVFP4_DEV_LAUNCH);
            return;
        }
    }
    uint8_t* epi_stage = smem + STAGES * STAGE_BYTES;
    uint64_t* full_bar = reinterpret_cast<uint64_t*>(epi_stage + (TMA_EPI ? EPI_BYTES : 0));
    uint64_t* sf_bar = full_bar + STAGES;        // scales of the stage are in TMEM
    uint64_t* empty_bar = sf_bar + STAGES;
    uint64_t* acc_full = empty_bar + STAGES;
    uint64_t* acc_empty = acc_full + 1;
    uint64_t* drain_bar = acc_empty + 1;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t leader = lane == 0 ? 1u : 0u;
    const int num_tiles = args.m_tiles * args.n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&sf_bar[s], 4);
            mbar_init(&empty_bar[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 4 * 32);
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
        tmem_alloc(tmem_holder, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        int stage = 0;
        uint32_t phase = 0;
        uint32_t fills[STAGES] = {};
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            const int m_blk = args.n_fastest ? tile / args.n_tiles : tile % args.m_tiles;
            const int n_blk = args.n_fastest ? tile % args.n_tiles : tile / args.m_tiles;
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (leader) {
                    uint8_t* sa = smem + stage * STAGE_BYTES;
                    uint8_t* sb = sa + A_BYTES;
                    uint8_t* ssfa = sb + B_BYTES;
                    uint8_t* ssfb = ssfa + SFA_BYTES;
                    // scale tiles: 3D tensor loads (zero-filled beyond the buffer)
                    mbar_arrive_expect_tx(&full_bar[stage], STAGE_BYTES);
                    tma_load_2d(sa, &tma_a, &full_bar[stage], kb * (BK / 2), m_blk * BM);
                    tma_load_3d(ssfa, &tma_sfa, &full_bar[stage], 0, kb * 4, m_blk);
                    tma_load_2d(sb, &tma_b, &full_bar[stage], kb * (BK / 2), n_blk * BN);
                    tma_load_3d(ssfb, &tma_sfb, &full_bar[stage], 0, kb * 4, n_blk * 2);
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
            // let every copy this warp issued land before the CTA exits
            for (int s = 0; s < STAGES; ++s)
                if (fills[s]) mbar_wait_bounded(&full_bar[s], (fills[s] - 1) & 1u, nullptr);
        }
    } else if (warp >= 6) {
        // --------------------------------------------- scale-factor warps --
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            for (int kb = 0; kb < args.k_blocks; ++kb) {
                if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                const uint32_t ssfa = smem_addr(smem + stage * STAGE_BYTES + A_BYTES + B_BYTES);
                const uint32_t ssfb = ssfa + SFA_BYTES;
                uint32_t r[48];
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint4 a = lds128(ssfa + ks * 512 + lane * 16);
                    r[ks * 4 + 0] = a.x; r[ks * 4 + 1] = a.y; r[ks * 4 + 2] = a.z; r[ks * 4 + 3] = a.w;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 b = lds128(ssfb + h * 2048 + ks * 512 + lane * 16);
                        const int c = 16 + ks * 8 + h * 4;
                        r[c + 0] = b.x; r[c + 1] = b.y; r[c + 2] = b.z; r[c + 3] = b.w;
                    }
                }
                const uint32_t t = tmem_base + lane_base + TMEM_SF_BASE + stage * SF_COLS_PER_STAGE;
                tmem_st_32x32b_x16(t, r);
                tmem_st_32x32b_x16(t + 16, r + 16);
                tmem_st_32x32b_x16(t + 32, r + 32);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (leader) mbar_arrive(&sf_bar[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ----
        constexpr uint32_t idesc = make_idesc();
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        bool issued = false;
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
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
                const uint32_t sa = smem_addr(smem + stage * STAGE_BYTES);
                const uint32_t sb = sa + A_BYTES;
                const uint32_t t_sf = tmem_base + TMEM_SF_BASE + stage * SF_COLS_PER_STAGE;
                const int nks = min(BK / 64, args.k_steps - kb * (BK / 64));
#pragma unroll
                for (int ks = 0; ks < BK / 64; ++ks) {
                    const uint64_t adesc = smem_desc(sa + ks * 32, 16, 1024, 2);
                    const uint64_t bdesc = smem_desc(sb + ks * 32, 16, 1024, 2);
                    tc_mma_nvf4_if(leader & (ks < nks ? 1u : 0u), tmem_base, adesc, bdesc, idesc,
                                   t_sf + ks * 4, t_sf + 16 + ks * 8, (kb | ks) != 0 ? 1u : 0u);
                }
                issued = true;
                tc_commit_if(leader, &empty_bar[stage]);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            tc_commit_if(leader, acc_full);
        }
        if (!ok && issued) {
            tc_commit_if(leader, drain_bar);
            mbar_wait_bounded(drain_bar, 0, nullptr);
        }
    } else {
        // --------------------------------------------------- epilogue ----
        const int quarter = warp & 3;
        const Alpha alpha = make_alpha(*args.gs_a, *args.gs_b);
        const uint32_t stg = smem_addr(epi_stage) + (uint32_t)(warp - 2) * EPI_WARP_BYTES;
        const uint64_t out_policy = l2_policy_evict_first();   // D is written once
        int local = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
            if (!mbar_wait_bounded(acc_full, (uint32_t)local & 1u, abort_flag)) break;
            tc_fence_after();
            const int m_blk = args.n_fastest ? tile / args.n_tiles : tile % args.m_tiles;
            const int n_blk = args.n_fastest ? tile % args.n_tiles : tile / args.m_tiles;
            const int64_t row = (int64_t)m_blk * BM + quarter * 32 + lane;
            const uint32_t t_row = tmem_base + ((uint32_t)(quarter * 32) << 16);
            if (TMA_EPI && local > 0) {
                if (leader) bulk_wait_read_all();          // staging tile free again
                __syncwarp();
            }
            uint32_t acc[32];
            for (int c = 0; c < BN / 32; ++c) {
                tmem_ld_32x32b_x32(t_row + c * 32, acc);
                tmem_ld_wait();
                if (c == BN / 32 - 1) {
                    tc_fence_before();
                    mbar_arrive(acc_empty);
                }
                if (TMA_EPI) {
                    stage_bf16_chunk(stg, c, lane, acc, alpha);
                } else {
                    const int64_t col0 = (int64_t)n_blk * BN + c * 32;
                    if (col0 < args.N) store_chunk(args, row, col0, acc, alpha);
                }
            }
            if (TMA_EPI) {
                fence_proxy_async_smem();
                __syncwarp();
                if (leader) {
                    const int y = m_blk * BM + quarter * 32;
                    for (int b = 0; b < BN / 64; ++b) {
                        const int x = n_blk * BN + b * 64;
                        if (x < args.N && y < args.M) tma_store_2d_hint(&tma_d, epi_stage + (warp - 2) * EPI_WARP_BYTES + b * 4096, x, y, out_policy);
                    }
                    bulk_commit_group();
                }
            }
        }
        if (TMA_EPI && leader) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace gemm
}  // namespace nvfp4
