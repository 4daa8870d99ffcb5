// gemm.cuh -- definitions shared by the block-scaled FP4 GEMMs (gemm2sm.cuh):
//
//   D[m, n] = alpha * sum_k (qa[m,k] * sa[m,k/16]) * (qb[n,k] * sb[n,k/16])
//
// with E2M1 codes qa/qb, E4M3 block scales sa/sb (one per 16 elements along
// k; E8M0 per 32 for MXFP4), FP32 accumulation in tensor memory and alpha =
// 1 / (S_A * S_B) applied in the epilogue (FP32 or BF16 output).  Source:
// NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and Speed and Efficiency
// of 4-Bit", Figure 1 (GEMMs of the linear layers dominate) and recipe
// bullets 1-2 (16-element blocks with E4M3 scales, natively supported by
// Blackwell tensor cores).
//
// Here: the tile shape, the kernel argument block, alpha and the plain-store
// epilogue chunk (FP32 output and ragged BF16 tiles).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include "codec.cuh"
#include "guard.cuh"
#include "ptx.cuh"
#include "status.cuh"

namespace nvfp4 {
namespace gemm {

constexpr int BM = 128;                       // output rows per CTA
constexpr int BN = 256;                       // output columns per tile
constexpr int BK = 256;                       // k elements per pipeline stage (128 bytes of codes)
constexpr int BAR_BYTES = 256;                // mbarriers and flags after the stage buffers
constexpr int SMEM_LIMIT = 232448;            // 227 KB opt-in maximum per CTA
constexpr int TMEM_COLS = 512;
constexpr int TMEM_SF_BASE = 256;             // [0, 256) accumulator, then the scale slots

struct Args {
    const float* gs_a;         // S_enc of A and B (device)
    const float* gs_b;
    void* d;
    int64_t ldd;
    int d_bf16;
    int M, N, K;
    int m_tiles, n_tiles;      // 128-row M tiles (even: CTA pairs) and 256-column N tiles
    int k_blocks;              // ceil(K / BK)
    int k_steps;               // ceil(K / 64): MMAs along k
    int n_fastest;             // tile walk: 1 = N blocks fastest (B stays in L2), 0 = M fastest
};

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

}  // namespace gemm
}  // namespace nvfp4
