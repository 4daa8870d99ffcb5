// dual.cuh -- dual-axis kernels: one read of a stored bf16 tensor S [R x C]
// serves both GEMM views of it.
//
//  * k_amax_dual: max |S| (the amax of either view) and max |RHT16(S^T)|
//    (the amax of the column-wise operand, transformed along K = R).
//  * k_quant_dual: the row-wise 1x16 operand S [R x C] (fprop / dgrad: blocks
//    along C) and the column-wise 1x16 operand S^T [C x R] (wgrad: blocks
//    along the tokens R, optionally after the 16-point random Hadamard
//    transform), from one shared-memory tile.
//
// Each output is bit for bit the one the separate calls make (the same
// per-block arithmetic in encode_block16, the same Philox indices), so the
// dual forms are pure traffic savings: S is read once instead of twice.
//
// Method: NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and Speed and
// Efficiency of 4-Bit", recipe bullets 1-5 (1x16 blocks with E4M3 scales,
// FP32 per-tensor scale, Hadamard transform on the wgrad inputs, stochastic
// rounding of gradients); prism.simon-ai.net article 7890, "Techniques
// against outliers and rounding error" (RHT along the reduction dimension).
#pragma once
#include <cstdint>
#include "codec.cuh"
#include "quantize.cuh"
#include "status.cuh"

namespace nvfp4 {

// Block-wide maxima of two non-negative float bit patterns, merged into two
// outputs with one atomic each per CTA.
__device__ __forceinline__ void block_max2_to_global(uint32_t m0, float* out0, uint32_t m1, float* out1) {
    __shared__ uint32_t red[2][kQuantThreads / 32];
    m0 = __reduce_max_sync(0xFFFFFFFFu, m0);
    m1 = __reduce_max_sync(0xFFFFFFFFu, m1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[0][warp] = m0;
        red[1][warp] = m1;
    }
    __syncthreads();
    if (warp == 0) {
        const bool in = lane < (int)(blockDim.x >> 5);
        m0 = __reduce_max_sync(0xFFFFFFFFu, in ? red[0][lane] : 0u);
        m1 = __reduce_max_sync(0xFFFFFFFFu, in ? red[1][lane] : 0u);
        if (lane == 0) {
            if (m0) atomicMax(reinterpret_cast<uint32_t*>(out0), m0);
            if (m1) atomicMax(reinterpret_cast<uint32_t*>(out1), m1);
        }
    }
}

// ============================================================ dual amax ====
// Thread item: 16 stored rows (one K block of the column-wise view) x 2
// stored columns, 4-byte loads (a warp covers 128 contiguous bytes of a row).
// The raw words feed the plain maximum (half-word SIMD max of the magnitude
// bits, NaN-propagating); the two columns are transformed one at a time.
__global__ void __launch_bounds__(kQuantThreads, 3) k_amax_dual(const uint16_t* __restrict__ p,
                                                                int64_t srows, int64_t scols, int64_t ld,
                                                                uint32_t mask, float* out_plain,
                                                                float* out_t) {
    constexpr uint32_t M = 0x7FFF7FFFu;
    uint32_t m = 0, m2 = 0;
    const int64_t ncp = (scols + 1) >> 1, nkb = srows >> 4;
    for (ItemWalk it((uint32_t)ncp); it.major < nkb; it.next()) {
        const int64_t c0 = (int64_t)it.minor * 2;
        const uint16_t* base = p + it.major * 16 * ld + c0;
        uint32_t w[16];
        if (c0 + 2 <= scols) {
#pragma unroll
            for (int t = 0; t < 16; ++t) w[t] = ldg_u32(base + t * ld);
        } else {
#pragma unroll
            for (int t = 0; t < 16; ++t) w[t] = (uint32_t)base[t * ld];
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) m2 = __vmaxu2(m2, w[t] & M);
        float v[16];
        if (mask) {
#pragma unroll
            for (int t = 0; t < 16; ++t) v[t] = bf16_lo(w[t]);
            m = max(m, rht16_absmax_bits_nan(v, mask));
#pragma unroll
            for (int t = 0; t < 16; ++t) v[t] = bf16_hi(w[t]);
            m = max(m, rht16_absmax_bits_nan(v, mask));
        }
    }
    const uint32_t plain = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    block_max2_to_global(plain, out_plain, mask ? m : plain, out_t);
}

// ======================================================== dual quantise ====
// CTA tile: 128 stored rows x 256 stored columns (64 KB of bf16), staged in
// shared memory as 16-byte chunks, chunk q of row r at position
// q ^ (((q >> 3) & 3) | ((r & 1) << 2)) of its row: the row stores (a warp
// per row), the row-wise reads (8 rows x 4 column groups per warp, 16-byte
// reads) and the column-pair reads (32 consecutive words of a row per warp)
// are all free of bank conflicts.
constexpr int kDualRows = 128, kDualCols = 256;
constexpr int kDualChunks = kDualCols / 8;                       // 16-byte chunks per row
constexpr int kDualSmem = kDualRows * kDualCols * 2;             // 64 KB

struct DualArgs {
    QuantArgs row;      // logical S [R x C]: x, rows = R, k = C, ld; codes/scales of out
    QuantArgs col;      // logical S^T [C x R]: rows = C, k = R; codes/scales of out_t; rht_mask
};

__device__ __forceinline__ int dual_chunk(int r, int q) {
    return r * kDualChunks + (q ^ (((q >> 3) & 3) | ((r & 1) << 2)));
}

template <bool SR1, bool SR2, bool RHT2>
__global__ void __launch_bounds__(kQuantThreads, 3) k_quant_dual(const DualArgs d) {
    extern __shared__ __align__(16) uint8_t dual_smem[];
    uint4* tile = reinterpret_cast<uint4*>(dual_smem);
    __shared__ float rtab1[128], rtab2[128];
    const QuantArgs& a1 = d.row;
    const QuantArgs& a2 = d.col;
    float s1, s2;
    const bool ok1 = resolve_scale(a1.scale_src, 0, a1.gs_out, nullptr, &s1);
    const bool ok2 = resolve_scale(a2.scale_src, 0, a2.gs_out, nullptr, &s2);
    if (!ok1 && !ok2) return;                                    // uniform over the grid
    for (int c = threadIdx.x; c < 128; c += blockDim.x) {
        rtab1[c] = ok1 ? encode_factor(s1, (uint32_t)c) : 0.0f;
        rtab2[c] = ok2 ? encode_factor(s2, (uint32_t)c) : 0.0f;
    }
    const int64_t R = a1.rows, C = a1.k;
    const int64_t r0 = (int64_t)blockIdx.y * kDualRows, c0 = (int64_t)blockIdx.x * kDualCols;
    // ---- stage the tile (zeros beyond the tensor)
    {
        const int q = threadIdx.x & 31;
        const bool col_ok = c0 + q * 8 < C;
#pragma unroll 4
        for (int k = 0; k < kDualRows / 8; ++k) {
            const int r = (threadIdx.x >> 5) + 8 * k;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (col_ok && r0 + r < R) v = ldg_stream(a1.x + (r0 + r) * a1.ld + c0 + q * 8);
            tile[dual_chunk(r, q)] = v;
        }
    }
    __syncthreads();

    // ---- row-wise operand: items (tile row, group of 4 blocks), 2 per thread
    if (ok1) {
        const int64_t nkb = C >> 4;
        const int64_t ngroups = (nkb + 3) >> 2;
        const int64_t rows_pad = (R + 127) & ~int64_t(127);
#pragma unroll 1
        for (int i = threadIdx.x; i < kDualRows * 4; i += blockDim.x) {
            const int r = i >> 2, g = i & 3;
            const int64_t rg = r0 + r;
            const int64_t G = c0 / 64 + g;
            if (rg >= rows_pad || G >= ngroups) continue;
            uint32_t* sdst = reinterpret_cast<uint32_t*>(a1.scales + scale_offset(rg, G * 4, ngroups));
            if (rg >= R) {
                *sdst = 0u;
                continue;
            }
            const int nblk = (int)min64(4, nkb - G * 4);
            uint32_t sw = 0, cw[8];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                cw[2 * b] = cw[2 * b + 1] = 0u;
                if (b < nblk) {
                    const uint4 lo = tile[dual_chunk(r, 8 * g + 2 * b)];
                    const uint4 hi = tile[dual_chunk(r, 8 * g + 2 * b + 1)];
                    float v[16];
                    unpack8(lo, v);
                    unpack8(hi, v + 8);
                    uint32_t sb;
                    encode_block16<false, SR1>(v, s1, rtab1, (uint64_t)(rg * C + G * 64 + b * 16), a1, &sb,
                                               &cw[2 * b], &cw[2 * b + 1], absmax_bits16_packed(lo, hi));
                    sw |= sb << (8 * b);
                }
            }
            uint8_t* cdst = a1.codes + rg * (C >> 1) + G * 32;
            if (nblk == 4 && (C & 31) == 0) {
                reinterpret_cast<uint4*>(cdst)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                reinterpret_cast<uint4*>(cdst)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
            } else {
#pragma unroll
                for (int b = 0; b < 4; ++b)
                    if (b < nblk) reinterpret_cast<uint2*>(cdst)[b] = make_uint2(cw[2 * b], cw[2 * b + 1]);
            }
            *sdst = sw;
        }
    }

    // ---- column-wise operand: item (column pair, half of the tile's rows)
    if (ok2) {
        const uint32_t* words = reinterpret_cast<const uint32_t*>(tile);
        const int pr = threadIdx.x & 127, h = threadIdx.x >> 7;
        const int64_t cc = c0 + 2 * pr;                       // logical rows cc, cc + 1
        const int64_t nkb = R >> 4;
        const int64_t ngroups = (nkb + 3) >> 2;
        const int64_t G = r0 / 64 + h;                        // group of 4 K blocks
        const int64_t rows_pad = (C + 127) & ~int64_t(127);
        if (G < ngroups && cc < rows_pad) {
            uint32_t* s0 = reinterpret_cast<uint32_t*>(a2.scales + scale_offset(cc, G * 4, ngroups));
            uint32_t* s1p = reinterpret_cast<uint32_t*>(a2.scales + scale_offset(cc + 1, G * 4, ngroups));
            if (cc >= C) {                                    // C is even: both rows are padding
                *s0 = 0u;
                *s1p = 0u;
            } else {
                const int nblk = (int)min64(4, nkb - G * 4);
                uint32_t sw0 = 0, sw1 = 0, c0w[8], c1w[8];
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    c0w[2 * b] = c0w[2 * b + 1] = c1w[2 * b] = c1w[2 * b + 1] = 0u;
                    if (b < nblk) {
                        uint32_t w[16];
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const int r = h * 64 + b * 16 + t;
                            w[t] = words[dual_chunk(r, pr >> 2) * 4 + (pr & 3)];
                        }
                        const int64_t kc = G * 64 + b * 16;
                        float v[16];
                        uint32_t sb;
#pragma unroll
                        for (int t = 0; t < 16; ++t) v[t] = bf16_lo(w[t]);
                        encode_block16<RHT2, SR2>(v, s2, rtab2, (uint64_t)(cc * R + kc), a2, &sb, &c0w[2 * b],
                                                  &c0w[2 * b + 1]);
                        sw0 |= sb << (8 * b);
#pragma unroll
                        for (int t = 0; t < 16; ++t) v[t] = bf16_hi(w[t]);
                        encode_block16<RHT2, SR2>(v, s2, rtab2, (uint64_t)((cc + 1) * R + kc), a2, &sb,
                                                  &c1w[2 * b], &c1w[2 * b + 1]);
                        sw1 |= sb << (8 * b);
                    }
                }
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const uint32_t* cw = rr ? c1w : c0w;
                    uint8_t* cdst = a2.codes + (cc + rr) * (R >> 1) + G * 32;
                    if (nblk == 4 && (R & 31) == 0) {
                        reinterpret_cast<uint4*>(cdst)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                        reinterpret_cast<uint4*>(cdst)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                    } else {
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            if (b < nblk)
                                reinterpret_cast<uint2*>(cdst)[b] = make_uint2(cw[2 * b], cw[2 * b + 1]);
                    }
                }
                *s0 = sw0;
                *s1p = sw1;
            }
        }
    }
}

}  // namespace nvfp4

namespace nvfp4 {

// ============================================ streamed (TMA-fed) amax ======
// max |S| and (RHT_COLS) max |RHT16 down the columns of S| for a stored bf16
// array S [srows x scols], streamed through shared memory: persistent CTAs
// walk 64-row x 256-column tiles (32 KB, loaded by one 2D TMA copy; zeros
// beyond the array) through a ring of kAmaxStages slots, so that up to
// kAmaxStages - 1 tiles per CTA are in flight while one is reduced.
// A tile is 128 column pairs x 4 blocks of 16 rows; each thread reduces two
// (pair, block) items with conflict-free 4-byte reads (a warp reads 128
// contiguous bytes of a tile row).
constexpr int kAmaxTileRows = 64, kAmaxTileCols = 256;
constexpr int kAmaxTileBytes = kAmaxTileRows * kAmaxTileCols * 2;
constexpr int kAmaxStages = 3;
constexpr int kAmaxSmem = kAmaxStages * kAmaxTileBytes + 64;

template <bool RHT_COLS>
__global__ void __launch_bounds__(kQuantThreads, 2) k_amax_stream(const __grid_constant__ CUtensorMap map,
                                                                  int64_t srows, int64_t scols, uint32_t mask,
                                                                  float* out_plain, float* out_t) {
    extern __shared__ __align__(128) uint8_t amax_smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(amax_smem + kAmaxStages * kAmaxTileBytes);
    __shared__ int abort_flag;
    const int64_t row_tiles = (srows + kAmaxTileRows - 1) / kAmaxTileRows;
    const int64_t col_tiles = (scols + kAmaxTileCols - 1) / kAmaxTileCols;
    const int64_t ntiles = row_tiles * col_tiles;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAmaxStages; ++s) mbar_init(&full[s], 1);
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&map);
    }
    __syncthreads();
    auto issue = [&](int64_t t, int s) {
        const int64_t tr = t / col_tiles, tc = t - tr * col_tiles;
        mbar_arrive_expect_tx(&full[s], kAmaxTileBytes);
        tma_load_2d(amax_smem + s * kAmaxTileBytes, &map, &full[s], (int32_t)(tc * kAmaxTileCols),
                    (int32_t)(tr * kAmaxTileRows));
    };
    if (threadIdx.x == 0)
        for (int s = 0; s < kAmaxStages; ++s) {
            const int64_t t = (int64_t)blockIdx.x + (int64_t)s * gridDim.x;
            if (t < ntiles) issue(t, s);
        }
    constexpr uint32_t M = 0x7FFF7FFFu;
    uint32_t m2 = 0, m = 0;
    const int pr = threadIdx.x & 127;                 // column pair of the tile
    const int kb0 = threadIdx.x >> 7;                 // blocks kb0 and kb0 + 2
    int i = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
        const int s = i % kAmaxStages;
        const uint32_t ph = (uint32_t)(i / kAmaxStages) & 1u;
        const bool ok = mbar_wait_bounded(&full[s], ph, &abort_flag);
        __syncthreads();                              // every thread saw the same outcome
        if (abort_flag || !ok) break;
        const uint32_t* words = reinterpret_cast<const uint32_t*>(amax_smem + s * kAmaxTileBytes);
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int kb = kb0 + 2 * j;
            uint32_t w[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) w[r] = words[(kb * 16 + r) * (kAmaxTileCols / 2) + pr];
#pragma unroll
            for (int r = 0; r < 16; ++r) m2 = __vmaxu2(m2, w[r] & M);
            if (RHT_COLS) {
                float v[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) v[r] = bf16_lo(w[r]);
                m = max(m, rht16_absmax_bits_nan(v, mask));
#pragma unroll
                for (int r = 0; r < 16; ++r) v[r] = bf16_hi(w[r]);
                m = max(m, rht16_absmax_bits_nan(v, mask));
            }
        }
        __syncthreads();                              // slot s fully read
        if (threadIdx.x == 0) {
            const int64_t tn = t + (int64_t)kAmaxStages * gridDim.x;
            if (tn < ntiles) issue(tn, s);
        }
    }
    // drain: no copy may still be writing into this CTA's shared memory
    if (threadIdx.x == 0 && abort_flag) {
        for (int k = 0; k < kAmaxStages; ++k) {
            const int ii = i + k;
            const int64_t t = (int64_t)blockIdx.x + (int64_t)ii * gridDim.x;
            if (t < ntiles && ii < i + kAmaxStages) mbar_wait_bounded(&full[ii % kAmaxStages], (uint32_t)(ii / kAmaxStages) & 1u, nullptr);
        }
    }
    const uint32_t plain = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    block_max2_to_global(plain, out_plain, RHT_COLS ? m : plain, out_t);
}

}  // namespace nvfp4
