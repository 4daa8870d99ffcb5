// dual.cuh -- dual-axis kernels: one read of a stored bf16 tensor S [R x C]
// serves both GEMM views of it.
//
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
#include <cuda.h>
#include <cstdint>
#include <type_traits>
#include "codec.cuh"
#include "guard.cuh"
#include "ptx.cuh"
#include "quantize.cuh"
#include "status.cuh"

namespace nvfp4 {

// Block-wide maxima of two non-negative float bit patterns, merged into two
// outputs with one atomic each per CTA (at most 32 warps per CTA).
__device__ __forceinline__ void block_max2_to_global(uint32_t m0, float* out0, uint32_t m1, float* out1) {
    __shared__ uint32_t red[2][32];
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
            if (m0 && out0 != nullptr) atomicMax(reinterpret_cast<uint32_t*>(out0), m0);
            if (m1 && out1 != nullptr) atomicMax(reinterpret_cast<uint32_t*>(out1), m1);
        }
    }
}

// ======================================================== dual quantise ====
// Persistent CTAs walk 64-row x 256-column tiles of S through a ring of
// kDqStages shared-memory slots.  A tile arrives as four 64 x 64 boxes (one
// TMA copy each, 128-byte swizzle: 16-byte chunk c of row r of a box sits at
// chunk c ^ (r & 7)); rows and columns beyond S read as zeros.  Row tiles
// cover S's 128-padded row count, so that the padding rows' scale words are
// written too.
//  * warp 8 (one lane) feeds the ring: it refills slot s as soon as all eight
//    encoding warps have arrived on empty[s];
//  * warps 0-7 encode.  They wait for full[s] and release the slot each on
//    its own, never for one another, so they drift apart in phase and the
//    Philox (integer), Hadamard (FP32) and conversion work of different warps
//    overlap on the SM's pipes.
// Each encoding thread takes one item of each kind per tile:
//  * row-wise item (tile row r, group g of 4 blocks = box g): 16-byte reads;
//    the 8 lanes of a quarter warp read one chunk of 8 consecutive rows,
//    which the swizzle spreads over all banks;
//  * column-wise item (column pair, half h of the tile's rows = 2 blocks):
//    4-byte reads, a warp reading the 128 bytes of one box row.
// Both item kinds carry 64 elements.
struct DualArgs {
    QuantArgs row;      // logical S [R x C]: x, rows = R, k = C, ld; codes/scales of out
    QuantArgs col;      // logical S^T [C x R]: rows = C, k = R; codes/scales of out_t; rht
};

constexpr int kDqRows = 64, kDqCols = 256, kDqBoxCols = 64;
constexpr int kDqBoxBytes = kDqRows * kDqBoxCols * 2;            // 8 KB
constexpr int kDqTileBytes = (kDqCols / kDqBoxCols) * kDqBoxBytes;  // 32 KB
constexpr int kDqStages = 3;
constexpr int kDqConsumerWarps = 8;
constexpr int kDqThreads = (kDqConsumerWarps + 1) * 32;
constexpr int kDqSmem = kDqStages * kDqTileBytes + 1024 + 128;     // + 1024-byte alignment slack, barriers

// Byte offset of 16-byte chunk c of row r of box b in a tile slot.
__device__ __forceinline__ uint32_t dq_chunk(int b, int r, int c) {
    return (uint32_t)(b * kDqBoxBytes + r * 128 + ((c ^ (r & 7)) << 4));
}

// SR1, SR2: rounding of each operand, 0 = RNE, 1 = NVFP4_SR, 2 = NVFP4_SR_HW.
// PATHS: bit 0 = the row-wise operand, bit 1 = the column-wise operand; a
// single path makes the kernel the TMA-fed 1x16 quantiser of one view (rows:
// a non-transposed view, with RHT1 for the transform along its k; columns: a
// transposed view, whose stored array is S).
template <int SR1, int SR2, bool RHT2, int PATHS = 3, bool RHT1 = false>
__global__ void __launch_bounds__(kDqThreads, 2) k_quant_dual(const __grid_constant__ CUtensorMap map,
                                                              const __grid_constant__ DualArgs d) {
    extern __shared__ uint8_t dq_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dq_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kDqStages * kDqTileBytes);
    uint64_t* empty = full + kDqStages;
    __shared__ float rtab1[128], rtab2[128];
    __shared__ int abort_flag;
    const QuantArgs& a1 = d.row;
    const QuantArgs& a2 = d.col;
    float s1, s2;
    constexpr bool ROWS = (PATHS & 1) != 0, COLS = (PATHS & 2) != 0;
    const bool ok1 = ROWS && resolve_scale(a1.scale_src, a1.src_is_senc, a1.gs_out, a1.gs_out2, &s1);
    const bool ok2 = COLS && resolve_scale(a2.scale_src, a2.src_is_senc, a2.gs_out, a2.gs_out2, &s2);
    if (!ok1 && !ok2) return;                                    // uniform over the grid
    for (int c = threadIdx.x; c < 128; c += blockDim.x) {
        rtab1[c] = ok1 ? encode_factor(s1, (uint32_t)c) : 0.0f;
        rtab2[c] = ok2 ? encode_factor(s2, (uint32_t)c) : 0.0f;
    }
    const int64_t R = a1.rows, C = a1.k;
    const int64_t rows_pad = (R + 127) & ~int64_t(127);
    const int64_t row_tiles = rows_pad / kDqRows;
    const int64_t col_tiles = (C + kDqCols - 1) / kDqCols;
    const int64_t ntiles = row_tiles * col_tiles;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDqStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kDqConsumerWarps);
        }
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&map);
    }
    __syncthreads();

    if (warp == kDqConsumerWarps) {
        // ------------------------------------------------------ producer --
        if ((threadIdx.x & 31) == 0) {
            int i = 0;
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int s = i % kDqStages;
                if (i >= kDqStages &&
                    !mbar_wait_bounded(&empty[s], (uint32_t)(i / kDqStages - 1) & 1u, &abort_flag))
                    break;
                if (abort_flag) break;
                const int64_t tr = t / col_tiles, tc = t - tr * col_tiles;
                mbar_arrive_expect_tx(&full[s], kDqTileBytes);
#pragma unroll
                for (int b = 0; b < kDqCols / kDqBoxCols; ++b)
                    tma_load_2d(ring + s * kDqTileBytes + b * kDqBoxBytes, &map, &full[s],
                                (int32_t)(tc * kDqCols + b * kDqBoxCols), (int32_t)(tr * kDqRows));
            }
            // every issued copy has landed before the CTA exits: copies before
            // the last kDqStages were waited for by the encoding warps (their
            // slots were released), the last kDqStages are waited for here
            for (int k = 1; k <= kDqStages && i - k >= 0; ++k) {
                const int ii = i - k;
                mbar_wait_bounded(&full[ii % kDqStages], (uint32_t)(ii / kDqStages) & 1u, nullptr);
            }
        }
        return;
    }

    // per-thread item coordinates (fixed over tiles)
    const int ri = threadIdx.x;
    const int rr = (ri & 7) | ((ri >> 5) << 3);                  // row-wise: tile row 0..63
    const int rg = (ri >> 3) & 3;                                // row-wise: 64-column group = box
    const int pc = threadIdx.x & 127;                            // column-wise: column pair
    const int ch = threadIdx.x >> 7;                             // column-wise: 32-row half
    const int pb = pc >> 5, pchunk = (pc & 31) >> 2, pword = pc & 3;

    const int64_t nkb = C >> 4, ngroups = (nkb + 3) >> 2;        // row-wise operand
    const int64_t nkb_t = R >> 4, ngroups_t = (nkb_t + 3) >> 2;  // column-wise operand
    const int64_t rows_pad_t = (C + 127) & ~int64_t(127);

    // The encoding loop, instantiated twice: with G32 the Philox block
    // indices are known to stay below 2^32 (the usual case, decided once per
    // launch) and the counter's constant words come folded.
    auto encode_tiles = [&](auto g32) {
        constexpr bool G32 = decltype(g32)::value;
        int i = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int s = i % kDqStages;
            const uint32_t ph = (uint32_t)(i / kDqStages) & 1u;
            // warp-uniform outcome: a lane that timed out stops its whole warp
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], ph, &abort_flag))) break;
            const uint8_t* tile = ring + s * kDqTileBytes;
            const int64_t tr = t / col_tiles, tc = t - tr * col_tiles;
            const int64_t r0 = tr * kDqRows, c0 = tc * kDqCols;

            // ---- row-wise operand
            if (ROWS && ok1) {
                const int64_t row = r0 + rr;
                const int64_t G = c0 / 64 + rg;
                if (G < ngroups) {
                    uint32_t* sdst = reinterpret_cast<uint32_t*>(a1.scales + scale_offset(row, G * 4, ngroups));
                    const bool s_ok =
                        NVFP4_GUARD(a1.scales, scales_extent(a1.rows, a1.k), sdst, 4, kGuardDualScales);
                    if (row >= R) {
                        if (s_ok) *sdst = 0u;
                    } else {
                        const int nblk = (int)min64(4, nkb - G * 4);
                        uint32_t sw = 0, cw[8];
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            cw[2 * b] = cw[2 * b + 1] = 0u;
                            if (b < nblk) {
                                const uint4 lo = *reinterpret_cast<const uint4*>(tile + dq_chunk(rg, rr, 2 * b));
                                const uint4 hi = *reinterpret_cast<const uint4*>(tile + dq_chunk(rg, rr, 2 * b + 1));
                                float v[16];
                                unpack8(lo, v);
                                unpack8(hi, v + 8);
                                uint32_t sb;
                                encode_block16<RHT1, SR1 != 0, SR1 == 2, G32>(
                                    v, s1, rtab1, (uint64_t)(row * C + G * 64 + b * 16), a1, &sb, &cw[2 * b],
                                    &cw[2 * b + 1], RHT1 ? ~0u : absmax_bits16_packed(lo, hi));
                                sw |= sb << (8 * b);
                            }
                        }
                        uint8_t* cdst = a1.codes + row * (C >> 1) + G * 32;
                        if (!NVFP4_GUARD(a1.codes, codes_extent(a1.rows, a1.k), cdst, 8 * nblk, kGuardDualCodes)) {
                        } else if (nblk == 4 && (C & 31) == 0) {
                            reinterpret_cast<uint4*>(cdst)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                            reinterpret_cast<uint4*>(cdst)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                        } else {
#pragma unroll
                            for (int b = 0; b < 4; ++b)
                                if (b < nblk) reinterpret_cast<uint2*>(cdst)[b] = make_uint2(cw[2 * b], cw[2 * b + 1]);
                        }
                        if (s_ok) *sdst = sw;
                    }
                }
            }

            // ---- column-wise operand: logical rows cc, cc + 1 of S^T, blocks kb0, kb0 + 1
            if (COLS && ok2) {
                const int64_t cc = c0 + 2 * pc;
                const int64_t G = r0 / 64;
                const int64_t kb0 = G * 4 + 2 * ch;
                if (G < ngroups_t && cc < rows_pad_t) {
                    uint16_t* s0 = reinterpret_cast<uint16_t*>(a2.scales + scale_offset(cc, kb0, ngroups_t));
                    uint16_t* s1p = reinterpret_cast<uint16_t*>(a2.scales + scale_offset(cc + 1, kb0, ngroups_t));
                    const int nblk = (int)max64(0, min64(2, nkb_t - kb0));
                    const bool s0_ok = NVFP4_GUARD(a2.scales, scales_extent(a2.rows, a2.k), s0, 2, kGuardDualScalesT);
                    const bool s1_ok = NVFP4_GUARD(a2.scales, scales_extent(a2.rows, a2.k), s1p, 2, kGuardDualScalesT);
                    // cc is even: cc >= C makes both rows padding; with an odd C the
                    // last pair's second row (column C, read as zeros) is padding too
                    if (cc >= C || nblk == 0) {
                        if (s0_ok) *s0 = 0;
                        if (s1_ok) *s1p = 0;
                    } else {
                        uint32_t sw0 = 0, sw1 = 0, c0w[4], c1w[4];
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            c0w[2 * b] = c0w[2 * b + 1] = c1w[2 * b] = c1w[2 * b + 1] = 0u;
                            if (b < nblk) {
                                uint32_t w[16];
#pragma unroll
                                for (int u = 0; u < 16; ++u) {
                                    const int r = ch * 32 + b * 16 + u;
                                    w[u] = *reinterpret_cast<const uint32_t*>(tile + dq_chunk(pb, r, pchunk) + pword * 4);
                                }
                                const int64_t kc = (kb0 + b) * 16;
                                float v[16];
                                uint32_t sb;
#pragma unroll
                                for (int u = 0; u < 16; ++u) v[u] = bf16_lo(w[u]);
                                encode_block16<RHT2, SR2 != 0, SR2 == 2, G32>(v, s2, rtab2, (uint64_t)(cc * R + kc), a2,
                                                                              &sb, &c0w[2 * b], &c0w[2 * b + 1]);
                                sw0 |= sb << (8 * b);
#pragma unroll
                                for (int u = 0; u < 16; ++u) v[u] = bf16_hi(w[u]);
                                encode_block16<RHT2, SR2 != 0, SR2 == 2, G32>(v, s2, rtab2, (uint64_t)((cc + 1) * R + kc),
                                                                              a2, &sb, &c1w[2 * b], &c1w[2 * b + 1]);
                                sw1 |= sb << (8 * b);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            if (cc + q >= C) break;              // no codes for a padding row
                            const uint32_t* cw = q ? c1w : c0w;
                            uint8_t* cdst = a2.codes + (cc + q) * (R >> 1) + kb0 * 8;
                            if (!NVFP4_GUARD(a2.codes, codes_extent(a2.rows, a2.k), cdst, 8 * nblk, kGuardDualCodesT)) {
                            } else if (nblk == 2 && (R & 31) == 0) {
                                *reinterpret_cast<uint4*>(cdst) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                            } else {
#pragma unroll
                                for (int b = 0; b < 2; ++b)
                                    if (b < nblk) reinterpret_cast<uint2*>(cdst)[b] = make_uint2(cw[2 * b], cw[2 * b + 1]);
                            }
                        }
                        if (s0_ok) *s0 = (uint16_t)sw0;
                        if (s1_ok) *s1p = (uint16_t)sw1;
                    }
                }
            }
            __syncwarp();                                        // this warp is done with slot s
            if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[s]);
        }
    };
    if ((!ROWS || a1.sr_g32) && (!COLS || a2.sr_g32)) encode_tiles(std::true_type{});
    else encode_tiles(std::false_type{});
}

}  // namespace nvfp4

namespace nvfp4 {

// ============================================ streamed (TMA-fed) amax ======
// max |S| and (RHT_COLS) max |RHT16 down the columns of S| for a stored bf16
// array S [srows x scols], streamed through shared memory: persistent CTAs
// walk 64-row x 256-column tiles (32 KB, loaded by one 2D TMA copy; zeros
// beyond the array) through a ring of kAmaxStages slots.  Warp 8 (one lane)
// feeds the ring and refills a slot as soon as the 8 reducing warps have
// arrived on its empty barrier; the reducing warps never wait for one
// another.  A tile is 128 column pairs x 4 blocks of 16 rows; each thread
// reduces two (pair, block) items with conflict-free 4-byte reads (a warp
// reads 128 contiguous bytes of a tile row).
constexpr int kAmaxTileRows = 64, kAmaxTileCols = 256;
constexpr int kAmaxTileBytes = kAmaxTileRows * kAmaxTileCols * 2;
constexpr int kAmaxStages = 3;
constexpr int kAmaxConsumerWarps = 8;
constexpr int kAmaxThreads = (kAmaxConsumerWarps + 1) * 32;
constexpr int kAmaxSmem = kAmaxStages * kAmaxTileBytes + 128;

// fi_skip_tile >= 0 (test-only fault injection): that tile's copy is never
// issued, so its consumers' bounded wait expires and the kernel reports
// NVFP4_DEV_TIMEOUT instead of hanging.
template <bool RHT_COLS>
__global__ void __launch_bounds__(kAmaxThreads, 2) k_amax_stream(const __grid_constant__ CUtensorMap map,
                                                                 int64_t srows, int64_t scols, const RhtSigns sg,
                                                                 float* out_plain, float* out_t,
                                                                 int64_t fi_skip_tile) {
    extern __shared__ __align__(128) uint8_t amax_smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(amax_smem + kAmaxStages * kAmaxTileBytes);
    uint64_t* empty = full + kAmaxStages;
    __shared__ int abort_flag;
    const int64_t row_tiles = (srows + kAmaxTileRows - 1) / kAmaxTileRows;
    const int64_t col_tiles = (scols + kAmaxTileCols - 1) / kAmaxTileCols;
    const int64_t ntiles = row_tiles * col_tiles;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAmaxStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kAmaxConsumerWarps);
        }
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&map);
    }
    __syncthreads();
    constexpr uint32_t M = 0x7FFF7FFFu;
    uint32_t m2 = 0, m = 0;
    if (warp == kAmaxConsumerWarps) {
        // ------------------------------------------------------ producer --
        if ((threadIdx.x & 31) == 0) {
            int i = 0;
            bool issued[kAmaxStages] = {};
            for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int s = i % kAmaxStages;
                if (i >= kAmaxStages &&
                    !mbar_wait_bounded(&empty[s], (uint32_t)(i / kAmaxStages - 1) & 1u, &abort_flag))
                    break;
                if (abort_flag) break;
                issued[s] = t != fi_skip_tile;
                if (!issued[s]) continue;              // test-only: this tile is never copied
                const int64_t tr = t / col_tiles, tc = t - tr * col_tiles;
                mbar_arrive_expect_tx(&full[s], kAmaxTileBytes);
                tma_load_2d(amax_smem + s * kAmaxTileBytes, &map, &full[s], (int32_t)(tc * kAmaxTileCols),
                            (int32_t)(tr * kAmaxTileRows));
            }
            // every issued copy lands before the CTA exits: the last kAmaxStages
            // issues (earlier ones were waited for by the reducing warps)
            for (int k = 1; k <= kAmaxStages && i - k >= 0; ++k) {
                const int ii = i - k;
                if (issued[ii % kAmaxStages])
                    mbar_wait_bounded(&full[ii % kAmaxStages], (uint32_t)(ii / kAmaxStages) & 1u, nullptr);
            }
        }
    } else {
        const int pr = threadIdx.x & 127;             // column pair of the tile
        const int kb0 = threadIdx.x >> 7;             // blocks kb0 and kb0 + 2
        int i = 0;
        for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int s = i % kAmaxStages;
            const uint32_t ph = (uint32_t)(i / kAmaxStages) & 1u;
            // warp-uniform outcome: a lane that timed out stops its whole warp
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[s], ph, &abort_flag))) break;
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
                    m = max(m, rht16_absmax_bits_nan(v, sg));
#pragma unroll
                    for (int r = 0; r < 16; ++r) v[r] = bf16_hi(w[r]);
                    m = max(m, rht16_absmax_bits_nan(v, sg));
                }
            }
            __syncwarp();                             // this warp is done with slot s
            if ((threadIdx.x & 31) == 0) mbar_arrive(&empty[s]);
        }
    }
    const uint32_t plain = max(m2 & 0xFFFFu, m2 >> 16) << 16;
    block_max2_to_global(plain, out_plain, RHT_COLS ? m : plain, out_t);
}

}  // namespace nvfp4
