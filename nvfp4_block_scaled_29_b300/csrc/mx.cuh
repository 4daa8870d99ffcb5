// mx.cuh -- MXFP4 quantisation and dequantisation: the comparison format of
// the NVFP4 recipe.
//
// MXFP4 (NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and Speed and
// Efficiency of 4-Bit", recipe bullets 1-2; prism.simon-ai.net article 7890,
// "MVFP4 and MXFP4" and "Core architectural changes of the MVFP4 format"):
// E2M1 elements, one power-of-two (E8M0) scale per 32 elements, no tensor
// scale.  The scale rule (the pages give none): block exponent
// X = floor(log2(amax_b)) - 2, the exponent of E2M1's largest value 6 = 1.5 *
// 2^2, clamped to [-127, 127]; for a float amax_b with biased exponent field
// E that is the E8M0 code max(E - 2, 0).  Elements v = fp32(x * 2^-X), RNE to
// E2M1 with saturation (the block's largest element lands in [4, 8), so
// values above 6 * 2^X clip).  An optional 16-point RHT transforms each
// 16-chunk along k first (two per block).
//
// Scales are stored in the block-scaled MMA layout with 32-element blocks:
// 512-byte tiles of 128 rows x 4 scales (128 k), read by kind::mxf4 with
// scale_vec::2X.
#pragma once
#include <cstdint>
#include "codec.cuh"
#include "guard.cuh"
#include "quantize.cuh"
#include "status.cuh"

namespace nvfp4 {

struct MxArgs {
    const uint16_t* x;
    int64_t rows, k, ld;       // logical [rows x k] = stored (non-transposed view)
    uint8_t* codes;            // [rows x k/2]
    uint8_t* scales;           // swizzled E8M0, 32-element blocks
    RhtSigns rht;              // RHT-16 sign multipliers (RHT variant only)
};

// E8M0 code of a block from its max |value| as float bits; 0xFF (NaN) for a
// non-finite block.
__device__ __forceinline__ uint32_t mx_scale_code(uint32_t amax_bits) {
    const uint32_t e = (amax_bits >> 23) & 0xFFu;
    if (e == 0xFFu) return 0xFFu;
    return e >= 2u ? e - 2u : 0u;
}

// 2^-X for E8M0 code X + 127 (code <= 252 for any finite block): exponent
// field 254 - code, always a normal float.
__device__ __forceinline__ float mx_inv_scale(uint32_t code) {
    return __uint_as_float((254u - code) << 23);
}

// Thread item: (row, group of 2 blocks = 64 elements): 8 x 16-byte loads,
// 32 bytes of codes and one 16-bit word of scales (the two blocks' scales are
// adjacent in the MMA layout).  Groups run to a whole 4-block scale tile so
// that the tile's padding bytes are written as 0.
template <bool RHT>
__global__ void __launch_bounds__(kQuantThreads, RHT ? 2 : 3) k_mx_quant_rows(const MxArgs a) {
    const int64_t nb = a.k >> 5;                                  // 32-element blocks per row
    const int64_t col_tiles = (nb + 3) >> 2;
    const uint32_t ngroups = (uint32_t)(col_tiles * 2);
    const int64_t rows_pad = (a.rows + 127) & ~int64_t(127);
    bool bad = false;
    for (ItemWalk w(ngroups); w.major < rows_pad; w.next()) {
        const int64_t r = w.major;
        const int64_t g = w.minor;
        uint16_t* sdst = reinterpret_cast<uint16_t*>(a.scales + scale_offset(r, g * 2, col_tiles));
        const int nblk = (int)min64(2, nb - g * 2);
        const bool s_ok = NVFP4_GUARD(a.scales, mx_scales_extent(a.rows, a.k), sdst, 2, kGuardMxScales);
        if (r >= a.rows || nblk <= 0) {
            if (s_ok) *sdst = 0;
            continue;
        }
        const uint4* src = reinterpret_cast<const uint4*>(a.x + r * a.ld + g * 64);
        const bool x_ok = NVFP4_GUARD(a.x, stored_extent(a.rows, a.k, a.ld, 2), src, 64 * nblk, kGuardMxX);
        uint4 raw[8];
#pragma unroll
        for (int b = 0; b < 2; ++b)
            if (b < nblk) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    raw[4 * b + q] = x_ok ? ldg_stream(src + 4 * b + q) : make_uint4(0, 0, 0, 0);
            }
        uint32_t sw = 0, cw[8];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
#pragma unroll
            for (int q = 0; q < 4; ++q) cw[4 * b + q] = 0u;
            if (b < nblk) {
                float v[32];
#pragma unroll
                for (int q = 0; q < 4; ++q) unpack8(raw[4 * b + q], v + 8 * q);
                // block max |value| as float bits by integer maxima of the
                // magnitude bit patterns, so that a NaN or Inf element (there
                // is no tensor amax to catch it) gives exponent field 0xFF
                uint32_t amax_bits;
                if (RHT) {
                    uint32_t m = 0;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        rht16_first3(v + 16 * h, a.rht);
                        float s[8];
                        rht16_pair_mags(v + 16 * h, s);
#pragma unroll
                        for (int i = 0; i < 8; ++i) m = max(m, __float_as_uint(s[i]));
                        rht16_last(v + 16 * h);
                    }
                    // max |y| = fp32(max pair magnitude * 1/4) (see rht16_pair_mags)
                    amax_bits = m >= 0x7F800000u ? m : __float_as_uint(__fmul_rn(__uint_as_float(m), 0.25f));
                } else {
                    constexpr uint32_t M = 0x7FFF7FFFu;
                    uint32_t m2 = 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 w = raw[4 * b + q];
                        m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(w.x & M, w.y & M), __vmaxu2(w.z & M, w.w & M)));
                    }
                    amax_bits = max(m2 & 0xFFFFu, m2 >> 16) << 16;
                }
                const uint32_t sc = mx_scale_code(amax_bits);
                if (sc == 0xFFu) bad = true;
                const float inv = mx_inv_scale(sc == 0xFFu ? 127u : sc);
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __fmul_rn(v[j], inv);
#pragma unroll
                for (int q = 0; q < 4; ++q) cw[4 * b + q] = e2m1x8_rne(v + 8 * q);
                sw |= sc << (8 * b);
            }
        }
        uint8_t* cdst = a.codes + r * (a.k >> 1) + g * 32;
        if (!NVFP4_GUARD(a.codes, codes_extent(a.rows, a.k), cdst, 16 * nblk, kGuardMxCodes)) {
        } else if (nblk == 2 && (a.k & 31) == 0 && ((r * (a.k >> 1)) & 15) == 0) {
            reinterpret_cast<uint4*>(cdst)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
            reinterpret_cast<uint4*>(cdst)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        } else {
#pragma unroll
            for (int b = 0; b < 2; ++b)
                if (b < nblk) {
                    reinterpret_cast<uint2*>(cdst)[2 * b] = make_uint2(cw[4 * b], cw[4 * b + 1]);
                    reinterpret_cast<uint2*>(cdst)[2 * b + 1] = make_uint2(cw[4 * b + 2], cw[4 * b + 3]);
                }
        }
        if (s_ok) *sdst = (uint16_t)sw;
    }
    if (bad) record_device_error(NVFP4_DEV_NONFINITE);
}

// x_hat = q * 2^X (exact) as fp32 or bf16 (RNE); the codes are decoded
// exactly (times an f16 one) and scaled in fp32.
template <bool BF16>
__global__ void __launch_bounds__(kQuantThreads) k_mx_dequant(const uint8_t* __restrict__ codes,
                                                              const uint8_t* __restrict__ scales,
                                                              int64_t rows, int64_t k, void* out, int64_t ld) {
    dequant_walk<BF16, 32>(codes, scales, mx_scales_extent(rows, k), rows, k, out, ld, kGuardMxDeqIn,
                           kGuardMxDeqOut, [](uint32_t cw, uint32_t sc, float* o) {
                               e2m1x8_times_scale(cw, 0x3C003C00u, o);                 // f16x2 (1, 1)
                               // 2^(sc - 127); code 0 is 2^-127 (subnormal), 0xFF NaN
                               const float s = sc == 0xFFu ? __int_as_float(0x7FC00000)
                                               : sc == 0u  ? 0x1p-127f
                                                           : __uint_as_float(sc << 23);
#pragma unroll
                               for (int j = 0; j < 8; ++j) o[j] = __fmul_rn(o[j], s);
                           });
}

}  // namespace nvfp4
