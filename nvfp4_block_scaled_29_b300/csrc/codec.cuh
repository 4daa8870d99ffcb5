// codec.cuh -- device-side number formats of the NVFP4 path (sm_103a).
//
// E2M1 element codes, E4M3 block scales, Philox4x32-10 stochastic-rounding
// bits and the in-register 16-point random Hadamard transform.  The numeric
// rules are those stated in include/nvfp4.h; every float operation that
// decides a code is a single IEEE binary32 operation (explicit __f*_rn
// intrinsics, no contraction, no flush-to-zero), so the results are
// reproducible bit for bit by any implementation that follows the same rules.
//
// Sources: NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and Speed and
// Efficiency of 4-Bit", recipe bullets 1-5 (micro-blocks, E4M3 scales,
// Hadamard transform, 2D weight blocks, stochastic rounding); prism.simon-ai.net
// article 7890, sections on the FP32 global scale and on stochastic rounding;
// Salmon et al., SC'11, for Philox4x32-10.
#pragma once
#include <cstdint>
#include <cfloat>

namespace nvfp4 {

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// ---------------------------------------------------------------- bf16 ----
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ----------------------------------------------------------- global scale --
// S_enc = 2688 / amax (448 * 6), 1 for amax == 0, FLT_MAX on overflow.
// Returns false when amax is not finite.
__device__ __forceinline__ bool global_encode_scale(float amax, float* s_enc) {
    if (!(fabsf(amax) <= FLT_MAX)) return false;   // NaN or Inf
    if (amax == 0.0f) { *s_enc = 1.0f; return true; }
    float s = __fdiv_rn(2688.0f, amax);
    if (s > FLT_MAX) s = FLT_MAX;
    *s_enc = s;
    return true;
}

// ------------------------------------------------------------------ E4M3 --
// t >= 0 -> E4M3 code, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_rne_satfinite(float t) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
    return r & 0xFFu;
}

// non-negative finite E4M3 code -> value (exact)
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0) return __fmul_rn((float)m, 0.001953125f);          // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Block decode scale and encode factor from the block amax.
__device__ __forceinline__ uint32_t block_scale(float amax_b, float s_enc, float* r_b) {
    float t = __fdiv_rn(amax_b, 6.0f);
    t = __fmul_rn(t, s_enc);
    uint32_t sb = e4m3_rne_satfinite(t);
    float sbv = e4m3_value(sb);
    float r = 0.0f;
    if (sbv != 0.0f) {
        r = __fdiv_rn(s_enc, sbv);
        if (r > FLT_MAX) r = FLT_MAX;
    }
    *r_b = r;
    return sb;
}

// ------------------------------------------------------------------ E2M1 --
// Eight floats -> eight RNE E2M1 codes, element 0 in the lowest nibble.
// cvt ...e2m1x2 d, a, b puts a in the high and b in the low nibble.
__device__ __forceinline__ uint32_t e2m1x8_rne(const float* v) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// Stochastic E2M1 rounding of one value with 16 random bits.  With lo <= |v|
// < hi the neighbouring grid values, the code moves up iff
// u16 < floor(frac * 2^16), frac = (|v| - lo) / (hi - lo).  Every step is
// exact: |v| - lo by Sterbenz (or lo == 0), the spacing is a power of two.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t u16) {
    uint32_t sign = (__float_as_uint(v) >> 28) & 8u;
    float a = fabsf(v);
    if (a >= 6.0f) return sign | 7u;
    uint32_t code;
    float lo, inv_step;
    if (a < 2.0f) {                    // grid 0, 0.5, 1, 1.5, (2): spacing 0.5
        code = (uint32_t)__fmul_rz(a, 2.0f);
        lo = __fmul_rn((float)code, 0.5f);
        inv_step = 2.0f;
    } else if (a < 4.0f) {             // grid 2, 3, (4): spacing 1
        uint32_t f = (uint32_t)a;
        code = f + 2u;
        lo = (float)f;
        inv_step = 1.0f;
    } else {                           // grid 4, 6: spacing 2
        code = 6u;
        lo = 4.0f;
        inv_step = 0.5f;
    }
    float frac = __fmul_rn(__fsub_rn(a, lo), inv_step);
    uint32_t F = (uint32_t)__fmul_rz(frac, 65536.0f);
    return sign | (code + (u16 < F ? 1u : 0u));
}

// ---------------------------------------------------------------- Philox --
// Philox4x32-10 (Salmon et al., SC'11): multipliers 0xD2511F53, 0xCD9E8D57,
// key increments 0x9E3779B9, 0xBB67AE85.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// Random bits of the 8 elements idx = 8*g .. 8*g+7 of a quantised operand.
__device__ __forceinline__ uint4 sr_bits8(uint64_t g, uint64_t seed, uint64_t stream_id) {
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), (uint32_t)stream_id,
                                    (uint32_t)(stream_id >> 32)),
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}

// Eight values -> eight SR codes (element 0 in the lowest nibble), r = the
// Philox block of these 8 elements.
__device__ __forceinline__ uint32_t e2m1x8_sr(const float* v, uint4 r) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t u = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu);
        out |= e2m1_sr(v[j], u) << (4 * j);
    }
    return out;
}

// -------------------------------------------------------------- RHT-16 ----
// y = H16 diag(s) x / 4 in place: sign flip, butterflies h = 1, 2, 4, 8,
// exact scaling by 1/4.
__device__ __forceinline__ void rht16(float* v, uint32_t mask) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
        v[j] = __uint_as_float(__float_as_uint(v[j]) ^ (((mask >> j) & 1u) << 31));
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            const float a = v[i], b = v[i + h];
            v[i] = __fadd_rn(a, b);
            v[i + h] = __fsub_rn(a, b);
        }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __fmul_rn(v[j], 0.25f);
}

// ------------------------------------------------------- scale layout -----
// Byte offset of (row, block column) in the swizzled scale layout.
__device__ __forceinline__ int64_t scale_offset(int64_t row, int64_t col, int64_t col_tiles) {
    return ((row >> 7) * col_tiles + (col >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 +
           (col & 3);
}

}  // namespace nvfp4
