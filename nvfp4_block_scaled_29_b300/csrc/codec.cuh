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
// u16 < F = floor(frac * 2^16), frac = (|v| - lo) / (hi - lo).  Branch-free
// on the bit pattern of |v| (exponent e, 23-bit mantissa m):
//   |v| >= 1   : lo = 2^e * (1 + m22/2), code_lo = 2 (e + 1) + m22, and frac
//                is the 22 mantissa bits below m22, so F = bits 21..6;
//   0.5..1     : lo = 0.5, code_lo = 1, frac = m / 2^23, so F = bits 22..7;
//   |v| < 0.5  : lo = 0, code_lo = 0, frac = 2|v|, F = floor(|v| * 2^17)
//                (an exact power-of-two scaling);
//   |v| >= 6   : saturates to code 7.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t u16) {
    const uint32_t bits = __float_as_uint(v);
    const uint32_t sign = (bits >> 28) & 8u;
    const uint32_t ab = bits & 0x7FFFFFFFu;
    const uint32_t code_n = ((ab >> 23) - 126u) * 2u + ((ab >> 22) & 1u);
    const uint32_t f_n = (ab >> 6) & 0xFFFFu;
    const uint32_t f_h = (ab >> 7) & 0xFFFFu;
    const uint32_t f_s = (uint32_t)__fmul_rz(__uint_as_float(ab), 131072.0f);
    const bool ge1 = ab >= 0x3F800000u, ge05 = ab >= 0x3F000000u;
    uint32_t code = ge1 ? code_n : (ge05 ? 1u : 0u);
    const uint32_t F = ge1 ? f_n : (ge05 ? f_h : f_s);
    code += (u16 < F) ? 1u : 0u;
    code = (ab >= 0x40C00000u) ? 7u : code;
    return sign | code;
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
        const uint64_t p0 = (uint64_t)c.x * 0xD2511F53u;
        const uint64_t p1 = (uint64_t)c.z * 0xCD9E8D57u;
        c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1,
                       (uint32_t)p0);
    }
    return c;
}

// Random bits of the 8 elements idx = 8*g .. 8*g+7 of a quantised operand.
__device__ __forceinline__ uint4 sr_bits8(uint64_t g, uint64_t seed, uint64_t stream_id) {
    return philox4x32_10(make_uint4((uint32_t)g, (uint32_t)(g >> 32), (uint32_t)stream_id,
                                    (uint32_t)(stream_id >> 32)),
                         (uint32_t)seed, (uint32_t)(seed >> 32));
}

// Stochastic rounding realised as "add random bits below the kept precision,
// then truncate".  On [1, 6) the E2M1 grid is 2^e x {1, 1.5}: the kept bits
// are the exponent and mantissa bit 22, and the 16 bits below them hold
// floor(frac * 2^16).  Adding rp = 65535 - u16 there carries into the kept
// bits exactly when floor(frac * 2^16) > u16, i.e. the rule above.  Values
// below 1 (grid 0, 0.5, 1: spacing 0.5) are first moved to [1, 2) by a
// round-toward-zero add of 1.0 -- the truncation is below 2^-17, so
// floor(frac * 2^16) is unchanged -- and moved back by an exact subtraction.
// |v| is clamped to 8 first (anything >= 6 saturates to 6).  The result is
// the chosen grid value (exact, sign kept), so RNE conversion returns its
// code unchanged.
__device__ __forceinline__ float sr_grid_value(float v, uint32_t rp) {
    const uint32_t bits = __float_as_uint(v);
    const float a = fminf(fabsf(v), 8.0f);
    const bool lt1 = a < 1.0f;
    const float a2 = lt1 ? __fadd_rz(a, 1.0f) : a;
    uint32_t qb;
    asm("mad.lo.u32 %0, %1, 64, %2;" : "=r"(qb) : "r"(rp), "r"(__float_as_uint(a2)));
    float q = __uint_as_float(qb & 0xFFC00000u);
    q = __fsub_rn(q, lt1 ? 1.0f : 0.0f);
    return __uint_as_float(__float_as_uint(q) | (bits & 0x80000000u));
}

// Eight values -> eight SR codes (element 0 in the lowest nibble), r = the
// Philox block of these 8 elements (slice j: word j/2, low half first).
__device__ __forceinline__ uint32_t e2m1x8_sr(const float* v, uint4 r) {
    const uint32_t w[4] = {~r.x, ~r.y, ~r.z, ~r.w};      // both halves become 65535 - u16
    float g[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t rp = (j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu);
        g[j] = sr_grid_value(v[j], rp);
    }
    return e2m1x8_rne(g);
}

// -------------------------------------------------------------- RHT-16 ----
// y = H16 diag(s) x / 4 in place: sign flip, butterflies h = 1, 2, 4, 8,
// exact scaling by 1/4.  The sign flip is folded into the first butterfly
// stage as fused multiply-adds by +-1: fma(s_b, b, s_a * a) rounds
// s_a a + s_b b once, exactly like the separate negate-then-add.
__device__ __forceinline__ void rht16(float* v, uint32_t mask) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float sa = ((mask >> i) & 1u) ? -1.0f : 1.0f;
        const float sb = ((mask >> (i + 1)) & 1u) ? -1.0f : 1.0f;
        const float a = __fmul_rn(v[i], sa), b = v[i + 1];
        v[i] = __fmaf_rn(sb, b, a);
        v[i + 1] = __fmaf_rn(-sb, b, a);
    }
#pragma unroll
    for (int h = 2; h < 16; h <<= 1) {
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
