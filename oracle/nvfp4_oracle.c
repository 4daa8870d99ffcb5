/*
 * nvfp4_oracle.c -- plain scalar CPU oracle of the NVFP4 linear-layer path.
 *
 * TEST INFRASTRUCTURE ONLY (see nvfp4_oracle.h for the rule and citations).
 * Built with -O2 -ffp-contract=off, no fast-math: every float operation
 * below is one IEEE-754 binary32 (or binary64 where stated) operation with
 * round-to-nearest-even, in the order written.
 *
 * Every step follows the method in the order the sources give it:
 *   1. per-tensor amax                         ([SAI] two-level scale)
 *   2. optional 16-point random Hadamard       ([NVB] bullet 3, [SAI] outliers)
 *   3. global encode scale S_enc = 448*6/amax  ([SAI] global FP32 scale)
 *   4. per-block E4M3 decode scale             ([NVB] bullets 1-2, [SAI])
 *   5. per-element E2M1 code, RNE or stochastic ([NVB] bullet 5, [SAI] 0.3 example)
 *   6. 16x16 weight blocks                     ([NVB] bullet 4, [SAI] 16x16 / 256 values)
 *   7. dequantisation and an FP64 GEMM reference.
 */
#include "nvfp4_oracle.h"
#include <float.h>
#include <math.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* E2M1: sign bit + 3-bit magnitude index into {0,.5,1,1.5,2,3,4,6}.        */
/* The magnitude table is the FP4 E2M1 value set (1 sign, 2 exponent, 1      */
/* mantissa bit, bias 1, one subnormal 0.5); 16 codes in total.              */
/* ------------------------------------------------------------------------ */
static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(uint8_t code) {
    double m = kE2M1Mag[code & 7u];
    return (code & 8u) ? -m : m;
}

/* Nearest representable magnitude by enumeration; on an exact tie the code
 * with an even mantissa bit (even code index) wins.  Magnitudes above 6
 * saturate to 6.  The sign of v (including -0) becomes the sign bit.       */
uint8_t orc_e2m1_rne(float v) {
    double a = fabs((double)v);
    uint8_t sign = signbit(v) ? 8u : 0u;
    if (a >= 6.0) return (uint8_t)(sign | 7u);
    int best = 0;
    double best_d = a;                       /* distance to code 0 (value 0) */
    for (int c = 1; c < 8; ++c) {
        double d = fabs(a - kE2M1Mag[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)(sign | (uint8_t)best);
}

/* Stochastic rounding: with lo <= |v| < hi the two neighbouring grid values,
 * round up with probability (|v|-lo)/(hi-lo).  The probability is realised
 * with 16 random bits: F = floor(frac * 2^16), up iff u16 < F.  frac is exact
 * in binary64 (|v| has 24 significant bits, hi-lo is a power of two).
 * Magnitudes of 6 and above saturate to 6; the sign of v (including -0) is
 * kept.                                                                    */
uint8_t orc_e2m1_sr(float v, uint32_t u16) {
    double a = fabs((double)v);
    uint8_t sign = signbit(v) ? 8u : 0u;
    if (a >= 6.0) return (uint8_t)(sign | 7u);
    int lo = 0;
    for (int c = 1; c < 8; ++c)
        if (kE2M1Mag[c] <= a) lo = c;
    double frac = (a - kE2M1Mag[lo]) / (kE2M1Mag[lo + 1] - kE2M1Mag[lo]);
    uint32_t F = (uint32_t)floor(frac * 65536.0);
    int code = ((u16 & 0xFFFFu) < F) ? lo + 1 : lo;
    return (uint8_t)(sign | (uint8_t)code);
}

/* ------------------------------------------------------------------------ */
/* E4M3 (FP8: 1 sign, 4 exponent bits bias 7, 3 mantissa bits, no infinity, */
/* 0x7F/0xFF NaN).  Value of a non-negative code by its definition.          */
/* ------------------------------------------------------------------------ */
float orc_e4m3_value(uint8_t code) {
    int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

/* Nearest of the 127 finite non-negative codes 0x00..0x7E by enumeration,
 * ties to the even code, anything above the largest finite value 448
 * saturates to 448 (code 0x7E).  t must be >= 0 and not NaN.  The values of
 * the codes are tabulated once, from orc_e4m3_value, when the library loads. */
static double g_e4m3_pos[0x7F];

__attribute__((constructor)) static void init_e4m3_table(void) {
    for (int c = 0; c < 0x7F; ++c) g_e4m3_pos[c] = (double)orc_e4m3_value((uint8_t)c);
}

uint8_t orc_e4m3_rne_satfinite(float t) {
    double a = (double)t;
    if (a >= 448.0) return 0x7E;
    int best = 0;
    double best_d = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double d = fabs(a - g_e4m3_pos[c]);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_d = d;
        }
    }
    return (uint8_t)best;
}

float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bfloat16 with round-to-nearest-even on the 16 dropped bits.  */
uint16_t orc_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if (isnan(f)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t hi = u >> 16, lo = u & 0xFFFFu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
    return (uint16_t)hi;
}

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 [PHX]: 10 rounds of the 4x32 Philox S-box with the paper's  */
/* multipliers and Weyl key increments.  One round maps                      */
/*   (c0,c1,c2,c3) -> (hi(M1*c2)^c1^k0, lo(M1*c2), hi(M0*c0)^c3^k1, lo(M0*c0)) */
/* with M0 = 0xD2511F53, M1 = 0xCD9E8D57; between rounds the key advances by  */
/* (0x9E3779B9, 0xBB67AE85).                                                 */
/* ------------------------------------------------------------------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

uint32_t orc_rht_mask_from_seed(uint64_t seed) {
    uint32_t ctr[4] = {0, 0, 0, 0};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    return o[0] & 0xFFFFu;
}

/* Element idx draws the (idx mod 8)-th 16-bit slice of the 128-bit output
 * of Philox(counter = (idx/8, stream_id), key = seed): word (idx%8)/2, low
 * half for even idx, high half for odd.                                     */
uint32_t orc_sr_bits16(uint64_t seed, uint64_t stream_id, uint64_t idx) {
    uint64_t g = idx >> 3;
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), (uint32_t)stream_id,
                       (uint32_t)(stream_id >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    uint32_t w = o[(idx & 7u) >> 1];
    return (idx & 1u) ? (w >> 16) : (w & 0xFFFFu);
}

/* Second layout (rounding mode 2): the layout in which the Blackwell FP4
 * stochastic-rounding conversion reads its 32 random bits for four values.
 * The word's bytes b3 b2 b1 b0 form two 16-bit integers, H = (b3, b1) and
 * L = (b2, b0) (first byte high); the four elements take r = L, L with its
 * 16 bits in reverse order, H, and H reversed, and round up iff
 * floor(frac * 2^16) + r >= 2^16, i.e. iff (65535 - r) < floor(frac * 2^16):
 * the u16 rule above with u16 = 65535 - r.  Each map from the 16 bits an
 * element reads to r is a bijection, so u16 is uniform when the word is.   */
static uint32_t rev16(uint32_t x) {
    uint32_t r = 0;
    for (int i = 0; i < 16; ++i) r |= ((x >> i) & 1u) << (15 - i);
    return r;
}

uint32_t orc_sr_r16_of_word(uint32_t w, int p) {
    uint32_t H = ((w >> 24) & 0xFFu) << 8 | ((w >> 8) & 0xFFu);
    uint32_t L = ((w >> 16) & 0xFFu) << 8 | (w & 0xFFu);
    switch (p & 3) {
        case 0: return L;
        case 1: return rev16(L);
        case 2: return H;
        default: return rev16(H);
    }
}

/* Element idx (mode 2) draws from the 128-bit output of Philox(counter =
 * (idx/16, stream_id), key = seed): word (idx%16)/4, element position idx%4
 * within that word; returned as the u16 of the rule above.                 */
uint32_t orc_sr_bits16_hw(uint64_t seed, uint64_t stream_id, uint64_t idx) {
    uint64_t g = idx >> 4;
    uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), (uint32_t)stream_id,
                       (uint32_t)(stream_id >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t o[4];
    orc_philox4x32_10(ctr, key, o);
    return 65535u - orc_sr_r16_of_word(o[(idx & 15u) >> 2], (int)(idx & 3u));
}

/* ------------------------------------------------------------------------ */
/* 16-point random Hadamard transform: y = H16 * diag(s) * x / 4, H16 the    */
/* Sylvester Hadamard matrix, s_j = -1 where bit j of the mask is set.       */
/* Evaluated as: sign flip; butterfly stages h = 1, 2, 4, 8 with             */
/* (a, b) -> (a + b, a - b) in binary32; then an exact scaling by 1/4.       */
/* ------------------------------------------------------------------------ */
void orc_rht16(const float in[16], uint32_t mask, float out[16]) {
    float y[16];
    for (int j = 0; j < 16; ++j) y[j] = ((mask >> j) & 1u) ? -in[j] : in[j];
    for (int h = 1; h < 16; h <<= 1) {
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            float a = y[i], b = y[i + h];
            y[i] = a + b;
            y[i + h] = a - b;
        }
    }
    for (int j = 0; j < 16; ++j) out[j] = y[j] * 0.25f;
}

/* element (r, c) of the logical [rows x k] operand */
static float load_elem(const uint16_t* x, int64_t ld, int transposed, int64_t r, int64_t c) {
    return orc_bf16_to_f32(transposed ? x[c * ld + r] : x[r * ld + c]);
}

/* the 16 (optionally transformed) values of row r, k-block kb */
static void load_block16(const uint16_t* x, int64_t ld, int transposed, uint32_t rht_mask,
                         int64_t r, int64_t kb, float v[16]) {
    float raw[16];
    for (int j = 0; j < 16; ++j) raw[j] = load_elem(x, ld, transposed, r, kb * 16 + j);
    if (rht_mask) orc_rht16(raw, rht_mask, v);
    else memcpy(v, raw, sizeof(raw));
}

/* ------------------------------------------------------------------------ */
/* Step 1: amax = max |x| (NaN if any element is NaN).                        */
/* ------------------------------------------------------------------------ */
float orc_amax(const uint16_t* x, int64_t rows, int64_t k, int64_t ld, int transposed,
               uint32_t rht_mask) {
    float amax = 0.0f;
    int saw_nan = 0;
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t kb = 0; kb < k / 16; ++kb) {
            float v[16];
            load_block16(x, ld, transposed, rht_mask, r, kb, v);
            for (int j = 0; j < 16; ++j) {
                if (isnan(v[j])) saw_nan = 1;
                else if (fabsf(v[j]) > amax) amax = fabsf(v[j]);
            }
        }
    }
    return saw_nan ? NAN : amax;
}

/* ------------------------------------------------------------------------ */
/* Step 3: global encode scale.                                               */
/* ------------------------------------------------------------------------ */
int orc_global_scale(float amax, float* s_enc) {
    if (!isfinite(amax)) {
        *s_enc = NAN;
        return -1;
    }
    if (amax == 0.0f) {
        *s_enc = 1.0f;
        return 0;
    }
    float s = 2688.0f / amax;          /* 2688 = 448 (E4M3 max) * 6 (E2M1 max) */
    if (!isfinite(s)) s = FLT_MAX;
    *s_enc = s;
    return 0;
}

/* Step 4: decode scale from a block amax, and the per-block encode factor. */
static uint8_t block_scale(float amax_b, float s_enc, float* r_b) {
    float t = amax_b / 6.0f;
    t = t * s_enc;
    uint8_t sb = orc_e4m3_rne_satfinite(t);
    float sbv = orc_e4m3_value(sb);
    if (sbv == 0.0f) {
        *r_b = 0.0f;
    } else {
        float r = s_enc / sbv;
        if (!isfinite(r)) r = FLT_MAX;
        *r_b = r;
    }
    return sb;
}

/* Step 5: one element. */
static uint8_t encode_elem(float x, float r_b, int round, uint64_t seed, uint64_t stream_id,
                           uint64_t idx) {
    float v = x * r_b;
    if (round == 0) return orc_e2m1_rne(v);
    if (round == 2) return orc_e2m1_sr(v, orc_sr_bits16_hw(seed, stream_id, idx));
    return orc_e2m1_sr(v, orc_sr_bits16(seed, stream_id, idx));
}

static void put_code(uint8_t* codes, int64_t k, int64_t r, int64_t c, uint8_t q) {
    uint8_t* p = codes + r * (k / 2) + c / 2;
    if (c & 1) *p = (uint8_t)((*p & 0x0Fu) | (q << 4));
    else       *p = (uint8_t)((*p & 0xF0u) | q);
}

int orc_quantize(const uint16_t* x, int64_t rows, int64_t k, int64_t ld, int transposed,
                 uint32_t rht_mask, int block2d, float amax, int round,
                 uint64_t seed, uint64_t stream_id,
                 int64_t row_begin, int64_t row_end,
                 uint8_t* codes, uint8_t* scales_plain) {
    float s_enc;
    if (orc_global_scale(amax, &s_enc) != 0) return -1;
    const int64_t nkb = k / 16;
    if (!block2d) {
        for (int64_t r = row_begin; r < row_end; ++r) {
            for (int64_t kb = 0; kb < nkb; ++kb) {
                float v[16];
                load_block16(x, ld, transposed, rht_mask, r, kb, v);
                float amax_b = 0.0f;
                for (int j = 0; j < 16; ++j)
                    if (fabsf(v[j]) > amax_b) amax_b = fabsf(v[j]);
                float r_b;
                uint8_t sb = block_scale(amax_b, s_enc, &r_b);
                scales_plain[r * nkb + kb] = sb;
                for (int j = 0; j < 16; ++j) {
                    int64_t c = kb * 16 + j;
                    put_code(codes, k, r, c,
                             encode_elem(v[j], r_b, round, seed, stream_id, (uint64_t)(r * k + c)));
                }
            }
        }
        return 0;
    }
    /* 16x16 blocks: 16 logical rows x 16 k-columns share one scale. */
    for (int64_t r0 = row_begin; r0 < row_end; r0 += 16) {
        int64_t r1 = r0 + 16 < rows ? r0 + 16 : rows;
        for (int64_t kb = 0; kb < nkb; ++kb) {
            float amax_b = 0.0f;
            for (int64_t r = r0; r < r1; ++r) {
                float v[16];
                load_block16(x, ld, transposed, rht_mask, r, kb, v);
                for (int j = 0; j < 16; ++j)
                    if (fabsf(v[j]) > amax_b) amax_b = fabsf(v[j]);
            }
            float r_b;
            uint8_t sb = block_scale(amax_b, s_enc, &r_b);
            for (int64_t r = r0; r < r1; ++r) {
                float v[16];
                load_block16(x, ld, transposed, rht_mask, r, kb, v);
                scales_plain[r * nkb + kb] = sb;
                for (int j = 0; j < 16; ++j) {
                    int64_t c = kb * 16 + j;
                    put_code(codes, k, r, c,
                             encode_elem(v[j], r_b, round, seed, stream_id, (uint64_t)(r * k + c)));
                }
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Swizzled scale layout read by the block-scaled GEMM: rows padded to 128, */
/* scale columns padded to 4.  Tile (row/128, col/4) is 512 bytes; tiles of */
/* one 128-row group are consecutive along the scale columns.  Inside a      */
/* tile, row r and column c sit at (r%32)*16 + ((r/32)%4)*4 + (c%4).          */
/* ------------------------------------------------------------------------ */
static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t orc_scale_bytes(int64_t rows, int64_t k) {
    int64_t row_tiles = ceil_div(rows, 128);
    int64_t col_tiles = ceil_div(k / 16, 4);
    return (size_t)(row_tiles * col_tiles * 512);
}

static int64_t swz_offset(int64_t r, int64_t c, int64_t col_tiles) {
    int64_t tile = (r / 128) * col_tiles + c / 4;
    return tile * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
}

void orc_swizzle_scales(const uint8_t* plain, int64_t rows, int64_t k, uint8_t* swz) {
    int64_t nkb = k / 16, col_tiles = ceil_div(nkb, 4);
    memset(swz, 0, orc_scale_bytes(rows, k));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < nkb; ++c)
            swz[swz_offset(r, c, col_tiles)] = plain[r * nkb + c];
}

void orc_unswizzle_scales(const uint8_t* swz, int64_t rows, int64_t k, uint8_t* plain) {
    int64_t nkb = k / 16, col_tiles = ceil_div(nkb, 4);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < nkb; ++c)
            plain[r * nkb + c] = swz[swz_offset(r, c, col_tiles)];
}

static uint8_t get_code(const uint8_t* codes, int64_t k, int64_t r, int64_t c) {
    uint8_t b = codes[r * (k / 2) + c / 2];
    return (c & 1) ? (uint8_t)(b >> 4) : (uint8_t)(b & 0x0Fu);
}

void orc_transpose_codes(const uint8_t* codes, int64_t rows, int64_t k, uint8_t* codes_t) {
    memset(codes_t, 0, (size_t)(k * (rows / 2)));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < k; ++c)
            put_code(codes_t, rows, c, r, get_code(codes, k, r, c));
}

/* ------------------------------------------------------------------------ */
/* Dequantisation: x_hat = fp32(fp32(q * s_b) * fp32(1 / S_enc)).            */
/* ------------------------------------------------------------------------ */
void orc_dequantize(const uint8_t* codes, const uint8_t* scales_swz, float s_enc,
                    int64_t rows, int64_t k, int64_t row_begin, int64_t row_end,
                    void* out, int out_is_bf16, int64_t ld) {
    int64_t col_tiles = ceil_div(k / 16, 4);
    float inv = 1.0f / s_enc;
    for (int64_t r = row_begin; r < row_end; ++r) {
        for (int64_t c = 0; c < k; ++c) {
            float q = (float)orc_e2m1_value(get_code(codes, k, r, c));
            float sb = orc_e4m3_value(scales_swz[swz_offset(r, c / 16, col_tiles)]);
            float p = q * sb;
            float v = p * inv;
            if (out_is_bf16) ((uint16_t*)out)[r * ld + c] = orc_f32_to_bf16_rne(v);
            else             ((float*)out)[r * ld + c] = v;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* GEMM reference: exact products in binary64, binary64 accumulation in k   */
/* order, one division by S_A * S_B (binary64) at the end.                   */
/* ------------------------------------------------------------------------ */
static void dot_point(const uint8_t* qa, const uint8_t* sa_swz, const uint8_t* qb,
                      const uint8_t* sb_swz, int64_t k, int64_t m, int64_t n,
                      double inv_scale, double* y, double* abs_sum) {
    int64_t col_tiles = ceil_div(k / 16, 4);
    double acc = 0.0, acc_abs = 0.0;
    for (int64_t c = 0; c < k; ++c) {
        double a = orc_e2m1_value(get_code(qa, k, m, c)) *
                   (double)orc_e4m3_value(sa_swz[swz_offset(m, c / 16, col_tiles)]);
        double b = orc_e2m1_value(get_code(qb, k, n, c)) *
                   (double)orc_e4m3_value(sb_swz[swz_offset(n, c / 16, col_tiles)]);
        acc += a * b;
        acc_abs += fabs(a * b);
    }
    *y = acc * inv_scale;
    *abs_sum = acc_abs * inv_scale;
}

void orc_gemm_points(const uint8_t* qa, const uint8_t* sa_swz, float s_a,
                     const uint8_t* qb, const uint8_t* sb_swz, float s_b,
                     int64_t m_rows, int64_t n_rows, int64_t k,
                     int64_t npts, const int64_t* ms, const int64_t* ns,
                     double* y, double* abs_sum) {
    (void)m_rows; (void)n_rows;
    double inv_scale = 1.0 / ((double)s_a * (double)s_b);
    for (int64_t i = 0; i < npts; ++i)
        dot_point(qa, sa_swz, qb, sb_swz, k, ms[i], ns[i], inv_scale, &y[i], &abs_sum[i]);
}

void orc_gemm_full(const uint8_t* qa, const uint8_t* sa_swz, float s_a,
                   const uint8_t* qb, const uint8_t* sb_swz, float s_b,
                   int64_t m_rows, int64_t n_rows, int64_t k,
                   int64_t m_begin, int64_t m_end, double* y, double* abs_sum) {
    (void)m_rows;
    double inv_scale = 1.0 / ((double)s_a * (double)s_b);
    for (int64_t m = m_begin; m < m_end; ++m)
        for (int64_t n = 0; n < n_rows; ++n)
            dot_point(qa, sa_swz, qb, sb_swz, k, m, n, inv_scale, &y[m * n_rows + n],
                      &abs_sum[m * n_rows + n]);
}

/* ------------------------------------------------------------------------ */
/* MXFP4: 32-element blocks, power-of-two (E8M0) scales, no tensor scale.    */
/* ------------------------------------------------------------------------ */
double orc_e8m0_value(uint8_t code) {
    if (code == 0xFF) return NAN;
    return ldexp(1.0, (int)code - 127);
}

uint8_t orc_mx_scale_code(float amax_b) {
    int X;
    if (amax_b == 0.0f) {
        X = -127;
    } else {
        int e;
        frexp((double)amax_b, &e);        /* amax_b = m 2^e, m in [0.5, 1) */
        X = (e - 1) - 2;                  /* floor(log2 amax_b) - emax(E2M1) */
        if (X < -127) X = -127;
        if (X > 127) X = 127;
    }
    return (uint8_t)(X + 127);
}

int orc_mx_quantize(const uint16_t* x, int64_t rows, int64_t k, int64_t ld, int transposed,
                    uint32_t rht_mask, int64_t row_begin, int64_t row_end,
                    uint8_t* codes, uint8_t* scales_plain) {
    int64_t nb = k / 32;
    for (int64_t r = row_begin; r < row_end; ++r) {
        for (int64_t b = 0; b < nb; ++b) {
            float v[32];
            load_block16(x, ld, transposed, rht_mask, r, 2 * b, v);
            load_block16(x, ld, transposed, rht_mask, r, 2 * b + 1, v + 16);
            float amax_b = 0.0f;
            for (int j = 0; j < 32; ++j) {
                if (!isfinite(v[j])) return -1;
                if (fabsf(v[j]) > amax_b) amax_b = fabsf(v[j]);
            }
            uint8_t sc = orc_mx_scale_code(amax_b);
            scales_plain[r * nb + b] = sc;
            double inv = ldexp(1.0, -((int)sc - 127));   /* 2^-X */
            for (int j = 0; j < 32; ++j) {
                float e = (float)((double)v[j] * inv);    /* exact product, one rounding */
                put_code(codes, k, r, b * 32 + j, orc_e2m1_rne(e));
            }
        }
    }
    (void)rows;
    return 0;
}

size_t orc_mx_scale_bytes(int64_t rows, int64_t k) {
    return (size_t)(ceil_div(rows, 128) * ceil_div(k / 32, 4) * 512);
}

void orc_mx_swizzle_scales(const uint8_t* plain, int64_t rows, int64_t k, uint8_t* swz) {
    int64_t nb = k / 32, col_tiles = ceil_div(nb, 4);
    memset(swz, 0, orc_mx_scale_bytes(rows, k));
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < nb; ++c)
            swz[swz_offset(r, c, col_tiles)] = plain[r * nb + c];
}

void orc_mx_unswizzle_scales(const uint8_t* swz, int64_t rows, int64_t k, uint8_t* plain) {
    int64_t nb = k / 32, col_tiles = ceil_div(nb, 4);
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < nb; ++c)
            plain[r * nb + c] = swz[swz_offset(r, c, col_tiles)];
}

void orc_mx_dequantize(const uint8_t* codes, const uint8_t* scales_swz, int64_t rows, int64_t k,
                       int64_t row_begin, int64_t row_end, float* out, int64_t ld) {
    int64_t col_tiles = ceil_div(k / 32, 4);
    (void)rows;
    for (int64_t r = row_begin; r < row_end; ++r)
        for (int64_t c = 0; c < k; ++c)
            out[r * ld + c] = (float)(orc_e2m1_value(get_code(codes, k, r, c)) *
                                      orc_e8m0_value(scales_swz[swz_offset(r, c / 32, col_tiles)]));
}

void orc_mx_gemm_points(const uint8_t* qa, const uint8_t* sa_swz, const uint8_t* qb,
                        const uint8_t* sb_swz, int64_t m_rows, int64_t n_rows, int64_t k,
                        int64_t npts, const int64_t* ms, const int64_t* ns,
                        double* y, double* abs_sum) {
    int64_t col_tiles = ceil_div(k / 32, 4);
    (void)m_rows; (void)n_rows;
    for (int64_t i = 0; i < npts; ++i) {
        double acc = 0.0, acc_abs = 0.0;
        for (int64_t c = 0; c < k; ++c) {
            double a = orc_e2m1_value(get_code(qa, k, ms[i], c)) *
                       orc_e8m0_value(sa_swz[swz_offset(ms[i], c / 32, col_tiles)]);
            double b = orc_e2m1_value(get_code(qb, k, ns[i], c)) *
                       orc_e8m0_value(sb_swz[swz_offset(ns[i], c / 32, col_tiles)]);
            acc += a * b;
            acc_abs += fabs(a * b);
        }
        y[i] = acc;
        abs_sum[i] = acc_abs;
    }
}
