/*
 * nvfp4_oracle.h -- plain, slow, scalar CPU oracle of the NVFP4 linear-layer path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library; the only thing both sides
 * see is the seeded synthetic input.
 *
 * Citations (sources of the method):
 *  [NVB]  NVIDIA technical blog "NVFP4 Trains with Precision of 16-Bit and
 *         Speed and Efficiency of 4-Bit" (Chinese edition), section
 *         "NVFP4 quantization recipe for pre-training", bullets 1-5.
 *  [SAI]  prism.simon-ai.net article 7890 "From MVFP4 to the essence of
 *         compute precision", sections "Core architectural changes of the
 *         MVFP4 format" (two-level scale), "Training stability and protection
 *         of sensitive layers" (16x16 weight blocks), "Techniques against
 *         outliers and rounding error" (Hadamard transform, stochastic
 *         rounding example 0.3 -> 1 with probability 30%).
 *  [PHX]  J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel random numbers:
 *         as easy as 1, 2, 3", SC'11 -- the Philox4x32-10 generator.
 *  The numeric constants that the pages leave open (E2M1 value set, the
 *  448*6 global-scale constant, the 16-point Hadamard size, Philox) are the
 *  readings of the path's specification, recorded in the design notes.
 *
 * Conventions shared with the library's public header *by specification*
 * (not by code): bf16 inputs are raw uint16 bit patterns; a quantised
 * operand is logical [rows x k], codes row-major with two E2M1 codes per
 * byte (lower k index in the low nibble); scales are E4M3 bytes, given here
 * either "plain" ([rows x k/16] row-major) or "swizzled" (the GEMM layout:
 * 128-row x 4-scale tiles of 512 bytes).
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ---------------------------------------------------- */
double  orc_e2m1_value(uint8_t code);              /* code 0..15 -> real value */
uint8_t orc_e2m1_rne(float v);                     /* nearest, ties to even code, |v|>6 -> 6, sign kept */
float   orc_e4m3_value(uint8_t code);              /* finite codes only (0x7F/0xFF are NaN) */
uint8_t orc_e4m3_rne_satfinite(float t);           /* t >= 0: nearest, ties to even, t > 448 -> 448 */
float   orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16_rne(float f);

/* ---- Philox4x32-10 [PHX] ------------------------------------------------ */
void     orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
uint32_t orc_rht_mask_from_seed(uint64_t seed);    /* low 16 bits of word 0 of Philox(ctr=0, key=seed) */
/* 16-bit random slice for element index idx of a quantised operand */
uint32_t orc_sr_bits16(uint64_t seed, uint64_t stream_id, uint64_t idx);
/* second layout (rounding mode 2): integer r of element p (0..3) of a
 * 32-bit word, and the u16 = 65535 - r of element idx */
uint32_t orc_sr_r16_of_word(uint32_t w, int p);
uint32_t orc_sr_bits16_hw(uint64_t seed, uint64_t stream_id, uint64_t idx);
/* stochastic E2M1 rounding of v given its 16 random bits: up iff u16 < floor(frac * 2^16) */
uint8_t  orc_e2m1_sr(float v, uint32_t u16);

/* ---- random Hadamard transform, 16 points ------------------------------ */
void orc_rht16(const float in[16], uint32_t mask, float out[16]);

/* ---- per-tensor amax and global scale ---------------------------------- */
/* x: bf16 view.  Stored as [rows x cols] with leading dimension ld when
 * transposed == 0 (logical operand = stored); when transposed == 1 the
 * stored array is [cols x rows]... i.e. the logical operand is [rows x k]
 * and element (r, c) sits at x[c*ld + r].  rht_mask == 0 means no RHT;
 * otherwise the max is taken over RHT16 of every 16-chunk along k.        */
float orc_amax(const uint16_t* x, int64_t rows, int64_t k, int64_t ld, int transposed,
               uint32_t rht_mask);
/* S_enc = 2688/amax, amax==0 -> 1, overflow -> FLT_MAX.  Returns 0 on
 * success, -1 if amax is not finite (then *s_enc is NaN).                  */
int   orc_global_scale(float amax, float* s_enc);

/* ---- quantisation ------------------------------------------------------- */
/* Quantise logical rows [row_begin, row_end) of the bf16 operand.
 *  block2d: 0 -> 1x16 blocks along k; 1 -> 16x16 blocks (row_begin/row_end
 *           must then be multiples of 16, except row_end == rows).
 *  round:   0 -> RNE, 1 -> stochastic (seed, stream_id), 2 -> stochastic with
 *           the second random-bit layout (orc_sr_bits16_hw).
 *  codes:   [rows x k/2] bytes (full-size buffer; only the range is written)
 *  scales:  plain [rows x k/16] E4M3 bytes (full-size buffer)
 * Returns 0, or -1 if amax is not finite.                                  */
int orc_quantize(const uint16_t* x, int64_t rows, int64_t k, int64_t ld, int transposed,
                 uint32_t rht_mask, int block2d, float amax, int round,
                 uint64_t seed, uint64_t stream_id,
                 int64_t row_begin, int64_t row_end,
                 uint8_t* codes, uint8_t* scales_plain);

/* Swizzled (GEMM) scale layout size for a [rows x k] operand, in bytes.   */
size_t orc_scale_bytes(int64_t rows, int64_t k);
/* plain [rows x k/16] -> swizzled (padding written as 0)                   */
void orc_swizzle_scales(const uint8_t* plain, int64_t rows, int64_t k, uint8_t* swz);
/* swizzled -> plain                                                        */
void orc_unswizzle_scales(const uint8_t* swz, int64_t rows, int64_t k, uint8_t* plain);

/* transpose of a quantised operand's codes: [rows x k] -> [k x rows]       */
void orc_transpose_codes(const uint8_t* codes, int64_t rows, int64_t k, uint8_t* codes_t);

/* ---- dequantisation ----------------------------------------------------- */
/* x_hat = fp32(fp32(q * s_b) * fp32(1 / S_enc)) for rows [row_begin,row_end);
 * out is fp32 [rows x ld] (out_is_bf16 == 0) or bf16 bits (out_is_bf16 == 1). */
void orc_dequantize(const uint8_t* codes, const uint8_t* scales_swz, float s_enc,
                    int64_t rows, int64_t k, int64_t row_begin, int64_t row_end,
                    void* out, int out_is_bf16, int64_t ld);

/* ---- GEMM reference in FP64 ---------------------------------------------- */
/* For each requested (m, n): y = sum_k a[m,k] b[n,k] / (S_A S_B) and
 * abs = sum_k |a[m,k] b[n,k]| / (S_A S_B), both in FP64, where
 * a = e2m1(qa) * e4m3(sa), b = e2m1(qb) * e4m3(sb).  Scales are swizzled.   */
void orc_gemm_points(const uint8_t* qa, const uint8_t* sa_swz, float s_a,
                     const uint8_t* qb, const uint8_t* sb_swz, float s_b,
                     int64_t m_rows, int64_t n_rows, int64_t k,
                     int64_t npts, const int64_t* ms, const int64_t* ns,
                     double* y, double* abs_sum);
/* Full GEMM for output rows [m_begin, m_end): y, abs_sum [M x N] row-major. */
void orc_gemm_full(const uint8_t* qa, const uint8_t* sa_swz, float s_a,
                   const uint8_t* qb, const uint8_t* sb_swz, float s_b,
                   int64_t m_rows, int64_t n_rows, int64_t k,
                   int64_t m_begin, int64_t m_end, double* y, double* abs_sum);

/* ---- MXFP4: the comparison format ---------------------------------------
 * [NVB] bullets 1-2 and [SAI] "MVFP4 and MXFP4" / "Core architectural
 * changes of the MVFP4 format": one shared power-of-two scale (E8M0) per 32
 * elements, no per-tensor scale.  The reading of the scale rule (the pages
 * give none): block exponent X = floor(log2(amax_b)) - 2, where 2 is the
 * E2M1 maximum's exponent (6 = 1.5 * 2^2), clamped to [-127, 127]; amax_b
 * == 0 gives X = -127.  Elements: v = x * 2^-X, E2M1 RNE with saturation.
 * Scales are E8M0 codes X + 127; the swizzled layout is the NVFP4 one with
 * 32-element blocks (512-byte tiles of 128 rows x 4 blocks = 128 k).      */
double  orc_e8m0_value(uint8_t code);               /* 2^(code - 127); code 255 is NaN */
uint8_t orc_mx_scale_code(float amax_b);            /* finite amax_b >= 0 */
/* Quantise logical rows [row_begin, row_end) in 1x32 blocks along k
 * (k % 32 == 0), RNE; rht_mask != 0 applies RHT16 to every 16-chunk along k
 * first.  codes [rows x k/2]; scales_plain [rows x k/32] E8M0 codes.
 * Returns 0, or -1 if a block's amax is not finite.                        */
int orc_mx_quantize(const uint16_t* x, int64_t rows, int64_t k, int64_t ld, int transposed,
                    uint32_t rht_mask, int64_t row_begin, int64_t row_end,
                    uint8_t* codes, uint8_t* scales_plain);
size_t orc_mx_scale_bytes(int64_t rows, int64_t k);
void   orc_mx_swizzle_scales(const uint8_t* plain, int64_t rows, int64_t k, uint8_t* swz);
void   orc_mx_unswizzle_scales(const uint8_t* swz, int64_t rows, int64_t k, uint8_t* plain);
/* x_hat = q * 2^X (exact) for rows [row_begin, row_end); fp32 [rows x ld]   */
void   orc_mx_dequantize(const uint8_t* codes, const uint8_t* scales_swz, int64_t rows, int64_t k,
                         int64_t row_begin, int64_t row_end, float* out, int64_t ld);
/* FP64 GEMM reference: y = sum_k a b, abs = sum_k |a b|, a = e2m1 * 2^Xa.   */
void   orc_mx_gemm_points(const uint8_t* qa, const uint8_t* sa_swz, const uint8_t* qb,
                          const uint8_t* sb_swz, int64_t m_rows, int64_t n_rows, int64_t k,
                          int64_t npts, const int64_t* ms, const int64_t* ns,
                          double* y, double* abs_sum);

#ifdef __cplusplus
}
#endif
#endif
