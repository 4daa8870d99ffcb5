/*
 * nvfp4.h -- C ABI of libnvfp4: the NVFP4 linear-layer hot path on one
 * NVIDIA B300 (sm_103a).
 *
 * The method (sources):
 *  [NVB] NVIDIA technical blog "NVFP4 Trains with Precision of 16-Bit and
 *        Speed and Efficiency of 4-Bit" (Chinese edition), section "NVFP4
 *        quantization recipe for pre-training": 16-element micro-blocks with
 *        one shared scale (bullet 1), E4M3 block scales (bullet 2), a
 *        Hadamard transform on GEMM inputs (bullet 3), 2D block quantisation
 *        of weights so forward and backward agree (bullet 4), stochastic
 *        rounding of gradients (bullet 5); Figure 1 (GEMMs dominate).
 *  [SAI] prism.simon-ai.net article 7890 "From MVFP4 to the essence of
 *        compute precision": section "Core architectural changes of the MVFP4
 *        format" (per-tensor FP32 scale over the E4M3 block scales), section
 *        "Training stability and protection of sensitive layers" (16x16
 *        weight blocks, 256 values per scale), section "Techniques against
 *        outliers and rounding error" (random Hadamard transform preserves the
 *        vector norm; stochastic rounding, 0.3 -> 1 with probability 30%).
 *
 * Numeric specification (the readings the pages leave open, fixed here):
 *  - amax: max |x| over the tensor (or over the 16-point RHT of every 16-chunk
 *    along k when an RHT mask is given).  NaN/Inf make the tensor invalid.
 *  - S_enc = fp32(2688 / amax) (2688 = 448 * 6, the E4M3 and E2M1 maxima);
 *    amax == 0 gives S_enc = 1; an overflowing S_enc saturates to FLT_MAX.
 *  - block decode scale s_b = E4M3_RNE_satfinite(fp32(fp32(amax_b / 6) * S_enc));
 *    encode factor r_b = fp32(S_enc / s_b) (0 when s_b == 0, FLT_MAX on
 *    overflow).
 *  - element: v = fp32(x * r_b); RNE: nearest E2M1 value, ties to the even
 *    code, saturating at +-6, sign kept (so small negatives give code 0x8);
 *    SR (NVFP4_SR): round |v| up from the grid value below to the one
 *    above iff u16 < floor(frac * 2^16), frac = (|v| - lo)/(hi - lo), where
 *    u16 is the element's 16-bit slice of Philox4x32-10 (key = seed,
 *    counter = (idx / 8, stream_id), slice idx % 8 = word (idx%8)/2, low
 *    half first), idx = r * k + c in the logical operand.
 *    SR_HW (NVFP4_SR_HW): the same rule with u16 = 65535 - r16, r16 drawn
 *    in the layout of the Blackwell FP4 stochastic-rounding conversion:
 *    word (idx % 16) / 4 of Philox4x32-10 (counter = (idx / 16,
 *    stream_id)), whose bytes b3 b2 b1 b0 give H = (b3, b1) and
 *    L = (b2, b0); element position idx % 4 = 0, 1, 2, 3 takes L, L
 *    bit-reversed, H, H bit-reversed.  32 random bits serve 4 elements
 *    (each element's u16 is uniform; the two elements sharing L or H are
 *    not independent).  Faster: one hardware conversion per 4 values.
 *    This layout is defined by the device's FP4 stochastic-rounding
 *    conversion (read off it with in-bounds probes), not by the pages,
 *    which give only the probability rule; NVFP4_SR is the path's mode.
 *  - RHT-16: y = H16 diag(s) x / 4, Sylvester order, s_j = -1 for set bit j of
 *    the 16-bit mask; evaluated sign flip, butterflies h = 1, 2, 4, 8 in fp32,
 *    then * 0.25.  Applied along k only.
 *  - dequantised value = fp32(fp32(q * s_b) * fp32(1 / S_enc)).
 *  - GEMM: D[m,n] = alpha * sum_k qa*sa*qb*sb with FP32 accumulation,
 *    alpha = fp32(1 / (S_enc_A * S_enc_B)); output FP32 or BF16 (RNE).
 *
 * Layouts.  A quantised operand is logical [rows x k], K-major:
 *  - codes:  rows x (k/2) bytes, row-major; element c of a row sits in byte
 *            c/2, the lower index in the low nibble.
 *  - scales: one E4M3 byte per (row, 16-column block), stored in the layout
 *            the block-scaled tensor-core MMA reads: rows padded to 128 and
 *            block columns padded to 4; 512-byte tiles, tile (row/128,
 *            col/4) at ((row/128) * ceil(k/64) + col/4) * 512, and inside a
 *            tile (row%32)*16 + ((row/32)%4)*4 + col%4.  Padding bytes are 0.
 *            Size: nvfp4_scale_bytes(rows, k).
 *  - global_scale: one float (S_enc) in device memory.
 *
 * Conventions for every call:
 *  - All pointers are DEVICE pointers owned by the caller; the library
 *    allocates no memory.  Buffers must not overlap unless stated.
 *  - Calls are asynchronous on `stream` and never synchronise with the host
 *    (except nvfp4_get_status).
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns an error and launches nothing.
 *  - Errors found on the device (non-finite amax reaching a quantiser, a
 *    pipeline wait that timed out) are recorded in a device status word,
 *    read and cleared by nvfp4_get_status().
 *  - No C++ exception crosses this interface.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_INVALID_ARG = 1,      /* null pointer, negative size, bad enum, aliasing   */
    NVFP4_ERR_UNSUPPORTED_SHAPE = 2,/* k not a multiple of 16 (32 for the GEMM), ...     */
    NVFP4_ERR_MISALIGNED = 3,       /* pointer or leading dimension not 16-byte aligned  */
    NVFP4_ERR_NONFINITE = 4,        /* amax was NaN or Inf (device-side, via get_status) */
    NVFP4_ERR_TIMEOUT = 5,          /* a bounded device wait expired (device-side)       */
    NVFP4_ERR_CUDA = 6,             /* a CUDA runtime call failed                        */
    NVFP4_ERR_LAUNCH = 7,           /* a kernel got less dynamic shared memory than it   */
                                    /* needs and returned early (device-side)            */
    NVFP4_ERR_GUARD = 8             /* debug build only: an index guard refused a global */
                                    /* access outside its buffer (device-side)           */
} nvfp4_status;

typedef enum { NVFP4_RNE = 0, NVFP4_SR = 1, NVFP4_SR_HW = 2 } nvfp4_round;

/* A bf16 tensor seen as the logical operand [rows x cols] (cols = k, the
 * GEMM reduction dimension).  transposed == 0: element (r, c) is at
 * ptr[r * ld + c] (ld >= cols).  transposed == 1: the array is stored as
 * [cols x rows] and element (r, c) is at ptr[c * ld + r] (ld >= rows) -- the
 * transpose-on-load used for the weight-gradient GEMM, where k is the token
 * dimension.  ptr must be 16-byte aligned and ld a multiple of 8.            */
typedef struct {
    const void* ptr;
    int64_t rows, cols, ld;
    int transposed;
} nvfp4_bf16_view;

/* A quantised operand (see Layouts).  block2d records the block shape it was
 * made with (0: 1x16, 1: 16x16); the GEMM does not depend on it.            */
typedef struct {
    uint8_t* codes;
    uint8_t* scales;
    float* global_scale;
    int64_t rows, k;
    int block2d;
} nvfp4_q;

/* Per-tensor amax ([SAI] two-level scale; step 1 of the path).
 * Writes max |x| of the logical operand (rht_mask == 0) or max |RHT16(x)|
 * over 16-chunks along k (rht_mask != 0, 16-bit mask) to *amax_dev.
 * x.cols must be a multiple of 16 when rht_mask != 0.  NaN inputs give a NaN
 * amax, Inf an Inf (no error here; the quantisers report it).               */
nvfp4_status nvfp4_amax(nvfp4_bf16_view x, uint32_t rht_mask, float* amax_dev,
                        cudaStream_t stream);

/* 1x16 quantisation ([NVB] bullets 1, 2, 5; [SAI] global scale).
 * x: logical [rows x k], k % 16 == 0.  amax_dev: the tensor's amax as written
 * by nvfp4_amax (same view, same RHT setting); NULL makes the call compute it
 * first, using out->global_scale as the temporary.  round: NVFP4_RNE,
 * NVFP4_SR or NVFP4_SR_HW (seed, stream_id select the Philox stream; ignored
 * for RNE).  out: rows and k must
 * equal x's; codes rows*k/2 bytes, scales nvfp4_scale_bytes(rows, k) bytes,
 * global_scale 1 float; all written (scale padding with 0).                 */
nvfp4_status nvfp4_quantize_1d(nvfp4_bf16_view x, const float* amax_dev, nvfp4_round round,
                               uint64_t seed, uint64_t stream_id, nvfp4_q* out,
                               cudaStream_t stream);

/* 16x16 quantisation of a weight ([NVB] bullet 4; [SAI] 16x16 blocks).
 * One scale per 16 rows x 16 columns (replicated into every row's slot of the
 * scale layout).  out_t (nullable) receives the transposed operand
 * [k x rows] made from the same codes and scales, so that the backward GEMM
 * sees exactly the forward's quantised weight; it needs rows % 16 == 0.
 * Stochastic rounding draws its bits by the index in x's logical layout, and
 * out_t holds the same codes transposed.                                    */
nvfp4_status nvfp4_quantize_2d(nvfp4_bf16_view w, const float* amax_dev, nvfp4_round round,
                               uint64_t seed, uint64_t stream_id, nvfp4_q* out,
                               nvfp4_q* out_t, cudaStream_t stream);

/* 16-point random Hadamard transform fused with quantisation ([NVB] bullet 3;
 * [SAI] Hadamard transform).  Each 16-chunk along k is replaced by
 * H16 diag(s) x / 4 before amax_b and encoding.  amax_dev must be the amax of
 * the transformed tensor (nvfp4_amax with the same mask) or NULL.
 * out->block2d selects 1x16 (0) or 16x16 (1) blocks.  The same mask must be
 * used for both operands of a GEMM so that their dot products are kept.     */
nvfp4_status nvfp4_rht_quantize(nvfp4_bf16_view x, uint32_t rht_mask, const float* amax_dev,
                                nvfp4_round round, uint64_t seed, uint64_t stream_id,
                                nvfp4_q* out, cudaStream_t stream);

/* Dual-axis amax: one read of a stored tensor S for both GEMM views of it
 * ([NVB] bullet 3 applies the Hadamard transform to the weight-gradient
 * inputs only; [SAI] per-tensor scale).  x must be a non-transposed view of
 * S [rows x cols] with rows % 16 == 0.  Writes
 *   *amax_dev   = max |S|                       (== nvfp4_amax(x, 0)),
 *   *amax_t_dev = max |RHT16 along rows of S|   (== nvfp4_amax of the
 *                 transposed view of S, k = rows, with rht_mask; the plain
 *                 max |S| when rht_mask == 0),
 * bit for bit.  The two outputs must be distinct floats.                    */
nvfp4_status nvfp4_amax_dual(nvfp4_bf16_view x, uint32_t rht_mask, float* amax_dev,
                             float* amax_t_dev, cudaStream_t stream);

/* Dual-axis 1x16 quantisation: one read of a stored tensor S [rows x cols]
 * emits both operands a training step takes from it ([NVB] bullets 1-3, 5):
 *   out   = logical S   [rows x cols], 1x16 blocks along cols, no RHT,
 *           rounding `round` with (seed, stream_id)          (fprop / dgrad);
 *   out_t = logical S^T [cols x rows], 1x16 blocks along rows (the tokens),
 *           RHT-16 with rht_mask_t (none when 0), rounding `round_t` with
 *           (seed_t, stream_id_t)                             (wgrad).
 * Each is bit for bit what nvfp4_quantize_1d(x, ...) and
 * nvfp4_rht_quantize / nvfp4_quantize_1d of the transposed view of S make.
 * x must be non-transposed with rows % 16 == 0 and cols % 16 == 0.
 * amax_dev / amax_t_dev: the amaxes of the two operands (nvfp4_amax_dual),
 * both required (no self-amax form).                                        */
nvfp4_status nvfp4_quantize_dual(nvfp4_bf16_view x, const float* amax_dev, nvfp4_round round,
                                 uint64_t seed, uint64_t stream_id, nvfp4_q* out,
                                 uint32_t rht_mask_t, const float* amax_t_dev, nvfp4_round round_t,
                                 uint64_t seed_t, uint64_t stream_id_t, nvfp4_q* out_t,
                                 cudaStream_t stream);

/* Dequantisation ([SAI] MXFP4 example: value = scale x code; with the global
 * scale divided out).  Writes q as fp32 (out_is_bf16 == 0) or bf16 (RNE) into
 * out[r * ld + c]; ld >= q->k, out 16-byte aligned, ld*elem a multiple of 16. */
nvfp4_status nvfp4_dequantize(const nvfp4_q* q, void* out, int out_is_bf16, int64_t ld,
                              cudaStream_t stream);

/* Block-scaled FP4 GEMM on the tensor cores ([NVB] Figure 1 and bullet 1).
 * D[m, n] = alpha * sum_k A[m,k] B[n,k] for A = a (M x K) and B = b (N x K),
 * both K-major; FP32 accumulation; alpha = 1/(S_A S_B) from the operands'
 * global scales.  d: M x N row-major with leading dimension ldd (elements),
 * fp32 or bf16 (d_is_bf16).  Needs a->k == b->k, K % 32 == 0, ldd >= N,
 * ldd * elem % 16 == 0, 16-byte aligned codes/scales/d.  M, N >= 1 arbitrary. */
nvfp4_status nvfp4_gemm(const nvfp4_q* a, const nvfp4_q* b, void* d, int d_is_bf16,
                        int64_t ldd, cudaStream_t stream);

/* ---- MXFP4, the comparison format ([NVB] bullets 1-2: 32-element blocks
 * with power-of-two E8M0 scales; [SAI] "MVFP4 and MXFP4", "Core
 * architectural changes of the MVFP4 format").  An MXFP4 operand uses
 * nvfp4_q with: codes as for NVFP4; scales = one E8M0 byte (2^(byte-127))
 * per (row, 32-column block) in the same 512-byte-tile layout with 32-element
 * blocks (nvfp4_mx_scale_bytes); global_scale unused (may be NULL); block2d 0.
 * Scale rule (the pages give none): X = floor(log2(block max)) - 2, clamped
 * to [-127, 127]; elements x * 2^-X rounded to E2M1 (RNE, saturating).     */
size_t nvfp4_mx_scale_bytes(int64_t rows, int64_t k);

/* 1x32 MXFP4 quantisation of a non-transposed view, k % 32 == 0, RNE;
 * rht_mask != 0 first applies RHT-16 to every 16-chunk along k.  A block
 * holding a NaN or Inf gets scale 0xFF and the call reports
 * NVFP4_ERR_NONFINITE through nvfp4_get_status.                              */
nvfp4_status nvfp4_mx_quantize(nvfp4_bf16_view x, uint32_t rht_mask, nvfp4_q* out, cudaStream_t stream);

/* x_hat = q * 2^X (exact), fp32 or bf16 (RNE), like nvfp4_dequantize.      */
nvfp4_status nvfp4_mx_dequantize(const nvfp4_q* q, void* out, int out_is_bf16, int64_t ld,
                                 cudaStream_t stream);

/* MXFP4 GEMM on the tensor cores (tcgen05.mma kind::mxf4, scale_vec::2X):
 * D[m, n] = sum_k A[m,k] B[n,k] with FP32 accumulation (no tensor scales).
 * Same shapes, layouts and rules as nvfp4_gemm (K % 32 == 0).               */
nvfp4_status nvfp4_mx_gemm(const nvfp4_q* a, const nvfp4_q* b, void* d, int d_is_bf16, int64_t ldd,
                           cudaStream_t stream);

/* Host helper: the 16-bit RHT sign mask of a seed = low 16 bits of word 0 of
 * Philox4x32-10(counter = 0, key = seed).                                   */
uint32_t nvfp4_rht_mask_from_seed(uint64_t seed);

/* Synchronises `stream`, returns the device-side status recorded since the
 * last call (NVFP4_ERR_GUARD before NVFP4_ERR_LAUNCH before NVFP4_ERR_TIMEOUT before
 * NVFP4_ERR_NONFINITE before NVFP4_OK, NVFP4_ERR_CUDA if the stream reports
 * a CUDA error) and clears it.                                              */
nvfp4_status nvfp4_get_status(cudaStream_t stream);

/* Size in bytes of the swizzled scale buffer of a [rows x k] operand.       */
size_t nvfp4_scale_bytes(int64_t rows, int64_t k);

/* Static text of a status code.                                             */
const char* nvfp4_status_string(nvfp4_status s);

/* Test-only fault injection for failure detection (no GPU fault, trap or
 * hang).  mode 1: the next streamed amax launch (nvfp4_amax_dual, or
 * nvfp4_amax on a strided view without RHT or on a transposed view with RHT)
 * does not issue the copy of its
 * first tile.  That tile's bounded wait expires after about 2 s, the kernel
 * drains its other copies and returns, and nvfp4_get_status then reports
 * NVFP4_ERR_TIMEOUT; the amax written by that call is undefined.  The
 * injection applies once and then clears.  mode 2: the next
 * nvfp4_quantize_dual takes its general path for Philox block indices of 64
 * bits (used only for operands of more than 2^35 elements) instead of the
 * path with 32-bit indices; the outputs must not change.  mode 0 clears
 * both.  Returns NVFP4_ERR_INVALID_ARG for any other mode. */
nvfp4_status nvfp4_debug_inject(int mode);

/* Test-only check of the block-scale arithmetic: the kernels compute
 * fp32(amax_b / 6) with a multiply and two FMAs (Markstein's correction,
 * P. Markstein, IBM J. Res. Dev. 34(1), 1990) instead of a division.  This
 * call evaluates that sequence and the IEEE-rounded division x / 6 (CUDA's
 * __fdiv_rn) for every float whose bit pattern b lies in [lo_bits, hi_bits)
 * (hi_bits <= 0x7F800000: non-negative finite floats), and writes the number
 * of patterns where they differ to *mismatches_dev and the smallest such
 * pattern (0xFFFFFFFF if none) to *first_bad_dev; both device pointers,
 * caller-owned (8- and 4-byte aligned).  Asynchronous on `stream`.        */
nvfp4_status nvfp4_debug_check_div6(uint32_t lo_bits, uint32_t hi_bits,
                                    unsigned long long* mismatches_dev, uint32_t* first_bad_dev,
                                    cudaStream_t stream);

/* Index guards (debug build).  The library built with NVFP4_DEBUG_GUARDS
 * defined (libnvfp4_guarded.so; same entry points, same results) checks
 * every plain global load and store of its kernels against the extent that
 * the layouts above give the buffer it addresses: codes rows * k/2 bytes,
 * scales nvfp4_scale_bytes (nvfp4_mx_scale_bytes for MXFP4), a bf16 or fp32
 * array ((outer - 1) * ld + inner) elements.  TMA copies are bounded by
 * their tensor maps and need no guard.  An access outside its extent is
 * skipped (a refused load reads zeros), nvfp4_get_status reports
 * NVFP4_ERR_GUARD, and the first refused access is recorded.  No access is
 * made outside the buffers in either build; the guards turn an indexing
 * error into a status instead of a memory fault.
 *
 * nvfp4_debug_guards_enabled: 1 in the guarded build, 0 otherwise.
 *
 * nvfp4_debug_guard_record: synchronises `stream`, writes the site of the
 * first refused access since the last call (0: none; 1..17 name the kernel
 * and buffer, listed in csrc/guard.cuh) and the low 48 bits of its byte
 * offset from the buffer's start to the host pointers, and clears the
 * record.  In the normal build it writes 0 and 0.  NVFP4_ERR_INVALID_ARG for
 * a null pointer.
 *
 * nvfp4_debug_guard_shrink (test-only): every guard checks against its extent
 * minus `bytes` (0 restores the extents), so that a test can make the guards
 * refuse in-bounds accesses near the end of a buffer and see them reported
 * and skipped, without any access leaving the buffer.  Synchronous.
 * NVFP4_ERR_INVALID_ARG in the normal build.                                */
int nvfp4_debug_guards_enabled(void);
nvfp4_status nvfp4_debug_guard_record(uint32_t* site, uint64_t* byte_offset, cudaStream_t stream);
nvfp4_status nvfp4_debug_guard_shrink(uint64_t bytes);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H */
