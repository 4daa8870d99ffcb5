// quantize.cuh -- HBM-bound kernels of the NVFP4 path: per-tensor amax,
// 1x16 and 16x16 quantisation (RNE or Philox stochastic rounding, optional
// fused 16-point random Hadamard transform, transpose-on-load, transposed
// emit for weights) and dequantisation.
//
// Method: NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and Speed and
// Efficiency of 4-Bit", recipe bullets 1-5; prism.simon-ai.net article 7890,
// sections "Core architectural changes of the MVFP4 format" (global FP32
// scale), "Training stability and protection of sensitive layers" (16x16
// weight blocks), "Techniques against outliers and rounding error" (RHT, SR).
//
// Work decomposition (the 1x16 quantiser, of a view or of its transpose, is
// the row-wise or the column-wise path of the dual kernel, dual.cuh):
//  * 2D variant (persistent, TMA-fed): a 16-lane half-warp holds one 16x64
//    strip (one row per lane); the 16x16 block amax is a 4-step shuffle
//    reduction.  The transposed operand is emitted from a shared-memory
//    nibble tile.
#pragma once
#include <cuda.h>
#include <cstdint>
#include "codec.cuh"
#include "guard.cuh"
#include "ptx.cuh"
#include "status.cuh"

namespace nvfp4 {

constexpr int kQuantThreads = 256;

// 16-byte streaming load that does not allocate in L1 (data read once).
__device__ __forceinline__ uint4 ldg_stream_na(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// A grid-stride walk over the items (major, minor) of a [nmajor x nminor]
// index space, minor fastest, without a division per step.
struct ItemWalk {
    int64_t major, dmajor;
    uint32_t minor, dminor, nminor;
    __device__ __forceinline__ ItemWalk(uint32_t nminor_) : nminor(nminor_) {
        const int64_t it0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        major = it0 / nminor;
        minor = (uint32_t)(it0 - major * nminor);
        dmajor = stride / nminor;
        dminor = (uint32_t)(stride - dmajor * nminor);
    }
    __device__ __forceinline__ void next() {
        minor += dminor;
        major += dmajor;
        if (minor >= nminor) {
            minor -= nminor;
            ++major;
        }
    }
};

__device__ __forceinline__ void unpack8(uint4 w, float* v) {
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x);
    v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
    v[4] = bf16_lo(w.z); v[5] = bf16_hi(w.z);
    v[6] = bf16_lo(w.w); v[7] = bf16_hi(w.w);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// max |v| over 16 finite values, as float bits (three-input maxima of the
// magnitudes; the inputs of a quantiser are finite because a non-finite amax
// stops it).
__device__ __forceinline__ uint32_t absmax_bits16(const float* v) {
    float m = fmax3(fabsf(v[0]), fabsf(v[1]), fabsf(v[2]));
#pragma unroll
    for (int j = 3; j < 15; j += 2) m = fmax3(m, fabsf(v[j]), fabsf(v[j + 1]));
    return __float_as_uint(fmaxf(m, fabsf(v[15])));
}

// max |v| over 16 values as float bits, NaN-propagating (integer max of the
// magnitude bit patterns): used by the amax kernels, whose inputs may hold
// NaN or Inf.
__device__ __forceinline__ uint32_t absmax_bits16_nan(const float* v) {
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) m = max(m, __float_as_uint(v[j]) & 0x7FFFFFFFu);
    return m;
}

// Reduce a per-thread maximum of non-negative float bit patterns and merge it
// into *out with one atomic per CTA (unsigned order == float order there).
__device__ __forceinline__ void block_max_to_global(uint32_t m, float* out) {
    __shared__ uint32_t red[kQuantThreads / 32];
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < (int)(blockDim.x >> 5) ? red[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0 && m) atomicMax(reinterpret_cast<uint32_t*>(out), m);
    }
}

// max |RHT16(v)| as float bits, NaN-propagating.  Finite blocks take the
// integer maximum of the non-negative pair magnitudes (see rht16_pair_mags);
// a non-finite magnitude (where a +-Inf pair can also make a NaN output)
// falls back to the full last stage.  v is clobbered.
__device__ __forceinline__ uint32_t rht16_absmax_bits_nan(float* v, const RhtSigns& sg) {
    rht16_first3(v, sg);
    float s[8];
    rht16_pair_mags(v, s);
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max(m, __float_as_uint(s[i]));
    if (m >= 0x7F800000u) {
        rht16_last(v);
        return absmax_bits16_nan(v);
    }
    return __float_as_uint(__fmul_rn(__uint_as_float(m), 0.25f));
}

// Resolve the global encode scale for a quantiser CTA.  src holds either the
// amax (src_is_senc == 0; CTA 0 then publishes S_enc to gs_out) or S_enc
// itself.  gs_out2 (nullable) receives a copy for a second operand made from
// the same encoding.  Returns false (after recording the error) when the
// scale is unusable.
__device__ __forceinline__ bool resolve_scale(const float* src, int src_is_senc, float* gs_out,
                                              float* gs_out2, float* s_enc) {
    const float v = *src;
    float s = v;
    bool ok = fabsf(v) <= FLT_MAX;
    if (!src_is_senc) ok = global_encode_scale(v, &s);
    if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
        const float pub = ok ? s : __int_as_float(0x7FC00000);
        if (!src_is_senc) {
            *gs_out = pub;
            if (!ok) record_device_error(NVFP4_DEV_NONFINITE);
        }
        if (gs_out2 != nullptr) *gs_out2 = pub;
    }
    *s_enc = s;
    return ok;
}

// Publish S_enc for an empty tensor (no quantiser CTA runs).
__global__ void k_publish_senc(const float* src, int src_is_senc, float* gs_out, float* gs_out2) {
    float s;
    resolve_scale(src, src_is_senc, gs_out, gs_out2, &s);
}

// ============================================================== amax ======
// max |x| (as bf16 magnitude bits) of a 16-byte aligned span, split over
// `nt` threads starting at `tid`: 16 independent 16-byte loads in flight per
// thread (HBM needs a few hundred KB in flight per SM), folded with
// half-word SIMD maxima of the magnitude bit patterns (order-free and
// NaN-propagating: a NaN pattern exceeds every finite one).
__device__ __forceinline__ uint32_t span_absmax(const uint16_t* base, int64_t len, int64_t tid,
                                                int64_t nt, const uint16_t* gbase, uint64_t gext) {
    constexpr uint32_t M = 0x7FFF7FFFu;
    constexpr int U = 16;
    uint32_t m2 = 0, m1 = 0;
    const int64_t nch = len >> 3;
    const uint4* v = reinterpret_cast<const uint4*>(base);
    int64_t i = tid;
    for (; i + (U - 1) * nt < nch; i += U * nt) {
        uint4 c[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            c[u] = NVFP4_GUARD(gbase, gext, v + i + u * nt, 16, kGuardAmaxX) ? ldg_stream_na(v + i + u * nt)
                                                                              : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < U; ++u)
            m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(c[u].x & M, c[u].y & M), __vmaxu2(c[u].z & M, c[u].w & M)));
    }
    for (; i < nch; i += nt) {
        const uint4 a = NVFP4_GUARD(gbase, gext, v + i, 16, kGuardAmaxX) ? ldg_stream_na(v + i)
                                                                         : make_uint4(0, 0, 0, 0);
        m2 = __vmaxu2(m2, __vmaxu2(__vmaxu2(a.x & M, a.y & M), __vmaxu2(a.z & M, a.w & M)));
    }
    for (int64_t j = (nch << 3) + tid; j < len; j += nt)
        if (NVFP4_GUARD(gbase, gext, base + j, 2, kGuardAmaxX)) m1 = max(m1, (uint32_t)(base[j] & 0x7FFFu));
    return max(max(m2 & 0xFFFFu, m2 >> 16), m1);
}

// max |x| of a bf16 array of nrows rows of len elements (leading dimension
// ld).  One row (contiguous data): the whole grid strides over it; several
// rows: CTAs stride over rows, threads over a row.
__global__ void __launch_bounds__(kQuantThreads, 3) k_amax_plain(const uint16_t* __restrict__ p,
                                                                 int64_t nrows, int64_t len,
                                                                 int64_t ld, float* out) {
    uint32_t m = 0;
    if (nrows == 1) {
        m = span_absmax(p, len, (int64_t)blockIdx.x * blockDim.x + threadIdx.x,
                        (int64_t)gridDim.x * blockDim.x, p, stored_extent(1, len, len, 2));
    } else {
        for (int64_t r = blockIdx.x; r < nrows; r += gridDim.x)
            m = max(m, span_absmax(p + r * ld, len, threadIdx.x, blockDim.x, p, stored_extent(nrows, len, ld, 2)));
    }
    block_max_to_global(m << 16, out);
}

// max |RHT16(x)| over 16-chunks along the stored rows (non-transposed view).
__global__ void __launch_bounds__(kQuantThreads) k_amax_rht_rows(const uint16_t* __restrict__ p,
                                                                 int64_t rows, int64_t k,
                                                                 int64_t ld, const RhtSigns sg,
                                                                 float* out) {
    uint32_t m = 0;
    const uint32_t nkb = (uint32_t)(k >> 4);
    const int64_t total = rows * (int64_t)nkb;
    for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < total;
         b += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = b / nkb, kb = b - r * nkb;
        const uint4* src = reinterpret_cast<const uint4*>(p + r * ld + kb * 16);
        float v[16];
        if (!NVFP4_GUARD(p, stored_extent(rows, k, ld, 2), src, 32, kGuardAmaxX)) continue;
        unpack8(ldg_stream(src), v);
        unpack8(ldg_stream(src + 1), v + 8);
        m = max(m, rht16_absmax_bits_nan(v, sg));
    }
    block_max_to_global(m, out);
}

// In-place amax -> S_enc (used when a quantiser computes its own amax).
__global__ void k_amax_to_senc(float* gs) {
    float s;
    if (!global_encode_scale(*gs, &s)) {
        s = __int_as_float(0x7FC00000);
        record_device_error(NVFP4_DEV_NONFINITE);
    }
    *gs = s;
}

// ====================================================== quantise 1x16 ======
struct QuantArgs {
    const uint16_t* x;
    int64_t rows, k, ld;        // logical operand [rows x k]; ld of the stored array
    const float* scale_src;     // amax, or S_enc when src_is_senc
    int src_is_senc;
    float* gs_out;
    float* gs_out2;             // copy of S_enc for the transposed operand (nullable)
    uint8_t* codes;             // [rows x k/2]
    uint8_t* scales;            // swizzled
    RhtSigns rht;               // RHT-16 sign multipliers (RHT kernels only)
    uint64_t stream_id;
    uint32_t sr_key[20];        // Philox round keys of the seed (philox4x32_10_not for
                                // NVFP4_SR, philox4x32_10 for NVFP4_SR_HW)
    int sr_hw;                  // 1: NVFP4_SR_HW random-bit layout (hardware conversion)
    int sr_g32;                 // 1: every Philox block index of the operand is below 2^32
    uint32_t sr_pre[4];         // rounds 0-1 constants of philox4x32_10_g32 (seed, stream_id)
    // 2D transposed emit (optional)
    uint8_t* codes_t;           // [k x rows/2]
    uint8_t* scales_t;
    int idx_transposed;         // SR index taken as (c * rows + r) (2D on a transposed view)
    int write_primary;
};

// |a| max |b| per bf16 half (the sign bits of the result are junk).
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// amax of 16 finite bf16 values held as 8 packed words, returned as a float
// bit pattern.
__device__ __forceinline__ uint32_t absmax_bits16_packed(uint4 a, uint4 b) {
    const uint32_t m = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(a.x, a.y), bf16x2_absmax(a.z, a.w)),
                                     bf16x2_absmax(bf16x2_absmax(b.x, b.y), bf16x2_absmax(b.z, b.w)));
    return max((m & 0x7FFFu) << 16, m & 0x7FFF0000u);
}

// Per-CTA table of the encode factor r_b for every E4M3 code 0..127 (the
// block scale is never negative, and 0x7F is never produced).
__device__ __forceinline__ void init_rtab(float* rtab, float s_enc) {
    for (int c = threadIdx.x; c < 128; c += blockDim.x) rtab[c] = encode_factor(s_enc, (uint32_t)c);
    __syncthreads();
}

// Encode one 16-element block.  amax_bits: the block's max |value| as float
// bits when already known (raw bf16 input), or ~0u to compute it here.
// HW: the stochastic rounding's random-bit layout, 1 = NVFP4_SR_HW, 0 =
// NVFP4_SR, -1 = taken from a.sr_hw at run time.  G32: the caller knows that
// a.sr_g32 holds (Philox block indices below 2^32), so the counter's constant
// words come folded (philox4x32_10_g32).
template <bool RHT, bool SR, int HW = -1, bool G32 = false>
__device__ __forceinline__ void encode_block16(float* v, float s_enc, const float* rtab, uint64_t idx0,
                                               const QuantArgs& a, uint32_t* sb_out,
                                               uint32_t* code_lo, uint32_t* code_hi,
                                               uint32_t amax_bits = ~0u) {
    if (RHT) {
        rht16_first3(v, a.rht);
        float s[8];
        rht16_pair_mags(v, s);
        const float m = fmaxf(fmax3(s[0], s[1], s[2]), fmax3(fmax3(s[3], s[4], s[5]), s[6], s[7]));
        amax_bits = __float_as_uint(__fmul_rn(m, 0.25f));
        rht16_last(v);
    } else if (amax_bits == ~0u) {
        amax_bits = absmax_bits16(v);
    }
    const uint32_t sb = block_scale_code(__uint_as_float(amax_bits), s_enc);
    const float r_b = rtab[sb];
    *sb_out = sb;
    scale16(v, r_b);
    if (SR) {
        if (HW == 1 || (HW < 0 && a.sr_hw)) {
            const uint4 w = G32 ? philox4x32_10_g32<false>((uint32_t)(idx0 >> 4), a.sr_key, a.sr_pre)
                                : sr_words16(idx0 >> 4, a.stream_id, a.sr_key);
            e2m1x16_sr(v, w, code_lo, code_hi);
        } else if (G32) {
            const uint32_t g = (uint32_t)(idx0 >> 3);
            *code_lo = e2m1x8_sr_cvt(v, philox4x32_10_g32<true>(g, a.sr_key, a.sr_pre));
            *code_hi = e2m1x8_sr_cvt(v + 8, philox4x32_10_g32<true>(g + 1, a.sr_key, a.sr_pre));
        } else {
            *code_lo = e2m1x8_sr_cvt(v, sr_rp8(idx0 >> 3, a.stream_id, a.sr_key));
            *code_hi = e2m1x8_sr_cvt(v + 8, sr_rp8((idx0 >> 3) + 1, a.stream_id, a.sr_key));
        }
    } else {
        *code_lo = e2m1x8_rne(v);
        *code_hi = e2m1x8_rne(v + 8);
    }
}

// ===================================================== quantise 16x16 ======
// CTA (128 threads) = 64 stored rows x 128 stored columns.  Warp w owns rows
// 16w..16w+15; lane l owns row 16w + (l & 15) and columns 64*(l >> 4) ..
// +63 of the CTA tile.  Grid: x over 128-column tiles, y over 64-row tiles
// (covering the 128-padded row count).
constexpr int k2DThreads = 128;

// In-register transpose of an 8x8 matrix of nibbles: on entry x[i] holds
// row i (nibble n = column n, low nibble first); on exit x[n] holds column n
// (nibble i = row i).  Three independent swaps of row and column index bits:
// bit 2 (16-bit halves) and bit 1 (bytes) by byte permutes, bit 0 (nibbles)
// by masks.
__device__ __forceinline__ void transpose8x8_nibbles(uint32_t* x) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = x[i], b = x[i + 4];
        x[i] = __byte_perm(a, b, 0x5410);
        x[i + 4] = __byte_perm(a, b, 0x7632);
    }
#pragma unroll
    for (int i = 0; i < 8; i += (i & 1) ? 3 : 1) {      // 0, 1, 4, 5
        const uint32_t a = x[i], b = x[i + 2];
        x[i] = __byte_perm(a, b, 0x6240);
        x[i + 2] = __byte_perm(a, b, 0x7351);
    }
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        const uint32_t a = x[i], b = x[i + 1];
        x[i] = (a & 0x0F0F0F0Fu) | ((b << 4) & 0xF0F0F0F0u);
        x[i + 1] = ((a >> 4) & 0x0F0F0F0Fu) | (b & 0xF0F0F0F0u);
    }
}

// Code tile of the transposed emit: 64 rows x 16 words (128 nibbles), stored
// swizzled so that both the producer's 16-byte row writes (8 consecutive rows
// per quarter-warp) and the transposer's word reads (8 row blocks x 4 word
// columns per warp) are free of bank conflicts.  Logical (row R, 16-byte
// chunk q, word u) lives at physical row R ^ bit3(R) and chunk
// q ^ ((R >> 1) ^ (R >> 4)) & 3.
__device__ __forceinline__ int tile_word(int R, int w) {
    const int rp = R ^ ((R >> 3) & 1);
    const int qp = (w >> 2) ^ (((R >> 1) ^ (R >> 4)) & 3);
    return rp * 16 + qp * 4 + (w & 3);
}

// Persistent CTAs walk the 64-row x 128-column tiles (covering the
// 128-padded row count) through a ring of kQ2Stages shared-memory slots.  A
// tile arrives as two 64 x 64 boxes (TMA, 128-byte swizzle: 16-byte chunk c
// of row r of a box at chunk c ^ (r & 7); zeros beyond the array), so that a
// quarter warp's reads of one chunk of 8 consecutive rows hit distinct banks.
constexpr int kQ2Stages = 3;
constexpr int kQ2BoxBytes = 64 * 64 * 2;                           // 8 KB
constexpr int kQ2TileBytes = 2 * kQ2BoxBytes;                      // 16 KB
constexpr int kQ2Smem = kQ2Stages * kQ2TileBytes + 1024 + 64;      // + alignment slack, barriers
constexpr int kQ2CtasPerSm = 4;

// Rounding of the 16x16 quantiser, a template parameter so that an
// instantiation carries only its own code: RNE; NVFP4_SR or NVFP4_SR_HW with
// the element index taken in the operand's layout; the same two with the
// index taken in the transposed layout (a transposed input view).
enum Q2Round : int { kQ2Rne = 0, kQ2Sr = 1, kQ2SrHw = 2, kQ2SrT = 3, kQ2SrHwT = 4 };

template <bool RHT, int SRM, bool EMIT_T>
__global__ void __launch_bounds__(k2DThreads, kQ2CtasPerSm) k_quant2d(const __grid_constant__ CUtensorMap map,
                                                                      const __grid_constant__ QuantArgs a) {
    constexpr bool SR = SRM != kQ2Rne;
    extern __shared__ uint8_t q2_raw[];
    uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(q2_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + kQ2Stages * kQ2TileBytes);
    __shared__ __align__(16) uint32_t tile_codes[64 * 16];
    __shared__ uint8_t tile_sb[4][8];          // [row block][k block]
    __shared__ int abort_flag;
    // encode factors r_b from a per-CTA table of the 128 E4M3 codes where the
    // kernel is bound by instructions (stochastic rounding, RHT, transposed
    // emit); the plain RNE kernel, bound by HBM, divides per block
    constexpr bool kTable = SR || RHT || EMIT_T;
    __shared__ float rtab[kTable ? 128 : 1];
    float s_enc;
    if (!resolve_scale(a.scale_src, a.src_is_senc, a.gs_out, a.gs_out2, &s_enc)) return;
    if constexpr (kTable) init_rtab(rtab, s_enc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nkb = a.k >> 4;
    const int64_t ngroups = (nkb + 3) >> 2;
    const int64_t row_tiles = ((a.rows + 127) & ~int64_t(127)) / 64;
    const int64_t col_tiles = (a.k + 127) / 128;
    const int64_t ntiles = row_tiles * col_tiles;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kQ2Stages; ++st) mbar_init(&full[st], 1);
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&map);
    }
    __syncthreads();
    auto issue = [&](int64_t t, int st) {
        const int64_t tr = t / col_tiles, tc = t - tr * col_tiles;
        mbar_arrive_expect_tx(&full[st], kQ2TileBytes);
        tma_load_2d(ring + st * kQ2TileBytes, &map, &full[st], (int32_t)(tc * 128), (int32_t)(tr * 64));
        tma_load_2d(ring + st * kQ2TileBytes + kQ2BoxBytes, &map, &full[st], (int32_t)(tc * 128 + 64),
                    (int32_t)(tr * 64));
    };
    if (threadIdx.x == 0)
        for (int st = 0; st < kQ2Stages; ++st) {
            const int64_t t = (int64_t)blockIdx.x + (int64_t)st * gridDim.x;
            if (t < ntiles) issue(t, st);
        }
    const int lr = warp * 16 + (lane & 15);    // tile row of this lane
    const int lg = lane >> 4;                  // 64-column half of the tile (= box)

    int it = 0;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x, ++it) {
        const int slot = it % kQ2Stages;
        const bool got = mbar_wait_bounded(&full[slot], (uint32_t)(it / kQ2Stages) & 1u, &abort_flag);
        __syncthreads();                       // every thread saw the same outcome
        if (abort_flag || !got) break;
        const int64_t tr = t / col_tiles, tc = t - tr * col_tiles;
        const int64_t row0 = tr * 64;
        const int64_t r = row0 + lr;
        const int64_t g = tc * 2 + lg;
        const bool row_ok = r < a.rows;
        const bool grp_ok = g < ngroups;
        const int nblk = grp_ok ? (int)min64(4, nkb - g * 4) : 0;

        float v[4][16];
        uint32_t lmax[4];
        {
            const uint8_t* tile = ring + slot * kQ2TileBytes + lg * kQ2BoxBytes + lr * 128;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                if (row_ok && b < nblk) {
                    unpack8(*reinterpret_cast<const uint4*>(tile + (((2 * b) ^ (lr & 7)) << 4)), v[b]);
                    unpack8(*reinterpret_cast<const uint4*>(tile + (((2 * b + 1) ^ (lr & 7)) << 4)), v[b] + 8);
                    if (RHT) rht16(v[b], a.rht);
                    lmax[b] = absmax_bits16(v[b]);
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[b][j] = 0.0f;
                    lmax[b] = 0u;
                }
            }
        }
        __syncthreads();                       // slot fully read: refill it
        if (threadIdx.x == 0) {
            const int64_t tn = t + (int64_t)kQ2Stages * gridDim.x;
            if (tn < ntiles) issue(tn, slot);
        }
        // 16x16 block amax: reduce over the 16 lanes holding the block's rows.
    #pragma unroll
        for (int b = 0; b < 4; ++b) {
    #pragma unroll
            for (int off = 1; off < 16; off <<= 1)
                lmax[b] = max(lmax[b], __shfl_xor_sync(0xFFFFFFFFu, lmax[b], off));
        }
        uint32_t sw = 0, cw[8];
    #pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t sb = (b < nblk) ? block_scale_code(__uint_as_float(lmax[b]), s_enc) : 0u;
            const float r_b = (b < nblk) ? (kTable ? rtab[sb] : encode_factor(s_enc, sb)) : 0.0f;
            sw |= sb << (8 * b);
            scale16(v[b], r_b);
            if (SR) {
                uint32_t lo = 0, hi = 0;
                if (row_ok && b < nblk) {
                    const int64_t c0 = g * 64 + b * 16;
                    if constexpr (SRM == kQ2SrHwT) {
                        // index in the transposed logical layout: (r, c) -> c * rows + r;
                        // rows is a multiple of 16, so every element of the strip
                        // takes the same word ((r % 16) / 4) and element position
                        // (r % 4) of its own Philox block.
                        const int wsel = (r >> 2) & 3, pos = r & 3;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint64_t idx = (uint64_t)((c0 + j) * a.rows + r);
                            const uint4 rb = sr_words16(idx >> 4, a.stream_id, a.sr_key);
                            const uint32_t w = wsel == 0 ? rb.x : wsel == 1 ? rb.y : wsel == 2 ? rb.z : rb.w;
                            const uint32_t q = e2m1_sr_at(v[b][j], w, pos);
                            if (j < 8) lo |= q << (4 * j);
                            else hi |= q << (4 * (j - 8));
                        }
                    } else if constexpr (SRM == kQ2SrT) {
                        // every element of the strip takes the same slice (r & 7)
                        // of its own Philox block
                        const uint32_t wsel = (uint32_t)(r & 7) >> 1;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint64_t idx = (uint64_t)((c0 + j) * a.rows + r);
                            const uint4 rb = sr_rp8(idx >> 3, a.stream_id, a.sr_key);
                            const uint32_t w = wsel == 0 ? rb.x : wsel == 1 ? rb.y : wsel == 2 ? rb.z : rb.w;
                            const uint32_t q = e2m1_sr_rp_at(v[b][j], w, (r & 1) != 0);
                            if (j < 8) lo |= q << (4 * j);
                            else hi |= q << (4 * (j - 8));
                        }
                    } else if constexpr (SRM == kQ2SrHw) {
                        const uint64_t idx0 = (uint64_t)(r * a.k + c0);
                        e2m1x16_sr(v[b], sr_words16(idx0 >> 4, a.stream_id, a.sr_key), &lo, &hi);
                    } else {
                        const uint64_t idx0 = (uint64_t)(r * a.k + c0);
                        if (a.sr_g32) {                      // uniform: block indices below 2^32
                            const uint32_t g8 = (uint32_t)(idx0 >> 3);
                            lo = e2m1x8_sr_cvt(v[b], philox4x32_10_g32<true>(g8, a.sr_key, a.sr_pre));
                            hi = e2m1x8_sr_cvt(v[b] + 8, philox4x32_10_g32<true>(g8 + 1, a.sr_key, a.sr_pre));
                        } else {
                            lo = e2m1x8_sr_cvt(v[b], sr_rp8(idx0 >> 3, a.stream_id, a.sr_key));
                            hi = e2m1x8_sr_cvt(v[b] + 8, sr_rp8((idx0 >> 3) + 1, a.stream_id, a.sr_key));
                        }
                    }
                }
                cw[2 * b] = lo;
                cw[2 * b + 1] = hi;
            } else {
                cw[2 * b] = e2m1x8_rne(v[b]);
                cw[2 * b + 1] = e2m1x8_rne(v[b] + 8);
            }
        }
        // primary operand
        if (a.write_primary && grp_ok) {
            uint32_t* sdst = reinterpret_cast<uint32_t*>(a.scales + scale_offset(r, g * 4, ngroups));
            if (r < ((a.rows + 127) & ~int64_t(127)) &&
                NVFP4_GUARD(a.scales, scales_extent(a.rows, a.k), sdst, 4, kGuardQ2dScales))
                *sdst = row_ok ? sw : 0u;
            if (row_ok) {
                uint8_t* cdst = a.codes + r * (a.k >> 1) + g * 32;
                if (!NVFP4_GUARD(a.codes, codes_extent(a.rows, a.k), cdst, 8 * nblk, kGuardQ2dCodes)) {
                } else if (nblk == 4 && (a.k & 31) == 0) {
                    reinterpret_cast<uint4*>(cdst)[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    reinterpret_cast<uint4*>(cdst)[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
                } else {
    #pragma unroll
                    for (int b = 0; b < 4; ++b)
                        if (b < nblk)
                            reinterpret_cast<uint2*>(cdst)[b] = make_uint2(cw[2 * b], cw[2 * b + 1]);
                }
            }
        }
        if (EMIT_T) {
            // transposed operand: rows = k, k = a.rows (a multiple of 16 here)
            {
                const int R = warp * 16 + (lane & 15);
                const bool live = row_ok && grp_ok;
                const int h = lane >> 4;
                *reinterpret_cast<uint4*>(&tile_codes[tile_word(R, 8 * h)]) =
                    live ? make_uint4(cw[0], cw[1], cw[2], cw[3]) : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(&tile_codes[tile_word(R, 8 * h + 4)]) =
                    live ? make_uint4(cw[4], cw[5], cw[6], cw[7]) : make_uint4(0, 0, 0, 0);
                if ((lane & 15) == 0) {
#pragma unroll
                    for (int b = 0; b < 4; ++b) tile_sb[warp][h * 4 + b] = (sw >> (8 * b)) & 0xFFu;
                }
            }
            __syncthreads();
            const int64_t kt = a.rows;                                 // k of the transposed operand
            const int64_t ngroups_t = ((kt >> 4) + 3) >> 2;
            const int64_t gt = row0 >> 6;                              // 4 blocks of 16 rows
            if (gt < ngroups_t) {                                      // else beyond the padded columns
                // scales: thread = one row (stored column) of the transposed operand
                const int64_t ct = tc * 128 + threadIdx.x;
                const int64_t ct_pad = (a.k + 127) & ~int64_t(127);
                if (ct < ct_pad) {
                    uint32_t* sdst_t =
                        reinterpret_cast<uint32_t*>(a.scales_t + scale_offset(ct, gt * 4, ngroups_t));
                    const int kb_local = threadIdx.x >> 4;
                    if (NVFP4_GUARD(a.scales_t, scales_extent(a.k, kt), sdst_t, 4, kGuardQ2dScalesT))
                        *sdst_t = ct >= a.k ? 0u
                                        : (uint32_t)tile_sb[0][kb_local] | ((uint32_t)tile_sb[1][kb_local] << 8) |
                                              ((uint32_t)tile_sb[2][kb_local] << 16) |
                                              ((uint32_t)tile_sb[3][kb_local] << 24);
                }
                // codes: thread = 8 stored rows (rb) x 8 stored columns (cb) of the
                // tile, transposed in registers; a warp writes 4 columns x 32
                // contiguous bytes.
                const int rb = threadIdx.x & 7, cb = threadIdx.x >> 3;
                const int64_t rows_here = min64(64, a.rows - row0);    // multiple of 16 when > 0
                if (rb * 8 < rows_here) {
                    uint32_t x[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) x[q] = tile_codes[tile_word(rb * 8 + q, cb)];
                    transpose8x8_nibbles(x);
                    const int64_t c0 = tc * 128 + cb * 8;
                    uint8_t* cdst = a.codes_t + c0 * (kt >> 1) + (row0 >> 1) + rb * 4;
#pragma unroll
                    for (int n = 0; n < 8; ++n)
                        if (c0 + n < a.k &&
                            NVFP4_GUARD(a.codes_t, codes_extent(a.k, kt), cdst + n * (kt >> 1), 4, kGuardQ2dCodesT))
                            *reinterpret_cast<uint32_t*>(cdst + n * (kt >> 1)) = x[n];
                }
            }
        }
    }
    // drain: no copy may still be writing into this CTA's shared memory
    if (threadIdx.x == 0 && abort_flag) {
        for (int k = 0; k < kQ2Stages; ++k) {
            const int ii = it + k;
            const int64_t t = (int64_t)blockIdx.x + (int64_t)ii * gridDim.x;
            if (t < ntiles) mbar_wait_bounded(&full[ii % kQ2Stages], (uint32_t)(ii / kQ2Stages) & 1u, nullptr);
        }
    }
}

// ======================================================== dequantise ======
// Two copies of the scale value as f16x2 (exact: a block scale is an E4M3
// value, at most 480 in magnitude with 4 significant bits).
__device__ __forceinline__ uint32_t f16x2_splat(float s) {
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(d) : "f"(s));
    return d;
}

// q * s_b for the 8 E2M1 codes of a word (element j in nibble j), exactly,
// as 8 floats: the hardware conversion decodes the codes in pairs to f16x2
// (exact), one f16x2 multiply per pair forms q * s_b (exact: |q s_b| <= 6 *
// 480 with at most 6 significant bits, and never below 2^-10, the f16
// normal range), and the products are widened to fp32 (exact).
__device__ __forceinline__ void e2m1x8_times_scale(uint32_t codes, uint32_t sb2, float* p) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
        "mov.b32 {c0, c1, c2, c3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, c0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, c2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(codes));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        asm("{\n\t.reg .f16 lo, hi;\n\t"
            "mul.rn.f16x2 %2, %2, %3;\n\t"
            "mov.b32 {lo, hi}, %2;\n\t"
            "cvt.f32.f16 %0, lo;\n\t"
            "cvt.f32.f16 %1, hi;\n\t}"
            : "=f"(p[2 * j]), "=f"(p[2 * j + 1]), "+r"(h[j])
            : "r"(sb2));
    }
}

// The walk of the dequantisers.  A warp takes 256 consecutive elements of a
// row at a time, 8 per lane, so that its code loads (4 bytes a lane) and its
// output stores (16 or 32 bytes a lane) each cover one contiguous span; the
// (row, chunk) walk is warp-uniform and free of 64-bit divides, and a warp
// gathers the loads of kDeqUnroll chunks before it converts and stores
// them.  decode(codes, scale byte, o) turns a lane's 8 codes and the scale
// byte of their block (BLOCK elements, swizzled layout) into 8 floats.
constexpr int kDeqUnroll = 4;

template <bool BF16, int BLOCK, class Decode>
__device__ __forceinline__ void dequant_walk(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                                             uint64_t scales_ext, int64_t rows, int64_t k, void* out, int64_t ld,
                                             uint32_t site_in, uint32_t site_out, Decode decode) {
    const int lane = threadIdx.x & 31;
    const int64_t col_tiles = ((k / BLOCK) + 3) >> 2;
    const uint32_t nchunks = (uint32_t)((k + 255) >> 8);
    const int64_t w0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    int64_t r = w0 / nchunks;
    uint32_t ch = (uint32_t)(w0 - r * nchunks);
    const int64_t dr = nw / nchunks;
    const uint32_t dch = (uint32_t)(nw - dr * nchunks);
    while (r < rows) {
        uint32_t cw[kDeqUnroll], sc[kDeqUnroll];
        int64_t e0[kDeqUnroll];
        bool ok[kDeqUnroll];
#pragma unroll
        for (int u = 0; u < kDeqUnroll; ++u) {
            const int64_t c = (int64_t)ch * 256 + lane * 8;            // c < k implies c + 8 <= k
            ok[u] = r < rows && c < k;
            cw[u] = 0u;
            sc[u] = 0u;
            e0[u] = r * ld + c;
            if (ok[u]) {
                const uint8_t* csrc = codes + r * (k >> 1) + (c >> 1);
                const uint8_t* ssrc = scales + scale_offset(r, c / BLOCK, col_tiles);
                if (NVFP4_GUARD(codes, codes_extent(rows, k), csrc, 4, site_in))
                    cw[u] = __ldg(reinterpret_cast<const uint32_t*>(csrc));
                if (NVFP4_GUARD(scales, scales_ext, ssrc, 1, site_in)) sc[u] = __ldg(ssrc);
            }
            ch += dch;
            r += dr;
            if (ch >= nchunks) {
                ch -= nchunks;
                ++r;
            }
        }
#pragma unroll
        for (int u = 0; u < kDeqUnroll; ++u) {
            if (!ok[u]) continue;
            float o[8];
            decode(cw[u], sc[u], o);
            if (BF16) {
                uint32_t p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * j], o[2 * j + 1]);
                    p[j] = *reinterpret_cast<const uint32_t*>(&h);
                }
                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(out) + e0[u]);
                if (NVFP4_GUARD(out, stored_extent(rows, k, ld, 2), dst, 16, site_out))
                    *dst = make_uint4(p[0], p[1], p[2], p[3]);
            } else {
                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + e0[u]);
                if (NVFP4_GUARD(out, stored_extent(rows, k, ld, 4), dst, 32, site_out)) {
                    dst[0] = make_float4(o[0], o[1], o[2], o[3]);
                    dst[1] = make_float4(o[4], o[5], o[6], o[7]);
                }
            }
        }
    }
}

// x_hat = fp32(fp32(q * s_b) * fp32(1 / S_enc)), as fp32 or bf16 (RNE).
template <bool BF16>
__global__ void __launch_bounds__(kQuantThreads) k_dequant(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales,
                                                           const float* __restrict__ gs,
                                                           int64_t rows, int64_t k, void* out,
                                                           int64_t ld) {
    const float inv = __frcp_rn(*gs);
    dequant_walk<BF16, 16>(codes, scales, scales_extent(rows, k), rows, k, out, ld, kGuardDeqIn, kGuardDeqOut,
                           [inv](uint32_t cw, uint32_t sc, float* o) {
                               e2m1x8_times_scale(cw, f16x2_splat(e4m3_value(sc)), o);
#pragma unroll
                               for (int j = 0; j < 8; ++j) o[j] = __fmul_rn(o[j], inv);
                           });
}

}  // namespace nvfp4
