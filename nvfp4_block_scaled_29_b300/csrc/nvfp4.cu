// nvfp4.cu -- the C ABI of libnvfp4 (declared in include/nvfp4.h).
//
// One translation unit: it includes every kernel header, validates arguments
// on the host, chooses launch shapes and encodes the TMA tensor maps.  The
// library allocates no memory; the only state is the device status word and
// small per-device caches of launch attributes.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <atomic>
#include <cstdint>
#include <cstring>

#include "../../include/nvfp4.h"
#include "codec.cuh"
#include "gemm.cuh"
#include "gemm2sm.cuh"
#include "dual.cuh"
#include "mx.cuh"
#include "quantize.cuh"
#include "status.cuh"

namespace {

using namespace nvfp4;

constexpr int kMaxDevices = 64;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int device_sm_count() {
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = 148;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

nvfp4_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

int grid_for(int64_t items, int threads, int per_sm) {
    const int64_t need = cdiv(items, threads);
    const int64_t cap = (int64_t)device_sm_count() * per_sm;
    return (int)std::max<int64_t>(1, std::min(need, cap));
}

// ------------------------------------------------------------- validation --
nvfp4_status check_view(const nvfp4_bf16_view& x, bool need_k16) {
    if (x.rows < 0 || x.cols < 0) return NVFP4_ERR_INVALID_ARG;
    if (x.transposed != 0 && x.transposed != 1) return NVFP4_ERR_INVALID_ARG;
    if (need_k16 && (x.cols % 16) != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (x.rows == 0 || x.cols == 0) return NVFP4_OK;
    if (x.ptr == nullptr) return NVFP4_ERR_INVALID_ARG;
    const int64_t min_ld = x.transposed ? x.rows : x.cols;
    if (x.ld < min_ld) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(x.ptr, 16) || (x.ld % 8) != 0) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

// A quantised operand of logical shape [rows x k]: NVFP4 operands need their
// global scale, MXFP4 operands (need_gs = false) have none.
nvfp4_status check_q(const nvfp4_q* q, int64_t rows, int64_t k, bool need_gs = true) {
    if (q == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (q->rows != rows || q->k != k) return NVFP4_ERR_INVALID_ARG;
    if (need_gs && (q->global_scale == nullptr || !aligned(q->global_scale, 4))) return NVFP4_ERR_INVALID_ARG;
    if (rows == 0 || k == 0) return NVFP4_OK;
    if (q->codes == nullptr || q->scales == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(q->codes, 16) || !aligned(q->scales, 16)) return NVFP4_ERR_MISALIGNED;
    return NVFP4_OK;
}

// ----------------------------------------------------------- tensor maps ---
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::atomic<EncodeTiledFn> fn{nullptr};
    EncodeTiledFn f = fn.load();
    if (f) return f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
        return nullptr;
    f = reinterpret_cast<EncodeTiledFn>(p);
    fn.store(f);
    return f;
}

// A stored bf16 array [rows x cols] (leading dimension ld) in the streamed
// amax's tiles: box 256 columns x 64 rows, no swizzle, zeros beyond.
// Test-only fault injection (nvfp4_debug_inject): 1 = the next streamed amax
// launch skips the copy of its first tile.
std::atomic<int> g_fault_injection{0};
// Test-only (nvfp4_debug_inject mode 2): the next dual quantise takes its
// general 64-bit Philox block-index path even though the indices fit 32 bits.
std::atomic<int> g_force_g64{0};

// 2D map of a stored bf16 array [rows x cols] (leading dimension ld) with a
// box of box_rows x box_cols elements.
bool make_bf16_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld, uint32_t box_cols,
                   uint32_t box_rows, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bf16_tile_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int64_t ld) {
    return make_bf16_map(m, ptr, rows, cols, ld, kAmaxTileCols, kAmaxTileRows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// RHT-16 sign multipliers of a 16-bit mask (all +1 for mask 0).
RhtSigns rht_signs(uint32_t mask) {
    RhtSigns sg;
    auto sgn = [&](int j) { return ((mask >> j) & 1u) ? -1.0f : 1.0f; };
    for (int k = 0; k < 8; ++k) {
        sg.p[k] = make_float2(sgn(k), sgn(k + 8));
        sg.n[k] = make_float2(-sgn(k), -sgn(k + 8));
    }
    return sg;
}

// Streamed amax of a stored array (plain, and with RHT down the columns when
// mask != 0); out_t may equal out_plain when mask == 0.
nvfp4_status launch_amax_stream(const void* ptr, int64_t srows, int64_t scols, int64_t ld, uint32_t mask,
                                float* out_plain, float* out_t, cudaStream_t st) {
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    if (!ready[dev].load()) {
        if (cudaFuncSetAttribute(k_amax_stream<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAmaxSmem) !=
                cudaSuccess ||
            cudaFuncSetAttribute(k_amax_stream<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAmaxSmem) !=
                cudaSuccess)
            return NVFP4_ERR_CUDA;
        ready[dev].store(1);
    }
    CUtensorMap map;
    if (!make_bf16_tile_map(&map, ptr, srows, scols, ld)) return NVFP4_ERR_CUDA;
    const int64_t tiles = cdiv(srows, kAmaxTileRows) * cdiv(scols, kAmaxTileCols);
    const int g = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)device_sm_count() * 2));
    const RhtSigns sg = rht_signs(mask);
    const int64_t skip = g_fault_injection.exchange(0) == 1 ? 0 : -1;   // test-only, one launch
    if (mask) k_amax_stream<true><<<g, kAmaxThreads, kAmaxSmem, st>>>(map, srows, scols, sg, out_plain, out_t, skip);
    else k_amax_stream<false><<<g, kAmaxThreads, kAmaxSmem, st>>>(map, srows, scols, sg, out_plain, out_t, skip);
    return launch_status();
}

// ------------------------------------------------------------------ amax ---
nvfp4_status launch_amax(const nvfp4_bf16_view& x, uint32_t mask, float* out, cudaStream_t st) {
    if (cudaMemsetAsync(out, 0, sizeof(float), st) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (x.rows == 0 || x.cols == 0) return NVFP4_OK;
    const uint16_t* p = static_cast<const uint16_t*>(x.ptr);
    const int64_t srows = x.transposed ? x.cols : x.rows;
    const int64_t scols = x.transposed ? x.rows : x.cols;
    if (mask == 0) {
        if (x.ld == scols || srows == 1) {
            const int64_t len = srows * scols;
            k_amax_plain<<<grid_for(cdiv(len, 128), kQuantThreads, 3), kQuantThreads, 0, st>>>(
                p, 1, len, x.ld, out);
        } else {
            return launch_amax_stream(p, srows, scols, x.ld, 0, out, out, st);
        }
    } else if (!x.transposed) {
        k_amax_rht_rows<<<grid_for(x.rows * (x.cols / 16), kQuantThreads, 8), kQuantThreads, 0, st>>>(
            p, x.rows, x.cols, x.ld, rht_signs(mask), out);
    } else {
        // transposed view: the RHT runs down the stored columns, the
        // column-wise half of the streamed dual amax (its plain half unused)
        return launch_amax_stream(p, x.cols, x.rows, x.ld, mask, nullptr, out, st);
    }
    return launch_status();
}

// -------------------------------------------------------------- quantise ---
// Philox round keys of the seed and the rounding mode's generator: NVFP4_SR
// runs philox4x32_10_not (complemented words, so that each half-word is
// 65535 - u16), whose round-9 pair is complemented; NVFP4_SR_HW runs the plain
// philox4x32_10.
void set_sr_keys(QuantArgs* a, uint64_t seed, uint64_t stream_id, nvfp4_round round, int64_t n_elems) {
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    const bool hw = round == NVFP4_SR_HW;
    for (int r = 0; r < 10; ++r) {
        a->sr_key[2 * r] = (r == 9 && !hw) ? ~k0 : k0;
        a->sr_key[2 * r + 1] = (r == 9 && !hw) ? ~k1 : k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    a->sr_hw = hw ? 1 : 0;
    a->stream_id = stream_id;
    // rounds 0 and 1 of Philox on the counter (g, 0, stream_lo, stream_hi):
    // everything but g is fixed per call (see philox4x32_10_g32)
    const uint32_t s_lo = (uint32_t)stream_id, s_hi = (uint32_t)(stream_id >> 32);
    const uint32_t k00 = (uint32_t)seed, k10 = (uint32_t)(seed >> 32);
    const uint32_t k01 = k00 + 0x9E3779B9u, k11 = k10 + 0xBB67AE85u;
    const uint64_t t = (uint64_t)s_lo * 0xCD9E8D57u;
    const uint32_t a0 = (uint32_t)(t >> 32) ^ k00, a1 = (uint32_t)t;
    const uint64_t p = (uint64_t)a0 * 0xD2511F53u;
    a->sr_pre[0] = s_hi ^ k10;
    a->sr_pre[1] = a1 ^ k01;
    a->sr_pre[2] = (uint32_t)(p >> 32) ^ k11;
    a->sr_pre[3] = (uint32_t)p;
    // the block index g = idx / 8 (idx / 16 for NVFP4_SR_HW) stays below 2^32
    a->sr_g32 = n_elems <= (int64_t(1) << 35) ? 1 : 0;
}

bool valid_round(nvfp4_round r) { return r == NVFP4_RNE || r == NVFP4_SR || r == NVFP4_SR_HW; }

template <bool RHT, int SRM, bool EMIT_T>
nvfp4_status launch_q2d_t(const CUtensorMap& map, const QuantArgs& a, int grid, cudaStream_t st) {
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    if (!ready[dev].load()) {
        if (cudaFuncSetAttribute(k_quant2d<RHT, SRM, EMIT_T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kQ2Smem) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ready[dev].store(1);
    }
    k_quant2d<RHT, SRM, EMIT_T><<<grid, k2DThreads, kQ2Smem, st>>>(map, a);
    return launch_status();
}

// 16x16 quantisation; srm is the kernel's rounding (Q2Round), emit_t the
// transposed emit.  The instantiations a call can reach: non-transposed views
// with or without the RHT (RNE, NVFP4_SR, NVFP4_SR_HW; the transposed emit
// without the RHT), transposed views with the emit (transposed-index modes).
nvfp4_status launch_q2d(const QuantArgs& a, bool rht, int srm, bool emit_t, cudaStream_t st) {
    CUtensorMap map;
    if (!make_bf16_map(&map, a.x, a.rows, a.k, a.ld, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return NVFP4_ERR_CUDA;
    const int64_t tiles = (cdiv(a.rows, 128) * 2) * cdiv(a.k, 128);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)device_sm_count() * kQ2CtasPerSm));
    if (rht) {
        if (emit_t) return NVFP4_ERR_INVALID_ARG;
        switch (srm) {
            case kQ2Rne: return launch_q2d_t<true, kQ2Rne, false>(map, a, grid, st);
            case kQ2Sr: return launch_q2d_t<true, kQ2Sr, false>(map, a, grid, st);
            case kQ2SrHw: return launch_q2d_t<true, kQ2SrHw, false>(map, a, grid, st);
            default: return NVFP4_ERR_INVALID_ARG;
        }
    }
    switch (srm) {
        case kQ2Rne: return emit_t ? launch_q2d_t<false, kQ2Rne, true>(map, a, grid, st)
                                   : launch_q2d_t<false, kQ2Rne, false>(map, a, grid, st);
        case kQ2Sr: return emit_t ? launch_q2d_t<false, kQ2Sr, true>(map, a, grid, st)
                                  : launch_q2d_t<false, kQ2Sr, false>(map, a, grid, st);
        case kQ2SrHw: return emit_t ? launch_q2d_t<false, kQ2SrHw, true>(map, a, grid, st)
                                    : launch_q2d_t<false, kQ2SrHw, false>(map, a, grid, st);
        case kQ2SrT: return emit_t ? launch_q2d_t<false, kQ2SrT, true>(map, a, grid, st) : NVFP4_ERR_INVALID_ARG;
        case kQ2SrHwT: return emit_t ? launch_q2d_t<false, kQ2SrHwT, true>(map, a, grid, st) : NVFP4_ERR_INVALID_ARG;
    }
    return NVFP4_ERR_INVALID_ARG;
}

template <int PATHS, bool RHT>
nvfp4_status launch_dual_single_sr(const DualArgs& d, int sr, cudaStream_t st);

nvfp4_status quantize_impl(const nvfp4_bf16_view& x, uint32_t mask, const float* amax_dev,
                           nvfp4_round round, uint64_t seed, uint64_t stream_id, nvfp4_q* out,
                           nvfp4_q* out_t, bool block2d, cudaStream_t st) {
    nvfp4_status s = check_view(x, true);
    if (s != NVFP4_OK) return s;
    if (mask > 0xFFFFu) return NVFP4_ERR_INVALID_ARG;
    if (!valid_round(round)) return NVFP4_ERR_INVALID_ARG;
    if ((s = check_q(out, x.rows, x.cols)) != NVFP4_OK) return s;
    if (out_t != nullptr) {
        if (!block2d || mask != 0) return NVFP4_ERR_INVALID_ARG;
        if ((s = check_q(out_t, x.cols, x.rows)) != NVFP4_OK) return s;
        if (x.rows % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    }
    if (block2d && x.transposed) {
        if (mask != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
        if (x.rows % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    }
    if (amax_dev != nullptr && (amax_dev == out->global_scale ||
                                (out_t != nullptr && amax_dev == out_t->global_scale)))
        return NVFP4_ERR_INVALID_ARG;
    if (amax_dev != nullptr && !aligned(amax_dev, 4)) return NVFP4_ERR_MISALIGNED;

    // global scale source
    const float* src = amax_dev;
    int src_is_senc = 0;
    if (amax_dev == nullptr) {
        if ((s = launch_amax(x, mask, out->global_scale, st)) != NVFP4_OK) return s;
        k_amax_to_senc<<<1, 1, 0, st>>>(out->global_scale);
        src = out->global_scale;
        src_is_senc = 1;
    }
    if (x.rows == 0 || x.cols == 0) {
        // nothing to encode: publish S_enc only
        k_publish_senc<<<1, 1, 0, st>>>(src, src_is_senc, out->global_scale,
                                        out_t ? out_t->global_scale : nullptr);
        return launch_status();
    }

    QuantArgs a{};
    a.x = static_cast<const uint16_t*>(x.ptr);
    a.ld = x.ld;
    a.scale_src = src;
    a.src_is_senc = src_is_senc;
    a.gs_out = out->global_scale;
    a.gs_out2 = out_t ? out_t->global_scale : nullptr;
    a.rht = rht_signs(mask);
    set_sr_keys(&a, seed, stream_id, round, x.rows * x.cols);
    const bool sr = round != NVFP4_RNE;

    if (!block2d) {
        a.rows = x.rows;
        a.k = x.cols;
        a.codes = out->codes;
        a.scales = out->scales;
        a.write_primary = 1;
        // TMA-fed persistent path (one path of the dual kernel): the stored
        // array is read in swizzled tiles; a transposed view is the
        // column-wise path over the stored array (logical rows in pairs, an
        // odd last row paired with a padding row)
        DualArgs d{};
        const int r = (int)round;
        if (!x.transposed) {
            d.row = a;
            return mask ? launch_dual_single_sr<1, true>(d, r, st) : launch_dual_single_sr<1, false>(d, r, st);
        }
        d.col = a;                              // the logical operand [x.rows x x.cols]
        d.row.x = a.x;                          // the stored array S = [x.cols x x.rows]
        d.row.rows = x.cols;
        d.row.k = x.rows;
        d.row.ld = x.ld;
        return mask ? launch_dual_single_sr<2, true>(d, r, st) : launch_dual_single_sr<2, false>(d, r, st);
    }
    if (!x.transposed) {
        a.rows = x.rows;
        a.k = x.cols;
        a.codes = out->codes;
        a.scales = out->scales;
        a.write_primary = 1;
        a.codes_t = out_t ? out_t->codes : nullptr;
        a.scales_t = out_t ? out_t->scales : nullptr;
        a.idx_transposed = 0;
        const bool emit = out_t != nullptr;
        const int srm = !sr ? kQ2Rne : round == NVFP4_SR_HW ? kQ2SrHw : kQ2Sr;
        return launch_q2d(a, mask != 0, srm, emit, st);
    }
    // 16x16 on a transposed view: quantise the stored [k x rows] array; its
    // primary output is the caller's out_t, its transposed emit the caller's out.
    a.rows = x.cols;
    a.k = x.rows;
    a.write_primary = out_t != nullptr;
    a.codes = out_t ? out_t->codes : nullptr;
    a.scales = out_t ? out_t->scales : nullptr;
    a.codes_t = out->codes;
    a.scales_t = out->scales;
    a.idx_transposed = 1;
    const int srm = !sr ? kQ2Rne : round == NVFP4_SR_HW ? kQ2SrHwT : kQ2SrT;
    return launch_q2d(a, false, srm, true, st);
}

// ------------------------------------------------------------------ dual ---
template <int SR1, int SR2, bool RHT2>
nvfp4_status launch_dual_t(const CUtensorMap& map, const DualArgs& d, int grid, cudaStream_t st) {
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    if (!ready[dev].load()) {
        if (cudaFuncSetAttribute(k_quant_dual<SR1, SR2, RHT2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDqSmem) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ready[dev].store(1);
    }
    k_quant_dual<SR1, SR2, RHT2><<<grid, kDqThreads, kDqSmem, st>>>(map, d);
    return launch_status();
}

template <int SR1, int SR2>
nvfp4_status launch_dual_rht(const CUtensorMap& map, const DualArgs& d, bool rht2, int grid, cudaStream_t st) {
    return rht2 ? launch_dual_t<SR1, SR2, true>(map, d, grid, st) : launch_dual_t<SR1, SR2, false>(map, d, grid, st);
}

template <int SR1>
nvfp4_status launch_dual_sr2(const CUtensorMap& map, const DualArgs& d, int sr2, bool rht2, int grid,
                             cudaStream_t st) {
    switch (sr2) {
        case 0: return launch_dual_rht<SR1, 0>(map, d, rht2, grid, st);
        case 1: return launch_dual_rht<SR1, 1>(map, d, rht2, grid, st);
        default: return launch_dual_rht<SR1, 2>(map, d, rht2, grid, st);
    }
}

// The TMA map and grid of the dual kernel: tiles of the stored array S, whose
// dimensions d.row carries (rows = S's rows, k = S's columns) for every path.
bool dual_map_grid(const DualArgs& d, CUtensorMap* map, int* grid) {
    if (!make_bf16_map(map, d.row.x, d.row.rows, d.row.k, d.row.ld, kDqBoxCols, kDqRows, CU_TENSOR_MAP_SWIZZLE_128B))
        return false;
    const int64_t rows_pad = cdiv(d.row.rows, 128) * 128;
    const int64_t tiles = (rows_pad / kDqRows) * cdiv(d.row.k, kDqCols);
    *grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, (int64_t)device_sm_count() * 2));
    return true;
}

// One path of the dual kernel as a 1x16 quantiser (PATHS 1: the row-wise
// operand, rounding SR and RHT along its k; PATHS 2: the column-wise one).
template <int PATHS, int SR, bool RHT>
nvfp4_status launch_dual_single(const DualArgs& d, cudaStream_t st) {
    constexpr int SR1 = PATHS == 1 ? SR : 0, SR2 = PATHS == 2 ? SR : 0;
    auto kern = k_quant_dual<SR1, SR2, PATHS == 2 && RHT, PATHS, PATHS == 1 && RHT>;
    static std::atomic<int> ready[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    if (!ready[dev].load()) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kDqSmem) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        ready[dev].store(1);
    }
    CUtensorMap map;
    int grid = 0;
    if (!dual_map_grid(d, &map, &grid)) return NVFP4_ERR_CUDA;
    kern<<<grid, kDqThreads, kDqSmem, st>>>(map, d);
    return launch_status();
}

template <int PATHS, bool RHT>
nvfp4_status launch_dual_single_sr(const DualArgs& d, int sr, cudaStream_t st) {
    switch (sr) {
        case 0: return launch_dual_single<PATHS, 0, RHT>(d, st);
        case 1: return launch_dual_single<PATHS, 1, RHT>(d, st);
        default: return launch_dual_single<PATHS, 2, RHT>(d, st);
    }
}

// sr1, sr2: 0 = RNE, 1 = NVFP4_SR, 2 = NVFP4_SR_HW
nvfp4_status launch_dual(const DualArgs& d, int sr1, int sr2, bool rht2, cudaStream_t st) {
    CUtensorMap map;
    int grid = 0;
    if (!dual_map_grid(d, &map, &grid)) return NVFP4_ERR_CUDA;
    switch (sr1) {
        case 0: return launch_dual_sr2<0>(map, d, sr2, rht2, grid, st);
        case 1: return launch_dual_sr2<1>(map, d, sr2, rht2, grid, st);
        default: return launch_dual_sr2<2>(map, d, sr2, rht2, grid, st);
    }
}

// [rows x k/2] bytes of E2M1 codes, box = 128 bytes x box_rows, 128-byte swizzle.
bool make_code_map(CUtensorMap* m, const uint8_t* codes, int64_t rows, int64_t k, int box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)(k / 2), (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(k / 2)};
    const cuuint32_t box[2] = {128u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1u, 1u};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(codes), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows x cols] bf16 output, box = 64 columns x 32 rows, 128-byte swizzle.
bool make_out_map(CUtensorMap* m, void* d, int64_t rows, int64_t cols, int64_t ld) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
    const cuuint32_t box[2] = {64u, 32u};
    const cuuint32_t estr[2] = {1u, 1u};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The swizzled scale buffer of a [rows x k] operand with `block`-element
// blocks (16: NVFP4, 32: MXFP4) as a 3D tensor of u32: [row tiles][512-byte
// tiles along k][128 words]; box = the tiles of one 256-wide k block (4 or 2)
// x `box_row_tiles` row tiles.  Out-of-range boxes read 0.
bool make_scale_map(CUtensorMap* m, const uint8_t* scales, int64_t rows, int64_t k, int box_row_tiles,
                    int block = 16) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const int64_t row_tiles = cdiv(rows, 128), col_tiles = cdiv(k / block, 4);
    const cuuint64_t dims[3] = {128u, (cuuint64_t)col_tiles, (cuuint64_t)row_tiles};
    const cuuint64_t strides[2] = {512u, (cuuint64_t)(col_tiles * 512)};
    const cuuint32_t box[3] = {128u, (cuuint32_t)(gemm::BK / (4 * block)), (cuuint32_t)box_row_tiles};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(scales), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemm_smem_ready() {
    static std::atomic<int> done[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    if (done[dev].load()) return true;
    if (cudaFuncSetAttribute(gemm2::k_gemm_nvfp4_2sm<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemm2::smem_bytes_for(true)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm2::k_gemm_nvfp4_2sm<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemm2::smem_bytes_for(false)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm2::k_gemm_nvfp4_2sm<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemm2::smem_bytes_for(true, true)) != cudaSuccess ||
        cudaFuncSetAttribute(gemm2::k_gemm_nvfp4_2sm<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             gemm2::smem_bytes_for(false, true)) != cudaSuccess)
        return false;
    done[dev].store(1);
    return true;
}

struct GemmMaps {
    CUtensorMap a, b, d, sfa, sfb;
};

// Launch the CTA-pair GEMM (clusters of 2 along M); MX selects the MXFP4
// (E8M0, 32-element blocks) scale format.
template <bool TMA, bool MX = false>
nvfp4_status launch_gemm_pair(const GemmMaps& mp, const gemm::Args& g, cudaStream_t stream) {
    const int64_t units = (int64_t)(g.m_tiles / 2) * g.n_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(gemm2::THREADS);
    cfg.dynamicSmemBytes = (size_t)gemm2::smem_bytes_for(TMA, MX);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    static std::atomic<int> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
    int n = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load() : 0;
    if (n <= 0) {
        cfg.gridDim = dim3((unsigned)(device_sm_count() / 2 * 2));
        if (cudaOccupancyMaxActiveClusters(&n, gemm2::k_gemm_nvfp4_2sm<TMA, MX>, &cfg) != cudaSuccess || n <= 0)
            return NVFP4_ERR_CUDA;
        if (dev >= 0 && dev < kMaxDevices) cache[dev].store(n);
    }
    const int clusters = (int)std::min<int64_t>(n, units);
    cfg.gridDim = dim3((unsigned)(clusters * 2));
    if (cudaLaunchKernelEx(&cfg, gemm2::k_gemm_nvfp4_2sm<TMA, MX>, mp.a, mp.b, mp.d, mp.sfa, mp.sfb, g) !=
        cudaSuccess)
        return NVFP4_ERR_CUDA;
    return NVFP4_OK;
}

// Test-only: compare div6_rn(x) with the IEEE division x / 6 (__fdiv_rn) for
// every float whose bit pattern lies in [lo, hi); counts the mismatches and
// keeps the smallest mismatching pattern.
__global__ void k_check_div6(uint32_t lo, uint32_t hi, unsigned long long* mismatches, uint32_t* first_bad) {
    unsigned long long local = 0;
    uint32_t first = 0xFFFFFFFFu;
    const uint64_t n = (uint64_t)(hi - lo);
    const uint64_t step = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += step) {
        const uint32_t bits = lo + (uint32_t)i;
        const float x = __uint_as_float(bits);
        if (__float_as_uint(div6_rn(x)) != __float_as_uint(__fdiv_rn(x, 6.0f))) {
            ++local;
            first = min(first, bits);
        }
    }
    if (local) {
        atomicAdd(mismatches, local);
        atomicMin(first_bad, first);
    }
}

// Host Philox4x32-10 (Salmon et al., SC'11), for the RHT sign mask.
uint32_t host_philox_word0(uint64_t seed) {
    uint32_t c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0, p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n1 = (uint32_t)p1;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1, n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    return c0;
}

}  // namespace

// =================================================================== ABI ===
extern "C" {

nvfp4_status nvfp4_amax(nvfp4_bf16_view x, uint32_t rht_mask, float* amax_dev,
                        cudaStream_t stream) {
    nvfp4_status s = check_view(x, rht_mask != 0);
    if (s != NVFP4_OK) return s;
    if (rht_mask > 0xFFFFu || amax_dev == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(amax_dev, 4)) return NVFP4_ERR_MISALIGNED;
    return launch_amax(x, rht_mask, amax_dev, stream);
}

nvfp4_status nvfp4_quantize_1d(nvfp4_bf16_view x, const float* amax_dev, nvfp4_round round,
                               uint64_t seed, uint64_t stream_id, nvfp4_q* out,
                               cudaStream_t stream) {
    return quantize_impl(x, 0, amax_dev, round, seed, stream_id, out, nullptr, false, stream);
}

nvfp4_status nvfp4_quantize_2d(nvfp4_bf16_view w, const float* amax_dev, nvfp4_round round,
                               uint64_t seed, uint64_t stream_id, nvfp4_q* out, nvfp4_q* out_t,
                               cudaStream_t stream) {
    return quantize_impl(w, 0, amax_dev, round, seed, stream_id, out, out_t, true, stream);
}

nvfp4_status nvfp4_rht_quantize(nvfp4_bf16_view x, uint32_t rht_mask, const float* amax_dev,
                                nvfp4_round round, uint64_t seed, uint64_t stream_id,
                                nvfp4_q* out, cudaStream_t stream) {
    if (rht_mask == 0 || out == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (out->block2d != 0 && out->block2d != 1) return NVFP4_ERR_INVALID_ARG;
    return quantize_impl(x, rht_mask, amax_dev, round, seed, stream_id, out, nullptr,
                         out->block2d == 1, stream);
}

nvfp4_status nvfp4_amax_dual(nvfp4_bf16_view x, uint32_t rht_mask, float* amax_dev,
                             float* amax_t_dev, cudaStream_t stream) {
    nvfp4_status s = check_view(x, false);
    if (s != NVFP4_OK) return s;
    if (x.transposed != 0 || rht_mask > 0xFFFFu || amax_dev == nullptr || amax_t_dev == nullptr ||
        amax_dev == amax_t_dev)
        return NVFP4_ERR_INVALID_ARG;
    if (x.rows % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(amax_dev, 4) || !aligned(amax_t_dev, 4)) return NVFP4_ERR_MISALIGNED;
    if (cudaMemsetAsync(amax_dev, 0, sizeof(float), stream) != cudaSuccess ||
        cudaMemsetAsync(amax_t_dev, 0, sizeof(float), stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (x.rows == 0 || x.cols == 0) return NVFP4_OK;
    return launch_amax_stream(x.ptr, x.rows, x.cols, x.ld, rht_mask, amax_dev, amax_t_dev, stream);
}

nvfp4_status nvfp4_quantize_dual(nvfp4_bf16_view x, const float* amax_dev, nvfp4_round round,
                                 uint64_t seed, uint64_t stream_id, nvfp4_q* out,
                                 uint32_t rht_mask_t, const float* amax_t_dev, nvfp4_round round_t,
                                 uint64_t seed_t, uint64_t stream_id_t, nvfp4_q* out_t,
                                 cudaStream_t stream) {
    nvfp4_status s = check_view(x, true);
    if (s != NVFP4_OK) return s;
    if (x.transposed != 0 || rht_mask_t > 0xFFFFu) return NVFP4_ERR_INVALID_ARG;
    if (!valid_round(round) || !valid_round(round_t))
        return NVFP4_ERR_INVALID_ARG;
    if (x.rows % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if ((s = check_q(out, x.rows, x.cols)) != NVFP4_OK) return s;
    if ((s = check_q(out_t, x.cols, x.rows)) != NVFP4_OK) return s;
    if (amax_dev == nullptr || amax_t_dev == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(amax_dev, 4) || !aligned(amax_t_dev, 4)) return NVFP4_ERR_MISALIGNED;
    if (amax_dev == out->global_scale || amax_dev == out_t->global_scale ||
        amax_t_dev == out->global_scale || amax_t_dev == out_t->global_scale ||
        out->global_scale == out_t->global_scale)
        return NVFP4_ERR_INVALID_ARG;
    if (x.rows == 0 || x.cols == 0) {
        k_publish_senc<<<1, 1, 0, stream>>>(amax_dev, 0, out->global_scale, nullptr);
        k_publish_senc<<<1, 1, 0, stream>>>(amax_t_dev, 0, out_t->global_scale, nullptr);
        return launch_status();
    }
    DualArgs d{};
    QuantArgs& a1 = d.row;
    a1.x = static_cast<const uint16_t*>(x.ptr);
    a1.ld = x.ld;
    a1.rows = x.rows;
    a1.k = x.cols;
    a1.scale_src = amax_dev;
    a1.gs_out = out->global_scale;
    a1.codes = out->codes;
    a1.scales = out->scales;
    a1.stream_id = stream_id;
    a1.write_primary = 1;
    set_sr_keys(&a1, seed, stream_id, round, x.rows * x.cols);
    QuantArgs& a2 = d.col;
    a2.x = a1.x;
    a2.ld = x.ld;
    a2.rows = x.cols;
    a2.k = x.rows;
    a2.scale_src = amax_t_dev;
    a2.gs_out = out_t->global_scale;
    a2.codes = out_t->codes;
    a2.scales = out_t->scales;
    a2.rht = rht_signs(rht_mask_t);
    a2.stream_id = stream_id_t;
    a2.write_primary = 1;
    set_sr_keys(&a2, seed_t, stream_id_t, round_t, x.rows * x.cols);
    if (g_force_g64.exchange(0) == 1) a1.sr_g32 = a2.sr_g32 = 0;    // test-only, one call
    return launch_dual(d, (int)round, (int)round_t, rht_mask_t != 0, stream);
}

nvfp4_status nvfp4_dequantize(const nvfp4_q* q, void* out, int out_is_bf16, int64_t ld,
                              cudaStream_t stream) {
    if (q == nullptr || (out_is_bf16 != 0 && out_is_bf16 != 1)) return NVFP4_ERR_INVALID_ARG;
    if (q->rows < 0 || q->k < 0) return NVFP4_ERR_INVALID_ARG;
    if (q->k % 16 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    nvfp4_status s = check_q(q, q->rows, q->k);
    if (s != NVFP4_OK) return s;
    if (q->rows == 0 || q->k == 0) return NVFP4_OK;
    if (out == nullptr || ld < q->k) return NVFP4_ERR_INVALID_ARG;
    const int64_t esz = out_is_bf16 ? 2 : 4;
    if (!aligned(out, 16) || (ld * esz) % 16 != 0) return NVFP4_ERR_MISALIGNED;
    // one warp per 256-element chunk of a row, kDeqUnroll chunks per pass
    const int g = grid_for(q->rows * cdiv(q->k, 256) * 32 / kDeqUnroll, kQuantThreads, 5);
    if (out_is_bf16)
        k_dequant<true><<<g, kQuantThreads, 0, stream>>>(q->codes, q->scales, q->global_scale,
                                                          q->rows, q->k, out, ld);
    else
        k_dequant<false><<<g, kQuantThreads, 0, stream>>>(q->codes, q->scales, q->global_scale,
                                                           q->rows, q->k, out, ld);
    return launch_status();
}

nvfp4_status nvfp4_gemm(const nvfp4_q* a, const nvfp4_q* b, void* d, int d_is_bf16, int64_t ldd,
                        cudaStream_t stream) {
    if (a == nullptr || b == nullptr || (d_is_bf16 != 0 && d_is_bf16 != 1))
        return NVFP4_ERR_INVALID_ARG;
    if (a->rows < 0 || b->rows < 0 || a->k < 0 || a->k != b->k) return NVFP4_ERR_INVALID_ARG;
    const int64_t M = a->rows, N = b->rows, K = a->k;
    if (K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    nvfp4_status s;
    if ((s = check_q(a, M, K)) != NVFP4_OK) return s;
    if ((s = check_q(b, N, K)) != NVFP4_OK) return s;
    if (M == 0 || N == 0) return NVFP4_OK;
    const int64_t esz = d_is_bf16 ? 2 : 4;
    if (d == nullptr || ldd < N) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(d, 16) || (ldd * esz) % 16 != 0) return NVFP4_ERR_MISALIGNED;
    if (K == 0) {
        return cudaMemset2DAsync(d, ldd * esz, 0, N * esz, M, stream) == cudaSuccess ? NVFP4_OK
                                                                                      : NVFP4_ERR_CUDA;
    }
    // CTA pairs run 256-row MMAs, each CTA holding half of every B tile
    GemmMaps mp;
    std::memset(&mp, 0, sizeof(mp));
    if (!make_code_map(&mp.a, a->codes, M, K, gemm::BM) || !make_code_map(&mp.b, b->codes, N, K, gemm::BN / 2) ||
        !make_scale_map(&mp.sfa, a->scales, M, K, 1) || !make_scale_map(&mp.sfb, b->scales, N, K, 2))
        return NVFP4_ERR_CUDA;
    if (d_is_bf16 && !make_out_map(&mp.d, d, M, N, ldd)) return NVFP4_ERR_CUDA;
    if (!gemm_smem_ready()) return NVFP4_ERR_CUDA;
    gemm::Args g{};
    g.gs_a = a->global_scale;
    g.gs_b = b->global_scale;
    g.d = d;
    g.ldd = ldd;
    g.d_bf16 = d_is_bf16;
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    // CTA pairs always: an odd last 128-row tile pairs with an empty one,
    // whose loads read zeros and whose rows are never stored
    g.m_tiles = (int)(cdiv(cdiv(M, gemm::BM), 2) * 2);
    g.n_tiles = (int)cdiv(N, gemm::BN);
    g.n_fastest = M > N ? 1 : 0;               // keep the smaller operand resident in L2
    g.k_blocks = (int)cdiv(K, gemm::BK);
    g.k_steps = (int)cdiv(K, 64);
    const nvfp4_status st = d_is_bf16 ? launch_gemm_pair<true>(mp, g, stream) : launch_gemm_pair<false>(mp, g, stream);
    if (st != NVFP4_OK) return st;
    return launch_status();
}

// ----------------------------------------------------------------- MXFP4 ---
size_t nvfp4_mx_scale_bytes(int64_t rows, int64_t k) {
    if (rows <= 0 || k <= 0) return 0;
    return (size_t)(cdiv(rows, 128) * cdiv(k / 32, 4) * 512);
}

nvfp4_status nvfp4_mx_quantize(nvfp4_bf16_view x, uint32_t rht_mask, nvfp4_q* out, cudaStream_t stream) {
    nvfp4_status s = check_view(x, true);
    if (s != NVFP4_OK) return s;
    if (x.transposed != 0 || rht_mask > 0xFFFFu || out == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (x.cols % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (out->rows != x.rows || out->k != x.cols) return NVFP4_ERR_INVALID_ARG;
    if (x.rows == 0 || x.cols == 0) return NVFP4_OK;
    if (out->codes == nullptr || out->scales == nullptr) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(out->codes, 16) || !aligned(out->scales, 16)) return NVFP4_ERR_MISALIGNED;
    MxArgs a{};
    a.x = static_cast<const uint16_t*>(x.ptr);
    a.rows = x.rows;
    a.k = x.cols;
    a.ld = x.ld;
    a.codes = out->codes;
    a.scales = out->scales;
    a.rht = rht_signs(rht_mask);
    const int64_t items = cdiv(x.rows, 128) * 128 * cdiv(x.cols / 32, 4) * 2;
    const int g = grid_for(items, kQuantThreads, 8);
    if (rht_mask) k_mx_quant_rows<true><<<g, kQuantThreads, 0, stream>>>(a);
    else k_mx_quant_rows<false><<<g, kQuantThreads, 0, stream>>>(a);
    return launch_status();
}

nvfp4_status nvfp4_mx_dequantize(const nvfp4_q* q, void* out, int out_is_bf16, int64_t ld, cudaStream_t stream) {
    if (q == nullptr || (out_is_bf16 != 0 && out_is_bf16 != 1)) return NVFP4_ERR_INVALID_ARG;
    if (q->rows < 0 || q->k < 0) return NVFP4_ERR_INVALID_ARG;
    if (q->k % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (q->rows == 0 || q->k == 0) return NVFP4_OK;
    if (q->codes == nullptr || q->scales == nullptr || out == nullptr || ld < q->k) return NVFP4_ERR_INVALID_ARG;
    const int64_t esz = out_is_bf16 ? 2 : 4;
    if (!aligned(q->codes, 16) || !aligned(out, 16) || (ld * esz) % 16 != 0) return NVFP4_ERR_MISALIGNED;
    const int g = grid_for(q->rows * cdiv(q->k, 256) * 32 / kDeqUnroll, kQuantThreads, 4);
    if (out_is_bf16) k_mx_dequant<true><<<g, kQuantThreads, 0, stream>>>(q->codes, q->scales, q->rows, q->k, out, ld);
    else k_mx_dequant<false><<<g, kQuantThreads, 0, stream>>>(q->codes, q->scales, q->rows, q->k, out, ld);
    return launch_status();
}

nvfp4_status nvfp4_mx_gemm(const nvfp4_q* a, const nvfp4_q* b, void* d, int d_is_bf16, int64_t ldd,
                           cudaStream_t stream) {
    if (a == nullptr || b == nullptr || (d_is_bf16 != 0 && d_is_bf16 != 1)) return NVFP4_ERR_INVALID_ARG;
    if (a->rows < 0 || b->rows < 0 || a->k < 0 || a->k != b->k) return NVFP4_ERR_INVALID_ARG;
    const int64_t M = a->rows, N = b->rows, K = a->k;
    if (K % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    nvfp4_status s;
    if ((s = check_q(a, M, K, false)) != NVFP4_OK) return s;
    if ((s = check_q(b, N, K, false)) != NVFP4_OK) return s;
    if (M == 0 || N == 0) return NVFP4_OK;
    const int64_t esz = d_is_bf16 ? 2 : 4;
    if (d == nullptr || ldd < N) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(d, 16) || (ldd * esz) % 16 != 0) return NVFP4_ERR_MISALIGNED;
    if (K == 0) {
        return cudaMemset2DAsync(d, ldd * esz, 0, N * esz, M, stream) == cudaSuccess ? NVFP4_OK
                                                                                      : NVFP4_ERR_CUDA;
    }
    GemmMaps mp;
    std::memset(&mp, 0, sizeof(mp));
    if (!make_code_map(&mp.a, a->codes, M, K, gemm::BM) || !make_code_map(&mp.b, b->codes, N, K, gemm::BN / 2) ||
        !make_scale_map(&mp.sfa, a->scales, M, K, 1, 32) || !make_scale_map(&mp.sfb, b->scales, N, K, 2, 32))
        return NVFP4_ERR_CUDA;
    if (d_is_bf16 && !make_out_map(&mp.d, d, M, N, ldd)) return NVFP4_ERR_CUDA;
    if (!gemm_smem_ready()) return NVFP4_ERR_CUDA;
    gemm::Args g{};
    g.d = d;
    g.ldd = ldd;
    g.d_bf16 = d_is_bf16;
    g.M = (int)M;
    g.N = (int)N;
    g.K = (int)K;
    // CTA pairs always: an odd last 128-row tile pairs with an empty one,
    // whose loads read zeros and whose rows are never stored
    g.m_tiles = (int)(cdiv(cdiv(M, gemm::BM), 2) * 2);
    g.n_tiles = (int)cdiv(N, gemm::BN);
    g.n_fastest = M > N ? 1 : 0;
    g.k_blocks = (int)cdiv(K, gemm::BK);
    g.k_steps = (int)cdiv(K, 64);
    nvfp4_status st = d_is_bf16 ? launch_gemm_pair<true, true>(mp, g, stream) : launch_gemm_pair<false, true>(mp, g, stream);
    if (st != NVFP4_OK) return st;
    return launch_status();
}

uint32_t nvfp4_rht_mask_from_seed(uint64_t seed) { return host_philox_word0(seed) & 0xFFFFu; }

nvfp4_status nvfp4_get_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_device_status, sizeof(word), 0, cudaMemcpyDeviceToHost,
                                  stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice,
                                stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    if (word & NVFP4_DEV_GUARD) return NVFP4_ERR_GUARD;
    if (word & NVFP4_DEV_LAUNCH) return NVFP4_ERR_LAUNCH;
    if (word & NVFP4_DEV_TIMEOUT) return NVFP4_ERR_TIMEOUT;
    if (word & NVFP4_DEV_NONFINITE) return NVFP4_ERR_NONFINITE;
    return NVFP4_OK;
}

size_t nvfp4_scale_bytes(int64_t rows, int64_t k) {
    if (rows <= 0 || k <= 0) return 0;
    return (size_t)(cdiv(rows, 128) * cdiv(k / 16, 4) * 512);
}

nvfp4_status nvfp4_debug_check_div6(uint32_t lo_bits, uint32_t hi_bits, unsigned long long* mismatches_dev,
                                    uint32_t* first_bad_dev, cudaStream_t stream) {
    if (lo_bits > hi_bits || hi_bits > 0x7F800000u || mismatches_dev == nullptr || first_bad_dev == nullptr)
        return NVFP4_ERR_INVALID_ARG;
    if (!aligned(mismatches_dev, 8) || !aligned(first_bad_dev, 4)) return NVFP4_ERR_MISALIGNED;
    if (cudaMemsetAsync(mismatches_dev, 0, sizeof(unsigned long long), stream) != cudaSuccess ||
        cudaMemsetAsync(first_bad_dev, 0xFF, sizeof(uint32_t), stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (lo_bits == hi_bits) return NVFP4_OK;
    k_check_div6<<<device_sm_count() * 8, 256, 0, stream>>>(lo_bits, hi_bits, mismatches_dev, first_bad_dev);
    return launch_status();
}

nvfp4_status nvfp4_debug_inject(int mode) {
    if (mode < 0 || mode > 2) return NVFP4_ERR_INVALID_ARG;
    if (mode == 2) {
        g_force_g64.store(1);
        return NVFP4_OK;
    }
    g_fault_injection.store(mode);
    if (mode == 0) g_force_g64.store(0);
    return NVFP4_OK;
}

int nvfp4_debug_guards_enabled(void) {
#ifdef NVFP4_DEBUG_GUARDS
    return 1;
#else
    return 0;
#endif
}

nvfp4_status nvfp4_debug_guard_record(uint32_t* site, uint64_t* byte_offset, cudaStream_t stream) {
    if (site == nullptr || byte_offset == nullptr) return NVFP4_ERR_INVALID_ARG;
    *site = 0;
    *byte_offset = 0;
#ifdef NVFP4_DEBUG_GUARDS
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    unsigned long long rec = 0;
    if (cudaMemcpyFromSymbolAsync(&rec, g_guard_record, sizeof(rec), 0, cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
        return NVFP4_ERR_CUDA;
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbolAsync(g_guard_record, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream) !=
        cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    *site = (uint32_t)(rec >> 48);
    *byte_offset = rec & 0xFFFFFFFFFFFFull;
#else
    (void)stream;
#endif
    return NVFP4_OK;
}

nvfp4_status nvfp4_debug_guard_shrink(uint64_t bytes) {
#ifdef NVFP4_DEBUG_GUARDS
    const unsigned long long v = bytes;
    if (cudaMemcpyToSymbol(g_guard_shrink, &v, sizeof(v)) != cudaSuccess) return NVFP4_ERR_CUDA;
    return NVFP4_OK;
#else
    (void)bytes;
    return NVFP4_ERR_INVALID_ARG;
#endif
}

const char* nvfp4_status_string(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_INVALID_ARG: return "invalid argument";
        case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case NVFP4_ERR_MISALIGNED: return "misaligned pointer or leading dimension";
        case NVFP4_ERR_NONFINITE: return "non-finite amax";
        case NVFP4_ERR_TIMEOUT: return "device wait timed out";
        case NVFP4_ERR_CUDA: return "CUDA error";
        case NVFP4_ERR_LAUNCH: return "kernel launched with too little dynamic shared memory";
        case NVFP4_ERR_GUARD: return "an index guard refused a global access (debug build)";
    }
    return "unknown status";
}

}  // extern "C"
