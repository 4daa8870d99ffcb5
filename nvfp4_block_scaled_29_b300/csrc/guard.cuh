// guard.cuh -- in-kernel index guards of the debug build.
//
// Compiled with -DNVFP4_DEBUG_GUARDS (the library libnvfp4_guarded.so), every
// plain global load and store of the kernels first checks that the bytes it
// touches lie inside the buffer that the public layouts define for that
// argument (TMA copies need no guard: their tensor maps bound them).  An access
// outside is skipped (a refused load reads zeros), NVFP4_DEV_GUARD is set in
// the status word, and the first refused access is recorded as its site and
// its byte offset from the buffer's start.  This stands in for a memory
// checker: a kernel whose index arithmetic leaves its layout reports it
// instead of corrupting memory or faulting.
//
// Without the macro NVFP4_GUARD is the constant true, its arguments are never
// evaluated, and the kernels compile to the same code as before.
#pragma once
#include <cstdint>

#include "status.cuh"

namespace nvfp4 {

// The access a guard protects: the site field of the guard record.
enum GuardSite : uint32_t {
    kGuardAmaxX = 1,       // amax kernels: loads of x
    kGuardQ2dCodes = 2,    // 16x16 quantise
    kGuardQ2dScales = 3,
    kGuardQ2dCodesT = 4,   // 16x16 quantise: the transposed operand
    kGuardQ2dScalesT = 5,
    kGuardDualCodes = 6,   // TMA-fed quantiser (dual and 1x16): the row-wise operand
    kGuardDualScales = 7,
    kGuardDualCodesT = 8,  // TMA-fed quantiser (dual and 1x16 of a transposed view): the column-wise operand
    kGuardDualScalesT = 9,
    kGuardDeqIn = 10,      // dequantise: loads of codes and scales
    kGuardDeqOut = 11,
    kGuardMxX = 12,        // MXFP4 quantise
    kGuardMxCodes = 13,
    kGuardMxScales = 14,
    kGuardMxDeqIn = 15,    // MXFP4 dequantise
    kGuardMxDeqOut = 16,
    kGuardGemmD = 17,      // GEMM epilogue: plain stores of D
};

// Byte extents of the public layouts.
__device__ __forceinline__ uint64_t codes_extent(int64_t rows, int64_t k) {
    return rows <= 0 || k <= 0 ? 0 : (uint64_t)(rows * (k >> 1));
}
// Swizzled E4M3 scales: 512-byte tiles of 128 rows x 4 blocks.
__device__ __forceinline__ uint64_t scales_extent(int64_t rows, int64_t k) {
    return rows <= 0 || k <= 0 ? 0 : (uint64_t)(((rows + 127) >> 7) * (((k >> 4) + 3) >> 2) * 512);
}
// MXFP4 scales: 512-byte tiles of 128 rows x 4 blocks of 32.
__device__ __forceinline__ uint64_t mx_scales_extent(int64_t rows, int64_t k) {
    return rows <= 0 || k <= 0 ? 0 : (uint64_t)(((rows + 127) >> 7) * (((k >> 5) + 3) >> 2) * 512);
}
// A stored array of `outer` rows of `inner` elements of `elem` bytes each,
// rows `ld` elements apart.
__device__ __forceinline__ uint64_t stored_extent(int64_t outer, int64_t inner, int64_t ld, int elem) {
    return outer <= 0 || inner <= 0 ? 0 : (uint64_t)((outer - 1) * ld + inner) * (uint64_t)elem;
}

#ifdef NVFP4_DEBUG_GUARDS
// (site << 48) | low 48 bits of the byte offset of the first refused access
__device__ unsigned long long g_guard_record;
// test-only: bytes taken off the end of every extent (nvfp4_debug_guard_shrink)
__device__ unsigned long long g_guard_shrink;

__device__ __forceinline__ bool guard_access(const void* base, uint64_t extent, const void* p, uint32_t nbytes,
                                             uint32_t site) {
    // an address below base wraps to a huge offset and is refused as well
    const uint64_t off = (uint64_t)(reinterpret_cast<uintptr_t>(p) - reinterpret_cast<uintptr_t>(base));
    const uint64_t shrink = g_guard_shrink;
    const uint64_t lim = extent > shrink ? extent - shrink : 0;
    if (off < lim && nbytes <= lim - off) return true;
    record_device_error(NVFP4_DEV_GUARD);
    atomicCAS(&g_guard_record, 0ull, ((unsigned long long)site << 48) | (off & 0xFFFFFFFFFFFFull));
    return false;
}
#define NVFP4_GUARD(base, extent, p, nbytes, site) \
    ::nvfp4::guard_access((base), (extent), (p), (nbytes), (site))
#else
#define NVFP4_GUARD(base, extent, p, nbytes, site) true
#endif

}  // namespace nvfp4
