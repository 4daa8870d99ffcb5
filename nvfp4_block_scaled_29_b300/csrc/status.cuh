// status.cuh -- the device-side status word of libnvfp4.
//
// Kernels never trap: a condition they cannot handle (a non-finite amax
// reaching a quantiser, a pipeline wait that exceeded its time limit, a launch
// with too little dynamic shared memory, in the debug build an access outside
// its buffer) sets a bit here and the kernel returns or skips the access.
// nvfp4_get_status() reads and clears it.
#pragma once
#include <cstdint>

namespace nvfp4 {

enum : uint32_t {
    NVFP4_DEV_NONFINITE = 1u,
    NVFP4_DEV_TIMEOUT = 2u,
    NVFP4_DEV_LAUNCH = 4u,     // a kernel was launched with less dynamic shared memory than it needs
    NVFP4_DEV_GUARD = 8u,      // debug build: an index guard refused a global access
};

// The library is one translation unit (nvfp4.cu includes every kernel
// header), so this is the only definition.
__device__ uint32_t g_device_status;

__device__ __forceinline__ void record_device_error(uint32_t bit) {
    atomicOr(&g_device_status, bit);
}

}  // namespace nvfp4
