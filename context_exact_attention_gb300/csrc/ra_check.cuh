// ra_check.cuh -- index checks of the debug build.
//
// Compiled with -DRA_DEBUG_BOUNDS (libringattn_debug.so), every global load and
// store of the kernels that is addressed by a computed index first asks
// in_bounds() whether the elements [i, i + n) lie inside the tensor's extent.  If
// they do not, the check records RA_STATUS_BOUNDS in the device status word and
// the access is skipped (a load yields 0), so a wrong index is reported instead of
// touching memory outside the tensor.  In the normal build in_bounds() is the
// constant true and the checks compile away.  (TMA tensor loads need no check:
// the tensor map bounds them in hardware, filling outside boxes with zeros.)
#pragma once

#include <cuda_runtime.h>

#define RA_STATUS_BOUNDS 4u   // a debug-build index check failed; the access was skipped

namespace ra {

#ifdef RA_DEBUG_BOUNDS
constexpr bool kCheckBounds = true;
#else
constexpr bool kCheckBounds = false;
#endif

__device__ __forceinline__ bool in_bounds(long long i, long long n, long long extent,
                                          unsigned int* status)
{
    if constexpr (kCheckBounds) {
        if (i < 0 || n < 0 || i > extent - n) {
            atomicOr(status, RA_STATUS_BOUNDS);
            return false;
        }
    }
    return true;
}

// base[i] through the read-only path, or 0 when the check fails.
__device__ __forceinline__ int checked_ldg(const int* base, long long i, long long extent,
                                           unsigned int* status)
{
    return in_bounds(i, 1, extent, status) ? __ldg(base + i) : 0;
}

}  // namespace ra
