// checks.cuh -- range checks of the data-dependent global stores, compiled
// in with -DW4_CHECK_BOUNDS (a test build of the library).
//
// W4_IN_BOUNDS(cond, status) is true when the store may go ahead.  In the
// checked build a false condition ORs W4_DEV_OUT_OF_BOUNDS into *status
// (when status is not NULL) and the caller skips the store: no trap, no
// assert.  In the normal build it is the constant true and costs nothing.
#pragma once

#include <cstdint>

namespace w4 {

constexpr int32_t kDevOutOfBounds = 0x10;

__device__ __forceinline__ bool check_in_bounds(bool ok, int32_t *status)
{
    if (!ok && status)
        atomicOr(status, kDevOutOfBounds);
    return ok;
}

}  // namespace w4

#ifdef W4_CHECK_BOUNDS
#define W4_IN_BOUNDS(cond, status) (::w4::check_in_bounds((cond), (status)))
#else
#define W4_IN_BOUNDS(cond, status) true
#endif
