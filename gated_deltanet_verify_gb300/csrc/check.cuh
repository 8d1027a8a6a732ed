// check.cuh -- bounds checks of a checked build (nvcc -DGDN_CHECKED=1).
//
// A checked build tests every global access of the verify-family and rollback
// kernels against the extent of its buffer before making it; an access that
// falls outside is skipped and the first such event writes GDN_ERR_BOUNDS to
// the caller's status word (no trap, no assert).  The ordinary build compiles
// every test away.  It stands in for a memory checker that cannot run here.
#pragma once

#include <cstddef>
#include <cstdint>

#include "gdn_verify.h"

#ifndef GDN_CHECKED
#define GDN_CHECKED 0
#endif

namespace gdn {

// true when [p, p + bytes) lies inside [base, base + extent)
__device__ __forceinline__ bool in_bounds(const void *p, size_t bytes, const void *base, size_t extent,
                                          int *status) {
    if constexpr (!GDN_CHECKED) {
        return true;
    } else {
        const uintptr_t q = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(base);
        if (base != nullptr && q >= b && q + bytes <= b + extent) return true;
        if (status) atomicCAS(status, int(GDN_OK), int(GDN_ERR_BOUNDS));
        return false;
    }
}

}  // namespace gdn
