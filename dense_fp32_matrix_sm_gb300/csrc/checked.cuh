// checked.cuh -- device-side bounds checks of the checked build.
//
// Built with -DSGEMM_CHECKED (build.py's checked library), every hand-
// computed shared-memory and global index the kernels form is tested
// against the extent of the buffer it addresses before the access; a
// failed test sets kStatusBounds in the per-device status word (which
// sgemm_device_status reports as SGEMM_ERR_BOUNDS) and skips the access, so
// an indexing mistake shows up as a status instead of a fault or a silent
// corruption.  In the normal build SG_CHK(cond, status) is the constant
// true and the compiled kernels are unchanged.
#pragma once

#include <stdint.h>

namespace sgemm {

enum : unsigned int { kStatusBounds = 16u };

#ifdef SGEMM_CHECKED
__device__ __forceinline__ bool checked_ok(bool ok, unsigned int* status) {
  if (!ok) atomicOr(status, kStatusBounds);
  return ok;
}
#define SG_CHK(cond, status) (::sgemm::checked_ok((cond), (status)))
#else
#define SG_CHK(cond, status) (true)
#endif

// index i of a buffer of n elements
#define SG_IN(i, n) (static_cast<int64_t>(i) >= 0 && static_cast<int64_t>(i) < static_cast<int64_t>(n))

}  // namespace sgemm
