// Device-side index checks of the bounds-checked build (compiled with
// -DCPATTN_BOUNDS_CHECK into libcpattn_checked.so; the normal build compiles
// them away).  A failing check records the first failure in the workspace
// status word (kStatusBounds and a site code naming the access) and tells the
// caller to skip the access; it never traps.  A skipped tensor load leaves its
// barrier incomplete, so the waiting role gives up through the kernel's
// bounded waits and the CTA leaves normally.
#pragma once
#include <stdint.h>

namespace cpattn {

constexpr int32_t kStatusBounds = 3;   // status word: a device-side index check failed

#ifdef CPATTN_BOUNDS_CHECK
__device__ __forceinline__ bool in_range_checked(long long v, long long lo, long long hi,
                                                 int32_t* status, int site) {
  if (v >= lo && v < hi) return true;
  if (status && atomicCAS(&status[0], 0, kStatusBounds) == 0) status[1] = site;
  return false;
}
#define CP_IN_RANGE(v, lo, hi, status, site) \
  ::cpattn::in_range_checked((long long)(v), (long long)(lo), (long long)(hi), (status), (site))
#else
#define CP_IN_RANGE(v, lo, hi, status, site) true
#endif

}  // namespace cpattn
