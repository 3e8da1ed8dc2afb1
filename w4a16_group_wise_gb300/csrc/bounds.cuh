// bounds.cuh -- the per-access bounds checks of the debug build.
//
// Compiled with -DW4A16_BOUNDS (the library _libw4a16_bounds.so), every kernel checks each global
// read of the packed weights, x, the ids and the AWQ tensors, and each global write of y, W, out
// and the split-K workspace, against the extent of its buffer as the call's sizes define it (the
// extent the entry point documents: w4a16_packed_bytes for the packed buffer, M*K halves for x,
// M*N halves for y, ...).  An access outside it records kErrBounds in the device error word and
// is skipped: a read gives zeros (a bulk copy is redirected to the buffer's first bytes, so that
// its barrier still completes), a write is dropped.  Nothing traps.  In the normal build
// in_extent() is the constant true and every check folds away.
//
// This stands in for a memory checker ("Race detection / sanitizers" of the test strategy): the
// guard-band tests see only stray writes that land next to the output buffers, these checks see
// every index the kernels form.
#pragma once
#include <cstddef>
#include <cstdint>

namespace w4a16 {

#ifdef W4A16_BOUNDS
constexpr bool kBoundsCheck = true;
#else
constexpr bool kBoundsCheck = false;
#endif

constexpr int kErrBounds = 8;  // device error word bit: an index outside its buffer (1 header, 2 timeout, 4 id)

// [p, p + bytes) inside the `extent` bytes at `base`?  A miss records kErrBounds.
__device__ __forceinline__ bool in_extent(const void *p, long long bytes, const void *base, long long extent,
                                          int *err) {
  if constexpr (!kBoundsCheck) {
    return true;
  } else {
    const long long off = static_cast<const char *>(p) - static_cast<const char *>(base);
    if (off >= 0 && bytes >= 0 && off + bytes <= extent) return true;
    atomicOr(err, kErrBounds);
    return false;
  }
}

}  // namespace w4a16
