// selftest.cu -- forced timeout of the library's bounded waits (failure detection, tested without
// a GPU fault).
//
// Every wait of the pipelined kernels (TMA, bulk-copy and tensor-core barriers) is a bounded poll
// that gives up after a time limit, records an error in the device error word and lets the
// kernel wind down, so that a lost arrival never hangs the GPU.  This kernel exercises exactly
// those helpers on an mbarrier that nothing arrives at: each wait must give up after the limit
// and report it, and the context must stay usable.  The analogue of the pages' harness that
// "records failures instead of dropping them" (vllm-omni commit "cpu_int4: dequantize prefill
// weights from the tinygemm layout, not a copy", the paragraph on the benchmark harness).
#include <cuda_runtime.h>

#include "bounds.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace w4a16 {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns, int *status, int *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);  // one arrival expected; none ever comes
  fence_mbar_init();
  int timed_out = 0;
  if (!mbar_wait_bounded(&bar, 0, limit_ns)) timed_out |= 1;        // polling wait
  if (!mbar_wait_sleep_bounded(&bar, 0, limit_ns)) timed_out |= 2;  // sleeping wait
  *status = timed_out;
  if (timed_out) atomicOr(err, 2);  // the kernels' timeout code
}

// The bounds check itself (bounds.cuh), on offsets from `base` that nothing dereferences: bit i of
// *status is set when case i is judged outside its extent.  Cases 0-1 lie inside a 64-byte
// buffer, cases 2-4 (one byte past the end, one before the start, a zero-length buffer) outside.
__global__ void __launch_bounds__(32) bounds_check_kernel(int *status, int *err) {
  if (threadIdx.x != 0) return;
  const long long off[5] = {0, 48, 49, -1, 0}, bytes[5] = {16, 16, 16, 1, 1}, ext[5] = {64, 64, 64, 64, 0};
  const char *base = reinterpret_cast<const char *>(status);
  int out = 0;
#pragma unroll
  for (int i = 0; i < 5; ++i)
    if (!in_extent(base + off[i], bytes[i], base, ext[i], err)) out |= 1 << i;
  *status = out;
}

}  // namespace

bool bounds_checked() { return kBoundsCheck; }

cudaError_t launch_bounds_selftest(int *status, int *err, cudaStream_t stream) {
  bounds_check_kernel<<<1, 32, 0, stream>>>(status, err);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(uint64_t limit_ns, int *status, int *err, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns, status, err);
  return cudaGetLastError();
}

}  // namespace w4a16
