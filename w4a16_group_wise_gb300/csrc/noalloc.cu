// noalloc.cu -- w4a16_gemm_noalloc: the layer's GEMM for callers that cannot allocate device
// memory.
//
// The tensor-core path of w4a16_gemm needs scratch memory when it splits K across CTAs (fp32
// partial tiles and per-tile arrival counters), which w4a16_gemm takes from a caller-provided
// workspace.  Some callers have no way to provide one: an inference runtime that plans all
// device memory up front and hands a layer only its input and output buffers, a plugin host that
// forbids device allocation after start-up, or a latency-critical path where an allocation could
// block or fail at the worst moment.  For them this entry point keeps its scratch in a fixed
// array that is part of the library itself: every GPU that loads the library holds these
// kScratchBytes for as long as the process lives, and no call ever allocates or frees memory.
//
// Rules that follow from one shared, static scratch area:
//  - every call uses the same array, which keeps whatever the last call left in it; the only
//    part that must start at zero (the arrival counters at its head) starts at zero when the
//    library's device code is loaded, is cleared again (ordered on the caller's stream, before
//    the call's kernel) when a device is first set up, and is left at zero by every call that
//    completes;
//  - calls that overlap on the GPU (on different streams, or from different host threads) race
//    on the array and give wrong results: serialize them;
//  - the first call on a device sets it up (looks up the array's device address and clears the
//    counters); make that first call before capturing the stream into a graph;
//  - CUDA loads a library's device code, and with it this array, on a device when the library is
//    first used there, which may be inside the first call here: that call can then fail for lack
//    of device memory.  A caller that must not see that make one call at start-up;
//  - the call plans its launch once and checks that plan's scratch against kScratchBytes, so a
//    split-K option changed by another thread meanwhile cannot make the kernel use more than was
//    checked; problems whose scratch would exceed it are rejected with W4A16_ERR_WORKSPACE.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/w4a16.h"
#include "kernels.h"
#include "layout.cuh"

using namespace w4a16;

namespace {

constexpr size_t kScratchBytes = (size_t)W4A16_NOALLOC_SCRATCH_BYTES;
static_assert(kScratchBytes > kSplitCounterBytes, "the scratch holds the split-K arrival counters");

// The scratch itself.  In host code `g_scratch` only names the symbol; its device address comes
// from cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_mu;

// Device address of the scratch on the current device; null on failure.  The first call on a
// device looks the address up and clears the arrival counters on `stream`, ahead of the kernel
// the caller launches next on that stream.
void *scratch_on_current_device(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return nullptr;
    if (cudaMemsetAsync(p, 0, kSplitCounterBytes, stream) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

#pragma GCC visibility push(default)
extern "C" int w4a16_gemm_noalloc(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
                                  void *stream) {
  if (M < 0 || K <= 0 || N <= 0 || g == 0 || g < -1) return W4A16_ERR_INVALID;
  if (N % 8 != 0 || layout_group(K, g) == 0) return W4A16_ERR_UNSUPPORTED;
  if (M == 0) return W4A16_OK;
  if (!x || !packed || !y) return W4A16_ERR_INVALID;
  if (!aligned16(x) || !aligned16(packed) || !aligned16(y)) return W4A16_ERR_MISALIGNED;
  // one plan per call: the scratch checked here is the scratch the launch uses
  TcPlan plan = {};
  size_t need = 0;
  if (M > kDecodeMaxM) {
    plan = plan_gemm_tc(M, N, K);
    need = gemm_tc_workspace_bytes(plan);
  }
  if (need > kScratchBytes) return W4A16_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void *scratch = scratch_on_current_device(s);
  int *err = device_error_word();
  if (!scratch || !err) return W4A16_ERR_CUDA;
  const int gl = layout_group(K, g);
  cudaError_t e = (M <= kDecodeMaxM) ? launch_gemv(x, packed, M, N, K, gl, kDtypeF16, y, err, s)
                                     : launch_gemm_tc(plan, x, packed, M, N, K, gl, kDtypeF16, y, err, scratch, s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  return W4A16_OK;
}
#pragma GCC visibility pop
