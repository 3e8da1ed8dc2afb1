// kernels.h -- host-side launchers of the library's CUDA kernels (internal; the public ABI is
// include/w4a16.h).  Every launcher has been handed validated arguments and returns the
// cudaError_t of its launch.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace w4a16 {

// `dtype` below is the layer's element type (kDtypeF16 or kDtypeBf16 of layout.cuh): that of x,
// the scales, the dequantized weights and y, all 16-bit.  Kernels check it against the packed
// header's dtype word.

// Repack columns [n0, n1) of AWQ tensors (slices starting at column n0, row strides in
// elements) into their n-blocks of `packed`, and write the header.  g is the layout's group
// size (32, 64, 128); the source tensors' scales and zeros have one row per gsrc rows of K
// (gsrc == g, or gsrc == K for one group over all of K).
cudaError_t launch_repack(const int32_t *qweight, int64_t ldq, const int32_t *qzeros, int64_t ldz,
                          const uint16_t *scales, int64_t lds, int K, int N, int g, int gsrc, int dtype,
                          int n0, int n1, void *packed, int *err, cudaStream_t stream);

// packed -> W[K][N].
cudaError_t launch_dequant(const void *packed, int K, int N, int g, int dtype, uint16_t *W, int *err,
                           cudaStream_t stream);

// Decode path: y = x . W for 1 <= M (rows are processed 16 at a time).
cudaError_t launch_gemv(const uint16_t *x, const void *packed, int M, int N, int K, int g, int dtype,
                        uint16_t *y, int *err, cudaStream_t stream);

// Tensor-core path (tcgen05): y = x . W for M > kDecodeMaxM.  A call plans its launch once
// (plan_gemm_tc, which reads the split-K reduction mode once), checks the workspace against that
// plan's gemm_tc_workspace_bytes, and launches exactly that plan, so the scratch the kernel uses
// is the scratch that was checked.  `workspace` holds gemm_tc_workspace_bytes(plan) bytes (may be
// null when that is 0); its first kSplitCounterBytes (the arrival counters) must be zero before
// the first call and are left zero by every completed call.
constexpr size_t kSplitCounterBytes = 4096;
struct TcPlan {
  int bm, stages, tmem_cols, splits, stages_per_split, tiles, a_col0;
  bool cluster, persist, dbl;
  size_t partial_bytes;  // fp32 partial tiles of the workspace reduction (0: none)
};
TcPlan plan_gemm_tc(int M, int N, int K);
size_t gemm_tc_workspace_bytes(const TcPlan &plan);
cudaError_t launch_gemm_tc(const TcPlan &plan, const uint16_t *x, const void *packed, int M, int N, int K, int g,
                           int dtype, uint16_t *y, int *err, void *workspace, cudaStream_t stream);
// W4A16_SPLITK_AUTO or W4A16_SPLITK_GLOBAL (include/w4a16.h); returns a W4A16 status.
int set_splitk_mode(int mode);

// The driver's cuTensorMapEncodeTiled (looked up once); null if the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Tied-embedding gather: out[t][k] = W[k][ids[t]] for t < T (grid T x ceil(KT / 8)).
cudaError_t launch_embed(const int32_t *ids, int T, const void *packed, int K, int N, int g, int dtype,
                         uint16_t *out, int *err, cudaStream_t stream);

// AWQ -> GPTQ-style standard packing: qweight [K/8][N] packed along K in plain order, qzeros
// [zero_rows][N/8] in plain order along N.
cudaError_t launch_awq_to_standard(const int32_t *qweight_awq, const int32_t *qzeros_awq, int K, int N,
                                   int zero_rows, int32_t *qweight_std, int32_t *qzeros_std, int *err,
                                   cudaStream_t stream);

// Forced timeout of the bounded waits: one thread waits (polling, then sleeping) on an mbarrier
// that nothing arrives at, with the given limit; *status gets a bit per wait that gave up.
cudaError_t launch_wait_timeout(uint64_t limit_ns, int *status, int *err, cudaStream_t stream);

// Whether this is the bounds-checked debug build (bounds.cuh), and a one-thread run of its check
// on five fixed cases (bit i of *status: case i judged outside its buffer).
bool bounds_checked();
cudaError_t launch_bounds_selftest(int *status, int *err, cudaStream_t stream);

// The packed layout's group size for a caller's g (32, 64 or 128; or one group over all of K,
// g == K or g == -1, stored as the largest of 128, 64, 32 dividing K); 0 when unsupported.
int layout_group(int K, int g);

// Device address of the library's per-device error word on the current device (null on failure).
int *device_error_word();

// Largest M the decode path takes: the measured crossover on GB300.  In chains of 8 layers
// the decode path was faster than the tensor-core path for every decoder shape up to M = 32
// and slower for each of them from M = 96 (at 48 and 64 it depends on the shape).
constexpr int kDecodeMaxM = 32;

}  // namespace w4a16
