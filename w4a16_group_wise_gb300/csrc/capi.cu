// capi.cu -- the extern "C" entry points of include/w4a16.h: argument validation (the analogue
// of vLLM's verify_marlin_supported, "Carga de capas cuantizadas", section "Limites y
// fallos"), the choice between the decode and the tensor-core path by M (vllm-omni commit
// "Add cpu_int4 ...": two paths over one set of weights), and the per-device error word.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "../../include/w4a16.h"
#include "kernels.h"
#include "layout.cuh"

using namespace w4a16;

// Per-device error word: kernels record device-side failures here (never trap).
static __device__ int g_device_error;

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int *> g_err_ptr[kMaxDevices];
std::mutex g_err_mu;
}  // namespace

// The per-device error word of the current device (resolved once per device; later calls read
// the cached address without taking the lock).
int *w4a16::device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  int *p = g_err_ptr[dev].load(std::memory_order_acquire);
  if (p) return p;
  std::lock_guard<std::mutex> lock(g_err_mu);
  p = g_err_ptr[dev].load(std::memory_order_relaxed);
  if (!p) {
    void *q = nullptr;
    if (cudaGetSymbolAddress(&q, g_device_error) != cudaSuccess) return nullptr;
    p = static_cast<int *>(q);
    g_err_ptr[dev].store(p, std::memory_order_release);
  }
  return p;
}

// The group size the packed layout uses for a caller's g: g itself for 32, 64, 128 (K % g == 0);
// for one group over all of K (g == K or g == -1, the pages' group_size = -1), the largest of
// 128, 64, 32 that divides K, every layout group then carrying the column's one scale and zero.
// 0 when unsupported.
int w4a16::layout_group(int K, int g) {
  if (K <= 0) return 0;
  if (g == 32 || g == 64 || g == 128) return K % g == 0 ? g : 0;
  if (g == K || g == -1)
    return K % 128 == 0 ? 128 : K % 64 == 0 ? 64 : K % 32 == 0 ? 32 : 0;
  return 0;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_shape(int K, int N, int g) {
  if (K <= 0 || N <= 0 || g == 0 || g < -1) return W4A16_ERR_INVALID;
  if (N % 8 != 0 || layout_group(K, g) == 0) return W4A16_ERR_UNSUPPORTED;
  return W4A16_OK;
}

int map_launch(cudaError_t e) {
  if (e == cudaSuccess) return W4A16_OK;
  cudaGetLastError();  // clear a sticky-free launch error so the next call starts clean
  return W4A16_ERR_CUDA;
}

// The entry points' bodies, shared by the fp16 and bf16 variants (dtype: kDtypeF16 / kDtypeBf16).
int repack_chunk_impl(const int32_t *qweight_c, int64_t ld_qweight, const int32_t *qzeros_c, int64_t ld_qzeros,
                      const uint16_t *scales_c, int64_t ld_scales, int K, int N, int g, int n0, int n1, int dtype,
                      void *packed, void *stream) {
  int st = check_shape(K, N, g);
  if (st != W4A16_OK) return st;
  if (!qweight_c || !qzeros_c || !scales_c || !packed) return W4A16_ERR_INVALID;
  if (n0 < 0 || n1 > N || n0 >= n1 || n0 % kBlockN != 0 || (n1 % kBlockN != 0 && n1 != N))
    return W4A16_ERR_INVALID;
  int64_t w = (n1 - n0) / 8;
  if (ld_qweight < w || ld_qzeros < w || ld_scales < (int64_t)(n1 - n0)) return W4A16_ERR_INVALID;
  if (!aligned16(packed) || (reinterpret_cast<uintptr_t>(qweight_c) & 3u) ||
      (reinterpret_cast<uintptr_t>(qzeros_c) & 3u) || (reinterpret_cast<uintptr_t>(scales_c) & 1u))
    return W4A16_ERR_MISALIGNED;
  const int gl = layout_group(K, g);
  const int gsrc = (g == -1) ? K : g;  // rows of K per row of the source scales and zeros
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  return map_launch(launch_repack(qweight_c, ld_qweight, qzeros_c, ld_qzeros, scales_c, ld_scales, K, N, gl, gsrc,
                                  dtype, n0, n1, packed, err, static_cast<cudaStream_t>(stream)));
}

int repack_impl(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales, int K, int N, int g,
                int dtype, void *packed, void *stream) {
  int st = check_shape(K, N, g);
  if (st != W4A16_OK) return st;
  if (!qweight || !qzeros || !scales || !packed) return W4A16_ERR_INVALID;
  if (!aligned16(qweight) || !aligned16(qzeros) || !aligned16(scales) || !aligned16(packed))
    return W4A16_ERR_MISALIGNED;
  return repack_chunk_impl(qweight, N / 8, qzeros, N / 8, scales, N, K, N, g, 0, N, dtype, packed, stream);
}

int gemm_impl(const uint16_t *x, const void *packed, int M, int N, int K, int g, int dtype, uint16_t *y,
              void *workspace, size_t workspace_bytes, void *stream) {
  if (M < 0) return W4A16_ERR_INVALID;
  int st = check_shape(K, N, g);
  if (st != W4A16_OK) return st;
  if (M == 0) return W4A16_OK;
  if (!x || !packed || !y) return W4A16_ERR_INVALID;
  if (!aligned16(x) || !aligned16(packed) || !aligned16(y)) return W4A16_ERR_MISALIGNED;
  // one plan per call: the workspace is checked against the plan that is launched
  TcPlan plan = {};
  size_t need = 0;
  if (M > kDecodeMaxM) {
    plan = plan_gemm_tc(M, N, K);
    need = gemm_tc_workspace_bytes(plan);
  }
  if (need > 0 && (!workspace || workspace_bytes < need)) return W4A16_ERR_WORKSPACE;
  if (need > 0 && !aligned16(workspace)) return W4A16_ERR_MISALIGNED;
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int gl = layout_group(K, g);
  if (M <= kDecodeMaxM) return map_launch(launch_gemv(x, packed, M, N, K, gl, dtype, y, err, s));
  return map_launch(launch_gemm_tc(plan, x, packed, M, N, K, gl, dtype, y, err, need > 0 ? workspace : nullptr, s));
}

int embed_impl(const int32_t *ids, int T, const void *packed, int K, int N, int g, int dtype, uint16_t *out,
               void *stream) {
  int st = check_shape(K, N, g);
  if (st != W4A16_OK) return st;
  if (T < 0) return W4A16_ERR_INVALID;
  if (T == 0) return W4A16_OK;
  if (!ids || !packed || !out) return W4A16_ERR_INVALID;
  if (!aligned16(packed) || !aligned16(out) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return W4A16_ERR_MISALIGNED;
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  return map_launch(launch_embed(ids, T, packed, K, N, layout_group(K, g), dtype, out, err,
                                 static_cast<cudaStream_t>(stream)));
}

int dequant_impl(const void *packed, int K, int N, int g, int dtype, uint16_t *W, void *stream) {
  int st = check_shape(K, N, g);
  if (st != W4A16_OK) return st;
  if (!packed || !W) return W4A16_ERR_INVALID;
  if (!aligned16(packed) || !aligned16(W)) return W4A16_ERR_MISALIGNED;
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  return map_launch(launch_dequant(packed, K, N, layout_group(K, g), dtype, W, err, static_cast<cudaStream_t>(stream)));
}

}  // namespace

// Only the entry points of include/w4a16.h are exported; everything else is hidden.
#pragma GCC visibility push(default)
extern "C" {

size_t w4a16_packed_bytes(int K, int N, int g) {
  if (check_shape(K, N, g) != W4A16_OK) return 0;
  return (size_t)packed_extent(K, N, layout_group(K, g));
}

size_t w4a16_workspace_bytes(int M, int N, int K, int g) {
  if (M < 0 || check_shape(K, N, g) != W4A16_OK) return 0;
  if (M <= kDecodeMaxM) return 0;
  return gemm_tc_workspace_bytes(plan_gemm_tc(M, N, K));
}

int w4a16_repack_chunk(const int32_t *qweight_c, int64_t ld_qweight, const int32_t *qzeros_c,
                       int64_t ld_qzeros, const uint16_t *scales_c, int64_t ld_scales, int K, int N,
                       int g, int n0, int n1, void *packed, void *stream) {
  return repack_chunk_impl(qweight_c, ld_qweight, qzeros_c, ld_qzeros, scales_c, ld_scales, K, N, g, n0, n1,
                           kDtypeF16, packed, stream);
}

int w4a16_repack_chunk_bf16(const int32_t *qweight_c, int64_t ld_qweight, const int32_t *qzeros_c,
                            int64_t ld_qzeros, const uint16_t *scales_c, int64_t ld_scales, int K, int N,
                            int g, int n0, int n1, void *packed, void *stream) {
  return repack_chunk_impl(qweight_c, ld_qweight, qzeros_c, ld_qzeros, scales_c, ld_scales, K, N, g, n0, n1,
                           kDtypeBf16, packed, stream);
}

int w4a16_repack(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales, int K,
                 int N, int g, void *packed, void *stream) {
  return repack_impl(qweight, qzeros, scales, K, N, g, kDtypeF16, packed, stream);
}

int w4a16_repack_bf16(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales, int K,
                      int N, int g, void *packed, void *stream) {
  return repack_impl(qweight, qzeros, scales, K, N, g, kDtypeBf16, packed, stream);
}

int w4a16_gemm(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
               void *workspace, size_t workspace_bytes, void *stream) {
  return gemm_impl(x, packed, M, N, K, g, kDtypeF16, y, workspace, workspace_bytes, stream);
}

int w4a16_gemm_bf16(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
                    void *workspace, size_t workspace_bytes, void *stream) {
  return gemm_impl(x, packed, M, N, K, g, kDtypeBf16, y, workspace, workspace_bytes, stream);
}

int w4a16_embed(const int32_t *ids, int T, const void *packed, int K, int N, int g, uint16_t *out,
                void *stream) {
  return embed_impl(ids, T, packed, K, N, g, kDtypeF16, out, stream);
}

int w4a16_embed_bf16(const int32_t *ids, int T, const void *packed, int K, int N, int g, uint16_t *out,
                     void *stream) {
  return embed_impl(ids, T, packed, K, N, g, kDtypeBf16, out, stream);
}

int w4a16_awq_to_standard(const int32_t *qweight_awq, const int32_t *qzeros_awq, int K, int N, int g,
                          int32_t *qweight_std, int32_t *qzeros_std, void *stream) {
  int st = check_shape(K, N, g);
  if (st != W4A16_OK) return st;
  if (!qweight_awq || !qzeros_awq || !qweight_std || !qzeros_std) return W4A16_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(qweight_awq) & 3u) || (reinterpret_cast<uintptr_t>(qzeros_awq) & 3u) ||
      !aligned16(qweight_std) || (reinterpret_cast<uintptr_t>(qzeros_std) & 3u))
    return W4A16_ERR_MISALIGNED;
  const int zero_rows = (g == -1 || g == K) ? 1 : K / g;
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  return map_launch(launch_awq_to_standard(qweight_awq, qzeros_awq, K, N, zero_rows, qweight_std, qzeros_std, err,
                                           static_cast<cudaStream_t>(stream)));
}

int w4a16_dequant(const void *packed, int K, int N, int g, uint16_t *W, void *stream) {
  return dequant_impl(packed, K, N, g, kDtypeF16, W, stream);
}

int w4a16_dequant_bf16(const void *packed, int K, int N, int g, uint16_t *W, void *stream) {
  return dequant_impl(packed, K, N, g, kDtypeBf16, W, stream);
}

const char *w4a16_status_string(int status) {
  switch (status) {
    case W4A16_OK: return "ok";
    case W4A16_ERR_INVALID: return "invalid argument (null pointer, non-positive size or bad n-range)";
    case W4A16_ERR_UNSUPPORTED:
      return "unsupported shape (need N % 8 == 0 and g in {32, 64, 128} with K % g == 0, or g == K or -1 with "
             "K % 32 == 0)";
    case W4A16_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case W4A16_ERR_WORKSPACE: return "workspace smaller than w4a16_workspace_bytes";
    case W4A16_ERR_CUDA: return "CUDA call or kernel launch failed";
    case W4A16_ERR_DEVICE:
      return "device-side error (packed buffer of another shape or element type, token id out of range, or a "
             "wait that timed out)";
    default: return "unknown status";
  }
}

int w4a16_last_device_error(void *stream) {
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return W4A16_ERR_CUDA;
  }
  int v = 0;
  if (cudaMemcpy(&v, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return W4A16_ERR_CUDA;
  if (v != 0) {
    int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return W4A16_ERR_CUDA;
    return W4A16_ERR_DEVICE;
  }
  return W4A16_OK;
}

int w4a16_layout_version(void) { return (int)kLayoutVersion; }

int w4a16_selftest_wait_timeout(int64_t limit_ns, int *status, void *stream) {
  if (limit_ns <= 0 || limit_ns > 100000000 || !status) return W4A16_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(status) & 3u) return W4A16_ERR_MISALIGNED;
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  return map_launch(launch_wait_timeout((uint64_t)limit_ns, status, err, static_cast<cudaStream_t>(stream)));
}

int w4a16_bounds_checked(void) { return bounds_checked() ? 1 : 0; }

int w4a16_selftest_bounds(int *status, void *stream) {
  if (!status) return W4A16_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(status) & 3u) return W4A16_ERR_MISALIGNED;
  int *err = device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  return map_launch(launch_bounds_selftest(status, err, static_cast<cudaStream_t>(stream)));
}

int w4a16_set_option(int option, int value) {
  if (option == W4A16_OPT_SPLITK_REDUCTION) return set_splitk_mode(value);
  return W4A16_ERR_INVALID;
}

}  // extern "C"
#pragma GCC visibility pop
