/*
 * w4a16.h -- C ABI of the GB300 (sm_103a) asymmetric group-wise W4A16 linear layer.
 *
 *   y[M,N] = x[M,K] . W,   W[k,n] = (q[k,n] - z[k/g,n]) * s[k/g,n]
 *
 * q and z are 4-bit codes (0..15) packed eight to an int32 along N in the AWQ checkpoint order,
 * s is fp16, x and y are fp16, and one group covers g consecutive rows of K.  The *_bf16 entry
 * points are the same layer with s, x, W and y in bfloat16.
 *
 * Where the operations come from:
 *  - "Carga de capas cuantizadas: AWQ / GPTQ / Marlin / fp8" (vLLM architecture walkthrough):
 *    section "Responsabilidades" splits a quantized linear into create_weights, a one-time
 *    process_weights_after_loading reorder, and apply (the GEMM); w4a16_repack is the one-time
 *    reorder and w4a16_gemm is apply.  Section "Flujo de datos" gives the tensors w4a16_repack
 *    takes: qweight int32 [K, N/8], qzeros int32 [K/g, N/8] (both packed along the output
 *    dimension) and scales [K/g, N].  Section "Limites y fallos" (verify_marlin_supported)
 *    rejects unsupported group sizes and types with an error: here, a status code.
 *  - vllm-omni commit "Add cpu_int4, an asymmetric 4-bit weight path for vLLM's CPU backend":
 *    the asymmetric grid, and the two paths over one set of weights (a decode path for few
 *    rows, a dense path for many), which w4a16_gemm picks between by M.
 *  - vllm-omni commit "cpu_int4: dequantize prefill weights from the tinygemm layout, not a
 *    copy": the packed layout need not be opaque; decoding it back is w4a16_dequant, which is
 *    bit-exact against the straightforward dequantizer.  The N = 80 case (64 + a 16 tail) must
 *    be handled, not misread.
 *  - vllm-omni commit "cpu_int4: repack weights in n-blocks, to bound the load-time peak":
 *    n-blocks are independent, so w4a16_repack_chunk packs one n-range at a time and gives the
 *    same bytes as packing the whole matrix.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library allocates
 *    nothing and keeps no pointer after the call returns.  Every call is asynchronous and
 *    ordered on `stream` (a cudaStream_t; NULL means the legacy default stream).  Apart from
 *    w4a16_last_device_error, no call synchronizes.
 *  - Shapes are int; K, N > 0.  Supported group sizes: g in {32, 64, 128} with K % g == 0, or
 *    one group over all of K (per-channel: g == K or g == -1, the group_size = -1 of section
 *    "Limites y fallos", with K % 32 == 0; the scales and zeros then have one row).  N % 8 == 0.
 *    The packed layout stores per-channel weights with g = the largest of 128, 64, 32 dividing
 *    K, every group carrying the column's one scale and zero, so the weights are unchanged;
 *    pass the same g (K or -1) to every call on that buffer.
 *    N need not be a multiple of 64 and K need not be a multiple of 128.
 *  - Device pointers must be 16-byte aligned.
 *  - Return value: W4A16_OK or a negative status (below).  No C++ exception crosses the ABI.
 *    A status other than W4A16_OK means nothing was launched.  Errors raised on the device
 *    (a packed buffer whose header does not match the call's K, N, g, or a bounded wait that
 *    ran out) are recorded in a per-device error word read by w4a16_last_device_error.
 *    A packed buffer's header also records the element type it was packed for (fp16 or
 *    bf16), and the calls of the other type reject it the same way.
 */
#ifndef W4A16_GB300_H
#define W4A16_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define W4A16_OK 0
#define W4A16_ERR_INVALID (-1)     /* null pointer, K/N <= 0, g 0 or < -1, M < 0, bad n-range */
#define W4A16_ERR_UNSUPPORTED (-2) /* N % 8 != 0, K % g != 0, g not 32/64/128/K/-1            */
#define W4A16_ERR_MISALIGNED (-3)  /* a device pointer is not 16-byte aligned                */
#define W4A16_ERR_WORKSPACE (-4)   /* workspace smaller than w4a16_workspace_bytes           */
#define W4A16_ERR_CUDA (-5)        /* a CUDA call or kernel launch failed                    */
#define W4A16_ERR_DEVICE (-6)      /* device-side error, reported by w4a16_last_device_error */

/* Version of the packed layout written by w4a16_repack; stored in every packed buffer's
 * header and checked on the device by w4a16_gemm and w4a16_dequant. */
#define W4A16_LAYOUT_VERSION 1

/*
 * Packed layout, version 1 (own design; the layouts of the pages' other kernels are prior
 * art).  All offsets in bytes from the start of the buffer.
 *   [0, 256)      header: uint32 magic 0x36314134, uint32 version, int32 K, int32 N, int32 g,
 *                 int32 dtype (0: fp16 layer, 1: bf16 layer), then zeros.
 *   [256, ...)    NB = ceil(N/64) n-blocks, each of KT = ceil(K/128) chunks of
 *                 CB = 4096 + (128/g) * 160 bytes; chunk (b, t) starts at 256 + (b*KT + t)*CB
 *                 and covers columns [64b, 64b+64) and rows k in [128t, 128t+128).
 *   chunk codes   [0, 4096): 64 column-rows of 64 bytes; row r is column n = 64b + r and holds
 *                 128 consecutive k as 16 little-endian uint32 words.  Word w holds
 *                 k = 128t + 8w + {0,2,4,6,1,3,5,7}[j] in nibble slot j (bits 4j..4j+3).
 *   chunk meta    [4096, CB): for each of the 128/g groups l of the chunk, 160 bytes:
 *                 64 scales (the layer's fp16 or bf16) then 32 bytes of zero codes, both in
 *                 "lane order": position
 *                 p = 8*(r%8) + 2*(r/16) + (r/8)%2 holds column-row r; the zero of position p
 *                 is nibble p%8 (bits 4(p%8)..) of little-endian uint32 word p/8.
 *   padding       columns n >= N and rows k >= K have code 0, zero code 0 and scale +0.0, so
 *                 the buffer's bytes are a pure function of (qweight, qzeros, scales, K, N, g).
 */

/* Bytes of the packed buffer for a K x N layer with group size g; 0 if the shape is invalid
 * or unsupported. */
size_t w4a16_packed_bytes(int K, int N, int g);

/* Bytes of device workspace w4a16_gemm needs for this problem on the current device under the
 * current options; 0 means none (workspace may then be NULL).  The tensor-core path splits K
 * across up to 8 CTAs when the output tiles alone would leave SMs idle, and adds the fp32
 * partial tiles in split order.  By default the CTAs of a tile form a thread-block cluster
 * and add them through distributed shared memory: no workspace.  The workspace reduction
 * (W4A16_SPLITK_GLOBAL, or a GPU that cannot run the clusters) needs 4096 bytes of per-tile
 * arrival counters at offset 0 followed by the partial tiles.  Stable for given arguments,
 * options and device.  The first 4096 bytes must be zero before the first use; every call that
 * completes leaves them zero (whatever its shape), so one buffer, sized for the largest
 * problem, serves call after call.  Calls that share a workspace must not overlap on the GPU
 * (one workspace per concurrent stream).  After a device-side error, zero the first 4096 bytes
 * again.  Both reductions give bit-identical results. */
size_t w4a16_workspace_bytes(int M, int N, int K, int g);

/* One-time repack of AWQ tensors into the packed layout (integer-exact; scales copied bit for
 * bit).  qweight int32 [K][N/8], qzeros int32 [K/g][N/8], scales fp16 bits [K/g][N], all
 * row-major and contiguous; packed: w4a16_packed_bytes(K, N, g) bytes, fully written. */
int w4a16_repack(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                 int K, int N, int g, void *packed, void *stream);

/* Repack only columns [n0, n1) into their n-blocks of `packed` (and the header).  n0 must be
 * a multiple of 64; n1 a multiple of 64 or equal to N; 0 <= n0 < n1 <= N.  The inputs are the
 * slices starting at column n0: qweight_c points at qweight[0][n0/8] with a row stride of
 * ld_qweight int32 elements, qzeros_c at qzeros[0][n0/8] (stride ld_qzeros), scales_c at
 * scales[0][n0] (stride ld_scales fp16 elements); a caller that holds only the slice passes
 * its compact strides.  Repacking every n-range of a partition of [0, N) yields the same
 * bytes as w4a16_repack. */
int w4a16_repack_chunk(const int32_t *qweight_c, int64_t ld_qweight,
                       const int32_t *qzeros_c, int64_t ld_qzeros,
                       const uint16_t *scales_c, int64_t ld_scales,
                       int K, int N, int g, int n0, int n1, void *packed, void *stream);

/* y = x . W.  x fp16 bits [M][K] row-major, y fp16 bits [M][N] row-major (fully written),
 * packed from w4a16_repack with the same K, N, g.  M == 0 is a no-op.  M <= 32 takes the
 * decode path (fused dequant + skinny GEMM streaming the packed weights once); larger M the
 * tensor-core path (weights dequantized to fp16 tile by tile into tensor memory, tcgen05 MMAs
 * with fp32 accumulation in tensor memory).  Accumulation is in fp32; the result is rounded
 * once to fp16 and is bit-identical from run to run.  workspace: w4a16_workspace_bytes(M, N,
 * K, g) bytes of 16-byte aligned device memory (may be NULL when that is 0), see there.
 * A w4a16_gemm may start reading `packed` while the previous w4a16_gemm on the same stream is
 * still running (programmatic dependent launch); it reads x and writes y only after that one
 * has completed. */
int w4a16_gemm(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
               void *workspace, size_t workspace_bytes, void *stream);

/* W = fp16((q - z) * s) for every k < K, n < N, written as fp16 bits [K][N] row-major: one
 * round-to-nearest-even rounding of the exact product, bit-identical to the straightforward
 * dequantizer. */
int w4a16_dequant(const void *packed, int K, int N, int g, uint16_t *W, void *stream);

/* Gather of the quantized tied embedding (the LM head's weight doubles as the embedding table:
 * vllm-omni commit "cpu_int4: repack weights in n-blocks, to bound the load-time peak", whose
 * transient table lists the embedding as "tied, so it is also the head"; commit "Add cpu_int4
 * ...": "the quantized tied embedding").  For t < T, row t of out (fp16 bits [T][K], row-major,
 * fully written) is column ids[t] of W: out[t][k] = fp16((q[k][n] - z[k/g][n]) * s[k/g][n]) with
 * n = ids[t], one round-to-nearest-even rounding, bit-identical to w4a16_dequant's column n.
 * ids: int32 [T] device array, 4-byte aligned.  T == 0 is a no-op.  An id outside [0, N) gives
 * a row of zeros and a device-side error (w4a16_last_device_error). */
int w4a16_embed(const int32_t *ids, int T, const void *packed, int K, int N, int g, uint16_t *out,
                void *stream);

/* AWQ packing -> the GPTQ-style "standard" packing ("Carga de capas cuantizadas: AWQ / GPTQ /
 * Marlin / fp8", section "Motivacion de diseno": AWQ packs along the output dimension in a
 * non-standard order, the standard format along the input dimension in plain order), integer
 * exact.  In: qweight_awq int32 [K][N/8], qzeros_awq int32 [K/g][N/8] (one row per-channel).
 * Out (fully written): qweight_std int32 [K/8][N], nibble j of word (r, n) = q[8r + j][n];
 * qzeros_std int32 [K/g][N/8], nibble j of word (G, c) = z[G][8c + j].  The scales are shared
 * by both formats.  qweight_std 16-byte aligned, the other pointers 4-byte aligned; the outputs
 * must not overlap the inputs. */
int w4a16_awq_to_standard(const int32_t *qweight_awq, const int32_t *qzeros_awq, int K, int N, int g,
                          int32_t *qweight_std, int32_t *qzeros_std, void *stream);

/* Size of the scratch array built into the library for w4a16_gemm_noalloc (24 MiB): every GPU
 * that loads the library keeps this much device memory for the life of the process. */
#define W4A16_NOALLOC_SCRATCH_BYTES (24u << 20)

/* y = x . W like w4a16_gemm, for callers that cannot allocate device memory at all -- a runtime
 * that plans every device buffer ahead and hands a layer only its inputs and outputs, a plugin
 * host that forbids allocation after start-up, a latency-critical path where an allocation could
 * stall or fail.  No workspace is passed: when the tensor-core path adds split-K partial tiles
 * through memory (the workspace reduction), they live in an array of
 * W4A16_NOALLOC_SCRATCH_BYTES inside the library (no counterpart on the pages; this entry point
 * exists only for such callers).  The caller still provides x, packed and y as for
 * w4a16_gemm.  Returns W4A16_ERR_WORKSPACE when the problem's scratch (w4a16_workspace_bytes)
 * exceeds that size.  All calls share the one array, so calls that overlap on the GPU race with
 * each other and must be serialized.  The first call on a device sets that device up (looks up
 * the array and clears the counters at its head, ordered on `stream` before the call's kernel),
 * so make it before capturing the stream; every completed call leaves those counters cleared
 * again.  Never calls cudaMalloc, cudaFree or any other allocating routine.  The array's device
 * memory is not free, though: CUDA commits the library's device code and this array on a device
 * when the library is first used there, which can be inside the first call, and that call then
 * fails with W4A16_ERR_CUDA if the device is out of memory; a caller that must not fail later
 * makes one call (or any other call of this library) on each device at start-up. */
int w4a16_gemm_noalloc(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
                       void *stream);

/* Process-wide options, read by the host when a call launches its kernels. */
#define W4A16_OPT_SPLITK_REDUCTION 1 /* how split-K partial tiles are added:              */
#define W4A16_SPLITK_AUTO 0          /*   cluster + distributed shared memory if possible */
#define W4A16_SPLITK_GLOBAL 1        /*   always through the caller's workspace           */

/* Set an option (W4A16_OPT_*) to a value; W4A16_ERR_INVALID for an unknown option or value.
 * Changes what w4a16_workspace_bytes reports for split-K problems: size workspaces after
 * setting it.  Not a per-call or per-thread setting: set it before issuing work. */
int w4a16_set_option(int option, int value);

/* The bfloat16 layer.  Same operation, shapes, layout, alignment and error behaviour as the
 * entry point without the suffix, with the scales, x, the weights W and y in bfloat16 (bits as
 * uint16) instead of fp16: W = bf16((q - z) * s) with one round-to-nearest-even rounding, and
 * y accumulated in fp32 and rounded once to bf16.  The pages' own CPU path computes in bf16
 * (vllm-omni commit "Add cpu_int4, an asymmetric 4-bit weight path for vLLM's CPU backend":
 * wider batches unpack the weight to bf16 once, and bf16 is the reference it is measured
 * against).  A buffer packed by w4a16_repack_bf16 / w4a16_repack_chunk_bf16 records dtype 1 in
 * its header and is accepted only by the *_bf16 calls (and an fp16 buffer only by the others):
 * a mismatch is a device-side error and nothing is written.  M <= 32 takes the decode path
 * (bf16 mma.sync), larger M the tensor-core path (tcgen05 kind::f16 with bf16 operands); the
 * workspace is that of w4a16_workspace_bytes. */
int w4a16_repack_bf16(const int32_t *qweight, const int32_t *qzeros, const uint16_t *scales,
                      int K, int N, int g, void *packed, void *stream);
int w4a16_repack_chunk_bf16(const int32_t *qweight_c, int64_t ld_qweight,
                            const int32_t *qzeros_c, int64_t ld_qzeros,
                            const uint16_t *scales_c, int64_t ld_scales,
                            int K, int N, int g, int n0, int n1, void *packed, void *stream);
int w4a16_gemm_bf16(const uint16_t *x, const void *packed, int M, int N, int K, int g, uint16_t *y,
                    void *workspace, size_t workspace_bytes, void *stream);
int w4a16_dequant_bf16(const void *packed, int K, int N, int g, uint16_t *W, void *stream);
int w4a16_embed_bf16(const int32_t *ids, int T, const void *packed, int K, int N, int g, uint16_t *out,
                     void *stream);

/* Self-test of failure detection, faulting nothing: one thread waits, with the library's bounded
 * waits (polling, then sleeping), on a barrier that never completes, each giving up after
 * limit_ns nanoseconds (0 < limit_ns <= 100 ms).  *status (a 4-byte aligned device int) gets
 * bit 0 if the polling wait gave up and bit 1 if the sleeping one did (3 when both work), and
 * the device error word records the timeout as the GEMM kernels do: w4a16_last_device_error then
 * returns W4A16_ERR_DEVICE, and the context stays usable.  The analogue of the pages' benchmark
 * harness that records failures instead of dropping them (vllm-omni commit "cpu_int4:
 * dequantize prefill weights from the tinygemm layout, not a copy"). */
int w4a16_selftest_wait_timeout(int64_t limit_ns, int *status, void *stream);

/* 1 if this library is the bounds-checked debug build, else 0.  That build (the same sources
 * compiled with W4A16_BOUNDS defined, shipped as _libw4a16_bounds.so beside the normal library,
 * with the same entry points) checks every global read of the packed weights, x, ids and the AWQ
 * tensors, and every global write of y, W, out and the split-K workspace, against the extent of
 * its buffer as the call's arguments define it (w4a16_packed_bytes for a packed buffer, M*K
 * elements for x, M*N for y, the slices' rows times their strides for w4a16_repack_chunk, ...).
 * An access outside it is skipped (a read gives zeros) and recorded in the device error word:
 * w4a16_last_device_error then returns W4A16_ERR_DEVICE.  Nothing traps.  It stands in for a
 * memory checker (the test strategy's "Race detection / sanitizers"); it is slower and is not
 * meant for production. */
int w4a16_bounds_checked(void);

/* Self-test of the bounds check, dereferencing nothing: one thread runs the check on five fixed
 * (offset, size, extent) cases, two inside their buffer and three outside (one byte past the end,
 * one byte before the start, any byte of an empty buffer), and writes to *status (a 4-byte aligned
 * device int) bit i for each case judged outside.  The bounds-checked build writes 0x1C and
 * records the misses in the device error word; the normal build, whose check is compiled out,
 * writes 0 and records nothing. */
int w4a16_selftest_bounds(int *status, void *stream);

/* Static description of a status code. */
const char *w4a16_status_string(int status);

/* Synchronizes `stream`, then returns W4A16_ERR_DEVICE if a kernel of this library recorded a
 * device-side error on the current device since the last call (and clears the record),
 * W4A16_ERR_CUDA if the synchronization itself failed, else W4A16_OK. */
int w4a16_last_device_error(void *stream);

/* W4A16_LAYOUT_VERSION of the library actually loaded. */
int w4a16_layout_version(void);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_GB300_H */
