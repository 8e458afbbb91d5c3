/*
 * qlora_nf4.h -- C ABI of the B300 (sm_103a) QLoRA NF4 + LoRA linear-layer library.
 *
 * The method (QLoRA tutorial pages):
 *   - infivelines.com "QLoRA", mechanism paragraphs: the frozen base is stored in 4 bits
 *     as NormalFloat4 (16 levels at normal quantiles), each block of 64 weights carries
 *     its own scale, the block scales are quantized again in blocks of 256 (about 0.127
 *     bits per weight), the base is dequantized to bf16 one block at a time inside the
 *     matrix multiply, and gradients flow through the frozen base into the adapters.
 *   - junaidshaukat.com "QLoRA -- the democratization event", recipe items 1-4: 4-bit NF4
 *     frozen base, 16-bit LoRA adapters, on-the-fly dequantization, double quantization.
 *   - addaly.com "QLoRA on one card", "What each setting is doing": weights stored in
 *     4 bits, dequantized to bfloat16 for each matrix multiply.
 *
 * Conventions for every entry point:
 *   - Ownership: the caller allocates and owns every buffer (device memory unless stated);
 *     the library never allocates or frees memory.
 *   - Asynchrony: device work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and the call returns without synchronizing.
 *   - Validation: all arguments are checked on the host before any launch; on a negative
 *     status nothing has been enqueued.
 *   - bf16 buffers are passed as uint16_t (raw bfloat16 bits), row-major.
 *   - Inputs must be finite; NaN/Inf inputs give unspecified (but memory-safe) results.
 *   - Layout: W is [N, K] row-major (out x in, the PyTorch Linear layout), X is [M, K],
 *     Y is [M, N], A is [r, K], B is [N, r], s = scale = alpha / r.
 */
#ifndef QLORA_NF4_H
#define QLORA_NF4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  0 is success; every failure is negative. */
#define QLORA_OK 0
#define QLORA_ERR_INVALID_ARG (-1)    /* null pointer, non-positive size, bad scale      */
#define QLORA_ERR_UNSUPPORTED (-2)    /* blocksize != 64, dq_block not 256 or 0, r > 128, or a
                                         GEMM shape the kernels do not cover            */
#define QLORA_ERR_MISALIGNED (-3)     /* a pointer is not 16-byte aligned                */
#define QLORA_ERR_WORKSPACE (-4)      /* workspace smaller than the *_workspace_bytes size */
#define QLORA_ERR_CUDA (-5)           /* a CUDA runtime call or kernel launch failed     */
#define QLORA_ERR_DEVICE_TIMEOUT (-6) /* a kernel gave up a bounded wait (see
                                         qlora_device_status)                            */
#define QLORA_ERR_NO_DEVICE (-7)      /* current device is not a compute-capability 10.3
                                         GPU                                             */
#define QLORA_ERR_TOO_LARGE (-8)      /* tensor larger than nf4_quantize_noalloc's fixed
                                         scratch allows (NF4_NOALLOC_MAX_NUMEL)          */

#define NF4_BLOCKSIZE 64  /* weights per first-level block (one absmax scale each)   */
#define NF4_DQ_BLOCK 256  /* first-level scales per second-level (double-quant) group */
#define NF4_NO_DQ 0       /* dq_block value of the variant without double quantization */
#define NF4_DQ_INT8 0     /* dq_type: second-level codes are int8 steps around the mean  */
#define NF4_DQ_FP8 1      /* dq_type: second-level codes are 8-bit floats (E4M3)          */

/*
 * A blockwise NF4 tensor with double-quantized scales: views into caller-owned device
 * memory.  numel = rows * cols, flattened row-major; block b covers flat elements
 * [64 b, 64 b + 64); group g covers blocks [256 g, 256 g + 256).
 *   codes        [ceil(numel / 2)] uint8: two 4-bit level indices per byte, the even flat
 *                element in the high nibble (an odd numel leaves the last low nibble 0).
 *   scale_codes  [ceil(numel / 64)] int8 in [-127, 127]: second-level code of each block's
 *                absmax, relative to scale_mean.
 *   scale_steps  [ceil(numel / 16384)] fp32: second-level step of each group.
 *   scale_mean   [1] fp32 on the device: the per-tensor mean of the block absmax values.
 * The recovered block scale is fmaf(scale_codes[b], scale_steps[b / 256], scale_mean[0]),
 * and weight e dequantizes to bf16_rne(level[code_e] * scale) (one fp32 multiply).
 * All four pointers must be 16-byte aligned.
 * Variant without double quantization (dq_block = NF4_NO_DQ; junaidshaukat.com recipe item 4
 * and addaly.com "What each setting is doing" present double quantization as a separate,
 * optional saving; infivelines.com "QLoRA": without it the block scales cost 32/64 = 0.5 bits
 * per weight): scale_steps holds the fp32 absmax of every block [ceil(numel / 64)], the block
 * scale is that absmax, and scale_codes and scale_mean are unused (may be NULL).
 * Variant with an 8-bit-float second level (dq_type = NF4_DQ_FP8; the QLoRA paper, which the
 * pages cite, quantizes the constants to 8-bit floats in blocks of 256): scale_codes holds
 * E4M3 bytes (sign, 4 exponent bits of bias 7, 3 mantissa bits, largest finite 448), the
 * group step is max |a - mean| / 448 and the block scale is
 * fmaf(e4m3_value(scale_codes[b]), scale_steps[b / 256], scale_mean[0]).
 * Every call taking an nf4_tensor accepts each variant.
 */
typedef struct nf4_tensor {
  uint8_t* codes;
  int8_t* scale_codes;
  float* scale_steps;
  float* scale_mean;
  int64_t rows; /* N */
  int64_t cols; /* K */
  int32_t blocksize; /* must be NF4_BLOCKSIZE */
  int32_t dq_block;  /* NF4_DQ_BLOCK, or NF4_NO_DQ */
  int32_t dq_type;   /* NF4_DQ_INT8 or NF4_DQ_FP8 (with dq_block = NF4_DQ_BLOCK) */
} nf4_tensor;

/*
 * Sizes in bytes of the four nf4_tensor buffers for a rows x cols tensor:
 * sizes[0] codes, sizes[1] scale_codes, sizes[2] scale_steps, sizes[3] scale_mean (with
 * dq_block = NF4_NO_DQ: codes, 0, 4 * ceil(numel / 64), 0); *total
 * is their sum (4.127 bits per weight: infivelines.com "QLoRA", the 0.127 bits/weight
 * figure for scales per 64 quantized again per 256).  Either output may be NULL.
 * Host only.  Returns QLORA_ERR_INVALID_ARG for rows or cols < 1,
 * QLORA_ERR_UNSUPPORTED for another blocksize, or a dq_block other than 256 and 0.
 */
int nf4_storage_bytes(int64_t rows, int64_t cols, int32_t blocksize, int32_t dq_block,
                      uint64_t sizes[4], uint64_t* total);

/* Device workspace nf4_quantize needs for numel weights (host only). */
int nf4_quantize_workspace_bytes(int64_t numel, uint64_t* out);

/*
 * Quantize fp32 weights W [rows*cols] (device) to NF4 with double-quantized scales into
 * the caller's nf4_tensor `out` (infivelines.com "QLoRA": NF4 levels, blocks of 64,
 * scales quantized again in blocks of 256; digipro.cn "QLoRA: Fine-Tuning a 7B Model on a
 * 16GB GPU": the weights are quantized as they are loaded).
 * Per block: absmax a, x = w / a (IEEE fp32 division; a = 0 gives x = 0), code = index of
 * the nearest of the 16 levels (ties to the lower index).  Then mean = fp64 pairwise sum of
 * all a / count (rounded to fp32); per group step = max |a - mean| / 127 and
 * scale_code = clamp(rint((a - mean) / step), -127, 127) (0 when step = 0).  With
 * out->dq_block = NF4_NO_DQ the block absmax values are stored as they are (no second level);
 * with out->dq_type = NF4_DQ_FP8, step = max |a - mean| / 448 and the code is
 * (a - mean) / step rounded to the nearest E4M3 value (ties to even, saturating at 448).
 * `workspace` (device, >= nf4_quantize_workspace_bytes) is scratch that the call
 * overwrites.  W, out buffers and workspace must be 16-byte aligned.  Any numel >= 1.
 */
int nf4_quantize(const float* W, const nf4_tensor* out, void* workspace,
                 uint64_t workspace_bytes, void* stream);

/*
 * nf4_quantize without a workspace argument, for callers that must not allocate device
 * memory when they quantize: a plugin inside a host application that owns every device
 * allocation, or a service that reserves its memory at start-up and keeps cudaMalloc (and
 * its implicit synchronization) off the request path.  The QLoRA pages have no counterpart
 * to this call; it computes exactly what nf4_quantize computes (bit-identical outputs).
 * Its scratch is a file-scope device array of the library sized for NF4_NOALLOC_MAX_NUMEL
 * weights (about 5.2 MB, held by every GPU that loads the library until exit); the call
 * itself allocates nothing.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current (again after the device's context is
 * created anew, e.g. after cudaDeviceReset), so make that first call before any stream
 * capture.  `stream` must belong to the current device (QLORA_ERR_INVALID_ARG otherwise).
 * All calls share the array: calls that overlap on the GPU (for example on two streams)
 * race and must be ordered by the caller.  rows * cols above
 * NF4_NOALLOC_MAX_NUMEL returns QLORA_ERR_TOO_LARGE with nothing enqueued.
 */
#define NF4_NOALLOC_MAX_NUMEL 67108864LL /* 2^26 weights, e.g. one 8192 x 8192 matrix */
int nf4_quantize_noalloc(const float* W, const nf4_tensor* out, void* stream);

/*
 * Dequantize an nf4_tensor to bf16 W_out [rows*cols] (device), bit-exactly the rule in
 * the nf4_tensor comment (addaly.com "QLoRA on one card": 4-bit storage dequantized to
 * bfloat16).  W_out 16-byte aligned.  Any numel >= 1.
 */
int nf4_dequantize(const nf4_tensor* q, uint16_t* W_out, void* stream);

/*
 * nf4_dequantize with fp16 output (the fp16 compute type: digipro.cn "QLoRA: Fine-Tuning a
 * 7B Model on a 16GB GPU", "The QLoRA insight", where the compute-dtype flag dequantizes to
 * fp16 for the matrix multiplies).  Each weight is the same fp32 product L[c] * absmax_hat
 * rounded once to fp16 (nearest, ties to even; fp16 subnormals kept).  Arguments, alignment
 * and errors as nf4_dequantize.
 */
int nf4_dequantize_f16(const nf4_tensor* q, uint16_t* W_out, void* stream);

/* Device workspace (bytes) qlora_linear_fwd / qlora_linear_bwd need for these sizes. */
int qlora_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r, uint64_t* out);

/*
 * LoRA-wrapped NF4 linear layer, forward (junaidshaukat.com recipe items 2-3; infivelines
 * "QLoRA": dequantized to bf16 one block at a time inside the matrix multiply):
 *     U = X A^T (fp32),   Y = bf16( X W'^T + scale * U B^T )
 * where W' is the bf16 dequantization of Wq.  X [M, K], A [r, K], B [N, r], Y [M, N] are
 * bf16 device buffers; U_save, if not NULL, receives U as fp32 [M, r] for the backward.
 * M >= 1; N = Wq->rows and K = Wq->cols must be multiples of 64; 1 <= r <= 128.
 * M <= 16 runs the decode (GEMV-shaped) kernel, larger M the tensor-core GEMM.
 * The product accumulates in fp32; the LoRA term enters the accumulator as bf16(scale*U).
 * ws: device scratch of at least qlora_workspace_bytes(M, N, K, r).
 */
int qlora_linear_fwd(const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                     const uint16_t* A, const uint16_t* B, int32_t r, float scale,
                     uint16_t* Y, float* U_save, void* ws, uint64_t ws_bytes, void* stream);

/*
 * qlora_linear_fwd in the fp16 compute type (digipro.cn "QLoRA: Fine-Tuning a 7B Model on a
 * 16GB GPU", "The QLoRA insight": the compute-dtype flag set to fp16).  X, A, B and Y are
 * fp16; W' is the fp16 dequantization (as nf4_dequantize_f16); the LoRA term enters the fp32
 * accumulator as fp16(scale*U) and Y is rounded once to fp16.  Everything else (shapes,
 * decode path for M <= 16, U_save, ws, errors) as qlora_linear_fwd.  Values beyond the fp16
 * range become infinities, as in any fp16 matrix multiply.
 */
int qlora_linear_fwd_f16(const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                         const uint16_t* A, const uint16_t* B, int32_t r, float scale,
                         uint16_t* Y, float* U_save, void* ws, uint64_t ws_bytes,
                         void* stream);

/*
 * qlora_linear_fwd for M <= 16 tokens that each choose their own adapter over one shared NF4
 * base (addaly.com "QLoRA on one card", "Merging a QLoRA adapter, and the subtlety": keep the
 * adapter separate and load it over the base, which also lets you swap adapters):
 *     Y_t = bf16( X_t W'^T + s_a (X_t A_a^T) B_a^T ),  a = adapter_idx[t]
 * A_all [n_adapters, r, K] and B_all [n_adapters, N, r] bf16; adapter_idx [M] int32 and
 * scales [n_adapters] fp32 are device buffers (4-byte aligned).  A token whose index is
 * outside [0, n_adapters) gets the base product only.  U_t is formed in fp32 (fixed-order
 * split over K), the adapter term s_a U_t B_a^T in fp32 and added to the fp32 base product
 * before the one rounding to bf16.  Shapes as for qlora_linear_fwd; M > 16 returns
 * QLORA_ERR_UNSUPPORTED.  ws: qlora_workspace_bytes(M, N, K, r).
 */
int qlora_linear_fwd_multi(const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                           const uint16_t* A_all, const uint16_t* B_all, int32_t r,
                           int32_t n_adapters, const int32_t* adapter_idx, const float* scales,
                           uint16_t* Y, void* ws, uint64_t ws_bytes, void* stream);

/*
 * Backward of qlora_linear_fwd with the base frozen (junaidshaukat.com recipe item 3 and
 * infivelines "QLoRA": gradients flow back through the quantized weights without updating
 * them -- there is no dW):
 *     V  = dY B (fp32 [M, r])
 *     dX = bf16( dY W' + scale * V A )      [M, K]  (skipped when dX is NULL)
 *     dA = scale * V^T X                     [r, K]  fp32
 *     dB = scale * dY^T U                    [N, r]  fp32
 * U_saved is the fp32 U from the forward, or NULL to recompute it from X and A.
 * dY [M, N], X [M, K] bf16.  Shapes and ws as for the forward.  The NF4 buffers are only
 * read.
 */
int qlora_linear_bwd(const uint16_t* dY, const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                     const uint16_t* A, const uint16_t* B, int32_t r, float scale,
                     const float* U_saved, uint16_t* dX, float* dA, float* dB, void* ws,
                     uint64_t ws_bytes, void* stream);

/*
 * qlora_linear_bwd in the fp16 compute type: dY, X, A, B and dX are fp16, W' is the fp16
 * dequantization, and the fp32 side products enter the tensor cores as fp16(scale*V) and
 * fp16(U); dA and dB are fp32 as in qlora_linear_bwd.  Everything else as qlora_linear_bwd.
 */
int qlora_linear_bwd_f16(const uint16_t* dY, const uint16_t* X, int64_t M,
                         const nf4_tensor* Wq, const uint16_t* A, const uint16_t* B, int32_t r,
                         float scale, const float* U_saved, uint16_t* dX, float* dA, float* dB,
                         void* ws, uint64_t ws_bytes, void* stream);

/*
 * Fold a LoRA adapter into the NF4 base (junaidshaukat.com "QLoRA -- the democratization
 * event", the deployment-subtlety paragraph: dequantize, merge, maybe requantize;
 * infivelines.com "QLoRA": merging into a 4-bit base and saving loses precision twice;
 * addaly.com "QLoRA on one card", "Merging a QLoRA adapter, and the subtlety"):
 *     W_merged[n, k] = bf16( W'[n, k] + scale * sum_j B[n, j] A[j, k] )
 * with W' the bf16 dequantization of Wq (as nf4_dequantize), the rank-r sum in fp32 in
 * ascending j, then one fp32 multiply by scale, one fp32 add and one round to bf16.
 * A [r, K], B [N, r] bf16; W_merged [N, K] bf16 and W_merged_f32 [N, K] fp32 (the same values,
 * ready for nf4_quantize to requantize) are each optional but not both NULL.  N = Wq->rows,
 * K = Wq->cols with K % 8 == 0; 1 <= r <= 128.  All pointers 16-byte aligned.
 */
int nf4_merge_lora(const nf4_tensor* Wq, const uint16_t* A, const uint16_t* B, int32_t r,
                   float scale, uint16_t* W_merged, float* W_merged_f32, void* stream);

/*
 * NF4 against INT4 on the same weights (aicurriculum.codextroop.com "QLoRA -- Module 12.4",
 * "Design Details That Matter": NF4 is often better than naive INT4; addaly.com "QLoRA on one
 * card", "What each setting is doing"): for fp32 W [numel] (device), per block of 64 with its
 * absmax a (no second-level quantization), out[0] = sum w^2, out[1] = sum (w - level[c] a)^2
 * with c the nearest NF4 level of RN(w / a), out[2] = sum (w - q RN(a / 7))^2 with
 * q = clamp(rint(RN(7 RN(w / a))), -7, 7) (symmetric absmax INT4).  Each thread sums its 16
 * weights in fp32, the rest is summed in fp64; out is 3 doubles of device memory.
 * workspace: device scratch of nf4_int4_error_workspace_bytes (current device).  W and
 * workspace 16-byte aligned; any numel >= 1.
 */
int nf4_int4_error_workspace_bytes(uint64_t* out);
int nf4_int4_error_stats(const float* W, int64_t numel, double* out, void* workspace,
                         uint64_t workspace_bytes, void* stream);

/*
 * The fp32 constants the kernels use (host only): levels[16], the NF4 levels in ascending
 * order, and thresholds[15], the midpoints of adjacent levels rounded toward -inf
 * (code = number of thresholds strictly below x).  Either pointer may be NULL.
 */
int nf4_level_table(float levels[16], float thresholds[15]);

/*
 * Reads and clears the device error word that kernels set when a bounded wait on an
 * mbarrier gives up (instead of hanging).  Synchronizes `stream`.  *out = 0 when clean,
 * else a nonzero code naming the wait (1..6), 7 when the decode kernel found a shared
 * window that its fixed layout does not fit and returned without work, or 8 after
 * qlora_wait_timeout_selftest.  Returns QLORA_ERR_DEVICE_TIMEOUT if it was set.
 */
int qlora_device_status(int32_t* out, void* stream);

/*
 * Self-test of the bounded waits (the pages have no counterpart; every kernel here waits on
 * mbarriers for its TMA copies and stages, and a wait that never completes must end in a
 * status, not a hang).  Enqueues on `stream` one CTA that waits, with the same bounded wait
 * the kernels use, on an mbarrier that nothing ever arrives on.  After the wait limit (about
 * 2 s) the wait gives up, records code 8 in the device error word and the kernel returns; the
 * device and its context stay usable.  The next qlora_device_status returns
 * QLORA_ERR_DEVICE_TIMEOUT with *out = 8 and clears the word.  Returns QLORA_OK once the
 * kernel is enqueued, QLORA_ERR_NO_DEVICE without a compute-capability 10.3 device.
 */
int qlora_wait_timeout_selftest(void* stream);

/*
 * Opt-in per-kernel device timing (host only; a measurement aid, not thread-safe).
 * qlora_profile_start: from now on every kernel the library launches is bracketed by CUDA
 * events recorded on the launch's own stream.  qlora_profile_stop: waits for those events,
 * writes one entry per kernel name (launch count, summed device milliseconds) into
 * out[0 .. capacity), sets *count to the number of distinct kernels and turns timing off.
 * Profiling creates CUDA events (driver objects) but never device memory.
 */
typedef struct qlora_kernel_time {
  char name[48];
  int32_t launches;
  double total_ms;
} qlora_kernel_time;

int qlora_profile_start(void);
int qlora_profile_stop(qlora_kernel_time* out, int32_t capacity, int32_t* count);

/* Human-readable text for a status code (static storage, host only). */
const char* qlora_status_str(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
int qlora_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QLORA_NF4_H */
