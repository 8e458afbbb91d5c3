// api.cu -- the C ABI (include/qlora_nf4.h): host-side validation, then launches.
#include <cstring>

#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "nf4_device.cuh"

using namespace qlora;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QLORA_ERR_NO_DEVICE;
  static thread_local int cached_dev = -1, cached_ok = 0;
  if (dev != cached_dev) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return QLORA_ERR_NO_DEVICE;
    cached_dev = dev;
    cached_ok = (major == 10 && minor == 3);
  }
  return cached_ok ? QLORA_OK : QLORA_ERR_NO_DEVICE;
}

int check_tensor(const nf4_tensor* q) {
  if (!q) return QLORA_ERR_INVALID_ARG;
  if (q->rows < 1 || q->cols < 1) return QLORA_ERR_INVALID_ARG;
  if (q->blocksize != NF4_BLOCKSIZE || (q->dq_block != NF4_DQ_BLOCK && q->dq_block != NF4_NO_DQ) ||
      (q->dq_type != NF4_DQ_INT8 && q->dq_type != NF4_DQ_FP8))
    return QLORA_ERR_UNSUPPORTED;
  const bool dq = q->dq_block != NF4_NO_DQ;
  if (!q->codes || !q->scale_steps || (dq && (!q->scale_codes || !q->scale_mean)))
    return QLORA_ERR_INVALID_ARG;
  if (!aligned16(q->codes) || !aligned16(q->scale_steps) ||
      (dq && (!aligned16(q->scale_codes) || !aligned16(q->scale_mean))))
    return QLORA_ERR_MISALIGNED;
  return QLORA_OK;
}

// The bf16 and fp16 entry points share their validation and launch; `half` selects the
// 16-bit type of the activations, adapters and outputs.
int dequantize_impl(const nf4_tensor* q, uint16_t* W_out, bool half, void* stream) {
  int st = check_tensor(q);
  if (st) return st;
  if (!W_out) return QLORA_ERR_INVALID_ARG;
  if (!aligned16(W_out)) return QLORA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  return launch_dequantize(*q, q->rows * q->cols, W_out, half,
                           static_cast<cudaStream_t>(stream));
}

int linear_fwd_impl(const uint16_t* X, int64_t M, const nf4_tensor* Wq, const uint16_t* A,
                    const uint16_t* B, int32_t r, float scale, uint16_t* Y, float* U_save,
                    void* ws, uint64_t ws_bytes, bool half, void* stream) {
  int st = check_tensor(Wq);
  if (st) return st;
  if (!X || !A || !B || !Y || !ws || M < 1 || r < 1) return QLORA_ERR_INVALID_ARG;
  if (!(scale == scale)) return QLORA_ERR_INVALID_ARG;
  if (r > kMaxRank) return QLORA_ERR_UNSUPPORTED;
  const int64_t N = Wq->rows, K = Wq->cols;
  if (N % 64 != 0 || K % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(Y) || !aligned16(ws) ||
      (U_save && !aligned16(U_save)))
    return QLORA_ERR_MISALIGNED;
  if (ws_bytes < linear_workspace_bytes(M, N, K, r)) return QLORA_ERR_WORKSPACE;
  if ((st = check_device())) return st;
  LinearArgs a{};
  a.M = M; a.N = N; a.K = K; a.r = r; a.scale = scale;
  a.X = X; a.A = A; a.B = B; a.Y = Y; a.U = U_save; a.q = *Wq;
  a.ws = ws; a.ws_bytes = ws_bytes; a.half = half;
  return linear_forward(a, static_cast<cudaStream_t>(stream));
}

int linear_bwd_impl(const uint16_t* dY, const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                    const uint16_t* A, const uint16_t* B, int32_t r, float scale,
                    const float* U_saved, uint16_t* dX, float* dA, float* dB, void* ws,
                    uint64_t ws_bytes, bool half, void* stream) {
  int st = check_tensor(Wq);
  if (st) return st;
  if (!dY || !X || !A || !B || !dA || !dB || !ws || M < 1 || r < 1) return QLORA_ERR_INVALID_ARG;
  if (!(scale == scale)) return QLORA_ERR_INVALID_ARG;
  if (r > kMaxRank) return QLORA_ERR_UNSUPPORTED;
  const int64_t N = Wq->rows, K = Wq->cols;
  if (N % 64 != 0 || K % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  if (!aligned16(dY) || !aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(dA) ||
      !aligned16(dB) || !aligned16(ws) || (dX && !aligned16(dX)) ||
      (U_saved && !aligned16(U_saved)))
    return QLORA_ERR_MISALIGNED;
  if (ws_bytes < linear_workspace_bytes(M, N, K, r)) return QLORA_ERR_WORKSPACE;
  if ((st = check_device())) return st;
  LinearArgs a{};
  a.M = M; a.N = N; a.K = K; a.r = r; a.scale = scale;
  a.X = X; a.A = A; a.B = B; a.dY = dY; a.dX = dX; a.dA = dA; a.dB = dB;
  a.U_in = U_saved; a.q = *Wq; a.ws = ws; a.ws_bytes = ws_bytes; a.half = half;
  return linear_backward(a, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int qlora_version(void) { return 10000; }

const char* qlora_status_str(int status) {
  switch (status) {
    case QLORA_OK: return "ok";
    case QLORA_ERR_INVALID_ARG: return "invalid argument";
    case QLORA_ERR_UNSUPPORTED: return "unsupported shape or format";
    case QLORA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case QLORA_ERR_WORKSPACE: return "workspace too small";
    case QLORA_ERR_CUDA: return "CUDA runtime or launch error";
    case QLORA_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case QLORA_ERR_NO_DEVICE: return "current device is not compute capability 10.3";
    case QLORA_ERR_TOO_LARGE: return "tensor exceeds the fixed scratch of the no-allocation call";
    default: return "unknown status";
  }
}

int nf4_level_table(float levels[16], float thresholds[15]) {
  static const float L[16] = QLORA_NF4_LEVELS;
  static const float T[15] = QLORA_NF4_THRESHOLDS;
  if (levels) std::memcpy(levels, L, sizeof(L));
  if (thresholds) std::memcpy(thresholds, T, sizeof(T));
  return QLORA_OK;
}

int nf4_storage_bytes(int64_t rows, int64_t cols, int32_t blocksize, int32_t dq_block,
                      uint64_t sizes[4], uint64_t* total) {
  if (rows < 1 || cols < 1) return QLORA_ERR_INVALID_ARG;
  if (blocksize != NF4_BLOCKSIZE || (dq_block != NF4_DQ_BLOCK && dq_block != NF4_NO_DQ))
    return QLORA_ERR_UNSUPPORTED;
  const uint64_t numel = (uint64_t)rows * (uint64_t)cols;
  const uint64_t nb = (numel + NF4_BLOCKSIZE - 1) / NF4_BLOCKSIZE;
  const uint64_t ng = (nb + NF4_DQ_BLOCK - 1) / NF4_DQ_BLOCK;
  const bool dq = dq_block != NF4_NO_DQ;
  const uint64_t s[4] = {(numel + 1) / 2, dq ? nb : 0, dq ? ng * 4 : nb * 4, dq ? 4u : 0u};
  if (sizes) std::memcpy(sizes, s, sizeof(s));
  if (total) *total = s[0] + s[1] + s[2] + s[3];
  return QLORA_OK;
}

int nf4_quantize_workspace_bytes(int64_t numel, uint64_t* out) {
  if (numel < 1 || !out) return QLORA_ERR_INVALID_ARG;
  *out = quantize_workspace_bytes(numel);
  return QLORA_OK;
}

int nf4_quantize(const float* W, const nf4_tensor* out, void* workspace,
                 uint64_t workspace_bytes, void* stream) {
  int st = check_tensor(out);
  if (st) return st;
  if (!W || !workspace) return QLORA_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(workspace)) return QLORA_ERR_MISALIGNED;
  const int64_t numel = out->rows * out->cols;
  if (workspace_bytes < quantize_workspace_bytes(numel)) return QLORA_ERR_WORKSPACE;
  if ((st = check_device())) return st;
  return launch_quantize(W, numel, *out, workspace, static_cast<cudaStream_t>(stream));
}

int nf4_dequantize(const nf4_tensor* q, uint16_t* W_out, void* stream) {
  return dequantize_impl(q, W_out, false, stream);
}

int nf4_dequantize_f16(const nf4_tensor* q, uint16_t* W_out, void* stream) {
  return dequantize_impl(q, W_out, true, stream);
}

int nf4_merge_lora(const nf4_tensor* Wq, const uint16_t* A, const uint16_t* B, int32_t r,
                   float scale, uint16_t* W_merged, float* W_merged_f32, void* stream) {
  int st = check_tensor(Wq);
  if (st) return st;
  if (!A || !B || (!W_merged && !W_merged_f32) || r < 1) return QLORA_ERR_INVALID_ARG;
  if (!(scale == scale)) return QLORA_ERR_INVALID_ARG;
  if (r > kMaxRank || Wq->cols % 8 != 0) return QLORA_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || (W_merged && !aligned16(W_merged)) ||
      (W_merged_f32 && !aligned16(W_merged_f32)))
    return QLORA_ERR_MISALIGNED;
  if ((st = check_device())) return st;
  return launch_merge(*Wq, A, B, r, scale, W_merged, W_merged_f32,
                      static_cast<cudaStream_t>(stream));
}

int nf4_int4_error_workspace_bytes(uint64_t* out) {
  if (!out) return QLORA_ERR_INVALID_ARG;
  int st = check_device();
  if (st) return st;
  *out = static_cast<uint64_t>(error_stats_parts()) * 3 * sizeof(double);
  return QLORA_OK;
}

int nf4_int4_error_stats(const float* W, int64_t numel, double* out, void* workspace,
                         uint64_t workspace_bytes, void* stream) {
  if (!W || !out || !workspace || numel < 1) return QLORA_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(out) & 7u))
    return QLORA_ERR_MISALIGNED;
  int st = check_device();
  if (st) return st;
  if (workspace_bytes < static_cast<uint64_t>(error_stats_parts()) * 3 * sizeof(double))
    return QLORA_ERR_WORKSPACE;
  return launch_error_stats(W, numel, out, workspace, static_cast<cudaStream_t>(stream));
}

int qlora_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t r, uint64_t* out) {
  if (M < 1 || N < 1 || K < 1 || r < 1 || !out) return QLORA_ERR_INVALID_ARG;
  if (r > kMaxRank) return QLORA_ERR_UNSUPPORTED;
  *out = linear_workspace_bytes(M, N, K, r);
  return QLORA_OK;
}

int qlora_linear_fwd(const uint16_t* X, int64_t M, const nf4_tensor* Wq, const uint16_t* A,
                     const uint16_t* B, int32_t r, float scale, uint16_t* Y, float* U_save,
                     void* ws, uint64_t ws_bytes, void* stream) {
  return linear_fwd_impl(X, M, Wq, A, B, r, scale, Y, U_save, ws, ws_bytes, false, stream);
}

int qlora_linear_fwd_f16(const uint16_t* X, int64_t M, const nf4_tensor* Wq, const uint16_t* A,
                         const uint16_t* B, int32_t r, float scale, uint16_t* Y, float* U_save,
                         void* ws, uint64_t ws_bytes, void* stream) {
  return linear_fwd_impl(X, M, Wq, A, B, r, scale, Y, U_save, ws, ws_bytes, true, stream);
}

int qlora_linear_fwd_multi(const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                           const uint16_t* A_all, const uint16_t* B_all, int32_t r,
                           int32_t n_adapters, const int32_t* adapter_idx, const float* scales,
                           uint16_t* Y, void* ws, uint64_t ws_bytes, void* stream) {
  int st = check_tensor(Wq);
  if (st) return st;
  if (!X || !A_all || !B_all || !adapter_idx || !scales || !Y || !ws || M < 1 || r < 1 ||
      n_adapters < 1)
    return QLORA_ERR_INVALID_ARG;
  if (r > kMaxRank || M > kSkinnyMaxM) return QLORA_ERR_UNSUPPORTED;
  const int64_t N = Wq->rows, K = Wq->cols;
  if (N % 64 != 0 || K % 64 != 0) return QLORA_ERR_UNSUPPORTED;
  if (!aligned16(X) || !aligned16(A_all) || !aligned16(B_all) || !aligned16(Y) ||
      !aligned16(ws) || (reinterpret_cast<uintptr_t>(adapter_idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(scales) & 3u))
    return QLORA_ERR_MISALIGNED;
  if (ws_bytes < linear_workspace_bytes(M, N, K, r)) return QLORA_ERR_WORKSPACE;
  if ((st = check_device())) return st;
  LinearArgs a{};
  a.M = M; a.N = N; a.K = K; a.r = r; a.scale = 1.0f;
  a.X = X; a.A = A_all; a.B = B_all; a.Y = Y; a.q = *Wq;
  a.ws = ws; a.ws_bytes = ws_bytes;
  a.adapter_idx = adapter_idx; a.n_adapters = n_adapters; a.scales = scales;
  return linear_forward(a, static_cast<cudaStream_t>(stream));
}

int qlora_linear_bwd(const uint16_t* dY, const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                     const uint16_t* A, const uint16_t* B, int32_t r, float scale,
                     const float* U_saved, uint16_t* dX, float* dA, float* dB, void* ws,
                     uint64_t ws_bytes, void* stream) {
  return linear_bwd_impl(dY, X, M, Wq, A, B, r, scale, U_saved, dX, dA, dB, ws, ws_bytes, false,
                         stream);
}

int qlora_linear_bwd_f16(const uint16_t* dY, const uint16_t* X, int64_t M, const nf4_tensor* Wq,
                         const uint16_t* A, const uint16_t* B, int32_t r, float scale,
                         const float* U_saved, uint16_t* dX, float* dA, float* dB, void* ws,
                         uint64_t ws_bytes, void* stream) {
  return linear_bwd_impl(dY, X, M, Wq, A, B, r, scale, U_saved, dX, dA, dB, ws, ws_bytes, true,
                         stream);
}

int qlora_device_status(int32_t* out, void* stream) {
  if (!out) return QLORA_ERR_INVALID_ARG;
  int st = check_device();
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return QLORA_ERR_CUDA;
  if ((st = read_and_clear_gemm_error(&v))) return st;
  int w = 0, d = 0, t = 0;
  if ((st = read_and_clear_side_error(&w))) return st;
  if ((st = read_and_clear_decode_error(&d))) return st;
  if ((st = read_and_clear_selftest_error(&t))) return st;
  if (!v) v = w;
  if (!v) v = d;
  if (!v) v = t;
  *out = v;
  return v ? QLORA_ERR_DEVICE_TIMEOUT : QLORA_OK;
}

int qlora_wait_timeout_selftest(void* stream) {
  const int st = check_device();
  if (st) return st;
  return launch_wait_selftest(static_cast<cudaStream_t>(stream));
}

}  // extern "C"
