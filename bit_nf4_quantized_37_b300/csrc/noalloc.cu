// noalloc.cu -- nf4_quantize_noalloc: the NF4 quantizer with its scratch in a fixed
// library-owned device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they quantize: a plugin
// running inside a host application that owns every device allocation through its own
// pool, or a service that reserves all of its memory at start-up and must never call
// cudaMalloc (with its implicit synchronization and its chance of failing) on the request
// path.  They pass only W and the output buffers; the absmax values and group sums the
// quantizer needs between its passes live in g_noalloc_quant_scratch below.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds
// it (about 5.2 MB) until the process exits.  Host code cannot hand the symbol itself to a
// kernel (on the host it is only a stand-in), so the first call on each device looks up
// its device address with cudaGetSymbolAddress while that device is current and caches it
// for that device's context; make that first call before any stream capture.  The stream
// passed must belong to the current device (checked; QLORA_ERR_INVALID_ARG otherwise).
// Every call shares the array and it keeps the last call's contents; the quantizer writes
// every scratch entry it later reads, so nothing needs clearing between calls.  Calls that
// overlap on the GPU (for instance on two streams) race on the array.
#include "common.cuh"
#include "launch.h"

namespace qlora {
namespace {

constexpr int64_t kNoallocMaxNumel = NF4_NOALLOC_MAX_NUMEL;
// absmax fp32 for whole groups of 256 blocks, one fp64 sum per 8 blocks, then the mean's
// tail: the layout of nf4_quantize's workspace, for the largest tensor
constexpr uint64_t kNoallocScratchBytes =
    ((kNoallocMaxNumel + 64 * 256 - 1) / (64 * 256)) * (256 * 4 + 32 * 8) + kQuantizeTailBytes;

__device__ __align__(256) unsigned char g_noalloc_quant_scratch[kNoallocScratchBytes];

// Device address of the scratch array on the current device: looked up with that device
// current, once per device and context (a context created again after cudaDeviceReset
// looks it up again).
int scratch_for_current_device(void** out) {
  static DeviceCache<void*> scratch;
  const int st = scratch.get(device_context_key, out, [](void** v) -> int {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_quant_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return QLORA_ERR_CUDA;
    }
    *v = p;
    return QLORA_OK;
  });
  return st == -1 ? QLORA_ERR_NO_DEVICE : st;
}

// The stream must belong to the current device: the scratch address is that device's.
// The legacy and per-thread default streams (handles 0, 1, 2) always do.
int check_stream_device(cudaStream_t stream, int dev) {
  const uintptr_t h = reinterpret_cast<uintptr_t>(stream);
  if (h <= 2) return QLORA_OK;
  int sdev = -1;
  if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) {
    cudaGetLastError();
    return QLORA_ERR_INVALID_ARG;
  }
  return sdev == dev ? QLORA_OK : QLORA_ERR_INVALID_ARG;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace qlora

using namespace qlora;

extern "C" int nf4_quantize_noalloc(const float* W, const nf4_tensor* out, void* stream) {
  if (!out || !W) return QLORA_ERR_INVALID_ARG;
  if (out->rows < 1 || out->cols < 1) return QLORA_ERR_INVALID_ARG;
  if (out->blocksize != NF4_BLOCKSIZE ||
      (out->dq_block != NF4_DQ_BLOCK && out->dq_block != NF4_NO_DQ) ||
      (out->dq_type != NF4_DQ_INT8 && out->dq_type != NF4_DQ_FP8))
    return QLORA_ERR_UNSUPPORTED;
  const bool dq = out->dq_block != NF4_NO_DQ;
  if (!out->codes || !out->scale_steps || (dq && (!out->scale_codes || !out->scale_mean)))
    return QLORA_ERR_INVALID_ARG;
  if (!aligned16(W) || !aligned16(out->codes) || !aligned16(out->scale_steps) ||
      (dq && (!aligned16(out->scale_codes) || !aligned16(out->scale_mean))))
    return QLORA_ERR_MISALIGNED;
  if (out->rows > kNoallocMaxNumel / out->cols) return QLORA_ERR_TOO_LARGE;
  const int64_t numel = out->rows * out->cols;
  if (quantize_workspace_bytes(numel) > kNoallocScratchBytes) return QLORA_ERR_TOO_LARGE;
  int major = 0, minor = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      major != 10 || minor != 3)
    return QLORA_ERR_NO_DEVICE;
  int st = check_stream_device(static_cast<cudaStream_t>(stream), dev);
  if (st) return st;
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch))) return st;
  return launch_quantize(W, numel, *out, scratch, static_cast<cudaStream_t>(stream));
}
