// launch.h -- host-side declarations shared by the translation units of the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qlora_nf4.h"
#include "device_cache.h"

namespace qlora {

// Device ordinal and id of its current context (the key of the per-device set-up caches).
DeviceKey device_context_key();

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Sets `kernel`'s dynamic shared-memory limit to `bytes` on the current device, once per
// device and context; `cache` is the call site's own (one per kernel).
template <typename Kernel>
int ensure_dynamic_smem(DeviceCache<int>& cache, Kernel kernel, int bytes) {
  int have = 0;
  const int st = cache.get(device_context_key, &have, [&](int* v) -> int {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
        cudaSuccess) {
      cudaGetLastError();
      return QLORA_ERR_CUDA;
    }
    *v = bytes;
    return QLORA_OK;
  });
  if (st == -1) return QLORA_ERR_NO_DEVICE;
  if (st) return st;
  return have >= bytes ? QLORA_OK : QLORA_ERR_CUDA;
}

// Reads and clears the fused GEMMs' device error word (umma_gemm.cu).
int read_and_clear_gemm_error(int* out);
// Reads and clears the side kernels' device error word (lora_side.cu).
int read_and_clear_side_error(int* out);
// Reads and clears the decode kernel's device error word (skinny.cu).
int read_and_clear_decode_error(int* out);
// Reads and clears the wait self-test's device error word, and launches that self-test: one
// bounded wait on an mbarrier nothing arrives on (selftest.cu).
int read_and_clear_selftest_error(int* out);
int launch_wait_selftest(cudaStream_t stream);

// Quantize / dequantize (nf4_codec.cu).
// The quantize workspace: absmax fp32 for whole groups of 256 blocks, one fp64 sum per 8
// blocks, then a tail of kQuantizeMeanParts fp64 subtree sums of the mean and the arrival
// ticket of the pass that combines them.
constexpr int kQuantizeMeanParts = 128;  // a power of two
constexpr uint64_t kQuantizeTailBytes = kQuantizeMeanParts * 8 + 16;
uint64_t quantize_workspace_bytes(int64_t numel);
int launch_quantize(const float* W, int64_t numel, const nf4_tensor& q, void* ws,
                    cudaStream_t stream);
// out: bf16, or fp16 when half.  dependent: launched as a programmatic dependent of the
// kernel before it in the stream (it reads nothing that kernel writes, and its CTAs wait for
// that kernel before they exit, so its completion implies the other's).
int launch_dequantize(const nf4_tensor& q, int64_t numel, uint16_t* out, bool half,
                      cudaStream_t stream, bool dependent = false);

// Adapter merge and NF4-vs-INT4 error statistics (merge.cu).
int launch_merge(const nf4_tensor& q, const uint16_t* A, const uint16_t* B, int r, float scale,
                 uint16_t* out16, float* out32, cudaStream_t stream);
int error_stats_parts();
int launch_error_stats(const float* W, int64_t numel, double* out, void* ws, cudaStream_t stream);

// 2-D tiled tensor map over a row-major matrix (tensormap.cu).  `inner` is the contiguous
// extent in elements, `outer` the row count, `row_bytes` the row pitch; the box is
// box_inner x box_outer elements.  Returns false when the driver rejects the map.
enum class MapSwizzle { None, B32, B64, B128 };
bool make_tensor_map_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype,
                        int elem_bytes, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_outer, MapSwizzle sw);

}  // namespace qlora
