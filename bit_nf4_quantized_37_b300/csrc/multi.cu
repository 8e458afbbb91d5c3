// multi.cu -- the decode path with per-token adapters: one NF4 base, several LoRA adapters
// kept separate and chosen per token (addaly.com "QLoRA on one card", "Merging a QLoRA
// adapter, and the subtlety": keeping the adapter separate and loading it over the base lets
// you swap adapters, which merging forfeits; junaidshaukat.com "QLoRA -- the democratization
// event", deployment-subtlety paragraph: serve the 4-bit base plus a separate adapter).
//   U_t = X_t A_{a(t)}^T              multi_u: split over K in 256-wide chunks, the chunks of
//                                     a token summed in chunk order by its last CTA
//   Z_t = s_{a(t)} U_t B_{a(t)}^T     multi_z: fp32, one thread per (token, output column)
//   Y_t = bf16( X_t W'^T + Z_t )      the decode GEMV (skinny.cu), adding Z before rounding
// Tokens whose index is outside [0, n_adapters) get no adapter term.
#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "profile.h"

namespace qlora {
namespace multi {

constexpr int KC = 256;  // contraction chunk of one multi_u CTA

__device__ __forceinline__ float bf16f(uint32_t h) { return __uint_as_float(h << 16); }

__global__ void __launch_bounds__(256) multi_u(const uint16_t* __restrict__ X, int64_t K,
                                               const uint16_t* __restrict__ A_all, int r,
                                               int n_adapters, const int32_t* __restrict__ idx,
                                               float* __restrict__ part, int* __restrict__ tickets,
                                               float* __restrict__ U) {
  __shared__ float sx[KC];
  __shared__ int s_last;
  const int t = blockIdx.y, c = blockIdx.x, nchunks = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int a = __ldg(idx + t);
  const bool live = a >= 0 && a < n_adapters;
  const int64_t k0 = static_cast<int64_t>(c) * KC;
  sx[tid] = k0 + tid < K ? bf16f(__ldg(X + t * K + k0 + tid)) : 0.0f;
  __syncthreads();
  float* mine = part + (static_cast<int64_t>(t) * nchunks + c) * r;
  if (live) {
    const uint16_t* Aa = A_all + static_cast<int64_t>(a) * r * K;
    const int64_t k = k0 + 8 * lane;
    for (int j = warp; j < r; j += 8) {
      float s = 0.0f;
      if (k < K) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(Aa + j * K + k));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          s = __fmaf_rn(bf16f(w[e] & 0xFFFFu), sx[8 * lane + 2 * e], s);
          s = __fmaf_rn(bf16f(w[e] >> 16), sx[8 * lane + 2 * e + 1], s);
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) mine[j] = s;
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&tickets[t], 1) == nchunks - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int j = tid; j < r; j += 256) {
    float u = 0.0f;
    if (live)
      for (int cc = 0; cc < nchunks; ++cc)
        u += __ldcg(part + (static_cast<int64_t>(t) * nchunks + cc) * r + j);
    U[t * r + j] = u;
  }
  if (tid == 0) tickets[t] = 0;  // ready for the next launch
}

__global__ void __launch_bounds__(128) multi_z(const float* __restrict__ U, int64_t N,
                                               const uint16_t* __restrict__ B_all, int r,
                                               int n_adapters, const int32_t* __restrict__ idx,
                                               const float* __restrict__ scales,
                                               float* __restrict__ Z) {
  extern __shared__ float su[];  // U row of this CTA's token [r]
  const int t = blockIdx.y;
  for (int j = threadIdx.x; j < r; j += 128) su[j] = U[t * r + j];
  __syncthreads();
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 128 + threadIdx.x;
  if (n >= N) return;
  const int a = __ldg(idx + t);
  float z = 0.0f;
  if (a >= 0 && a < n_adapters) {
    const uint16_t* Brow = B_all + (static_cast<int64_t>(a) * N + n) * r;
    float acc = 0.0f;  // ascending j
    if ((r & 7) == 0) {
      for (int j8 = 0; j8 < r; j8 += 8) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(Brow + j8));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc = __fmaf_rn(su[j8 + 2 * e], bf16f(w[e] & 0xFFFFu), acc);
          acc = __fmaf_rn(su[j8 + 2 * e + 1], bf16f(w[e] >> 16), acc);
        }
      }
    } else {
      for (int j = 0; j < r; ++j) acc = __fmaf_rn(su[j], bf16f(__ldg(Brow + j)), acc);
    }
    z = __fmul_rn(__ldg(scales + a), acc);
  }
  Z[t * N + n] = z;
}

}  // namespace multi

int launch_multi_fwd(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  float* U = reinterpret_cast<float*>(ws + L.U32);
  float* Z = reinterpret_cast<float*>(ws + L.Z);
  const unsigned nchunks = (unsigned)((a.K + multi::KC - 1) / multi::KC);
  {
    ProfileScope ps("multi_u", stream);
    multi::multi_u<<<dim3(nchunks, (unsigned)a.M), 256, 0, stream>>>(
        a.X, a.K, a.A, a.r, a.n_adapters, a.adapter_idx, reinterpret_cast<float*>(ws + L.part),
        reinterpret_cast<int*>(ws + L.tickets), U);
    if (cudaGetLastError() != cudaSuccess) return QLORA_ERR_CUDA;
  }
  {
    ProfileScope ps("multi_z", stream);
    multi::multi_z<<<dim3((unsigned)((a.N + 127) / 128), (unsigned)a.M), 128, (size_t)a.r * 4,
                     stream>>>(U, a.N, a.B, a.r, a.n_adapters, a.adapter_idx, a.scales, Z);
    if (cudaGetLastError() != cudaSuccess) return QLORA_ERR_CUDA;
  }
  return launch_decode_gemv(a, L, Z, stream);
}

}  // namespace qlora
