// nf4_codec.cu -- blockwise NF4 quantization with double-quantized scales, and
// dequantization to bf16 (infivelines.com "QLoRA": 16 normal-quantile levels, one absmax
// scale per 64 weights, scales quantized again in blocks of 256; digipro.cn "QLoRA:
// Fine-Tuning a 7B Model on a 16GB GPU": quantized on the fly during load).
//
// Three launches quantize a tensor, all HBM-bound, no host synchronization:
//   nf4_quant_blocks   reads W once: per-64 absmax (half-warp shuffle max), the nearest
//                      level of w/absmax, 4-bit packing; writes the codes, the absmax values
//                      and, per group of 256 blocks, the fp64 pairwise sum of its absmax.
//   nf4_absmax_mean    one CTA: the pairwise sum over the group sums -> mean (fp32).
//   nf4_double_quant   one CTA per group: step = max|a - mean| / 127, int8 codes.
// Dequantization is one launch (nf4_dequant_kernel) built on the byte-permute table
// dequantizer shared with the GEMM producers.
#include "common.cuh"
#include "nf4_device.cuh"
#include "launch.h"
#include "profile.h"

namespace qlora {

constexpr int kBlock = NF4_BLOCKSIZE;               // 64 weights per block
constexpr int kGroup = NF4_DQ_BLOCK;                // 256 blocks per group
constexpr int64_t kGroupElems = (int64_t)kBlock * kGroup;  // 16384 weights
constexpr int kQuantThreads = 256;

// -------------------------------------------------------------------- pass 1
// One CTA per group of 256 blocks (16384 weights).  A half-warp covers one block with one
// float4 per lane; each warp walks 32 of the group's blocks, 4 pairs per iteration so that
// four 512-byte loads are in flight per warp.
__global__ void __launch_bounds__(kQuantThreads) nf4_quant_blocks(
    const float* __restrict__ W, int64_t numel, uint8_t* __restrict__ codes,
    float* __restrict__ absmax, double* __restrict__ group_sum) {
  __shared__ float s_abs[kGroup];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int half = lane >> 4, hl = lane & 15;
  const int64_t g = blockIdx.x;
  const int64_t nblocks = (numel + kBlock - 1) / kBlock;

#pragma unroll 1
  for (int it = 0; it < 4; ++it) {
    float4 v[4];
    int64_t e0[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int local_block = warp * 32 + it * 8 + u * 2 + half;
      const int64_t b = g * kGroup + local_block;
      e0[u] = b * kBlock + hl * 4;
      if (e0[u] + 3 < numel) {
        v[u] = __ldg(reinterpret_cast<const float4*>(W + e0[u]));
      } else {
        v[u].x = e0[u] + 0 < numel ? W[e0[u] + 0] : 0.0f;
        v[u].y = e0[u] + 1 < numel ? W[e0[u] + 1] : 0.0f;
        v[u].z = e0[u] + 2 < numel ? W[e0[u] + 2] : 0.0f;
        v[u].w = e0[u] + 3 < numel ? W[e0[u] + 3] : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float m = fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)), fmaxf(fabsf(v[u].z), fabsf(v[u].w)));
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      const int local_block = warp * 32 + it * 8 + u * 2 + half;
      const int64_t b = g * kGroup + local_block;
      if (hl == 0) {
        s_abs[local_block] = m;  // blocks past the end hold 0 (all their inputs read as 0)
        if (b < nblocks) absmax[b] = m;
      }
      uint32_t c0, c1, c2, c3;
      if (m == 0.0f) {
        c0 = c1 = c2 = c3 = nf4_code(0.0f);
      } else {
        c0 = nf4_code(__fdiv_rn(v[u].x, m));
        c1 = nf4_code(__fdiv_rn(v[u].y, m));
        c2 = nf4_code(__fdiv_rn(v[u].z, m));
        c3 = nf4_code(__fdiv_rn(v[u].w, m));
      }
      // even element in the high nibble
      const uint32_t byte0 = (c0 << 4) | c1, byte1 = (c2 << 4) | c3;
      const int64_t e = e0[u];
      if (e + 3 < numel) {
        *reinterpret_cast<uint16_t*>(codes + e / 2) = static_cast<uint16_t>(byte0 | (byte1 << 8));
      } else {
        if (e < numel) codes[e / 2] = static_cast<uint8_t>(e + 1 < numel ? byte0 : (c0 << 4));
        if (e + 2 < numel) codes[e / 2 + 1] = static_cast<uint8_t>(e + 3 < numel ? byte1 : (c2 << 4));
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // Perfect binary tree over the 256 absmax values in block order: each lane sums 8
    // neighbours pairwise, then the xor butterfly combines lanes (x+y == y+x in IEEE).
    const float* a = s_abs + lane * 8;
    double s = (((double)a[0] + (double)a[1]) + ((double)a[2] + (double)a[3])) +
               (((double)a[4] + (double)a[5]) + ((double)a[6] + (double)a[7]));
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) group_sum[g] = s;
  }
}

// -------------------------------------------------------------------- pass 2
// One CTA of 1024 threads: the pairwise tree over the group sums (zero-padded to a power of
// two) -> mean = (float)(total / nblocks).  Each thread first folds a run of `run` leaves
// (a power of two) with a binary-counter stack, which is exactly the pairwise tree of the
// run; the runs then combine through warp butterflies and a final warp.
__global__ void __launch_bounds__(1024) nf4_absmax_mean(const double* __restrict__ group_sum,
                                                        int64_t ngroups, int64_t nblocks,
                                                        int64_t run, float* __restrict__ mean) {
  __shared__ double s_warp[32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  double stack[32];
  int depth = 0;
  const int64_t lo = (int64_t)t * run;
  for (int64_t i = 0; i < run; ++i) {
    double v = (lo + i < ngroups) ? group_sum[lo + i] : 0.0;
    // merge equal-sized subtrees, like incrementing a binary counter
    int64_t k = i + 1;
    while ((k & 1) == 0) {
      v = stack[--depth] + v;
      k >>= 1;
    }
    stack[depth++] = v;
  }
  double s = stack[0];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) s_warp[warp] = s;
  __syncthreads();
  if (warp == 0) {
    double w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (lane == 0) mean[0] = (float)(w / (double)nblocks);
  }
}

// -------------------------------------------------------------------- pass 3
__global__ void __launch_bounds__(kGroup) nf4_double_quant(const float* __restrict__ absmax,
                                                           int64_t nblocks,
                                                           const float* __restrict__ mean,
                                                           int8_t* __restrict__ scale_codes,
                                                           float* __restrict__ steps) {
  __shared__ float s_max[kGroup / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t b = (int64_t)blockIdx.x * kGroup + t;
  const float mu = mean[0];
  const float d = (b < nblocks) ? __fsub_rn(absmax[b], mu) : 0.0f;
  float m = fabsf(d);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_max[warp] = m;
  __syncthreads();
  float s2 = s_max[0];
#pragma unroll
  for (int i = 1; i < kGroup / 32; ++i) s2 = fmaxf(s2, s_max[i]);
  const float step = __fdiv_rn(s2, 127.0f);
  if (t == 0) steps[blockIdx.x] = step;
  if (b < nblocks) {
    int q = 0;
    if (step > 0.0f) {
      q = __float2int_rn(__fdiv_rn(d, step));  // round half to even
      q = q > 127 ? 127 : (q < -127 ? -127 : q);
    }
    scale_codes[b] = static_cast<int8_t>(q);
  }
}

// -------------------------------------------------------------------- dequantize
// Grid-stride over 16-weight pieces: 8 code bytes in, 32 bytes of bf16 out per thread; the
// four threads of a 64-block each build the block's byte table.
__global__ void __launch_bounds__(256) nf4_dequant_kernel(const uint8_t* __restrict__ codes,
                                                          const int8_t* __restrict__ scale_codes,
                                                          const float* __restrict__ steps,
                                                          const float* __restrict__ mean,
                                                          int64_t numel, uint16_t* __restrict__ out) {
  const float mu = __ldg(mean);
  const int64_t npieces = (numel + 15) / 16;
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < npieces;
       p += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e0 = p * 16;
    const int64_t b = e0 / kBlock;
    const float scale = __fmaf_rn((float)__ldg(scale_codes + b), __ldg(steps + b / kGroup), mu);
    const Nf4ByteTable tab = nf4_make_table(scale);
    uint32_t q[2];
    if (e0 + 16 <= numel) {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(codes + e0 / 2));
      q[0] = raw.x;
      q[1] = raw.y;
    } else {
      uint8_t bytes[8];
      const int64_t nbytes = (numel + 1) / 2;
#pragma unroll
      for (int i = 0; i < 8; ++i) bytes[i] = (e0 / 2 + i < nbytes) ? codes[e0 / 2 + i] : 0;
      q[0] = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | ((uint32_t)bytes[3] << 24);
      q[1] = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | ((uint32_t)bytes[7] << 24);
    }
    uint32_t o0[4], o1[4];
    nf4_dequant8(tab, q[0], o0);
    nf4_dequant8(tab, q[1], o1);
    if (e0 + 16 <= numel) {
      uint4* dst = reinterpret_cast<uint4*>(out + e0);
      dst[0] = make_uint4(o0[0], o0[1], o0[2], o0[3]);
      dst[1] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    } else {
      for (int i = 0; i < 16 && e0 + i < numel; ++i) {
        const uint32_t w = i < 8 ? o0[i / 2] : o1[(i - 8) / 2];
        out[e0 + i] = static_cast<uint16_t>((w >> (16 * (i & 1))) & 0xFFFFu);
      }
    }
  }
}

// -------------------------------------------------------------------- launchers
uint64_t quantize_workspace_bytes(int64_t numel) {
  const int64_t nb = (numel + kBlock - 1) / kBlock;
  const int64_t ng = (nb + kGroup - 1) / kGroup;
  // absmax fp32 [ngroups * 256] (padded to whole groups), then group sums fp64 [ngroups]
  return (uint64_t)ng * kGroup * 4 + (uint64_t)ng * 8 + 256;
}

int launch_quantize(const float* W, int64_t numel, const nf4_tensor& q, void* ws,
                    cudaStream_t stream) {
  const int64_t nb = (numel + kBlock - 1) / kBlock;
  const int64_t ng = (nb + kGroup - 1) / kGroup;
  float* absmax = reinterpret_cast<float*>(ws);
  double* gsum = reinterpret_cast<double*>(reinterpret_cast<char*>(ws) + ng * kGroup * 4);
  {
    ProfileScope ps("nf4_quant_blocks", stream);
    nf4_quant_blocks<<<(unsigned)ng, kQuantThreads, 0, stream>>>(W, numel, q.codes, absmax, gsum);
  }
  int64_t p2 = 1;
  while (p2 < ng) p2 *= 2;
  const int64_t run = p2 > 1024 ? p2 / 1024 : 1;
  {
    ProfileScope ps("nf4_absmax_mean", stream);
    nf4_absmax_mean<<<1, 1024, 0, stream>>>(gsum, ng, nb, run, q.scale_mean);
  }
  {
    ProfileScope ps("nf4_double_quant", stream);
    nf4_double_quant<<<(unsigned)ng, kGroup, 0, stream>>>(absmax, nb, q.scale_mean, q.scale_codes,
                                                          q.scale_steps);
  }
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

int launch_dequantize(const nf4_tensor& q, int64_t numel, uint16_t* out, cudaStream_t stream) {
  const int64_t npieces = (numel + 15) / 16;
  const int threads = 256;
  int64_t blocks = (npieces + threads - 1) / threads;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (blocks > cap) blocks = cap;
  ProfileScope ps("nf4_dequant", stream);
  nf4_dequant_kernel<<<(unsigned)blocks, threads, 0, stream>>>(q.codes, q.scale_codes,
                                                               q.scale_steps, q.scale_mean,
                                                               numel, out);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
