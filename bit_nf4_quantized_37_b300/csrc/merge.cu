// merge.cu -- folding a LoRA adapter into the NF4 base, and the NF4-vs-INT4 error statistics.
//
// Merge (junaidshaukat.com "QLoRA -- the democratization event", the deployment-subtlety
// paragraph: merging means dequantize, merge, maybe requantize; infivelines.com "QLoRA": a
// bf16 adapter merged into a 4-bit base and saved loses precision twice; addaly.com "QLoRA on
// one card", "Merging a QLoRA adapter, and the subtlety"):
//     W_merged = bf16( W' + s * B A )          W' = the bf16 dequantization of the NF4 base
// One pass over the packed codes: each CTA stages its [r x 128] slice of A (16-byte slots
// swizzled against bank conflicts) and [32 x r] slice of B in shared memory as fp32, a thread
// forms the rank-r product of eight consecutive columns of one row with fp32 multiply-adds
// (each bf16 x bf16 product is exact in fp32), dequantizes the same eight codes exactly as
// nf4_dequantize does, adds RN(s * delta) in fp32 and rounds once to bf16.  The fp32 copy
// (the same values) feeds nf4_quantize for the requantized artifact.
//
// Error statistics (aicurriculum.codextroop.com "QLoRA -- Module 12.4", "Design Details That
// Matter": NF4 places levels at normal quantiles and is often better than naive INT4;
// addaly.com "QLoRA on one card", "What each setting is doing": NF4 keeps more information
// than plain 4-bit integers at the same size): for fp32 weights, per block of 64 with its
// absmax a, the squared error of the NF4 reconstruction level[c] * a (c = nearest level of
// w / a) and of the symmetric absmax INT4 reconstruction q * (a / 7), q = clamp(rint(7 w / a),
// -7, 7), summed over the tensor together with sum w^2 (fp32 within a thread's 16 weights,
// fp64 across threads and CTAs).
#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "nf4_device.cuh"
#include "profile.h"

namespace qlora {
namespace merge {

constexpr int ROWS = 64;      // output rows per CTA
constexpr int COLS = 128;     // output columns per CTA
constexpr int THREADS = 256;  // 16 threads per row (8 columns each); a thread takes 4 rows
constexpr int RPT = ROWS / (THREADS / 16);  // rows per thread, sharing each A load

inline int smem_bytes(int r) { return (r * COLS + ROWS * (r + 1)) * 4; }

// 16-byte slot of columns 8 c8 + 4 h .. + 3 within a staged row of A: the low slot bit is
// flipped for c8 & 4, so the eight lanes of a 128-bit shared load hit eight distinct bank
// quads (unswizzled, lanes c8 and c8 + 4 collide)
__device__ __forceinline__ int a_slot(int c8, int h) { return (2 * c8 + h) ^ ((c8 >> 2) & 1); }

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__global__ void __launch_bounds__(THREADS) nf4_merge_kernel(
    const uint8_t* __restrict__ codes, const int8_t* __restrict__ qs,
    const float* __restrict__ steps, const float* __restrict__ mean,
    int dq, int fp8, const uint16_t* __restrict__ A, const uint16_t* __restrict__ B, int64_t N,
    int64_t K, int r, float scale, uint16_t* __restrict__ out16, float* __restrict__ out32) {
  extern __shared__ float msm[];
  float* sA = msm;               // [r][COLS]
  float* sB = msm + r * COLS;    // [ROWS][r + 1]
  const int tid = threadIdx.x;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * COLS;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * ROWS;
  for (int i = tid; i < r * (COLS / 8); i += THREADS) {
    const int j = i / (COLS / 8), c8 = i % (COLS / 8);
    const int64_t k = k0 + 8 * c8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (k < K) v = __ldg(reinterpret_cast<const uint4*>(A + j * K + k));
    float* row = sA + j * COLS;
    *reinterpret_cast<float4*>(row + 4 * a_slot(c8, 0)) =
        make_float4(bf16_bits_to_f32(v.x & 0xFFFFu), bf16_bits_to_f32(v.x >> 16),
                    bf16_bits_to_f32(v.y & 0xFFFFu), bf16_bits_to_f32(v.y >> 16));
    *reinterpret_cast<float4*>(row + 4 * a_slot(c8, 1)) =
        make_float4(bf16_bits_to_f32(v.z & 0xFFFFu), bf16_bits_to_f32(v.z >> 16),
                    bf16_bits_to_f32(v.w & 0xFFFFu), bf16_bits_to_f32(v.w >> 16));
  }
  for (int i = tid; i < ROWS * r; i += THREADS) {
    const int rr = i / r, j = i % r;
    const int64_t n = n0 + rr;
    sB[rr * (r + 1) + j] = n < N ? bf16_bits_to_f32(__ldg(B + n * r + j)) : 0.0f;
  }
  __syncthreads();
  const float mu = dq ? __ldg(mean) : 0.0f;
  const int c8 = tid & 15;
  const int64_t kk = k0 + 8 * c8;
  if (kk >= K) return;
  // rows (tid >> 4) + 16 p, p < RPT: each A value read from shared memory feeds RPT rows
  float d[RPT][8];
#pragma unroll
  for (int p = 0; p < RPT; ++p)
#pragma unroll
    for (int i = 0; i < 8; ++i) d[p][i] = 0.f;
  const int rr0 = tid >> 4;
  const float* acol0 = sA + 4 * a_slot(c8, 0);
  const float* acol1 = sA + 4 * a_slot(c8, 1);
#pragma unroll 2
  for (int j = 0; j < r; ++j) {  // ascending j: a fixed fp32 summation order
    const float4 a0 = *reinterpret_cast<const float4*>(acol0 + j * COLS);
    const float4 a1 = *reinterpret_cast<const float4*>(acol1 + j * COLS);
#pragma unroll
    for (int p = 0; p < RPT; ++p) {
      const float b = sB[(rr0 + 16 * p) * (r + 1) + j];
      d[p][0] = __fmaf_rn(b, a0.x, d[p][0]);
      d[p][1] = __fmaf_rn(b, a0.y, d[p][1]);
      d[p][2] = __fmaf_rn(b, a0.z, d[p][2]);
      d[p][3] = __fmaf_rn(b, a0.w, d[p][3]);
      d[p][4] = __fmaf_rn(b, a1.x, d[p][4]);
      d[p][5] = __fmaf_rn(b, a1.y, d[p][5]);
      d[p][6] = __fmaf_rn(b, a1.z, d[p][6]);
      d[p][7] = __fmaf_rn(b, a1.w, d[p][7]);
    }
  }
#pragma unroll
  for (int p = 0; p < RPT; ++p) {
    const int64_t n = n0 + rr0 + 16 * p;
    if (n >= N) break;
    // the eight base weights (n, kk .. kk + 7): one code word, one block scale
    const int64_t e = n * K + kk;
    const uint32_t word = __ldg(reinterpret_cast<const uint32_t*>(codes + e / 2));
    const int64_t blk = e / 64;
    const float a_hat =
        dq ? __fmaf_rn(nf4_second_level(static_cast<uint8_t>(__ldg(qs + blk)), fp8),
                       __ldg(steps + (blk >> 8)), mu)
           : __ldg(steps + blk);
    uint32_t wd[4];
    nf4_dequant8(nf4_make_table(a_hat), word, wd);
    uint32_t o16[4];
    float o32[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float v0 = __fadd_rn(bf16_bits_to_f32(wd[i] & 0xFFFFu), __fmul_rn(scale, d[p][2 * i]));
      const float v1 = __fadd_rn(bf16_bits_to_f32(wd[i] >> 16), __fmul_rn(scale, d[p][2 * i + 1]));
      const __nv_bfloat162 h = __floats2bfloat162_rn(v0, v1);
      o16[i] = *reinterpret_cast<const uint32_t*>(&h);
      o32[2 * i] = bf16_bits_to_f32(o16[i] & 0xFFFFu);
      o32[2 * i + 1] = bf16_bits_to_f32(o16[i] >> 16);
    }
    if (out16) *reinterpret_cast<uint4*>(out16 + e) = make_uint4(o16[0], o16[1], o16[2], o16[3]);
    if (out32) {
      reinterpret_cast<float4*>(out32 + e)[0] = make_float4(o32[0], o32[1], o32[2], o32[3]);
      reinterpret_cast<float4*>(out32 + e)[1] = make_float4(o32[4], o32[5], o32[6], o32[7]);
    }
  }
}

// ---------------------------------------------------------------- error statistics
constexpr int ES_THREADS = 256;

__global__ void __launch_bounds__(ES_THREADS) nf4_int4_error_kernel(
    const float* __restrict__ W, int64_t numel, double* __restrict__ part) {
  __shared__ double s_red[ES_THREADS / 32][3];
  constexpr float L[16] = QLORA_NF4_LEVELS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ql = lane & 3;  // quarter of a 64-block: 16 weights
  const int64_t nblocks = (numel + 63) / 64;
  const int64_t gwarps = static_cast<int64_t>(gridDim.x) * (ES_THREADS / 32);
  double acc[3] = {0.0, 0.0, 0.0};  // sum w^2, sum e_nf4^2, sum e_int4^2
  // a warp takes eight blocks at a time, four lanes per block
  for (int64_t b0 = (static_cast<int64_t>(blockIdx.x) * (ES_THREADS / 32) + warp) * 8;
       b0 < nblocks; b0 += gwarps * 8) {
    const int64_t b = b0 + (lane >> 2);
    const int64_t e0 = b * 64 + ql * 16;
    float w[16];
    if (b < nblocks && e0 + 16 <= numel) {
      const float4* src = reinterpret_cast<const float4*>(W + e0);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const float4 f = __ldg(src + v);
        w[4 * v] = f.x; w[4 * v + 1] = f.y; w[4 * v + 2] = f.z; w[4 * v + 3] = f.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = (b < nblocks && e0 + i < numel) ? W[e0 + i] : 0.0f;
    }
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(w[i]));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    const float a7 = __fdiv_rn(a, 7.0f);
    float s_w = 0.f, s_n = 0.f, s_i = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float x = a > 0.0f ? __fdiv_rn(w[i], a) : 0.0f;
      const float en = __fsub_rn(w[i], __fmul_rn(L[nf4_code(x)], a));
      const float q = fminf(fmaxf(rintf(__fmul_rn(7.0f, x)), -7.0f), 7.0f);
      const float ei = __fsub_rn(w[i], __fmul_rn(q, a7));
      s_w = __fmaf_rn(w[i], w[i], s_w);
      s_n = __fmaf_rn(en, en, s_n);
      s_i = __fmaf_rn(ei, ei, s_i);
    }
    acc[0] += s_w;
    acc[1] += s_n;
    acc[2] += s_i;
  }
#pragma unroll
  for (int k = 0; k < 3; ++k)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], o);
  if (lane == 0)
    for (int k = 0; k < 3; ++k) s_red[warp][k] = acc[k];
  __syncthreads();
  if (threadIdx.x < 3) {
    double v = 0.0;
    for (int i = 0; i < ES_THREADS / 32; ++i) v += s_red[i][threadIdx.x];
    part[blockIdx.x * 3 + threadIdx.x] = v;
  }
}

__global__ void nf4_int4_error_sum(const double* __restrict__ part, int nparts,
                                   double* __restrict__ out) {
  if (threadIdx.x < 3) {
    double v = 0.0;
    for (int i = 0; i < nparts; ++i) v += part[i * 3 + threadIdx.x];
    out[threadIdx.x] = v;
  }
}

}  // namespace merge

int launch_merge(const nf4_tensor& q, const uint16_t* A, const uint16_t* B, int r, float scale,
                 uint16_t* out16, float* out32, cudaStream_t stream) {
  const int smem = merge::smem_bytes(r);
  static DeviceCache<int> attr;  // set once per device to the largest rank's need
  if (smem > 48 * 1024) {
    const int st = ensure_dynamic_smem(attr, merge::nf4_merge_kernel, merge::smem_bytes(kMaxRank));
    if (st) return st;
  }
  const dim3 grid((unsigned)((q.cols + merge::COLS - 1) / merge::COLS),
                  (unsigned)((q.rows + merge::ROWS - 1) / merge::ROWS));
  ProfileScope ps("nf4_merge", stream);
  merge::nf4_merge_kernel<<<grid, merge::THREADS, smem, stream>>>(
      q.codes, q.scale_codes, q.scale_steps, q.scale_mean, q.dq_block != 0 ? 1 : 0,
      q.dq_type == NF4_DQ_FP8 ? 1 : 0, A, B, q.rows, q.cols, r, scale, out16, out32);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

int error_stats_parts() { return 4 * num_sms(); }

int launch_error_stats(const float* W, int64_t numel, double* out, void* ws, cudaStream_t stream) {
  const int64_t nblocks = (numel + 63) / 64;
  int64_t ctas = (nblocks + 63) / 64;  // eight warps of eight blocks each
  if (ctas > error_stats_parts()) ctas = error_stats_parts();
  if (ctas < 1) ctas = 1;
  double* part = static_cast<double*>(ws);
  ProfileScope ps("nf4_int4_error", stream);
  merge::nf4_int4_error_kernel<<<(unsigned)ctas, merge::ES_THREADS, 0, stream>>>(W, numel, part);
  if (cudaGetLastError() != cudaSuccess) return QLORA_ERR_CUDA;
  merge::nf4_int4_error_sum<<<1, 32, 0, stream>>>(part, static_cast<int>(ctas), out);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
