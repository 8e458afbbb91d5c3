// nf4_codec.cu -- blockwise NF4 quantization with double-quantized scales, and
// dequantization to bf16 (infivelines.com "QLoRA": 16 normal-quantile levels, one absmax
// scale per 64 weights, scales quantized again in blocks of 256; digipro.cn "QLoRA:
// Fine-Tuning a 7B Model on a 16GB GPU": quantized on the fly during load).
//
// Three launches quantize a tensor, no host synchronization:
//   nf4_quant_blocks   reads W once: per-64 absmax, the nearest level of w/absmax (exactly as
//                      with an IEEE division, see below), 4-bit packing; writes the codes, the
//                      absmax values and, per run of 8 blocks, the fp64 pairwise sum of their
//                      absmax (a warp's perfect 8-leaf subtree, by shuffles).
//   nf4_absmax_mean    up to 128 CTAs: aligned subtrees of the pairwise sum over those
//                      8-block sums.
//   nf4_double_quant   a warp per group: mean (fp32) from the subtree sums, then
//                      step = max|a - mean| / 127, int8 codes.
// Dequantization is one launch (nf4_dequant_kernel) built on the byte-permute table
// dequantizer shared with the GEMM producers.
#include <algorithm>

#include "common.cuh"
#include "nf4_device.cuh"
#include "launch.h"
#include "profile.h"

namespace qlora {

constexpr int kBlock = NF4_BLOCKSIZE;               // 64 weights per block
constexpr int kGroup = NF4_DQ_BLOCK;                // 256 blocks per group
constexpr int64_t kGroupElems = (int64_t)kBlock * kGroup;  // 16384 weights
constexpr int kQuantThreads = 256;
constexpr int kUnit = 64;                               // blocks per pass-1 work unit
constexpr int64_t kUnitElems = (int64_t)kBlock * kUnit;  // 4096 weights

// -------------------------------------------------------------------- pass 1
// Persistent CTAs, each taking units of 64 blocks (4096 weights) in a grid-stride loop: units
// a quarter of a scale group keep the CTAs' shares even on tensors of a few thousand groups
// (1024 groups on 592 resident CTAs left every CTA one or two).
//
// Full units: four lanes per 64-block, 16 weights per lane (four float4 loads, the next
// unit's loads in flight across the unit boundary), so a block's absmax is 15 max
// operations and two shuffles; a warp's eight blocks are a perfect subtree of the mean's
// pairwise tree, summed by three more shuffles, so full units need no CTA barrier.  The exact quotient x = RN(w / a) is never needed away from a
// threshold: y = RN(w * RN(1/a)) is within 3 * 2^-24 * |x| of x, so whenever y is more than
// 2^-20 from every threshold, y and x fall between the same two thresholds and the level
// follows from y.  The level comes from a shared-memory table over cells of y (sign; cell 0
// for |y| < 2^-5, then binade and top 4 mantissa bits for |y| in [2^-5, 1.0625)): each cell
// holds at most one threshold T, the level is c_lo + (y > T), and |y - T| < 2^-20 sends the
// lane's 16 weights to the exact division (thresholds lie >= 2.3e-4 inside their cells, so
// a threshold between x and y is always the one in y's cell); so does an absmax without a
// finite reciprocal, which leaves every y of the fast path finite and inside the table.  The
// table is built once per CTA, one interleaved copy per lane (entry i of copy l at word pair
// 32 i + l), so the 8-byte lookups of a half-warp never collide on a bank.
// The last, partial unit takes the element-by-element path with the exact division.
constexpr int kCells = 82;                  // per sign: [0, 2^-5), then 5 binades x 16, [1, 1.0625)
constexpr int kCopies = 32;                 // one table copy per lane
constexpr uint32_t kCellBase = 0x3D000000u;  // bits of 2^-5
constexpr float kGuard = 0x1p-20f;
constexpr int kCellBytes = 2 * kCells * kCopies * 8;  // 41 KB of dynamic shared memory

__device__ __forceinline__ uint32_t code_exact(float w, float a) {
  return a == 0.0f ? nf4_code(0.0f) : nf4_code(__fdiv_rn(w, a));
}

// cell table entry: (threshold inside the cell or +inf, lowest level of the cell), entry i of
// copy c at tab[i * kCopies + c]
__device__ void build_cells(float2* tab) {
  constexpr float T[15] = QLORA_NF4_THRESHOLDS;
  for (int i = threadIdx.x; i < 2 * kCells; i += blockDim.x) {
    const int neg = i / kCells, idx = i % kCells;
    int c_lo = 7;                            // |y| < 2^-5: level 7 (every threshold is farther)
    float thr = __int_as_float(0x7f800000);  // +inf: no threshold in the cell
    if (idx > 0) {
      const float lo = __uint_as_float(kCellBase + (static_cast<uint32_t>(idx - 1) << 19));
      const float hi = __uint_as_float(kCellBase + (static_cast<uint32_t>(idx) << 19));
      c_lo = 0;
      for (int t = 0; t < 15; ++t) {
        if (!neg) {  // y in [lo, hi)
          if (T[t] < lo) ++c_lo;
          else if (T[t] < hi) thr = T[t];
        } else {     // y in (-hi, -lo]
          if (T[t] <= -hi) ++c_lo;
          else if (T[t] <= -lo) thr = T[t];
        }
      }
    }
    const float2 e = make_float2(thr, __int_as_float(c_lo));
#pragma unroll
    for (int c = 0; c < kCopies; ++c) tab[i * kCopies + c] = e;
  }
}

// Level of a finite y = RN(w * RN(1/a)), |y| <= 1 + 2^-23, from the cell table.  tab_b is
// the shared-window address of this lane's copy of entry 0, less the bias of the cell
// index, so the entry address is two multiply-adds of the sign bit and of the top bits of
// max(|y|, bottom of cell 1).  dmin collects |T - y|, which decides whether the exact
// division is needed.  The level is c_lo + (y > T), and y > T exactly when T - y is
// negative (T = +inf for a cell without threshold gives +inf).
constexpr uint32_t kCellBias = (kCellBase >> 19) - 1u;       // top bits of cell 0
constexpr uint32_t kEntryBytes = kCopies * 8;                // one entry, all copies
__device__ __forceinline__ uint32_t code_fast(float y, uint32_t tab_b, float& dmin) {
  const float ay = fmaxf(fabsf(y), __uint_as_float(kCellBase - (1u << 19)));  // tiny -> cell 0
  const uint32_t addr = tab_b + (__float_as_uint(y) >> 31) * (kCells * kEntryBytes) +
                        (__float_as_uint(ay) >> 19) * kEntryBytes;
  float t, lo;
  asm("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(t), "=f"(lo) : "r"(addr));
  const float nd = t - y;
  dmin = fminf(dmin, fabsf(nd));
  return __float_as_uint(lo) + (__float_as_uint(nd) >> 31);
}

__global__ void __launch_bounds__(kQuantThreads, 4) nf4_quant_blocks(
    const float* __restrict__ W, int64_t numel, uint8_t* __restrict__ codes,
    float* __restrict__ absmax, double* __restrict__ sum8, int* ticket) {
  __shared__ float s_abs[kUnit];  // the partial last unit's absmax values
  extern __shared__ float2 s_cells[];  // 2 * kCells * kCopies entries
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nblocks = (numel + kBlock - 1) / kBlock;
  const int64_t nunits = (nblocks + kUnit - 1) / kUnit;
  const int64_t nfull = numel / kUnitElems;  // units with all 4096 weights present
  launch_dependents();  // pass 2 may be scheduled meanwhile (it waits for this grid)
  if (ticket && blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0;  // pass 2's arrival count
  build_cells(s_cells);
  __syncthreads();
  const uint32_t tab_b = smem_u32(s_cells) + static_cast<uint32_t>(lane) * 8u - kCellBias * kEntryBytes;
  const int ql = lane & 3, bw = lane >> 2;  // quarter of the block, block within the warp
  auto load16 = [&](int64_t u, float4 (&f)[4]) {
    const int64_t b = u * kUnit + warp * 8 + bw;
    const float4* src = reinterpret_cast<const float4*>(W + b * kBlock + ql * 16);
#pragma unroll
    for (int v = 0; v < 4; ++v) f[v] = __ldg(src + v);
  };
  float4 nxt[4];
  if (blockIdx.x < nfull) load16(blockIdx.x, nxt);
  // the unit after is pulled into L2 ahead of its register loads (one bulk prefetch per unit)
  if (threadIdx.x == 0 && blockIdx.x + gridDim.x < nfull)
    prefetch_l2_bulk(W + (blockIdx.x + gridDim.x) * kUnitElems, kUnitElems * 4);

#pragma unroll 1
  for (int64_t u = blockIdx.x; u < nunits; u += gridDim.x) {
    if (u < nfull) {
      const int local_block = warp * 8 + bw;
      const int64_t b = u * kUnit + local_block;
      float w[16];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        w[4 * v + 0] = nxt[v].x; w[4 * v + 1] = nxt[v].y; w[4 * v + 2] = nxt[v].z; w[4 * v + 3] = nxt[v].w;
      }
      // the next unit's loads in flight during this one, the one after that on its way to L2
      if (u + gridDim.x < nfull) load16(u + gridDim.x, nxt);
      if (threadIdx.x == 0 && u + 2 * gridDim.x < nfull)
        prefetch_l2_bulk(W + (u + 2 * gridDim.x) * kUnitElems, kUnitElems * 4);
      float m = fabsf(w[0]);
#pragma unroll
      for (int i = 1; i < 16; ++i) m = fmaxf(m, fabsf(w[i]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      if (ql == 0) absmax[b] = m;
      {
        // blocks warp*8 .. warp*8+7 sit at lanes 4 bw: pair sums over bw bits 0, 1, 2 build
        // the perfect binary tree of the eight (x + y == y + x in IEEE)
        double t = static_cast<double>(m);
        t += __shfl_xor_sync(0xffffffffu, t, 4);
        t += __shfl_xor_sync(0xffffffffu, t, 8);
        t += __shfl_xor_sync(0xffffffffu, t, 16);
        if (lane == 0) sum8[u * 8 + warp] = t;
      }
      uint32_t c[16];
      // a tiny, infinite or NaN absmax has no usable reciprocal: exact division
      bool near = !(m >= 0x1p-100f && m <= 0x1.fffffep127f);
      if (!near) {
        const float rcp = __frcp_rn(m);
        float dmin = __int_as_float(0x7f800000);
#pragma unroll
        for (int i = 0; i < 16; ++i) c[i] = code_fast(__fmul_rn(w[i], rcp), tab_b, dmin);
        near = !(dmin >= kGuard);
      }
      if (near) {
#pragma unroll
        for (int i = 0; i < 16; ++i) c[i] = code_exact(w[i], m);
      }
      // byte j = (c[2j] << 4) | c[2j+1], little endian: the nibbles from the top are
      // c6 c7 c4 c5 c2 c3 c0 c1, accumulated as a multiply-add chain (multiply-add pipe)
      uint32_t lo = c[6], hi = c[14];
#pragma unroll
      for (int t = 1; t < 8; ++t) {
        const int e = 6 - 2 * (t >> 1) + (t & 1);  // 7, 4, 5, 2, 3, 0, 1
        lo = lo * 16u + c[e];
        hi = hi * 16u + c[8 + e];
      }
      *reinterpret_cast<uint2*>(codes + b * (kBlock / 2) + ql * 8) = make_uint2(lo, hi);
    } else {
      // partial last unit: half a warp per block, one float4 per lane, exact division
      const int half = lane >> 4, hl = lane & 15;
#pragma unroll 1
      for (int it = 0; it < kUnit / 16; ++it) {
        const int local_block = it * 16 + warp * 2 + half;
        const int64_t b = u * kUnit + local_block;
        const int64_t e = b * kBlock + hl * 4;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = e + i < numel ? W[e + i] : 0.0f;
        float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (hl == 0) {
          s_abs[local_block] = m;  // blocks past the end hold 0 (all their inputs read as 0)
          if (b < nblocks) absmax[b] = m;
        }
        const uint32_t c0 = code_exact(v[0], m), c1 = code_exact(v[1], m);
        const uint32_t c2 = code_exact(v[2], m), c3 = code_exact(v[3], m);
        if (e < numel) codes[e / 2] = static_cast<uint8_t>(e + 1 < numel ? ((c0 << 4) | c1) : (c0 << 4));
        if (e + 2 < numel) codes[e / 2 + 1] = static_cast<uint8_t>(e + 3 < numel ? ((c2 << 4) | c3) : (c2 << 4));
      }
      __syncthreads();  // the partial unit's absmax values are all in s_abs
      if (warp == 0 && lane < 8) {  // its eight 8-block subtrees
        const float* a = s_abs + lane * 8;
        sum8[u * 8 + lane] = (((double)a[0] + (double)a[1]) + ((double)a[2] + (double)a[3])) +
                             (((double)a[4] + (double)a[5]) + ((double)a[6] + (double)a[7]));
      }
    }
  }
}

// -------------------------------------------------------------------- pass 2
// The pairwise tree over the 8-block sums, zero-padded to a power of two P, is cut into
// nparts <= 128 aligned subtrees of P / nparts leaves, one CTA of 1024 threads each; pass 3
// combines the subtree sums (the top levels of the same tree) and forms
// mean = (float)(total / nblocks).  Each thread folds a run of kRun consecutive leaves (a
// power of two) with a register tree -- exactly the pairwise tree of the run -- and the runs
// combine through warp butterflies and a final warp.
template <int kRun>
__device__ __forceinline__ double fold_run(const double* __restrict__ leaf, int64_t lo, int64_t n) {
  double v[kRun];
#pragma unroll
  for (int i = 0; i < kRun; ++i) v[i] = (lo + i < n) ? leaf[lo + i] : 0.0;
#pragma unroll
  for (int w = 1; w < kRun; w <<= 1)
#pragma unroll
    for (int i = 0; i < kRun; i += 2 * w) v[i] = v[i] + v[i + w];
  return v[0];
}

__global__ void __launch_bounds__(1024) nf4_absmax_mean(const double* __restrict__ leaf_sum,
                                                        int64_t nleaves, int64_t run,
                                                        double* __restrict__ part, int* ticket,
                                                        int64_t nblocks, float* __restrict__ mean) {
  __shared__ double s_warp[32];
  __shared__ int s_last;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  launch_dependents();     // pass 3 may be scheduled meanwhile (it waits for this grid)
  grid_dependency_wait();  // the 8-block sums of pass 1
  const int64_t lo = ((int64_t)blockIdx.x * 1024 + t) * run;
  double s;
  switch (run) {
    case 1: s = fold_run<1>(leaf_sum, lo, nleaves); break;
    case 2: s = fold_run<2>(leaf_sum, lo, nleaves); break;
    case 4: s = fold_run<4>(leaf_sum, lo, nleaves); break;
    case 8: s = fold_run<8>(leaf_sum, lo, nleaves); break;
    case 16: s = fold_run<16>(leaf_sum, lo, nleaves); break;
    default: {  // very large tensors: binary-counter fold of the run, still the pairwise tree
      double stack[48];
      int depth = 0;
      for (int64_t i = 0; i < run; ++i) {
        double v = (lo + i < nleaves) ? leaf_sum[lo + i] : 0.0;
        int64_t k = i + 1;
        while ((k & 1) == 0) {
          v = stack[--depth] + v;
          k >>= 1;
        }
        stack[depth++] = v;
      }
      s = stack[0];
    }
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) s_warp[warp] = s;
  __syncthreads();
  if (warp == 0) {
    double w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) w += __shfl_xor_sync(0xffffffffu, w, o);
    if (lane == 0) {
      part[blockIdx.x] = w;
      __threadfence();
      s_last = atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1;
    }
  }
  __syncthreads();
  if (!s_last || warp != 0) return;
  // the last CTA: the top levels of the tree over the nparts subtree sums -- a lane folds
  // nparts / 32 consecutive sums (past 32 parts), then a butterfly over the lanes holding
  // one -- and mean = (float)(total / nblocks); the ticket is left at zero for the next call
  __threadfence();
  const int nparts = static_cast<int>(gridDim.x);
  double v = 0.0;
  if (nparts <= 32) {
    if (lane < nparts) v = __ldcg(part + lane);
  } else if (nparts == 64) {
    v = __ldcg(part + 2 * lane) + __ldcg(part + 2 * lane + 1);
  } else {  // 128
    v = (__ldcg(part + 4 * lane) + __ldcg(part + 4 * lane + 1)) +
        (__ldcg(part + 4 * lane + 2) + __ldcg(part + 4 * lane + 3));
  }
  const int lanes = nparts < 32 ? nparts : 32;
  for (int o = 1; o < lanes; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) {
    mean[0] = (float)(v / (double)nblocks);
    *ticket = 0;
  }
}

// -------------------------------------------------------------------- pass 3
// A warp per group of 256 blocks (8 per lane), 8 groups per CTA, with the mean that pass 2
// stored.
__global__ void __launch_bounds__(256) nf4_double_quant(const float* __restrict__ absmax,
                                                        int64_t nblocks, int64_t ngroups,
                                                        const float* mean, int fp8,
                                                        int8_t* __restrict__ scale_codes,
                                                        float* __restrict__ steps) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t g = (int64_t)blockIdx.x * 8 + warp;
  grid_dependency_wait();  // the mean of pass 2 (and with it the absmax of pass 1)
  const int64_t b0 = g * kGroup + lane * 8;
  const bool whole = b0 + 8 <= nblocks;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (g < ngroups) {
    if (whole) {
      const float4* src = reinterpret_cast<const float4*>(absmax + b0);
      const float4 x = __ldg(src), y = __ldg(src + 1);
      a[0] = x.x; a[1] = x.y; a[2] = x.z; a[3] = x.w;
      a[4] = y.x; a[5] = y.y; a[6] = y.z; a[7] = y.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (b0 + i < nblocks) a[i] = absmax[b0 + i];
    }
  }
  if (g >= ngroups) return;
  const float mu = __ldcg(mean);
  float d[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) d[i] = (whole || b0 + i < nblocks) ? __fsub_rn(a[i], mu) : 0.0f;
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(d[i]));
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // int8: 127 steps each side; fp8: the E4M3 range, 448 at the largest |a - mean|
  const float step = __fdiv_rn(m, fp8 ? 448.0f : 127.0f);
  if (lane == 0) steps[g] = step;
  uint32_t q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (fp8) {  // nearest E4M3 value, ties to even, saturating at 448 (code 0 when step = 0)
      q[i] = step > 0.0f
                 ? static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(d[i], step), __NV_SATFINITE, __NV_E4M3))
                 : 0u;
    } else {
      int v = 0;
      if (step > 0.0f) {
        v = __float2int_rn(__fdiv_rn(d[i], step));  // round half to even
        v = v > 127 ? 127 : (v < -127 ? -127 : v);
      }
      q[i] = static_cast<uint32_t>(v) & 0xFFu;
    }
  }
  if (whole) {
    *reinterpret_cast<uint2*>(scale_codes + b0) =
        make_uint2(q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24),
                   q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24));
  } else {
    for (int i = 0; i < 8; ++i)
      if (b0 + i < nblocks) scale_codes[b0 + i] = static_cast<int8_t>(q[i]);
  }
}

// -------------------------------------------------------------------- dequantize
// Grid-stride over 16-weight pieces: 8 code bytes in, 32 bytes of bf16 (fp16 when H) out per
// thread; the four threads of a 64-block each build the block's byte table.  Without double
// quantization (dq = 0) `steps` holds the fp32 absmax of every block, and the block scale is
// fmaf(1, absmax, 0) = absmax through the same arithmetic.
template <bool H, bool kDependent>
__global__ void __launch_bounds__(256) nf4_dequant_kernel(const uint8_t* __restrict__ codes,
                                                          const int8_t* __restrict__ scale_codes,
                                                          const float* __restrict__ steps,
                                                          const float* __restrict__ mean,
                                                          int64_t numel, int dq, int fp8,
                                                          uint16_t* __restrict__ out) {
  if (kDependent) launch_dependents();  // the GEMM streaming the output waits for this grid
  const float mu = dq ? __ldg(mean) : 0.0f;
  const int64_t npieces = (numel + 15) / 16;
  for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < npieces;
       p += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e0 = p * 16;
    const int64_t b = e0 / kBlock;
    const float scale =
        dq ? __fmaf_rn(nf4_second_level(static_cast<uint8_t>(__ldg(scale_codes + b)), fp8),
                       __ldg(steps + b / kGroup), mu)
           : __ldg(steps + b);
    const Nf4ByteTable tab = nf4_make_table<H>(scale);
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
  // launched as a programmatic dependent (the staged base of a GEMM): the kernel before it
  // (the rank-r product the GEMM reads) must be complete when this grid is; one thread per
  // CTA waits, so its CTA completes no earlier.  A separate instantiation: the wait raised
  // the kernel from 30 to 40 registers, 6 instead of 8 resident CTAs per SM (the standalone
  // 28672 x 8192 dequantization took 137 instead of 104 us).
  if (kDependent && threadIdx.x == 0) grid_dependency_wait();
}

// -------------------------------------------------------------------- launchers
constexpr int kMeanParts = kQuantizeMeanParts;  // most CTAs of pass 2

uint64_t quantize_workspace_bytes(int64_t numel) {
  const int64_t nb = (numel + kBlock - 1) / kBlock;
  const int64_t ng = (nb + kGroup - 1) / kGroup;
  // absmax fp32 [ngroups * 256] (padded to whole groups), 8-block sums fp64 [<= 32 ngroups],
  // then the mean's subtree sums fp64 [<= kMeanParts] and the arrival ticket of pass 2
  return (uint64_t)ng * kGroup * 4 + (uint64_t)ng * (kGroup / 8) * 8 + kQuantizeTailBytes;
}

int launch_quantize(const float* W, int64_t numel, const nf4_tensor& q, void* ws,
                    cudaStream_t stream) {
  const int64_t nb = (numel + kBlock - 1) / kBlock;
  const int64_t ng = (nb + kGroup - 1) / kGroup;
  const bool dq = q.dq_block != 0;
  // without double quantization pass 1 writes the block absmax straight into the tensor
  float* absmax = dq ? reinterpret_cast<float*>(ws) : q.scale_steps;
  const int64_t nu = (nb + kUnit - 1) / kUnit;
  const int64_t nleaves = nu * (kUnit / 8);  // 8-block sums
  double* usum = reinterpret_cast<double*>(reinterpret_cast<char*>(ws) + ng * kGroup * 4);
  double* part = usum + ng * (kGroup / 8);
  int* ticket = reinterpret_cast<int*>(part + kMeanParts);  // zeroed by pass 1
  {
    ProfileScope ps("nf4_quant_blocks", stream);
    // persistent: as many CTAs as are resident at once, or fewer units
    static DeviceCache<int> occupancy;  // resident CTAs per SM, per device
    int per_sm = 0;
    const int st = occupancy.get(device_context_key, &per_sm, [](int* v) -> int {
      if (cudaFuncSetAttribute(nf4_quant_blocks, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kCellBytes) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, nf4_quant_blocks, kQuantThreads,
                                                        kCellBytes) != cudaSuccess) {
        cudaGetLastError();
        return QLORA_ERR_CUDA;
      }
      if (*v < 1) *v = 1;
      return QLORA_OK;
    });
    if (st) return st == -1 ? QLORA_ERR_NO_DEVICE : st;
    const int64_t resident = (int64_t)per_sm * num_sms();
    const int64_t ctas = nu < resident ? nu : resident;
    nf4_quant_blocks<<<(unsigned)ctas, kQuantThreads, kCellBytes, stream>>>(
        W, numel, q.codes, absmax, usum, dq ? ticket : nullptr);
  }
  if (!dq) return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
  int64_t p2 = 1;
  while (p2 < nleaves) p2 *= 2;
  const int nparts =
      p2 > 1024 ? static_cast<int>(p2 / 1024 < kMeanParts ? p2 / 1024 : kMeanParts) : 1;
  const int64_t run = p2 > 1024 * nparts ? p2 / (1024 * nparts) : 1;
  // passes 2 and 3 are programmatic dependents: launched while the pass before finishes,
  // they wait for it (griddepcontrol.wait) before reading its output
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  {
    ProfileScope ps("nf4_absmax_mean", stream);
    cfg.gridDim = dim3(nparts);
    cfg.blockDim = dim3(1024);
    if (cudaLaunchKernelEx(&cfg, nf4_absmax_mean, static_cast<const double*>(usum), nleaves, run,
                           part, ticket, nb, q.scale_mean) != cudaSuccess)
      return QLORA_ERR_CUDA;
  }
  {
    ProfileScope ps("nf4_double_quant", stream);
    cfg.gridDim = dim3((unsigned)((ng + 7) / 8));
    cfg.blockDim = dim3(256);
    if (cudaLaunchKernelEx(&cfg, nf4_double_quant, static_cast<const float*>(absmax), nb, ng,
                           static_cast<const float*>(q.scale_mean),
                           q.dq_type == NF4_DQ_FP8 ? 1 : 0, q.scale_codes, q.scale_steps) != cudaSuccess)
      return QLORA_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

// Resident CTAs per SM of the dequantize kernel (per device and context).
template <bool H, bool kDependent>
static int dequant_resident(int* per_sm) {
  static DeviceCache<int> occupancy;
  const int st = occupancy.get(device_context_key, per_sm, [](int* v) -> int {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, nf4_dequant_kernel<H, kDependent>, 256,
                                                      0) != cudaSuccess) {
      cudaGetLastError();
      return QLORA_ERR_CUDA;
    }
    if (*v < 1) *v = 1;
    return QLORA_OK;
  });
  return st == -1 ? QLORA_ERR_NO_DEVICE : st;
}

int launch_dequantize(const nf4_tensor& q, int64_t numel, uint16_t* out, bool half,
                      cudaStream_t stream, bool dependent) {
  const int64_t npieces = (numel + 15) / 16;
  const int threads = 256;
  int64_t blocks = (npieces + threads - 1) / threads;
  // one wave of the grid-stride loop: as many CTAs as are resident (at most 8 per SM; as a
  // programmatic dependent it launches once every CTA of the kernel before it is running, so
  // its CTAs only take what is left)
  int per_sm = 0;
  const int ost = dependent ? (half ? dequant_resident<true, true>(&per_sm)
                                    : dequant_resident<false, true>(&per_sm))
                            : (half ? dequant_resident<true, false>(&per_sm)
                                    : dequant_resident<false, false>(&per_sm));
  if (ost) return ost;
  const int64_t cap = (int64_t)num_sms() * std::min(per_sm, 8);
  if (blocks > cap) blocks = cap;
  ProfileScope ps("nf4_dequant", stream);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  const int dq = q.dq_block != 0 ? 1 : 0, fp8 = q.dq_type == NF4_DQ_FP8 ? 1 : 0;
  const auto kernel = dependent ? (half ? nf4_dequant_kernel<true, true> : nf4_dequant_kernel<false, true>)
                                : (half ? nf4_dequant_kernel<true, false> : nf4_dequant_kernel<false, false>);
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, q.codes, q.scale_codes, q.scale_steps,
                                           q.scale_mean, numel, dq, fp8, out);
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
