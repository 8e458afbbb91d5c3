// merge.cu -- folding a LoRA adapter into the NF4 base, and the NF4-vs-INT4 error statistics.
//
// Merge (junaidshaukat.com "QLoRA -- the democratization event", the deployment-subtlety
// paragraph: merging means dequantize, merge, maybe requantize; infivelines.com "QLoRA": a
// bf16 adapter merged into a 4-bit base and saved loses precision twice; addaly.com "QLoRA on
// one card", "Merging a QLoRA adapter, and the subtlety"):
//     W_merged = bf16( W' + s * B A )          W' = the bf16 dequantization of the NF4 base
// One pass over the packed codes: each CTA stages its [r x 128] slice of A and [64 x r] slice
// of B in shared memory, forms the rank-r product of its 64 x 128 tile on the tensor cores
// (mma.sync, bf16 x bf16 products exact, fp32 accumulation), and each thread then
// dequantizes its base weights exactly as nf4_dequantize does, adds RN(s * delta) in fp32 and
// rounds once to bf16.  The fp32 copy (the same values) feeds nf4_quantize for the
// requantized artifact.
//
// Error statistics (aicurriculum.codextroop.com "QLoRA -- Module 12.4", "Design Details That
// Matter": NF4 places levels at normal quantiles and is often better than naive INT4;
// addaly.com "QLoRA on one card", "What each setting is doing": NF4 keeps more information
// than plain 4-bit integers at the same size): for fp32 weights, per block of 64 with its
// absmax a, the squared error of the NF4 reconstruction level[c] * a (c = nearest level of
// w / a) and of the symmetric absmax INT4 reconstruction q * (a / 7), q = clamp(rint(7 w / a),
// -7, 7), summed over the tensor together with sum w^2 (fp32 within a thread's 16 weights,
// fp64 across threads and CTAs).
#include <algorithm>

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

// Rank padded to the MMA contraction (16) and the shared-memory pitches (in bf16 / fp32
// elements; the +8 / +4 pads make the ldmatrix rows and the fp32 tile's float2 stores
// conflict-free).
__host__ __device__ inline int rank16(int r) { return (r + 15) / 16 * 16; }
constexpr int A_PITCH = COLS + 8;   // sA [r16][COLS] bf16
constexpr int D_PITCH = COLS + 4;   // sD [ROWS][COLS] fp32
inline int b_pitch(int r) { return rank16(r) + 8; }  // sB [ROWS][r16] bf16
inline int smem_bytes(int r) {
  return rank16(r) * A_PITCH * 2 + ROWS * b_pitch(r) * 2 + ROWS * D_PITCH * 4;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&v)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(addr));
}

// The persistent form's fp32 tile is [ROWS][COLS] with no pad; the 16-byte piece J of row R
// sits at piece J ^ x(R, b), b = the 64-column half of J.  x takes bits 0-1 from R and bit 2
// from b ^ R, so the MMA's float2 stores (rows g = 0..3 of a half-warp in distinct piece pairs)
// and the epilogue's float4 loads (two rows x two halves x two threads per quarter-warp) both
// cover all 32 banks.
__device__ __forceinline__ int swz_col(int R, int C) {
  const int x = (R & 3) | ((((C >> 6) ^ R) & 1) << 2);
  return C ^ (x << 2);
}

// delta = B A for one 64 x 128 tile on the tensor cores (mma.sync m16n8k16, bf16 x bf16
// products exact, fp32 accumulation): warp w takes rows 16 (w & 3) .. + 15 and columns
// 64 (w >> 2) .. + 63 from the staged slices sA [r16][A_PITCH] and sB [ROWS][bp], and writes
// its fp32 results to sD ([ROWS][D_PITCH], or the swizzled [ROWS][COLS] when kSwz).
template <bool kSwz>
__device__ __forceinline__ void merge_tile_mma(const uint16_t* sA, const uint16_t* sB, float* sD,
                                               int r16, int bp, int warp, int lane) {
  const int mt = warp & 3, nh = warp >> 2;
  float acc[8][4];
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  const uint32_t sA0 = smem_u32(sA), sB0 = smem_u32(sB);
  for (int j0 = 0; j0 < r16; j0 += 16) {
    uint32_t a[4];  // rows 16 mt + (lane & 15), rank j0 + 8 (lane >> 4) .. + 7
    ldsm_x4(sB0 + ((16 * mt + (lane & 15)) * bp + j0 + 8 * (lane >> 4)) * 2, a);
#pragma unroll
    for (int t = 0; t < 8; t += 2) {
      // n-tiles t, t + 1 of this warp's 64 columns; rank halves j0 .. + 7, j0 + 8 .. + 15
      uint32_t b[4];
      const int jr = j0 + (lane & 7) + 8 * ((lane >> 3) & 1);
      const int col = 64 * nh + 8 * (t + (lane >> 4));
      ldsm_x4_t(sA0 + (jr * A_PITCH + col) * 2, b);
      const uint32_t b0[2] = {b[0], b[1]}, b1[2] = {b[2], b[3]};
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
          " {%8, %9}, {%0, %1, %2, %3};"
          : "+f"(acc[t][0]), "+f"(acc[t][1]), "+f"(acc[t][2]), "+f"(acc[t][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0[0]), "r"(b0[1]));
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
          " {%8, %9}, {%0, %1, %2, %3};"
          : "+f"(acc[t + 1][0]), "+f"(acc[t + 1][1]), "+f"(acc[t + 1][2]), "+f"(acc[t + 1][3])
          : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b1[0]), "r"(b1[1]));
    }
  }
  const int g = lane >> 2, q = lane & 3;
  const int r0 = 16 * mt + g, r1 = r0 + 8;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const int col = 64 * nh + 8 * t + 2 * q;
    if (kSwz) {
      *reinterpret_cast<float2*>(sD + r0 * COLS + swz_col(r0, col)) = make_float2(acc[t][0], acc[t][1]);
      *reinterpret_cast<float2*>(sD + r1 * COLS + swz_col(r1, col)) = make_float2(acc[t][2], acc[t][3]);
    } else {
      *reinterpret_cast<float2*>(sD + r0 * D_PITCH + col) = make_float2(acc[t][0], acc[t][1]);
      *reinterpret_cast<float2*>(sD + r1 * D_PITCH + col) = make_float2(acc[t][2], acc[t][3]);
    }
  }
}

// The base weights of one thread in a tile: rows rr0 + 16 p (p < RPT), columns kk .. kk + 7
// (one code word and one block scale each), zero outside W.
struct MergeCodes {
  uint32_t word[RPT];
  uint8_t scode[RPT];
  float sstep[RPT];
};
__device__ __forceinline__ void merge_load_codes(MergeCodes& mc, const uint8_t* codes,
                                                 const int8_t* qs, const float* steps, int dq,
                                                 int64_t N, int64_t K, int64_t n0, int64_t kk,
                                                 int rr0) {
#pragma unroll
  for (int p = 0; p < RPT; ++p) {
    const int64_t n = n0 + rr0 + 16 * p;
    mc.word[p] = 0;
    mc.scode[p] = 0;
    mc.sstep[p] = 0.f;
    if (n < N && kk < K) {
      const int64_t e = n * K + kk;
      const int64_t blk = e / 64;
      mc.word[p] = __ldg(reinterpret_cast<const uint32_t*>(codes + e / 2));
      if (dq) {
        mc.scode[p] = static_cast<uint8_t>(__ldg(qs + blk));
        mc.sstep[p] = __ldg(steps + (blk >> 8));
      } else {
        mc.sstep[p] = __ldg(steps + blk);
      }
    }
  }
}

// One thread's outputs of a tile: dequantize its eight base weights of each row exactly as
// nf4_dequantize does, add RN(s * delta) in fp32, round once to bf16.
__device__ __forceinline__ void merge_tile_epilogue(const MergeCodes& mc, const float* sD, float mu,
                                                    int dq, int fp8, float scale, int64_t N,
                                                    int64_t K, int64_t n0, int64_t kk, int rr0,
                                                    int c8, uint16_t* out16, float* out32) {
  if (kk >= K) return;
#pragma unroll
  for (int p = 0; p < RPT; ++p) {
    const int rr = rr0 + 16 * p;
    const int64_t n = n0 + rr;
    if (n >= N) break;
    const int64_t e = n * K + kk;
    // the thread's two 16-byte pieces, in an order that alternates by groups of 4 lanes, so
    // the 16 lanes of a row cover all 8 bank groups in each load (in column order, only the
    // even pieces in the first load: 4-way conflicts)
    const int sw = (c8 >> 2) & 1;
    const float4 e0 = *reinterpret_cast<const float4*>(sD + rr * D_PITCH + 8 * c8 + 4 * sw);
    const float4 e1 = *reinterpret_cast<const float4*>(sD + rr * D_PITCH + 8 * c8 + 4 * (1 - sw));
    const float4 d0 = sw ? e1 : e0, d1 = sw ? e0 : e1;
    const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    const float a_hat = dq ? __fmaf_rn(nf4_second_level(mc.scode[p], fp8), mc.sstep[p], mu) : mc.sstep[p];
    uint32_t wd[4];
    nf4_dequant8(nf4_make_table(a_hat), mc.word[p], wd);
    uint32_t o16[4];
    float o32[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float v0 = __fadd_rn(bf16_bits_to_f32(wd[i] & 0xFFFFu), __fmul_rn(scale, d[2 * i]));
      const float v1 = __fadd_rn(bf16_bits_to_f32(wd[i] >> 16), __fmul_rn(scale, d[2 * i + 1]));
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

// One CTA per tile (output rows n0 .. n0 + 63, columns k0 .. k0 + 127): the general form
// (any rank up to 128; ranks past 32 or not multiples of 8, and K not a multiple of 64).
__global__ void __launch_bounds__(THREADS) nf4_merge_kernel(
    const uint8_t* __restrict__ codes, const int8_t* __restrict__ qs,
    const float* __restrict__ steps, const float* __restrict__ mean,
    int dq, int fp8, const uint16_t* __restrict__ A, const uint16_t* __restrict__ B, int64_t N,
    int64_t K, int r, float scale, uint16_t* __restrict__ out16, float* __restrict__ out32) {
  extern __shared__ __align__(16) uint8_t msm[];
  const int r16 = rank16(r), bp = r16 + 8;
  uint16_t* sA = reinterpret_cast<uint16_t*>(msm);              // [r16][A_PITCH]
  uint16_t* sB = sA + r16 * A_PITCH;                            // [ROWS][bp]
  float* sD = reinterpret_cast<float*>(sB + ROWS * bp);         // [ROWS][D_PITCH]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t k0 = static_cast<int64_t>(blockIdx.x) * COLS;
  const int64_t n0 = static_cast<int64_t>(blockIdx.y) * ROWS;
  const int c8 = tid & 15;
  const int64_t kk = k0 + 8 * c8;
  const int rr0 = tid >> 4;
  // the base weights first, so they arrive while the adapters are staged and multiplied
  MergeCodes mc;
  merge_load_codes(mc, codes, qs, steps, dq, N, K, n0, kk, rr0);
  // A [r][K] -> sA[j][0, COLS) (16-byte pieces; zero past r and past K)
  for (int i = tid; i < r16 * (COLS / 8); i += THREADS) {
    const int j = i / (COLS / 8), c = i % (COLS / 8);
    const int64_t k = k0 + 8 * c;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (j < r && k < K) v = __ldg(reinterpret_cast<const uint4*>(A + j * K + k));
    *reinterpret_cast<uint4*>(sA + j * A_PITCH + 8 * c) = v;
  }
  // B [N][r] -> sB[row][0, r16): 16-byte pieces when the rows are 16-byte multiples, else
  // element by element
  if (r % 8 == 0) {
    const int per = r16 / 8;  // pieces per staged row
    for (int i = tid; i < ROWS * per; i += THREADS) {
      const int rr = i / per, j8 = i % per;
      const int64_t n = n0 + rr;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < N && 8 * j8 < r) v = __ldg(reinterpret_cast<const uint4*>(B + n * r + 8 * j8));
      *reinterpret_cast<uint4*>(sB + rr * bp + 8 * j8) = v;
    }
  } else {
    for (int i = tid; i < ROWS * r16; i += THREADS) {
      const int rr = i / r16, j = i % r16;
      const int64_t n = n0 + rr;
      sB[rr * bp + j] = (n < N && j < r) ? __ldg(B + n * r + j) : static_cast<uint16_t>(0);
    }
  }
  __syncthreads();
  merge_tile_mma<false>(sA, sB, sD, r16, bp, warp, lane);
  __syncthreads();
  const float mu = dq ? __ldg(mean) : 0.0f;
  merge_tile_epilogue(mc, sD, mu, dq, fp8, scale, N, K, n0, kk, rr0, c8, out16, out32);
}

// The persistent form's thread layout: thread t takes row t / 4 of the tile and, in the
// 64-column half b = (t / 2) % 2 (one quantization block of W, K being a multiple of 64), the
// columns 8 h + 16 i .. + 7 (h = t % 2, i = 0..3): one block scale and one dequantization
// table for its 32 weights, and each 16-byte store of a thread pair fills a 32-byte sector.
struct RowCodes {
  uint32_t word[4];  // codes of columns 8 h + 16 i .. + 7
  uint8_t scode;
  float sstep;
};
__device__ __forceinline__ void merge_row_load(RowCodes& rc, const uint8_t* codes, const int8_t* qs,
                                               const float* steps, int dq, int64_t N, int64_t K,
                                               int64_t n, int64_t kb, int h) {
  rc.word[0] = rc.word[1] = rc.word[2] = rc.word[3] = 0;
  rc.scode = 0;
  rc.sstep = 0.f;
  if (n < N && kb < K) {
    const int64_t e = n * K + kb;  // a multiple of 64: the block's first weight
    const int64_t blk = e >> 6;
    const uint32_t* w = reinterpret_cast<const uint32_t*>(codes + (e >> 1)) + h;
#pragma unroll
    for (int i = 0; i < 4; ++i) rc.word[i] = __ldg(w + 2 * i);
    if (dq) {
      rc.scode = static_cast<uint8_t>(__ldg(qs + blk));
      rc.sstep = __ldg(steps + (blk >> 8));
    } else {
      rc.sstep = __ldg(steps + blk);
    }
  }
}

// One thread's 32 outputs: dequantize as nf4_dequantize does, add RN(s * delta) in fp32,
// round once to bf16 (sD: the swizzled tile).
__device__ __forceinline__ void merge_row_epilogue(const RowCodes& rc, const float* sD, float mu,
                                                   int dq, int fp8, float scale, int64_t N,
                                                   int64_t K, int64_t n, int64_t kb, int rr, int b,
                                                   int h, uint16_t* out16, float* out32) {
  if (n >= N || kb >= K) return;
  const float a_hat = dq ? __fmaf_rn(nf4_second_level(rc.scode, fp8), rc.sstep, mu) : rc.sstep;
  const Nf4ByteTable tab = nf4_make_table(a_hat);
  const float* row = sD + rr * COLS;
  const int64_t e = n * K + kb + 8 * h;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int c0 = 64 * b + 8 * h + 16 * i;  // this group's first column in the tile
    const float4 d0 = *reinterpret_cast<const float4*>(row + swz_col(rr, c0));
    const float4 d1 = *reinterpret_cast<const float4*>(row + swz_col(rr, c0 + 4));
    const float d[8] = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
    uint32_t wd[4];
    nf4_dequant8(tab, rc.word[i], wd);
    uint32_t o16[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float v0 = __fadd_rn(bf16_bits_to_f32(wd[j] & 0xFFFFu), __fmul_rn(scale, d[2 * j]));
      const float v1 = __fadd_rn(bf16_bits_to_f32(wd[j] >> 16), __fmul_rn(scale, d[2 * j + 1]));
      const __nv_bfloat162 o = __floats2bfloat162_rn(v0, v1);
      o16[j] = *reinterpret_cast<const uint32_t*>(&o);
    }
    if (out16) *reinterpret_cast<uint4*>(out16 + e + 16 * i) = make_uint4(o16[0], o16[1], o16[2], o16[3]);
    if (out32) {
      float4* o = reinterpret_cast<float4*>(out32 + e + 16 * i);
      o[0] = make_float4(bf16_bits_to_f32(o16[0] & 0xFFFFu), bf16_bits_to_f32(o16[0] >> 16),
                         bf16_bits_to_f32(o16[1] & 0xFFFFu), bf16_bits_to_f32(o16[1] >> 16));
      o[1] = make_float4(bf16_bits_to_f32(o16[2] & 0xFFFFu), bf16_bits_to_f32(o16[2] >> 16),
                         bf16_bits_to_f32(o16[3] & 0xFFFFu), bf16_bits_to_f32(o16[3] >> 16));
    }
  }
}

// Persistent form for ranks r <= 32 with r % 8 == 0 (R16 = 16 or 32) and K a multiple of 64:
// the resident CTAs take tiles t, t + grid, ...; the next tile's A / B slices (one or two
// 16-byte pieces per thread) and base-weight codes are loaded into registers before the
// current tile's MMA and epilogue, so their latency overlaps that work instead of opening
// every tile.
template <int R16>
__global__ void __launch_bounds__(THREADS, 3) nf4_merge_persistent(
    const uint8_t* __restrict__ codes, const int8_t* __restrict__ qs,
    const float* __restrict__ steps, const float* __restrict__ mean,
    int dq, int fp8, const uint16_t* __restrict__ A, const uint16_t* __restrict__ B, int64_t N,
    int64_t K, int r, float scale, uint16_t* __restrict__ out16, float* __restrict__ out32,
    int ntr, int kbl) {
  constexpr int BP = R16 + 8;
  constexpr int APT = R16 * (COLS / 8) / THREADS;  // A pieces per thread (1 or 2)
  constexpr int BPR = R16 / 8;                     // B pieces per staged row
  static_assert(ROWS * BPR <= THREADS, "one B piece per thread at most");
  __shared__ __align__(16) uint16_t sA[R16 * A_PITCH];
  __shared__ __align__(16) uint16_t sB[ROWS * BP];
  extern __shared__ __align__(16) uint8_t msm[];
  float* sD = reinterpret_cast<float*>(msm);  // [ROWS][COLS], swizzled
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rr = tid >> 2, b = (tid >> 1) & 1, h = tid & 1;
  const float mu = dq ? __ldg(mean) : 0.0f;
  // per-thread pieces of the A / B slices: A row j = tid / 16 + 16 u, columns 8 (tid % 16) ..;
  // B row tid / BPR, ranks 8 (tid % BPR) ..
  const int a_j = tid / (COLS / 8), a_c = tid % (COLS / 8);
  const int b_r = tid / BPR, b_j = tid % BPR;
  const bool b_on = tid < ROWS * BPR && 8 * b_j < r;
  uint4 av[APT], bv;
  RowCodes rc;
  // tile (tr, tc): rows 64 tr .., columns 128 tc ..
  auto load = [&](int tr, int tc, uint4 (&a)[APT], uint4& bb, RowCodes& c) {
    const int64_t n0 = static_cast<int64_t>(tr) * ROWS, k0 = static_cast<int64_t>(tc) * COLS;
    const int64_t k = k0 + 8 * a_c;
#pragma unroll
    for (int u = 0; u < APT; ++u) {
      const int j = a_j + u * (THREADS / (COLS / 8));
      a[u] = make_uint4(0, 0, 0, 0);
      if (j < r && k < K) a[u] = __ldg(reinterpret_cast<const uint4*>(A + j * K + k));
    }
    bb = make_uint4(0, 0, 0, 0);
    if (b_on && n0 + b_r < N)
      bb = __ldg(reinterpret_cast<const uint4*>(B + (n0 + b_r) * r + 8 * b_j));
    merge_row_load(c, codes, qs, steps, dq, N, K, n0 + rr, k0 + 64 * b, h);
  };
  auto stage = [&](const uint4 (&a)[APT], const uint4& bb) {
#pragma unroll
    for (int u = 0; u < APT; ++u)
      *reinterpret_cast<uint4*>(sA + (a_j + u * (THREADS / (COLS / 8))) * A_PITCH + 8 * a_c) = a[u];
    if (tid < ROWS * BPR) *reinterpret_cast<uint4*>(sB + b_r * BP + 8 * b_j) = bb;
  };
  // the CTA's tiles t, t + grid, ... (of ntr x kbl) as (row tile, column tile), advanced
  // without division
  const int step_r = static_cast<int>(gridDim.x) / kbl, step_c = static_cast<int>(gridDim.x) % kbl;
  int tr = static_cast<int>(blockIdx.x) / kbl, tc = static_cast<int>(blockIdx.x) % kbl;
  if (tr >= ntr) return;
  load(tr, tc, av, bv, rc);
  stage(av, bv);
  __syncthreads();
  while (true) {
    int nr = tr + step_r, nc = tc + step_c;
    if (nc >= kbl) {
      nc -= kbl;
      ++nr;
    }
    const bool more = nr < ntr;
    RowCodes nrc;
    if (more) load(nr, nc, av, bv, nrc);  // in flight during this tile's work
    {
      // the codes of the tile after that on their way to L2, so its register loads hit there
      int pr = nr + step_r, pc = nc + step_c;
      if (pc >= kbl) {
        pc -= kbl;
        ++pr;
      }
      const int64_t pn = static_cast<int64_t>(pr) * ROWS + rr, pk = static_cast<int64_t>(pc) * COLS + 64 * b;
      if (h == 0 && pr < ntr && pn < N && pk < K)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(codes + ((pn * K + pk) >> 1)));
    }
    merge_tile_mma<true>(sA, sB, sD, R16, BP, warp, lane);
    __syncthreads();
    const int64_t n0 = static_cast<int64_t>(tr) * ROWS, k0 = static_cast<int64_t>(tc) * COLS;
    merge_row_epilogue(rc, sD, mu, dq, fp8, scale, N, K, n0 + rr, k0 + 64 * b, rr, b, h, out16,
                       out32);
    if (!more) break;
    __syncthreads();  // every read of sA / sB / sD is done
    stage(av, bv);
    rc = nrc;
    tr = nr;
    tc = nc;
    __syncthreads();
  }
}

// ---------------------------------------------------------------- error statistics
constexpr int ES_THREADS = 256;

__global__ void __launch_bounds__(ES_THREADS) nf4_int4_error_kernel(
    const float* __restrict__ W, int64_t numel, double* __restrict__ part) {
  __shared__ double s_red[ES_THREADS / 32][3];
  // the levels in shared memory: a lane's level is one conflict-free load (16 words in 16
  // banks), where a per-lane index into a constant array is not
  __shared__ float s_L[16];
  {
    constexpr float L[16] = QLORA_NF4_LEVELS;
    if (threadIdx.x < 16) s_L[threadIdx.x] = L[threadIdx.x];
    __syncthreads();
  }
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
      const float en = __fsub_rn(w[i], __fmul_rn(s_L[nf4_code(x)], a));
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

// Resident CTAs per SM of the persistent merge (per instantiation, device and context).
template <int R16>
static int merge_resident(int* per_sm) {
  static DeviceCache<int> occupancy;
  const int st = occupancy.get(device_context_key, per_sm, [](int* v) -> int {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(v, merge::nf4_merge_persistent<R16>,
                                                      merge::THREADS,
                                                      merge::ROWS * merge::COLS * 4) !=
        cudaSuccess) {
      cudaGetLastError();
      return QLORA_ERR_CUDA;
    }
    if (*v < 1) *v = 1;
    return QLORA_OK;
  });
  return st == -1 ? QLORA_ERR_NO_DEVICE : st;
}

template <int R16>
static int launch_merge_persistent(const nf4_tensor& q, const uint16_t* A, const uint16_t* B,
                                   int r, float scale, uint16_t* out16, float* out32,
                                   cudaStream_t stream) {
  int per_sm = 0;
  const int st = merge_resident<R16>(&per_sm);
  if (st) return st;
  const int64_t kblocks = (q.cols + merge::COLS - 1) / merge::COLS;
  const int64_t rblocks = (q.rows + merge::ROWS - 1) / merge::ROWS;
  const int64_t ntiles = kblocks * rblocks;
  if (ntiles > INT32_MAX) return QLORA_ERR_UNSUPPORTED;
  const int64_t grid = std::min<int64_t>(ntiles, (int64_t)per_sm * num_sms());
  const int smem = merge::ROWS * merge::COLS * 4;  // the fp32 tile (32 KB)
  ProfileScope ps("nf4_merge", stream);
  merge::nf4_merge_persistent<R16><<<(unsigned)grid, merge::THREADS, smem, stream>>>(
      q.codes, q.scale_codes, q.scale_steps, q.scale_mean, q.dq_block != 0 ? 1 : 0,
      q.dq_type == NF4_DQ_FP8 ? 1 : 0, A, B, q.rows, q.cols, r, scale, out16, out32,
      static_cast<int>(rblocks), static_cast<int>(kblocks));
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

int launch_merge(const nf4_tensor& q, const uint16_t* A, const uint16_t* B, int r, float scale,
                 uint16_t* out16, float* out32, cudaStream_t stream) {
  // ranks up to 32 in whole 16-byte rows, rows of whole quantization blocks: the persistent form
  if (r % 8 == 0 && q.cols % 64 == 0) {
    if (r <= 16) return launch_merge_persistent<16>(q, A, B, r, scale, out16, out32, stream);
    if (r <= 32) return launch_merge_persistent<32>(q, A, B, r, scale, out16, out32, stream);
  }
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
