// skinny.cu -- the decode path: Y = X W'^T + s U B^T for M <= 16 tokens (junaidshaukat.com
// "QLoRA -- the democratization event": serve the 4-bit base plus a separate adapter;
// addaly.com "QLoRA on one card": keep the adapter separate and load it over the base).
// With so few tokens the layer is a stream over the packed weights: every weight byte is
// read once, dequantized in registers and consumed by the warp-level tensor cores with the
// tokens padded to 16 (mma.sync m16n8k16: tokens are the MMA rows, 8 weight rows the MMA
// columns).  Nothing of W' is written anywhere.
//
// Per warp: two groups of 8 weight rows.  Lane (g, q) = (lane/4, lane%4) owns weight row g of
// each group and, in every 256-wide k step, the 64-block q of that row -- so one byte table
// per block and per lane.  Inside an MMA the 16 contraction slots of lane class q map to the
// physical k of its own block (the contraction order is free as long as the X fragment uses
// the same map), which lets X come from shared memory as 16-byte loads.
// The k range is split over blockIdx.y; split partial sums go to the workspace and a second
// kernel adds them in a fixed order together with the LoRA term.
#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "profile.h"
#include "nf4_device.cuh"

namespace qlora {
namespace skinny {

constexpr int THREADS = 256;
constexpr int R = 2;                       // 8-row groups per warp
constexpr int ROWS_PER_CTA = 8 * R * (THREADS / 32);  // 128

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte chunk position of logical chunk `ch` of token row `row` in the X tile: xor by the
// 64-element window and the row so the 8 lanes of a quarter warp hit 8 distinct bank groups.
__device__ __forceinline__ int xchunk(int row, int ch) {
  return ch ^ ((2 * ((ch >> 3) & 3) + row) & 7);
}

struct Codes {
  uint4 c0, c1;
  float step;
  int q;
};

__global__ void __launch_bounds__(THREADS) nf4_decode_gemv(
    const uint16_t* __restrict__ X, int64_t M, int64_t N, int64_t K, const uint8_t* __restrict__ codes,
    const int8_t* __restrict__ qs, const float* __restrict__ steps, const float* __restrict__ mean,
    int64_t KS, float* __restrict__ part) {
  extern __shared__ __align__(16) uint4 xs[];  // [16][KS / 8] chunks
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int64_t k_begin = (int64_t)blockIdx.y * KS;
  const int64_t k_end = (k_begin + KS < K) ? k_begin + KS : K;
  const int cpr = static_cast<int>(KS / 8);  // chunks per token row

  // stage the tokens' k range (rows >= M and k >= K are zero)
  for (int i = tid; i < 16 * cpr; i += THREADS) {
    const int row = i / cpr, ch = i % cpr;
    const int64_t k = k_begin + (int64_t)ch * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < M && k < k_end) v = __ldg(reinterpret_cast<const uint4*>(X + row * K + k));
    xs[row * cpr + xchunk(row, ch)] = v;
  }
  __syncthreads();

  const float mu = __ldg(mean);
  const int64_t KB = K / 64;
  int64_t wrow[R];
#pragma unroll
  for (int rg = 0; rg < R; ++rg)
    wrow[rg] = (int64_t)blockIdx.x * ROWS_PER_CTA + warp * (8 * R) + rg * 8 + g;

  auto load_codes = [&](Codes (&c)[R], int64_t k0) {
    const int64_t kq = k0 + 64 * q;
#pragma unroll
    for (int rg = 0; rg < R; ++rg) {
      if (wrow[rg] < N && kq < k_end) {
        const uint4* src = reinterpret_cast<const uint4*>(codes + wrow[rg] * (K / 2) + kq / 2);
        c[rg].c0 = __ldg(src);
        c[rg].c1 = __ldg(src + 1);
        const int64_t b = wrow[rg] * KB + kq / 64;
        c[rg].q = __ldg(qs + b);
        c[rg].step = __ldg(steps + (b >> 8));
      } else {
        c[rg].c0 = c[rg].c1 = make_uint4(0, 0, 0, 0);
        c[rg].q = 0;
        c[rg].step = 0.f;
      }
    }
  };

  float acc[R][4];
#pragma unroll
  for (int rg = 0; rg < R; ++rg) acc[rg][0] = acc[rg][1] = acc[rg][2] = acc[rg][3] = 0.f;

  Codes cur[R], nxt[R];
  load_codes(cur, k_begin);
  for (int64_t k0 = k_begin; k0 < k_end; k0 += 256) {
    if (k0 + 256 < k_end) load_codes(nxt, k0 + 256);
    const bool kvalid = k0 + 64 * q < k_end;
    Nf4ByteTable tab[R];
#pragma unroll
    for (int rg = 0; rg < R; ++rg) {
      // invalid rows / k give a zero table -> zero weights
      const float sc = (wrow[rg] < N && kvalid) ? __fmaf_rn((float)cur[rg].q, cur[rg].step, mu) : 0.f;
      tab[rg] = nf4_make_table(sc);
    }
    const int chunk0 = static_cast<int>((k0 - k_begin) / 8) + 8 * q;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 xa = xs[g * cpr + xchunk(g, chunk0 + c)];
      const uint4 xb = xs[(g + 8) * cpr + xchunk(g + 8, chunk0 + c)];
#pragma unroll
      for (int rg = 0; rg < R; ++rg) {
        const uint32_t word = (c < 4) ? (&cur[rg].c0.x)[c] : (&cur[rg].c1.x)[c - 4];
        uint32_t w[4];
        nf4_dequant8(tab[rg], word, w);
        mma_bf16_16816(acc[rg], xa.x, xb.x, xa.y, xb.y, w[0], w[1]);
        mma_bf16_16816(acc[rg], xa.z, xb.z, xa.w, xb.w, w[2], w[3]);
      }
    }
#pragma unroll
    for (int rg = 0; rg < R; ++rg) cur[rg] = nxt[rg];
  }

  // acc[rg]: [0] token g / row 2q, [1] token g / row 2q+1, [2] token g+8 / 2q, [3] token g+8 / 2q+1
  float* out = part + (int64_t)blockIdx.y * M * N;
#pragma unroll
  for (int rg = 0; rg < R; ++rg) {
    const int64_t n = (int64_t)blockIdx.x * ROWS_PER_CTA + warp * (8 * R) + rg * 8 + 2 * q;
    if (n < N) {
      if (g < M) *reinterpret_cast<float2*>(out + g * N + n) = make_float2(acc[rg][0], acc[rg][1]);
      if (g + 8 < M)
        *reinterpret_cast<float2*>(out + (g + 8) * N + n) = make_float2(acc[rg][2], acc[rg][3]);
    }
  }
}

// Y[m][n] = bf16( sum_s part[s][m][n] + sum_j sU[m][j] B[n][j] ), splits in order.
__global__ void __launch_bounds__(256) decode_finalize(const float* __restrict__ part, int S,
                                                      int64_t M, int64_t N,
                                                      const uint16_t* __restrict__ sU,
                                                      const uint16_t* __restrict__ B, int r,
                                                      int64_t rp, uint16_t* __restrict__ Y) {
  extern __shared__ float su[];  // [M][r]
  for (int i = threadIdx.x; i < M * r; i += blockDim.x) {
    const int m = i / r, j = i % r;
    su[i] = __bfloat162float(__ushort_as_bfloat16(sU[m * rp + j]));
  }
  __syncthreads();
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  for (int64_t m = 0; m < M; ++m) {
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += part[((int64_t)s * M + m) * N + n];
    float l = 0.f;
    for (int j = 0; j < r; ++j)
      l = fmaf(su[m * r + j], __bfloat162float(__ushort_as_bfloat16(B[n * r + j])), l);
    Y[m * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v + l));
  }
}

}  // namespace skinny

namespace {

int64_t skinny_ks(int64_t N, int64_t K) {
  // k range per split: a multiple of 256 giving ~3 CTA waves, and at most 2048 (64 KB of X)
  const int64_t row_blocks = (N + skinny::ROWS_PER_CTA - 1) / skinny::ROWS_PER_CTA;
  const int64_t steps = (K + 255) / 256;
  const int64_t want = 3LL * num_sms();
  int64_t splits = (want + row_blocks - 1) / row_blocks;
  if (splits < 1) splits = 1;
  if (splits > steps) splits = steps;
  int64_t per = (steps + splits - 1) / splits;
  if (per > 8) per = 8;
  return per * 256;
}

}  // namespace

uint64_t skinny_partial_bytes(int64_t M, int64_t N, int64_t K) {
  if (M > kSkinnyMaxM) return 0;
  const int64_t ks = skinny_ks(N, K);
  const int64_t S = (K + ks - 1) / ks;
  return (uint64_t)S * M * N * 4;
}

int launch_skinny_fwd(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int64_t ks = skinny_ks(a.N, a.K);
  const int64_t S = (a.K + ks - 1) / ks;
  float* part = reinterpret_cast<float*>(ws + L.part);
  const int smem = static_cast<int>(16 * ks * 2);
  static bool attr = false;  // once: the largest X tile (2048 columns of 16 tokens)
  if (!attr) {
    if (cudaFuncSetAttribute(skinny::nf4_decode_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             16 * 2048 * 2) != cudaSuccess)
      return QLORA_ERR_CUDA;
    attr = true;
  }
  dim3 grid((unsigned)((a.N + skinny::ROWS_PER_CTA - 1) / skinny::ROWS_PER_CTA), (unsigned)S);
  {
  ProfileScope ps("decode_gemv", stream);
  skinny::nf4_decode_gemv<<<grid, skinny::THREADS, smem, stream>>>(
      a.X, a.M, a.N, a.K, a.q.codes, a.q.scale_codes, a.q.scale_steps, a.q.scale_mean, ks, part);
  }
  if (cudaGetLastError() != cudaSuccess) return QLORA_ERR_CUDA;
  ProfileScope ps("decode_finalize", stream);
  const int fsmem = static_cast<int>(a.M * a.r * 4);
  skinny::decode_finalize<<<(unsigned)((a.N + 255) / 256), 256, fsmem, stream>>>(
      part, (int)S, a.M, a.N, reinterpret_cast<const uint16_t*>(ws + L.sU),
      a.B, a.r, L.rp, a.Y);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
