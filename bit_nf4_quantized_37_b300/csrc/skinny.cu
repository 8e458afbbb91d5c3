// skinny.cu -- the decode path: Y = X W'^T + s U B^T for M <= 16 tokens (junaidshaukat.com
// "QLoRA -- the democratization event": serve the 4-bit base plus a separate adapter;
// addaly.com "QLoRA on one card": keep the adapter separate and load it over the base).
// With so few tokens the layer is a stream over the packed weights: every weight byte is
// read once, dequantized in registers and consumed by the warp-level tensor cores with the
// tokens padded to 16 (mma.sync m16n8k16: tokens are the MMA rows, 8 weight rows the MMA
// columns).  Nothing of W' is written anywhere.
//
// nf4_decode_gemv: a CTA owns 128 weight rows and a k range.  One thread streams the packed
// codes with TMA ([128 rows x 256 k] per stage, 128-byte swizzle, 4 stages in flight); every
// warp dequantizes two 8-row groups: lane (g, q) = (lane/4, lane%4) owns weight row g of each
// group and, per 256-wide stage, the 64-block q of that row -- one byte table per block and
// lane.  Inside an MMA the 16 contraction slots of lane class q map to the physical k of its
// own block (the contraction order is free as long as the X fragment uses the same map), so
// X comes from shared memory as 16-byte loads.  The k ranges of a row block are summed, in
// a fixed order, by the CTA that finishes last (atomic ticket), which also adds the LoRA
// term s U B^T and writes Y.
#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "nf4_device.cuh"
#include "profile.h"

namespace qlora {

// Device error word of the decode kernel (bounded waits that gave up).
__device__ int g_decode_error = 0;

int read_and_clear_decode_error(int* out) {
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_decode_error, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_decode_error, &zero, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  *out = v;
  return QLORA_OK;
}

namespace skinny {

constexpr int THREADS = 256;
constexpr int R = 2;                                 // 8-row groups per warp
constexpr int ROWS = 8 * R * (THREADS / 32);         // 128 weight rows per CTA
constexpr int KSTEP = 256;                           // k per stage
constexpr int STAGE_BYTES = ROWS * KSTEP / 2;        // 16 KB of packed codes
constexpr int STAGES = 4;
constexpr int KS_MAX = 1024;                         // k range per CTA (X tile <= 32 KB)
constexpr int X_BYTES = 16 * KS_MAX * 2;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + X_BYTES + 1024;

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

struct Params {
  const uint16_t* X;
  int64_t M, N, K;
  const int8_t* qs;
  const float* steps;
  const float* mean;
  int64_t KS;       // k range per CTA (multiple of 256)
  int S;            // k ranges per row block
  float* part;      // [S][M][N]
  int* tickets;     // [row blocks]
  const uint16_t* sU;  // [M][rp] bf16, scale * U
  int64_t rp;
  const uint16_t* B;   // [N][r]
  int r;
  uint16_t* Y;
};

__global__ void __launch_bounds__(THREADS, 2)
    nf4_decode_gemv(const __grid_constant__ CUtensorMap tmCodes, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sC = smem;                                               // STAGES x [128 rows][128 B]
  uint4* xs = reinterpret_cast<uint4*>(smem + STAGES * STAGE_BYTES);  // [16][KS / 8] chunks
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ int abort_flag, s_last;
  volatile int* abort_p = &abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, q = lane & 3;
  const int64_t n0 = (int64_t)blockIdx.x * ROWS;
  const int64_t k_begin = (int64_t)blockIdx.y * p.KS;
  const int64_t k_end = (k_begin + p.KS < p.K) ? k_begin + p.KS : p.K;
  const int nst = static_cast<int>((k_end - k_begin + KSTEP - 1) / KSTEP);
  const int cpr = static_cast<int>(p.KS / 8);  // X chunks per token row

  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) mbar_init(&full_bar[i], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  auto issue = [&](int st) {
    const int slot = st % STAGES;
    mbar_arrive_expect_tx(&full_bar[slot], STAGE_BYTES);
    tma_load_2d(sC + slot * STAGE_BYTES, &tmCodes, &full_bar[slot],
                static_cast<int32_t>((k_begin + (int64_t)st * KSTEP) / 2), static_cast<int32_t>(n0));
  };
  if (tid == 0) {
    tma_prefetch_desc(&tmCodes);
    for (int st = 0; st < STAGES && st < nst; ++st) issue(st);
  }
  // the tokens' k range (rows >= M and k >= K are zero)
  for (int i = tid; i < 16 * cpr; i += THREADS) {
    const int row = i / cpr, ch = i % cpr;
    const int64_t k = k_begin + (int64_t)ch * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < p.M && k < k_end) v = __ldg(reinterpret_cast<const uint4*>(p.X + row * p.K + k));
    xs[row * cpr + xchunk(row, ch)] = v;
  }
  __syncthreads();

  const float mu = __ldg(p.mean);
  const int64_t KB = p.K / 64;
  int lrow[R];
  int64_t wrow[R];
#pragma unroll
  for (int rg = 0; rg < R; ++rg) {
    lrow[rg] = warp * (8 * R) + rg * 8 + g;
    wrow[rg] = n0 + lrow[rg];
  }
  auto scale_of = [&](int rg, int st) -> float {
    const int64_t kq = k_begin + (int64_t)st * KSTEP + 64 * q;
    if (wrow[rg] >= p.N || kq >= k_end) return 0.f;  // zero table -> zero weights
    const int64_t b = wrow[rg] * KB + kq / 64;
    return __fmaf_rn((float)__ldg(p.qs + b), __ldg(p.steps + (b >> 8)), mu);
  };
  float sc_next[R];
#pragma unroll
  for (int rg = 0; rg < R; ++rg) sc_next[rg] = scale_of(rg, 0);

  float acc[R][4];
#pragma unroll
  for (int rg = 0; rg < R; ++rg) acc[rg][0] = acc[rg][1] = acc[rg][2] = acc[rg][3] = 0.f;

  bool ok = true;
  for (int st = 0; st < nst; ++st) {
    float sc[R];
#pragma unroll
    for (int rg = 0; rg < R; ++rg) sc[rg] = sc_next[rg];
    if (st + 1 < nst) {
#pragma unroll
      for (int rg = 0; rg < R; ++rg) sc_next[rg] = scale_of(rg, st + 1);
    }
    if (!mbar_wait(&full_bar[st % STAGES], (st / STAGES) & 1, kWaitTmaFull, abort_p,
                   &g_decode_error)) {
      ok = false;
      break;
    }
    const uint8_t* cs = sC + (st % STAGES) * STAGE_BYTES;
    Nf4ByteTable tab[R];
    uint4 cw[R][2];
#pragma unroll
    for (int rg = 0; rg < R; ++rg) {
      tab[rg] = nf4_make_table(sc[rg]);
      const int row = lrow[rg];
#pragma unroll
      for (int h = 0; h < 2; ++h)
        cw[rg][h] = *reinterpret_cast<const uint4*>(cs + row * 128 + (((2 * q + h) ^ (row & 7)) << 4));
    }
    const int chunk0 = static_cast<int>((int64_t)st * KSTEP / 8) + 8 * q;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 xa = xs[g * cpr + xchunk(g, chunk0 + c)];
      const uint4 xb = xs[(g + 8) * cpr + xchunk(g + 8, chunk0 + c)];
#pragma unroll
      for (int rg = 0; rg < R; ++rg) {
        const uint4& v = cw[rg][c >> 2];
        const uint32_t word = (c & 3) == 0 ? v.x : (c & 3) == 1 ? v.y : (c & 3) == 2 ? v.z : v.w;
        uint32_t w[4];
        nf4_dequant8(tab[rg], word, w);
        mma_bf16_16816(acc[rg], xa.x, xb.x, xa.y, xb.y, w[0], w[1]);
        mma_bf16_16816(acc[rg], xa.z, xb.z, xa.w, xb.w, w[2], w[3]);
      }
    }
    __syncthreads();  // every warp is done with this stage's buffer
    if (tid == 0 && st + STAGES < nst) {
      fence_proxy_async_smem();
      issue(st + STAGES);
    }
  }
  if (!ok) {
    __syncthreads();
    if (tid == 0)  // never release shared memory with a copy still landing in it
      for (int st = 0; st < nst && st < STAGES; ++st) mbar_drain(&full_bar[st], 0);
    return;
  }

  // acc[rg]: [0] token g / row 2q, [1] token g / row 2q+1, [2] token g+8 / 2q, [3] token g+8 / 2q+1
  float* mine = p.part + (int64_t)blockIdx.y * p.M * p.N;
#pragma unroll
  for (int rg = 0; rg < R; ++rg) {
    const int64_t n = n0 + warp * (8 * R) + rg * 8 + 2 * q;
    if (n < p.N) {
      if (g < p.M) __stcg(reinterpret_cast<float2*>(mine + g * p.N + n), make_float2(acc[rg][0], acc[rg][1]));
      if (g + 8 < p.M)
        __stcg(reinterpret_cast<float2*>(mine + (g + 8) * p.N + n), make_float2(acc[rg][2], acc[rg][3]));
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&p.tickets[blockIdx.x], 1) == p.S - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // Last CTA of this row block: sum the k ranges in order, add s U B^T, write Y (bf16).
  // B rows and sU are staged in the (now idle) code buffers.
  const int r = p.r;
  const int bp = r + 1;  // odd pitch in floats: conflict-free row reads
  float* sB = reinterpret_cast<float*>(sC);                // [128][r + 1]
  float* sUf = sB + ROWS * bp;                             // [M][r]
  for (int i = tid; i < ROWS * r; i += THREADS) {
    const int rr = i / r, j = i % r;
    const int64_t n = n0 + rr;
    sB[rr * bp + j] = n < p.N ? __bfloat162float(__ushort_as_bfloat16(p.B[n * r + j])) : 0.f;
  }
  for (int i = tid; i < p.M * r; i += THREADS) {
    const int m = i / r, j = i % r;
    sUf[i] = __bfloat162float(__ushort_as_bfloat16(p.sU[m * p.rp + j]));
  }
  __syncthreads();
  const int nl = tid % ROWS, half = tid / ROWS;  // 2 threads per row, tokens split in halves
  const int64_t n = n0 + nl;
  if (n < p.N) {
    for (int m = half; m < p.M; m += 2) {
      float v = 0.f;
      const float* src = p.part + m * p.N + n;
      int s = 0;
      for (; s + 4 <= p.S; s += 4) {
        const float a0 = __ldcg(src + (int64_t)(s + 0) * p.M * p.N);
        const float a1 = __ldcg(src + (int64_t)(s + 1) * p.M * p.N);
        const float a2 = __ldcg(src + (int64_t)(s + 2) * p.M * p.N);
        const float a3 = __ldcg(src + (int64_t)(s + 3) * p.M * p.N);
        v += a0; v += a1; v += a2; v += a3;
      }
      for (; s < p.S; ++s) v += __ldcg(src + (int64_t)s * p.M * p.N);
      float l = 0.f;
      for (int j = 0; j < r; ++j) l = fmaf(sUf[m * r + j], sB[nl * bp + j], l);
      p.Y[m * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v + l));
    }
  }
  if (tid == 0) p.tickets[blockIdx.x] = 0;  // ready for the next launch
}

// U = X A^T for a few tokens: one CTA per adapter row j (and zero columns r .. rp-1 of sU).
__global__ void __launch_bounds__(256) small_u(const uint16_t* __restrict__ X, int64_t M, int64_t K,
                                               const uint16_t* __restrict__ A, int r, int64_t rp,
                                               float scale, uint16_t* __restrict__ sU,
                                               float* __restrict__ U_out) {
  __shared__ float red[8][16];
  const int j = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (j >= r) {
    for (int m = tid; m < M; m += blockDim.x) sU[m * rp + j] = 0;
    return;
  }
  float acc[16];
#pragma unroll
  for (int m = 0; m < 16; ++m) acc[m] = 0.f;
  for (int64_t k = (int64_t)tid * 8; k < K; k += (int64_t)blockDim.x * 8) {
    const uint4 av = __ldg(reinterpret_cast<const uint4*>(A + (int64_t)j * K + k));
    const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
    float af[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      af[2 * e] = __uint_as_float(aw[e] << 16);
      af[2 * e + 1] = __uint_as_float(aw[e] & 0xFFFF0000u);
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      if (m < M) {
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(X + (int64_t)m * K + k));
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[m] = fmaf(__uint_as_float(xw[e] << 16), af[2 * e], acc[m]);
          acc[m] = fmaf(__uint_as_float(xw[e] & 0xFFFF0000u), af[2 * e + 1], acc[m]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < 16; ++m) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
  }
  if (lane == 0) {
#pragma unroll
    for (int m = 0; m < 16; ++m) red[warp][m] = acc[m];
  }
  __syncthreads();
  if (tid < M) {
    float u = 0.f;
    for (int w = 0; w < 8; ++w) u += red[w][tid];
    sU[tid * rp + j] = __bfloat16_as_ushort(__float2bfloat16_rn(u * scale));
    if (U_out) U_out[tid * r + j] = u;
  }
}

}  // namespace skinny

namespace {

int64_t skinny_ks(int64_t N, int64_t K) {
  // k range per CTA: a multiple of 256, at most 1024, small enough for ~2 CTAs per SM
  const int64_t row_blocks = (N + skinny::ROWS - 1) / skinny::ROWS;
  int64_t want = (2LL * num_sms() + row_blocks - 1) / row_blocks;
  if (want < 1) want = 1;
  int64_t ks = (K + want - 1) / want;
  ks = (ks + skinny::KSTEP - 1) / skinny::KSTEP * skinny::KSTEP;
  if (ks > skinny::KS_MAX) ks = skinny::KS_MAX;
  if (ks < skinny::KSTEP) ks = skinny::KSTEP;
  return ks;
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
  uint16_t* sU = reinterpret_cast<uint16_t*>(ws + L.sU);
  {
    ProfileScope ps("decode_u", stream);
    skinny::small_u<<<(unsigned)L.rp, 256, 0, stream>>>(a.X, a.M, a.K, a.A, a.r, L.rp, a.scale, sU,
                                                        a.U);
    if (cudaGetLastError() != cudaSuccess) return QLORA_ERR_CUDA;
  }
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(skinny::nf4_decode_gemv, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             skinny::SMEM_BYTES) != cudaSuccess)
      return QLORA_ERR_CUDA;
    attr = true;
  }
  CUtensorMap tm;
  if (!make_tensor_map_2d(&tm, a.q.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)(a.K / 2),
                          (uint64_t)a.N, (uint64_t)(a.K / 2), 128, skinny::ROWS, MapSwizzle::B128))
    return QLORA_ERR_CUDA;
  skinny::Params p{};
  p.X = a.X;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.qs = a.q.scale_codes;
  p.steps = a.q.scale_steps;
  p.mean = a.q.scale_mean;
  p.KS = skinny_ks(a.N, a.K);
  p.S = (int)((a.K + p.KS - 1) / p.KS);
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.tickets = reinterpret_cast<int*>(ws + L.tickets);
  p.sU = sU;
  p.rp = L.rp;
  p.B = a.B;
  p.r = a.r;
  p.Y = a.Y;
  dim3 grid((unsigned)((a.N + skinny::ROWS - 1) / skinny::ROWS), (unsigned)p.S);
  ProfileScope ps("decode_gemv", stream);
  skinny::nf4_decode_gemv<<<grid, skinny::THREADS, skinny::SMEM_BYTES, stream>>>(tm, p);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
