// lora_side.cu -- the rank-r side products of the LoRA branch (junaidshaukat.com recipe
// item 2: adapters kept in 16 bit; item 3: gradients flow into the adapters):
//   U  = X  A^T      [M, r]   forward, rows m, contraction over K
//   V  = dY B        [M, r]   backward, rows m, contraction over N  (B transposed to [r, N])
//   dB = s dY^T U    [N, r]   backward, rows n, contraction over M  (dY read column-wise)
//   dA^T = X^T sV    [K, r]   backward, rows k, contraction over M  (X read column-wise)
// Each is a tall-skinny product: one big operand read once from HBM, the other (rank r)
// tiny.  They run on the warp-level tensor-core path (mma.sync m16n8k16, bf16 in, fp32
// accumulate) fed by cp.async double buffering and ldmatrix (.trans for the column-wise
// operand), split over the contraction for occupancy.  The split partial sums are combined
// in a fixed order by the finalize kernels, so results are bit-reproducible.
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "profile.h"

namespace qlora {
namespace side {

constexpr int TR = 64;   // rows per CTA
constexpr int TC = 64;   // contraction per stage
constexpr int THREADS = 128;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = smem_u32(smem);
  const int n = valid ? 16 : 0;  // src-size 0 zero-fills the 16 bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Element offset of 16-byte chunk `ch` (0..7) of row `row` in a [rows][64] bf16 tile whose
// chunks are xor-swizzled by row (conflict-free ldmatrix).
__device__ __forceinline__ int swz(int row, int ch) { return row * 64 + ((ch ^ (row & 7)) << 3); }

// part[split][R][NJ] = sum over the split's contraction range of P(row, c) * Q[j][c].
// P: K-major (P[row * ldp + c]) or, with kPColumn, column-wise (P[c * ldp + row]).
// Q: [NJ rows][ldq] bf16, zero rows past the rank, columns valid up to round_up(C, 64).
template <bool kPColumn, int NJ>
__global__ void __launch_bounds__(THREADS) side_gemm(const uint16_t* __restrict__ P, int64_t R,
                                                     int64_t C, int64_t ldp,
                                                     const uint16_t* __restrict__ Q, int64_t ldq,
                                                     float* __restrict__ part, int64_t chunk) {
  extern __shared__ __align__(128) uint16_t sm[];
  uint16_t* sP = sm;                    // [2][64 * 64]
  uint16_t* sQ = sm + 2 * TR * TC;      // [2][NJ * 64]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r0 = (int64_t)blockIdx.x * TR;
  const int64_t c_begin = (int64_t)blockIdx.y * chunk;
  const int64_t c_pad = (C + TC - 1) / TC * TC;
  const int64_t c_end = (c_begin + chunk < c_pad) ? c_begin + chunk : c_pad;
  const int nstages = c_end > c_begin ? (int)((c_end - c_begin) / TC) : 0;

  auto load_stage = [&](int st, int buf) {
    const int64_t c0 = c_begin + (int64_t)st * TC;
    uint16_t* dP = sP + buf * TR * TC;
    uint16_t* dQ = sQ + buf * NJ * TC;
#pragma unroll
    for (int i = tid; i < TR * 8; i += THREADS) {
      const int a = i >> 3, ch = i & 7;
      if (!kPColumn) {  // a = row, chunk along c
        const int64_t row = r0 + a;
        const bool v = row < R;
        cp_async16(dP + swz(a, ch), P + (v ? row : 0) * ldp + c0 + ch * 8, v);
      } else {  // a = c, chunk along rows
        const int64_t c = c0 + a;
        const bool v = (c < C) && (r0 + ch * 8 < R);
        cp_async16(dP + swz(a, ch), P + (v ? c : 0) * ldp + (v ? r0 + ch * 8 : 0), v);
      }
    }
#pragma unroll
    for (int i = tid; i < NJ * 8; i += THREADS) {
      const int j = i >> 3, ch = i & 7;
      cp_async16(dQ + swz(j, ch), Q + (int64_t)j * ldq + c0 + ch * 8, true);
    }
  };

  float acc[NJ / 8][4];
#pragma unroll
  for (int t = 0; t < NJ / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  if (nstages > 0) load_stage(0, 0);
  cp_async_commit();
  for (int st = 0; st < nstages; ++st) {
    if (st + 1 < nstages) load_stage(st + 1, (st + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint16_t* tP = sP + (st & 1) * TR * TC;
    const uint16_t* tQ = sQ + (st & 1) * NJ * TC;
#pragma unroll
    for (int kk = 0; kk < TC / 16; ++kk) {
      uint32_t a[4];
      if (!kPColumn) {
        const int row = warp * 16 + (lane & 15);
        ldsm_x4(smem_u32(tP + swz(row, kk * 2 + (lane >> 4))), a);
      } else {
        const int i = lane >> 3, rr = lane & 7;
        const int c = kk * 16 + rr + 8 * (i >> 1);
        ldsm_x4_t(smem_u32(tP + swz(c, warp * 2 + (i & 1))), a);
      }
#pragma unroll
      for (int t = 0; t < NJ / 8; ++t) {
        uint32_t b[2];
        const int j = t * 8 + (lane & 7);
        ldsm_x2(smem_u32(tQ + swz(j, kk * 2 + ((lane >> 3) & 1))), b);
        mma_bf16_16816(acc[t], a, b);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  const int g = lane >> 2, q = lane & 3;
  float* out = part + (int64_t)blockIdx.y * R * NJ;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t row = r0 + warp * 16 + g + 8 * h;
    if (row < R) {
#pragma unroll
      for (int t = 0; t < NJ / 8; ++t)
        *reinterpret_cast<float2*>(out + row * NJ + t * 8 + 2 * q) =
            make_float2(acc[t][2 * h], acc[t][2 * h + 1]);
    }
  }
}

// ---------------------------------------------------------------- finalize kernels
// U / V rows: sum the splits in order; write fp32 (optional, pitch ldo), bf16(scale * x) into
// the [M, rp] operand buffer (zero past r) and bf16(scale_t * x) into the transposed
// [rp, Mp] buffer (zero past r and past M).
__global__ void finalize_rows(const float* __restrict__ part, int S, int64_t M, int NJ, int r,
                              int64_t rp, int64_t Mp, float* __restrict__ out32, int64_t ldo,
                              uint16_t* __restrict__ op, float op_scale,
                              uint16_t* __restrict__ opt, float opt_scale) {
  const int64_t total = Mp * rp;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = i / Mp, m = i % Mp;  // m fastest: coalesced transposed writes
    float v = 0.f;
    if (m < M && j < r) {
      for (int s = 0; s < S; ++s) v += part[((int64_t)s * M + m) * NJ + j];
    }
    if (opt) opt[j * Mp + m] = __bfloat16_as_ushort(__float2bfloat16_rn(v * opt_scale));
    if (m < M) {
      if (op) op[m * rp + j] = __bfloat16_as_ushort(__float2bfloat16_rn(v * op_scale));
      if (out32 && j < r) out32[m * ldo + j] = v;
    }
  }
}

// Adapter gradient from row partials: out[j * ld_j + row * ld_row] = scale * sum_s part.
__global__ void finalize_grad(const float* __restrict__ part, int S, int64_t R, int NJ, int r,
                              float scale, float* __restrict__ out, int64_t ld_row,
                              int64_t ld_j) {
  const int64_t total = R * r;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    int64_t row, j;
    if (ld_row == 1) { j = i / R; row = i % R; }   // transposed output: row fastest
    else { row = i / r; j = i % r; }
    float v = 0.f;
    for (int s = 0; s < S; ++s) v += part[((int64_t)s * R + row) * NJ + j];
    out[j * ld_j + row * ld_row] = v * scale;
  }
}

// Zero-padded / transposed adapter copies: Bp [N, rp], Bt [rp, N], Ap [rp, K].
__global__ void pad_adapters(const uint16_t* __restrict__ A, const uint16_t* __restrict__ B,
                             int64_t N, int64_t K, int r, int64_t rp, uint16_t* __restrict__ Bp,
                             uint16_t* __restrict__ Bt, uint16_t* __restrict__ Ap) {
  const int64_t nB = N * rp, nA = rp * K;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nB + nA;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nB) {
      const int64_t n = i / rp, j = i % rp;
      const uint16_t v = j < r ? B[n * r + j] : 0;
      Bp[i] = v;
      if (Bt) Bt[j * N + n] = v;
    } else {
      const int64_t t = i - nB, j = t / K;
      Ap[t] = j < r ? A[t] : 0;
    }
  }
}

}  // namespace side

// ---------------------------------------------------------------- host side
namespace {

int pick_nj(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : r <= 64 ? 64 : 128; }

// Splits of the contraction (multiples of 64) so the grid covers ~3 waves of CTAs.
int64_t pick_chunk(int64_t rows, int64_t C) {
  const int64_t row_tiles = (rows + side::TR - 1) / side::TR;
  const int64_t c_tiles = (C + side::TC - 1) / side::TC;
  const int64_t want = 3LL * num_sms();
  int64_t splits = std::max<int64_t>(1, std::min<int64_t>(c_tiles, (want + row_tiles - 1) / row_tiles));
  const int64_t per = (c_tiles + splits - 1) / splits;
  return per * side::TC;
}

template <bool kCol>
int run_side(const char* name, const uint16_t* P, int64_t R, int64_t C, int64_t ldp,
             const uint16_t* Q, int64_t ldq, int NJ, float* part, int64_t chunk,
             cudaStream_t stream) {
  ProfileScope ps(name, stream);
  const int64_t c_pad = (C + side::TC - 1) / side::TC * side::TC;
  dim3 grid((unsigned)((R + side::TR - 1) / side::TR), (unsigned)((c_pad + chunk - 1) / chunk));
  const int smem = 2 * (side::TR * side::TC + NJ * side::TC) * 2;
  switch (NJ) {
#define QLORA_SIDE_CASE(nj)                                                                     \
  case nj:                                                                                      \
    cudaFuncSetAttribute(side::side_gemm<kCol, nj>, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                         smem);                                                                 \
    side::side_gemm<kCol, nj><<<grid, side::THREADS, smem, stream>>>(P, R, C, ldp, Q, ldq, part,  \
                                                                     chunk);                    \
    break;
    QLORA_SIDE_CASE(16)
    QLORA_SIDE_CASE(32)
    QLORA_SIDE_CASE(64)
    QLORA_SIDE_CASE(128)
#undef QLORA_SIDE_CASE
    default: return QLORA_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

int splits_of(int64_t C, int64_t chunk) {
  const int64_t c_pad = (C + side::TC - 1) / side::TC * side::TC;
  return (int)((c_pad + chunk - 1) / chunk);
}

unsigned grid_for(int64_t n) {
  int64_t b = (n + 255) / 256;
  const int64_t cap = 8LL * num_sms();
  return (unsigned)std::max<int64_t>(1, std::min(b, cap));
}

}  // namespace

uint64_t side_partial_bytes(int64_t M, int64_t N, int64_t K, int r) {
  const int NJ = pick_nj(r);
  uint64_t worst = 0;
  auto upd = [&](int64_t rows, int64_t C) {
    const int64_t chunk = pick_chunk(rows, C);
    worst = std::max<uint64_t>(worst, (uint64_t)splits_of(C, chunk) * rows * NJ * 4);
  };
  upd(M, K);  // U
  upd(M, N);  // V
  upd(N, M);  // dB
  upd(K, M);  // dA^T
  return worst;
}

int launch_pad_adapters(const LinearArgs& a, const WorkspaceLayout& L, bool need_bt,
                        cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  ProfileScope ps("pad_adapters", stream);
  side::pad_adapters<<<grid_for(a.N * L.rp + L.rp * a.K), 256, 0, stream>>>(
      a.A, a.B, a.N, a.K, a.r, L.rp, reinterpret_cast<uint16_t*>(ws + L.Bp),
      need_bt ? reinterpret_cast<uint16_t*>(ws + L.Bt) : nullptr,
      reinterpret_cast<uint16_t*>(ws + L.Ap));
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

// U = X A^T -> sU = bf16(scale U) [M, rp], and U fp32 [M, r] when the caller keeps it.
int launch_lora_u(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int NJ = pick_nj(a.r);
  float* part = reinterpret_cast<float*>(ws + L.part);
  const int64_t chunk = pick_chunk(a.M, a.K);
  int st = run_side<false>("side_u", a.X, a.M, a.K, a.K, reinterpret_cast<const uint16_t*>(ws + L.Ap), a.K,
                           NJ, part, chunk, stream);
  if (st) return st;
  const int64_t Mp = round_up(a.M, 64);
  ProfileScope ps("finalize_rows", stream);
  side::finalize_rows<<<grid_for(Mp * L.rp), 256, 0, stream>>>(
      part, splits_of(a.K, chunk), a.M, NJ, a.r, L.rp, Mp, a.U, a.r,
      reinterpret_cast<uint16_t*>(ws + L.sU), a.scale, nullptr, 0.f);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

// Backward with a saved U: Ut = bf16(U) transposed (for dB).
__global__ void ut_from_saved(const float* __restrict__ U, int64_t M, int r, int64_t rp, int64_t Mp,
                              uint16_t* __restrict__ Ut) {
  const int64_t total = rp * Mp;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j = i / Mp, m = i % Mp;
    const float v = (m < M && j < r) ? U[m * r + j] : 0.f;
    Ut[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
  }
}

int launch_u_from_saved(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int64_t Mp = round_up(a.M, 64);
  if (a.U_in) {
    ProfileScope ps("ut_from_saved", stream);
    ut_from_saved<<<grid_for(L.rp * Mp), 256, 0, stream>>>(a.U_in, a.M, a.r, L.rp, Mp,
                                                           reinterpret_cast<uint16_t*>(ws + L.Ut));
    return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
  }
  // recompute U = X A^T straight into the transposed bf16 buffer
  const int NJ = pick_nj(a.r);
  float* part = reinterpret_cast<float*>(ws + L.part);
  const int64_t chunk = pick_chunk(a.M, a.K);
  int st = run_side<false>("side_u", a.X, a.M, a.K, a.K, reinterpret_cast<const uint16_t*>(ws + L.Ap),
                           a.K, NJ, part, chunk, stream);
  if (st) return st;
  ProfileScope ps("finalize_rows", stream);
  side::finalize_rows<<<grid_for(Mp * L.rp), 256, 0, stream>>>(
      part, splits_of(a.K, chunk), a.M, NJ, a.r, L.rp, Mp, nullptr, 0, nullptr, 0.f,
      reinterpret_cast<uint16_t*>(ws + L.Ut), 1.0f);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

// V = dY B -> sV = bf16(scale V) [M, rp] and its transpose [rp, Mp].
int launch_lora_v(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int NJ = pick_nj(a.r);
  float* part = reinterpret_cast<float*>(ws + L.part);
  const int64_t chunk = pick_chunk(a.M, a.N);
  int st = run_side<false>("side_v", a.dY, a.M, a.N, a.N, reinterpret_cast<const uint16_t*>(ws + L.Bt),
                           a.N, NJ, part, chunk, stream);
  if (st) return st;
  const int64_t Mp = round_up(a.M, 64);
  ProfileScope ps("finalize_rows", stream);
  side::finalize_rows<<<grid_for(Mp * L.rp), 256, 0, stream>>>(
      part, splits_of(a.N, chunk), a.M, NJ, a.r, L.rp, Mp, nullptr, 0,
      reinterpret_cast<uint16_t*>(ws + L.sV), a.scale, reinterpret_cast<uint16_t*>(ws + L.Vt),
      a.scale);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

// dB = scale * dY^T U  (rows n, contraction over m; dY read column-wise).
int launch_lora_db(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int NJ = pick_nj(a.r);
  float* part = reinterpret_cast<float*>(ws + L.part);
  const int64_t chunk = pick_chunk(a.N, a.M);
  const int64_t Mp = round_up(a.M, 64);
  int st = run_side<true>("side_db", a.dY, a.N, a.M, a.N, reinterpret_cast<const uint16_t*>(ws + L.Ut),
                          Mp, NJ, part, chunk, stream);
  if (st) return st;
  ProfileScope ps("finalize_grad", stream);
  side::finalize_grad<<<grid_for(a.N * a.r), 256, 0, stream>>>(part, splits_of(a.M, chunk), a.N, NJ,
                                                               a.r, a.scale, a.dB, a.r, 1);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

// dA = (X^T sV)^T  (rows k, contraction over m; X read column-wise; sV already scaled).
int launch_lora_da(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int NJ = pick_nj(a.r);
  float* part = reinterpret_cast<float*>(ws + L.part);
  const int64_t chunk = pick_chunk(a.K, a.M);
  const int64_t Mp = round_up(a.M, 64);
  int st = run_side<true>("side_da", a.X, a.K, a.M, a.K, reinterpret_cast<const uint16_t*>(ws + L.Vt),
                          Mp, NJ, part, chunk, stream);
  if (st) return st;
  ProfileScope ps("finalize_grad", stream);
  side::finalize_grad<<<grid_for(a.K * a.r), 256, 0, stream>>>(part, splits_of(a.M, chunk), a.K, NJ,
                                                               a.r, 1.0f, a.dA, 1, a.K);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
