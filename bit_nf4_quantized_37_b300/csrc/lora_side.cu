// lora_side.cu -- the rank-r side products of the LoRA branch (junaidshaukat.com recipe
// item 2: adapters kept in 16 bit; item 3: gradients flow into the adapters):
//   U    = X A^T        [M, r]  forward      rows m, contraction over K (X row-major)
//   V    = dY B         [M, r]  backward     rows m, contraction over N (dY row-major)
//   dB   = s dY^T U     [N, r]  backward     rows n, contraction over M (dY read by columns)
//   dA^T = X^T sV       [K, r]  backward     rows k, contraction over M (X read by columns)
// Each is tall and skinny: one big operand P read once from HBM, one rank-r operand Q that
// fits in shared memory.  One kernel serves all four: P streams through a 4-stage TMA
// ring of 128 x 64 tiles (two CTAs per SM) into the warp-level tensor cores (mma.sync m16n8k16, bf16 in, fp32
// accumulate; fp16 in the fp16 compute type; ldmatrix.trans reads the column-wise P), Q is
// staged once per CTA for its whole contraction range (converted to the 16-bit type on the
// way, zero past the rank), and the contraction
// is split over blockIdx.y.  The CTA that finishes a row tile last (atomic ticket) adds the
// split partial sums in split order and writes the outputs -- so results are
// bit-reproducible and no separate reduction launch is needed.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "nf4_device.cuh"
#include "profile.h"

namespace qlora {

// Device error word of the side kernels (bounded waits that gave up).
__device__ int g_side_error = 0;

int read_and_clear_side_error(int* out) {
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_side_error, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_side_error, &zero, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  *out = v;
  return QLORA_OK;
}

namespace side {

constexpr int THREADS = 256;  // 8 warps x 16 rows
constexpr int TR = 128;       // rows per CTA
constexpr int TC = 64;        // contraction per stage
constexpr int STAGES = 4;
constexpr int P_STAGE_BYTES = TR * TC * 2;
constexpr int Q_SMEM_MAX = 40 * 1024;

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
__device__ __forceinline__ void ldsm_x2_t(uint32_t addr, uint32_t (&r)[2]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
// bf16 operands, or fp16 when H; fp32 accumulate
template <bool H>
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4],
                                          const uint32_t (&b)[2]) {
  if constexpr (H)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Rank-r operand: Q(c, j) = src[c * ldc + j * ldj] (fp32, or the 16-bit type), zero for j >= r.
struct QSrc {
  const void* ptr;
  int64_t ldc, ldj;
  int fp32;
};

// Outputs of the last CTA of a row tile, for rows < R:
//   out32[row * ld_row + j * ld_j] = scale32 * v                 (j < r)
//   op[row * ld_op + j] = 16-bit(scale_op * v), zero for j >= r    (j < op_cols)
struct Epi {
  float* out32;
  int64_t ld_row, ld_j;
  float scale32;
  uint16_t* op;
  int64_t ld_op;
  int op_cols;
  float scale_op;
  // narrow V only (rank <= 16): with db_part set, also the partial products of
  // dB = dY^T U16 over this CTA's 128 rows, U16 = 16-bit(u_src) (fp32 [R][r]):
  // db_part[row tile][c][16] fp32 for every contraction index c of P
  const float* u_src;
  float* db_part;
  // narrow form only: CTA 0 zeroes zero_tickets[0, nzero) first (the arrival counters of the
  // split reductions later in the call), in place of a memset launch
  int* zero_tickets;
  int64_t nzero;
};

// One fp32 value rounded to the 16-bit type (bf16, or fp16 when H).
template <bool H>
__device__ __forceinline__ uint16_t round16(float v) {
  return static_cast<uint16_t>(pack_pair<H>(v, 0.0f) & 0xFFFFu);
}

// Stage Q(c, j), c in [c_begin, c_begin + clen), into sQ[c][j] (pitch NJ + 8).  Three vector
// layouts of the source: bf16 contiguous along c (A[j][k]), bf16 contiguous along j (B[n][j],
// sV[m][j]) and fp32 contiguous along j (U[m][j]); anything else element by element.
// kick() runs once, right after the first batch of loads is issued: the caller starts the
// big operand's TMA stream there, so the rank-r loads are not queued behind it.
template <int NJ, bool H, typename Kick>
__device__ __forceinline__ void stage_q(uint16_t* sQ, const QSrc& qs, int r, int64_t C,
                                        int64_t c_begin, int clen, int tid, Kick&& kick) {
  constexpr int QP = NJ + 8;
  constexpr int BATCH = 8;
  bool kicked = false;
  const uint16_t* b16 = static_cast<const uint16_t*>(qs.ptr);
  const float* f32 = static_cast<const float*>(qs.ptr);
  if (!qs.fp32 && qs.ldc == 1 && (qs.ldj % 8) == 0 && (c_begin % 8) == 0) {
    // A[j][c]: 8 consecutive c per load, scattered into 8 rows of sQ
    const int per_j = clen / 8, n = NJ * per_j;
    for (int base = tid; base < n; base += BATCH * THREADS) {
      uint4 v[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        const int c8 = idx / NJ, j = idx % NJ;  // consecutive threads: consecutive j (smem)
        v[u] = make_uint4(0, 0, 0, 0);
        if (idx < n && j < r && c_begin + 8 * c8 < C)
          v[u] = __ldg(reinterpret_cast<const uint4*>(b16 + (int64_t)j * qs.ldj + c_begin + 8 * c8));
      }
      if (!kicked) {
        kick();
        kicked = true;
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        if (idx >= n) break;
        const int c8 = idx / NJ, j = idx % NJ;
        const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
          sQ[(8 * c8 + e) * QP + j] = static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1)));
      }
    }
  } else if (!qs.fp32 && qs.ldj == 1 && (qs.ldc % 8) == 0 && (r % 8) == 0) {
    // src[c][j]: one 16-byte row piece of 8 j per load
    constexpr int J8 = NJ / 8;
    const int n = clen * J8;
    for (int base = tid; base < n; base += BATCH * THREADS) {
      uint4 v[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        const int c = idx / J8, j8 = idx % J8;
        v[u] = make_uint4(0, 0, 0, 0);
        if (idx < n && 8 * j8 < r && c_begin + c < C)
          v[u] = __ldg(reinterpret_cast<const uint4*>(b16 + (c_begin + c) * qs.ldc + 8 * j8));
      }
      if (!kicked) {
        kick();
        kicked = true;
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        if (idx >= n) break;
        const int c = idx / J8, j8 = idx % J8;
        *reinterpret_cast<uint4*>(sQ + c * QP + 8 * j8) = v[u];
      }
    }
  } else if (qs.fp32 && qs.ldj == 1 && (qs.ldc % 4) == 0 && (r % 4) == 0) {
    // fp32 src[c][j]: 4 j per load, converted to the 16-bit type
    constexpr int J4 = NJ / 4;
    const int n = clen * J4;
    for (int base = tid; base < n; base += BATCH * THREADS) {
      float4 v[BATCH];
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        const int c = idx / J4, j4 = idx % J4;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < n && 4 * j4 < r && c_begin + c < C)
          v[u] = __ldg(reinterpret_cast<const float4*>(f32 + (c_begin + c) * qs.ldc + 4 * j4));
      }
      if (!kicked) {
        kick();
        kicked = true;
      }
#pragma unroll
      for (int u = 0; u < BATCH; ++u) {
        const int idx = base + u * THREADS;
        if (idx >= n) break;
        const int c = idx / J4, j4 = idx % J4;
        *reinterpret_cast<uint2*>(sQ + c * QP + 4 * j4) =
            make_uint2(pack_pair<H>(v[u].x, v[u].y), pack_pair<H>(v[u].z, v[u].w));
      }
    }
  } else {
    kick();
    kicked = true;
    for (int i = tid; i < clen * NJ; i += THREADS) {
      const int c = i / NJ, j = i % NJ;
      const int64_t gc = c_begin + c;
      float v = 0.f;
      if (j < r && gc < C) {
        const int64_t off = gc * qs.ldc + (int64_t)j * qs.ldj;
        v = qs.fp32 ? __ldg(f32 + off) : widen16<H>(__ldg(b16 + off));
      }
      sQ[c * QP + j] = round16<H>(v);
    }
  }
  if (!kicked) kick();
}

// The outputs of one float4 piece (row, columns j0 .. j0 + 3) of the summed tile.
template <bool H>
__device__ __forceinline__ void epi_store(const Epi& epi, int r, int64_t row, int j0, float4 v) {
  const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = j0 + e;
    const float x = j < r ? vv[e] : 0.f;
    if (epi.out32 && j < r) epi.out32[row * epi.ld_row + j * epi.ld_j] = x * epi.scale32;
    if (epi.op && j < epi.op_cols) epi.op[row * epi.ld_op + j] = round16<H>(x * epi.scale_op);
  }
}

template <bool kPCol, int NJ, bool H>
__global__ void __launch_bounds__(THREADS, 2)
    side_gemm(const __grid_constant__ CUtensorMap tmP, int64_t R, int64_t C, QSrc qs, int r,
              float* __restrict__ part, int* __restrict__ tickets, int64_t chunk, int S, Epi epi,
              int64_t part_cap, int64_t ticket_cap) {
  constexpr int QP = NJ + 8;  // Q row pitch in elements (+16 bytes: conflict-free ldmatrix)
  extern __shared__ uint8_t smem_raw[];
  // TMA writes 128-byte-swizzled tiles: stage buffers start on 1024-byte boundaries
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint16_t* sP = reinterpret_cast<uint16_t*>(smem);
  uint16_t* sQ = reinterpret_cast<uint16_t*>(smem + STAGES * P_STAGE_BYTES);
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ int s_last;
  __shared__ int abort_flag;
  volatile int* abort_p = &abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t r0 = (int64_t)blockIdx.x * TR;
  const int64_t c_pad = (C + TC - 1) / TC * TC;
  const int64_t c_begin = (int64_t)blockIdx.y * chunk;
  const int64_t c_end = (c_begin + chunk < c_pad) ? c_begin + chunk : c_pad;
  const int nst = c_end > c_begin ? static_cast<int>((c_end - c_begin) / TC) : 0;

  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) mbar_init(&full_bar[i], 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  launch_dependents();  // the fused GEMM that reads this output may be scheduled meanwhile
  __syncthreads();

  // One thread streams P with TMA: K-major tiles are one [64 c x 128 rows] box (row r at
  // r*128 bytes, 16-byte chunk ^ (r & 7)); column-wise tiles are two [64 rows x 64 c] boxes
  // (c at c*128 bytes within each half).  Out-of-range rows / columns arrive as zeros.
  auto issue = [&](int st) {
    const int slot = st % STAGES;
    uint16_t* d = sP + slot * (TR * TC);
    const int32_t c0 = static_cast<int32_t>(c_begin + (int64_t)st * TC);
    mbar_arrive_expect_tx(&full_bar[slot], P_STAGE_BYTES);
    if (!kPCol) {
      tma_load_2d(d, &tmP, &full_bar[slot], c0, static_cast<int32_t>(r0));
    } else {
      tma_load_2d(d, &tmP, &full_bar[slot], static_cast<int32_t>(r0), c0);
      tma_load_2d(d + TR * TC / 2, &tmP, &full_bar[slot], static_cast<int32_t>(r0 + 64), c0);
    }
  };
  int issued = 0;
  if (tid == 0) tma_prefetch_desc(&tmP);
  // rank-r operand for the whole contraction range, as [c][j] bf16 (zero past the rank),
  // loaded with 16-byte vectors in batches of 8 per thread so the loads overlap; its first
  // loads go out before the big operand's stream starts
  stage_q<NJ, H>(sQ, qs, r, C, c_begin, static_cast<int>(c_end - c_begin), tid, [&]() {
    if (tid == 0)
      for (; issued < STAGES - 1 && issued < nst; ++issued) issue(issued);
  });

  float acc[NJ / 8][4];
#pragma unroll
  for (int t = 0; t < NJ / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  bool ok = true;
  for (int st = 0; st < nst; ++st) {
    ok = mbar_wait(&full_bar[st % STAGES], (st / STAGES) & 1, kWaitTmaFull, abort_p, &g_side_error);
    __syncthreads();  // every warp is past stage st - 1: its buffer can be refilled
    if (!ok || *abort_p) {
      ok = false;
      break;
    }
    if (tid == 0 && st + STAGES - 1 < nst) {
      fence_proxy_async_smem();  // the generic-proxy reads of that buffer precede the refill
      issue(st + STAGES - 1);
      ++issued;
    }
    const uint16_t* tP = sP + (st % STAGES) * (TR * TC);
#pragma unroll
    for (int kk = 0; kk < TC / 16; ++kk) {
      uint32_t a[4];
      if (!kPCol) {
        const int row = warp * 16 + (lane & 15);
        ldsm_x4(smem_u32(tP + row * TC + (((kk * 2 + (lane >> 4)) ^ (row & 7)) << 3)), a);
      } else {
        const int i = lane >> 3;
        const int c = kk * 16 + (lane & 7) + 8 * (i >> 1);
        const int chunk16 = warp * 2 + (i & 1);  // 8-row group of the 128 rows
        ldsm_x4_t(smem_u32(tP + (chunk16 >> 3) * (TR * TC / 2) + c * 64 +
                           (((chunk16 & 7) ^ (c & 7)) << 3)), a);
      }
      const int qc = st * TC + kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
      for (int t = 0; t < NJ / 8; ++t) {
        uint32_t b[2];
        ldsm_x2_t(smem_u32(sQ + qc * QP + t * 8), b);
        mma_16816<H>(acc[t], a, b);
      }
    }
  }
  if (!ok) {
    // give up without a result (the row tile's ticket never completes), but never leave a
    // copy in flight into this CTA's shared memory
    if (tid == 0)
      for (int st = issued - (STAGES - 1) < 0 ? 0 : issued - (STAGES - 1); st < issued; ++st)
        mbar_drain(&full_bar[st % STAGES], (st / STAGES) & 1);
    __syncthreads();
    return;
  }

  const int g = lane >> 2, q = lane & 3;
  // this CTA's partial sums
  float* mine = part + (int64_t)blockIdx.y * R * NJ;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t row = r0 + warp * 16 + g + 8 * h;
    if (row < R && QLORA_CHECK((int64_t)blockIdx.y * R * NJ + row * NJ + NJ <= part_cap, &g_side_error,
                               kBoundsPartial)) {
#pragma unroll
      for (int t = 0; t < NJ / 8; ++t)
        __stcg(reinterpret_cast<float2*>(mine + row * NJ + t * 8 + 2 * q),
               make_float2(acc[t][2 * h], acc[t][2 * h + 1]));
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    s_last = 0;
    if (QLORA_CHECK(blockIdx.x < ticket_cap, &g_side_error, kBoundsTicket)) {
      const int before = atomicAdd(&tickets[blockIdx.x], 1);
      (void)QLORA_CHECK(before < S, &g_side_error, kBoundsTicket);
      s_last = before == S - 1;
    }
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last CTA of this row tile: fixed-order sum over the splits, then the outputs.  Each
  // thread owns PER float4 pieces; 16 partial loads are in flight per batch.
  constexpr int V4 = NJ / 4;
  constexpr int PER = TR * V4 / THREADS;
  constexpr int PB = PER < 2 ? PER : 2;  // pieces per pass
  constexpr int SB = 16 / PB;            // splits per batch
  const int64_t sstride = R * NJ / 4;    // float4 stride between splits
  // the last split's rows of this tile lie inside the partial buffer
  if (!QLORA_CHECK((int64_t)(S - 1) * R * NJ + min(R, r0 + TR) * NJ <= part_cap, &g_side_error,
                   kBoundsPartial))
    return;
#pragma unroll 1
  for (int p0 = 0; p0 < PER; p0 += PB) {
    const float4* src[PB];
    bool live[PB];
    float4 v[PB];
#pragma unroll
    for (int b = 0; b < PB; ++b) {
      const int i = tid + (p0 + b) * THREADS;
      const int64_t row = r0 + i / V4;
      live[b] = row < R;
      src[b] = reinterpret_cast<const float4*>(part + (live[b] ? row : r0) * NJ + (i % V4) * 4);
      v[b] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // batches of SB splits, the last one partial (its loads and adds predicated): one L2
    // round trip per batch
    for (int s = 0; s < S; s += SB) {
      const int n = S - s < SB ? S - s : SB;
      float4 a[PB][SB];
#pragma unroll
      for (int b = 0; b < PB; ++b)
#pragma unroll
        for (int u = 0; u < SB; ++u)
          if (u < n) a[b][u] = __ldcg(src[b] + (s + u) * sstride);
#pragma unroll
      for (int b = 0; b < PB; ++b)
#pragma unroll
        for (int u = 0; u < SB; ++u)
          if (u < n) {
            v[b].x += a[b][u].x; v[b].y += a[b][u].y; v[b].z += a[b][u].z; v[b].w += a[b][u].w;
          }
    }
#pragma unroll
    for (int b = 0; b < PB; ++b) {
      if (!live[b]) continue;
      const int i = tid + (p0 + b) * THREADS;
      epi_store<H>(epi, r, r0 + i / V4, (i % V4) * 4, v[b]);
    }
  }
  if (epi.op && epi.op_cols > NJ) {  // zero columns of the operand copy past NJ
    const int extra = epi.op_cols - NJ;
    for (int i = tid; i < TR * extra; i += THREADS) {
      const int64_t row = r0 + i / extra;
      if (row < R) epi.op[row * epi.ld_op + NJ + i % extra] = 0;
    }
  }
  if (tid == 0) tickets[blockIdx.x] = 0;  // ready for the next launch
}

// Narrow form of the row-wise products U = X A^T and V = dY B, for launches whose row tiles
// alone leave most SMs free: one CTA per 128-row tile takes the whole contraction, so there
// are no split partials and no ticket, and the rank-r operand streams beside P in the same
// TMA ring instead of being staged up front.  A fused GEMM launched behind it as a
// programmatic dependent then finds most SMs free for its first wave and only needs this
// output at its LoRA stage, after its NF4 stages.
// P is row-major: one [64 c x 128 rows] box per stage, 128-byte swizzled.
//   kQRows: Q is [r rows][C] with c contiguous (A of U): one [64 c x NJ rows] box per stage,
//           128-byte swizzled, read with plain ldmatrix (rows j, 8 consecutive c);
//   else    Q is [C rows][rq] with j contiguous (B of V): one [NJ j x 64 c] box per stage,
//           read with ldmatrix.trans.
// Rows past r (or past rq) arrive as zeros.
// kDB (V with rank <= 16): the dY tile of each stage also feeds the partial products of
// dB = dY^T U over the CTA's 128 rows, on 8 more warps beside the 8 of V (measured: 39 us per
// launch with both on the same 8 warps).  dB warp w takes 16 columns of the stage (w & 3) and 8
// of the rank (w >> 2): an m16n8k16 with A = the tile read transposed (ldmatrix.trans) and
// B = the rows' U in the 16-bit type, held in registers for the whole launch.  A fixed-order
// sum of the row tiles' partials (db_reduce) finishes dB.
template <int NJ>
struct Narrow {
  static constexpr int Q_STAGE_BYTES = NJ * TC * 2;
  static constexpr int STAGE_BYTES = P_STAGE_BYTES + Q_STAGE_BYTES;
  static constexpr int STAGES = (216 * 1024) / STAGE_BYTES < 12 ? (216 * 1024) / STAGE_BYTES : 12;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024;
};

// The consumer warps (8 for U / V: 16 rows each; 16 with kDB: 8 more form the dB partials)
// and one producer warp.  Each stage's slot is released by an empty barrier that every
// consumer warp arrives on after its last read, so the warps drift freely across the ring
// (measured: a CTA-wide barrier per stage made the launch wait on its slowest warp every
// stage).
template <bool kDB>
struct NarrowWarps {
  static constexpr int kConsumers = kDB ? 2 * (THREADS / 32) : THREADS / 32;
  static constexpr int kThreads = (kConsumers + 1) * 32;
};

template <bool kQRows, int NJ, bool H, bool kDB>
__global__ void __launch_bounds__(NarrowWarps<kDB>::kThreads, 1)
    side_rows(const __grid_constant__ CUtensorMap tmP, const __grid_constant__ CUtensorMap tmQ,
              int64_t R, int64_t C, int r, Epi epi) {
  using G = Narrow<NJ>;
  constexpr int S = G::STAGES;
  constexpr int NWC = NarrowWarps<kDB>::kConsumers;
  constexpr int kThreads = NarrowWarps<kDB>::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sP = smem;                          // S x [128 rows x 64 c], 128-byte swizzled
  uint8_t* sQ = smem + S * P_STAGE_BYTES;      // S x Q tile (1 KB multiples: swizzle atoms)
  __shared__ __align__(8) uint64_t full_bar[S];
  __shared__ __align__(8) uint64_t empty_bar[S];
  __shared__ int abort_flag;
  volatile int* abort_p = &abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool v_warp = warp < THREADS / 32;       // forms U / V (rows 16 warp ..)
  const int dw = warp - THREADS / 32;            // kDB: dB warp index (0..7)
  const int64_t r0 = (int64_t)blockIdx.x * TR;
  const int nst = static_cast<int>((C + TC - 1) / TC);

  if (tid == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], NWC);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  // the tickets are zero (and visible device-wide) before the kernel behind this one, which
  // draws from them before it waits for this grid, may start
  if (blockIdx.x == 0 && epi.zero_tickets) {
    for (int64_t i = tid; i < epi.nzero; i += kThreads) epi.zero_tickets[i] = 0;
    __threadfence();
  }
  __syncthreads();
  launch_dependents();

  if (warp == NWC) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmP);
      tma_prefetch_desc(&tmQ);
      int issued = 0;
      for (; issued < nst; ++issued) {
        const int slot = issued % S, round = issued / S;
        if (round > 0 &&
            !mbar_wait(&empty_bar[slot], (round - 1) & 1, kWaitEmpty, abort_p, &g_side_error))
          break;
        fence_proxy_async_smem();  // the consumers' reads of the slot precede the refill
        const int32_t c0 = static_cast<int32_t>((int64_t)issued * TC);
        mbar_arrive_expect_tx(&full_bar[slot], G::STAGE_BYTES);
        tma_load_2d(sP + slot * P_STAGE_BYTES, &tmP, &full_bar[slot], c0, static_cast<int32_t>(r0));
        if (kQRows)
          tma_load_2d(sQ + slot * G::Q_STAGE_BYTES, &tmQ, &full_bar[slot], c0, 0);
        else
          tma_load_2d(sQ + slot * G::Q_STAGE_BYTES, &tmQ, &full_bar[slot], 0, c0);
      }
      // never leave with a copy in flight into this CTA's shared memory
      for (int st = issued - S < 0 ? 0 : issued - S; st < issued; ++st)
        mbar_drain(&full_bar[st % S], (st / S) & 1);
    }
    return;
  }

  float acc[NJ / 8][4];
#pragma unroll
  for (int t = 0; t < NJ / 8; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;

  // kDB: B fragments of U (rows r0 + 16 kc + 2 q (+1, +8, +9), rank 8 (dw >> 2) + g)
  uint32_t ub[kDB ? 8 : 1][2];
  if (kDB && !v_warp) {
    const int g = lane >> 2, q = lane & 3, j = 8 * (dw >> 2) + g;
#pragma unroll
    for (int kc = 0; kc < 8; ++kc)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t m = r0 + 16 * kc + 2 * q + 8 * h;
        const float lo = (j < r && m < R) ? __ldg(epi.u_src + m * r + j) : 0.f;
        const float hi = (j < r && m + 1 < R) ? __ldg(epi.u_src + (m + 1) * r + j) : 0.f;
        ub[kc][h] = pack_pair<H>(lo, hi);
      }
  }
  // Q rows of NJ j (2 NJ bytes) with the swizzle of that span (32 / 64 / 128 bytes; none for
  // wider rows): 16-byte chunk h of row c sits at chunk h ^ ((c * 2 NJ / 128) & (2 NJ / 16 - 1))
  constexpr int QSPAN = 2 * NJ;
  constexpr int QXOR = QSPAN <= 128 ? QSPAN / 16 - 1 : 0;

  for (int st = 0; st < nst; ++st) {
    const int slot = st % S;
    if (!mbar_wait(&full_bar[slot], (st / S) & 1, kWaitTmaFull, abort_p, &g_side_error)) return;
    const uint32_t tP = smem_u32(sP + slot * P_STAGE_BYTES);
    const uint32_t tQ = smem_u32(sQ + slot * G::Q_STAGE_BYTES);
    if (v_warp) {
#pragma unroll
      for (int kk = 0; kk < TC / 16; ++kk) {
        uint32_t a[4];
        {
          const int row = warp * 16 + (lane & 15);
          ldsm_x4(tP + row * 128 + ((((kk * 2 + (lane >> 4)) ^ (row & 7))) << 4), a);
        }
#pragma unroll
        for (int t = 0; t < NJ / 8; t += 2) {
          // lanes 0-15: n-tile t, lanes 16-31: n-tile t + 1; within each, c halves 0-7 / 8-15
          uint32_t b[4];
          if (kQRows) {
            const int j = 8 * (t + (lane >> 4)) + (lane & 7);
            const int chunk = kk * 2 + ((lane >> 3) & 1);
            ldsm_x4(tQ + j * 128 + ((chunk ^ (j & 7)) << 4), b);
          } else {
            const int c = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
            const int h = t + (lane >> 4);
            ldsm_x4_t(tQ + c * QSPAN + ((h ^ ((c * QSPAN / 128) & QXOR)) << 4), b);
          }
          const uint32_t b0[2] = {b[0], b[1]}, b1[2] = {b[2], b[3]};
          mma_16816<H>(acc[t], a, b0);
          mma_16816<H>(acc[t + 1], a, b1);
        }
      }
    }
    if (kDB && !v_warp) {
      // columns c = 64 st + 16 (dw & 3) .. + 15 of this stage against the tile's 128 rows
      const int nt = dw & 3, i = lane & 7, mat = lane >> 3;
      float d[4] = {0.f, 0.f, 0.f, 0.f}, d2[4] = {0.f, 0.f, 0.f, 0.f};  // two MMA chains
#pragma unroll
      for (int kc = 0; kc < 8; ++kc) {
        uint32_t a[4];  // A = tile^T: rows c (16 nt + 8 (mat & 1) + ..), columns m (16 kc + ..)
        const int m = 16 * kc + i + 8 * (mat >> 1);
        const int chunk = 2 * nt + (mat & 1);
        ldsm_x4_t(tP + m * 128 + ((chunk ^ (m & 7)) << 4), a);
        mma_16816<H>((kc & 1) ? d2 : d, a, ub[kc]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) d[e] += d2[e];
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);  // this warp's reads of the slot are done
      const int g = lane >> 2, q = lane & 3;
      float* dst = epi.db_part + (int64_t)blockIdx.x * C * 16 + 8 * (dw >> 2) + 2 * q;
      const int64_t c = (int64_t)st * TC + 16 * nt + g;
      if (c < C) __stcg(reinterpret_cast<float2*>(dst + c * 16), make_float2(d[0], d[1]));
      if (c + 8 < C) __stcg(reinterpret_cast<float2*>(dst + (c + 8) * 16), make_float2(d[2], d[3]));
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);  // this warp's reads of the slot are done
    }
  }

  // outputs straight from the accumulators: lane (g, q) holds rows g and g + 8 of the warp's
  // 16, columns 8t + 2q and 8t + 2q + 1
  if (!v_warp) return;
  const int g = lane >> 2, q = lane & 3;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t row = r0 + warp * 16 + g + 8 * h;
    if (row >= R) continue;
#pragma unroll
    for (int t = 0; t < NJ / 8; ++t)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = 8 * t + 2 * q + e;
        const float x = j < r ? acc[t][2 * h + e] : 0.f;
        if (epi.out32 && j < r) epi.out32[row * epi.ld_row + j * epi.ld_j] = x * epi.scale32;
        if (epi.op && j < epi.op_cols) epi.op[row * epi.ld_op + j] = round16<H>(x * epi.scale_op);
      }
    if (epi.op)
      for (int j = NJ + q; j < epi.op_cols; j += 4) epi.op[row * epi.ld_op + j] = 0;
  }
}

// dB[n][j] = scale * sum over the row tiles t (ascending) of part[t][n][j], j < r <= 16.
__global__ void __launch_bounds__(256) db_reduce(const float* __restrict__ part, int ntiles,
                                                 int64_t N, int r, float scale,
                                                 float* __restrict__ dB) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // (n, 4-column group)
  if (i >= N * 4) return;
  const int64_t n = i >> 2;
  const int j0 = 4 * static_cast<int>(i & 3);
  if (j0 >= r) return;
  const float4* src = reinterpret_cast<const float4*>(part + n * 16 + j0);
  const int64_t stride = N * 4;  // float4 per tile
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int t = 0;
  for (; t + 8 <= ntiles; t += 8) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcg(src + (t + u) * stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
    }
  }
  for (; t < ntiles; ++t) {
    const float4 v = __ldcg(src + t * stride);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  const float vv[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (j0 + e < r) dB[n * r + j0 + e] = scale * vv[e];
}

// Zero-padded copy Bp [N, rp] of B [N, r], for ranks whose rows are not 16-byte multiples.
__global__ void pad_b(const uint16_t* __restrict__ B, int64_t N, int r, int64_t rp,
                      uint16_t* __restrict__ Bp) {
  const int64_t total = N * rp;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = i / rp, j = i % rp;
    Bp[i] = j < r ? B[n * r + j] : 0;
  }
}

}  // namespace side

// ---------------------------------------------------------------- host side
namespace {

int pick_nj(int r) { return r <= 16 ? 16 : r <= 32 ? 32 : r <= 64 ? 64 : 128; }

struct Split {
  int64_t chunk;
  int S;
  unsigned row_tiles;
};

// Contraction split so that row tiles x splits fill the SMs once (one CTA per SM), within
// the shared-memory budget for the staged rank-r operand.
Split pick_split(int64_t R, int64_t C, int NJ) {
  Split sp;
  sp.row_tiles = (unsigned)((R + side::TR - 1) / side::TR);
  const int64_t c_tiles = (C + side::TC - 1) / side::TC;
  int64_t want = 2LL * num_sms() / (int64_t)sp.row_tiles;  // two CTAs per SM
  // With few row tiles that would cut the contraction into many short chunks, and the last
  // CTA of a row tile reads every split's TR x NJ fp32 partial tile alone.  A CTA reads
  // TR * 2 bytes per contraction column and the final sum TR * NJ * 4 per split: the two
  // balance at S = sqrt(C / (2 NJ)), the most splits taken (at M = 512 on the 4096^2 layer:
  // 11 instead of 64 for U; twice the balance point measured 3 us slower per step).
  const int64_t bal = static_cast<int64_t>(std::sqrt(static_cast<double>(C) / (2.0 * NJ)));
  if (want > bal) want = bal;
  if (want < 1) want = 1;
  if (want > c_tiles) want = c_tiles;
  int64_t per = (c_tiles + want - 1) / want;
  const int64_t qmax = side::Q_SMEM_MAX / ((NJ + 8) * 2) / side::TC;
  if (per > qmax) per = qmax;
  if (per < 1) per = 1;
  sp.chunk = per * side::TC;
  sp.S = (int)((c_tiles + per - 1) / per);
  return sp;
}

template <bool kCol, bool H>
int run_side_t(const char* name, const uint16_t* P, int64_t R, int64_t C, int64_t ldp, side::QSrc qs,
             int r, const side::Epi& epi, const LinearArgs& a, const WorkspaceLayout& L,
             cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int NJ = pick_nj(r);
  const Split sp = pick_split(R, C, NJ);
  float* part = reinterpret_cast<float*>(ws + L.part);
  int* tickets = reinterpret_cast<int*>(ws + L.tickets);
  const int64_t part_cap = static_cast<int64_t>(L.part_bytes / 4);
  const int64_t ticket_cap = static_cast<int64_t>(L.ntickets);
  CUtensorMap tm;
  // K-major: P is [R rows][C] and a box is 64 c x 128 rows; column-wise: P is [C][R] and a
  // box is 64 rows x 64 c
  const bool mapped =
      kCol ? make_tensor_map_2d(&tm, P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)R,
                                (uint64_t)C, (uint64_t)ldp * 2, 64, 64, MapSwizzle::B128)
           : make_tensor_map_2d(&tm, P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)C,
                                (uint64_t)R, (uint64_t)ldp * 2, 64, side::TR, MapSwizzle::B128);
  if (!mapped) return QLORA_ERR_CUDA;
  const int smem = side::STAGES * side::P_STAGE_BYTES + (int)sp.chunk * (NJ + 8) * 2 + 1024;
  dim3 grid(sp.row_tiles, (unsigned)sp.S);
  ProfileScope ps(name, stream);
  switch (NJ) {
#define QLORA_SIDE_CASE(nj)                                                                       \
  case nj:                                                                                        \
    {                                                                                             \
      static DeviceCache<int> attr; /* per instantiation and device: the largest configuration */ \
      const int st = ensure_dynamic_smem(attr, side::side_gemm<kCol, nj, H>,                      \
                                         side::STAGES * side::P_STAGE_BYTES + side::Q_SMEM_MAX + 1024); \
      if (st) return st;                                                                          \
    }                                                                                             \
    side::side_gemm<kCol, nj, H><<<grid, side::THREADS, smem, stream>>>(                          \
        tm, R, C, qs, r, part, tickets, sp.chunk, sp.S, epi, part_cap, ticket_cap);               \
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

// The 16-bit type of P, Q and op follows the call (bf16, or fp16 in the fp16 compute type).
template <bool kCol>
int run_side(const char* name, const uint16_t* P, int64_t R, int64_t C, int64_t ldp, side::QSrc qs,
             int r, const side::Epi& epi, const LinearArgs& a, const WorkspaceLayout& L,
             cudaStream_t stream) {
  return a.half ? run_side_t<kCol, true>(name, P, R, C, ldp, qs, r, epi, a, L, stream)
                : run_side_t<kCol, false>(name, P, R, C, ldp, qs, r, epi, a, L, stream);
}

// The narrow form serves U and V when their row tiles fill at most a quarter of the SMs, in
// front of a GEMM on CTA pairs: the GEMM has work for the other SMs from its first stage on and
// reads U / V only in its LoRA stage.  (A GEMM with a staged base waits for the kernels before
// it instead, and one-CTA tiles come at sizes where the split form is short.)  A narrow CTA
// streams at about 40 GB/s, so the narrow form is no use where its rows must finish quickly
// on few SMs: dB and dA keep the split form.
bool use_narrow(int64_t M, int64_t Nout, int64_t Kc) {
  return (M + side::TR - 1) / side::TR <= num_sms() / 4 && fused_plan(M, Nout, Kc).kind == 2;
}

template <bool kQRows, int NJ, bool H, bool kDB>
int launch_rows(const CUtensorMap& tmP, const CUtensorMap& tmQ, int64_t R, int64_t C, int r,
                const side::Epi& epi, cudaStream_t stream) {
  constexpr int smem = side::Narrow<NJ>::SMEM_BYTES;
  static DeviceCache<int> attr;  // per instantiation and device
  const int st = ensure_dynamic_smem(attr, side::side_rows<kQRows, NJ, H, kDB>, smem);
  if (st) return st;
  const dim3 grid((unsigned)((R + side::TR - 1) / side::TR));
  side::side_rows<kQRows, NJ, H, kDB><<<grid, side::NarrowWarps<kDB>::kThreads, smem, stream>>>(
      tmP, tmQ, R, C, r, epi);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

// P: [R rows][C] (ldp).  Q: kQRows -> [q_outer rows = r][q_inner = C] (A), 128-byte swizzled
// boxes of [64 c x NJ rows]; else [q_outer = C][q_inner] (B) in boxes of [NJ j x 64 c], with
// the swizzle of their 2 NJ-byte rows (none past 128 bytes).  kDB: the V form with the dB
// partials (rank <= 16).
template <bool kQRows, bool H, bool kDB>
int run_rows_t(const char* name, const uint16_t* P, int64_t R, int64_t C, int64_t ldp,
               const uint16_t* Q, int64_t q_outer, int64_t q_inner, int64_t q_pitch, int r,
               const side::Epi& epi, cudaStream_t stream) {
  const int NJ = pick_nj(r);
  CUtensorMap tmP, tmQ;
  if (!make_tensor_map_2d(&tmP, P, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)C, (uint64_t)R,
                          (uint64_t)ldp * 2, 64, side::TR, MapSwizzle::B128))
    return QLORA_ERR_CUDA;
  const MapSwizzle qsw = NJ == 16 ? MapSwizzle::B32
                       : NJ == 32 ? MapSwizzle::B64
                       : NJ == 64 ? MapSwizzle::B128
                                  : MapSwizzle::None;
  const bool qmap =
      kQRows ? make_tensor_map_2d(&tmQ, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)q_inner,
                                  (uint64_t)q_outer, (uint64_t)q_pitch * 2, 64, (uint32_t)NJ,
                                  MapSwizzle::B128)
             : make_tensor_map_2d(&tmQ, Q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)q_inner,
                                  (uint64_t)q_outer, (uint64_t)q_pitch * 2, (uint32_t)NJ, 64, qsw);
  if (!qmap) return QLORA_ERR_CUDA;
  ProfileScope ps(name, stream);
  if (kDB) return NJ == 16 ? launch_rows<kQRows, 16, H, kDB>(tmP, tmQ, R, C, r, epi, stream)
                           : QLORA_ERR_UNSUPPORTED;
  switch (NJ) {
    case 16: return launch_rows<kQRows, 16, H, false>(tmP, tmQ, R, C, r, epi, stream);
    case 32: return launch_rows<kQRows, 32, H, false>(tmP, tmQ, R, C, r, epi, stream);
    case 64: return launch_rows<kQRows, 64, H, false>(tmP, tmQ, R, C, r, epi, stream);
    case 128: return launch_rows<kQRows, 128, H, false>(tmP, tmQ, R, C, r, epi, stream);
    default: return QLORA_ERR_UNSUPPORTED;
  }
}

template <bool kQRows, bool kDB = false>
int run_rows(const char* name, const uint16_t* P, int64_t R, int64_t C, int64_t ldp,
             const uint16_t* Q, int64_t q_outer, int64_t q_inner, int64_t q_pitch, int r,
             const side::Epi& epi, const LinearArgs& a, cudaStream_t stream) {
  return a.half ? run_rows_t<kQRows, true, kDB>(name, P, R, C, ldp, Q, q_outer, q_inner, q_pitch,
                                                r, epi, stream)
                : run_rows_t<kQRows, false, kDB>(name, P, R, C, ldp, Q, q_outer, q_inner, q_pitch,
                                                 r, epi, stream);
}

side::Epi no_epi() {
  side::Epi e{};
  e.scale32 = 1.f;
  e.scale_op = 1.f;
  return e;
}

}  // namespace

uint64_t side_partial_bytes(int64_t M, int64_t N, int64_t K, int r) {
  const int NJ = pick_nj(r);
  uint64_t worst = 0;
  auto upd = [&](int64_t rows, int64_t C) {
    const Split sp = pick_split(rows, C, NJ);
    worst = std::max<uint64_t>(worst, (uint64_t)sp.S * rows * NJ * 4);
  };
  upd(M, K);  // U
  upd(M, N);  // V
  upd(N, M);  // dB
  upd(K, M);  // dA^T
  return worst;
}

uint64_t side_ticket_count(int64_t M, int64_t N, int64_t K) {
  const int64_t m = std::max(M, std::max(N, K));
  return (uint64_t)((m + side::TR - 1) / side::TR);
}

int launch_pad_b(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int64_t n = a.N * L.rp;
  unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 8LL * num_sms());
  ProfileScope ps("pad_b", stream);
  side::pad_b<<<blocks, 256, 0, stream>>>(a.B, a.N, a.r, L.rp, reinterpret_cast<uint16_t*>(ws + L.Bp));
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

bool side_narrow_u(const LinearArgs& a) { return use_narrow(a.M, a.N, a.K) && a.K % 8 == 0; }
bool side_narrow_v(const LinearArgs& a) { return use_narrow(a.M, a.K, a.N) && a.r % 8 == 0; }

// U = X A^T -> sU = 16-bit(scale U) [M, rp], and U fp32 [M, r] into u32 (caller's U_save or
// the workspace copy the backward recomputes), when given.  narrow_ok: the narrow form may be
// used (it zeroes the call's arrival tickets); the backward's recomputation, on the critical
// path, takes the split form.
int launch_lora_u(const LinearArgs& a, const WorkspaceLayout& L, float* u32, cudaStream_t stream,
                  bool narrow_ok) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  side::QSrc qs{a.A, 1, a.K, 0};  // Q(c = k, j) = A[j][k]
  side::Epi e = no_epi();
  e.out32 = u32;
  e.ld_row = a.r;
  e.ld_j = 1;
  e.op = reinterpret_cast<uint16_t*>(ws + L.sU);
  e.ld_op = L.rp;
  e.op_cols = a.r;  // readers see the columns past r as zeros (TMA fill)
  e.scale_op = a.scale;
  if (narrow_ok && side_narrow_u(a)) {
    e.zero_tickets = reinterpret_cast<int*>(ws + L.tickets);
    e.nzero = static_cast<int64_t>(L.nticket_words);
    return run_rows<true>("side_u", a.X, a.M, a.K, a.K, a.A, a.r, a.K, a.K, a.r, e, a, stream);
  }
  return run_side<false>("side_u", a.X, a.M, a.K, a.K, qs, a.r, e, a, L, stream);
}

// The narrow V also forms the dB partials (rank <= 16); launch_lora_db then only sums them.
bool fused_db(int64_t M, int64_t N, int64_t K, int r) {
  return use_narrow(M, K, N) && r % 8 == 0 && pick_nj(r) == 16;
}
static bool fused_db(const LinearArgs& a) { return fused_db(a.M, a.N, a.K, a.r); }

// V = dY B -> sV = 16-bit(scale V) [M, rp]; with fused_db also the partial products of dB over
// each 128-row tile of dY (U from u32), into the workspace.  The narrow form zeroes the call's
// arrival tickets.
int launch_lora_v(const LinearArgs& a, const WorkspaceLayout& L, const float* u32,
                  cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  side::QSrc qs{a.B, a.r, 1, 0};  // Q(c = n, j) = B[n][j]
  side::Epi e = no_epi();
  e.op = reinterpret_cast<uint16_t*>(ws + L.sV);
  e.ld_op = L.rp;
  e.op_cols = a.r;  // readers see the columns past r as zeros (TMA fill)
  e.scale_op = a.scale;
  if (side_narrow_v(a)) {
    e.zero_tickets = reinterpret_cast<int*>(ws + L.tickets);
    e.nzero = static_cast<int64_t>(L.nticket_words);
  }
  if (fused_db(a)) {
    if (L.dbpart_bytes < (uint64_t)((a.M + side::TR - 1) / side::TR) * a.N * 64)
      return QLORA_ERR_WORKSPACE;
    e.u_src = u32;
    e.db_part = reinterpret_cast<float*>(ws + L.dbpart);
    return run_rows<false, true>("side_v", a.dY, a.M, a.N, a.N, a.B, a.N, a.r, a.r, a.r, e, a,
                                 stream);
  }
  if (side_narrow_v(a))
    return run_rows<false>("side_v", a.dY, a.M, a.N, a.N, a.B, a.N, a.r, a.r, a.r, e, a, stream);
  return run_side<false>("side_v", a.dY, a.M, a.N, a.N, qs, a.r, e, a, L, stream);
}

// dB = scale * dY^T U  (rows n, contraction over m; U fp32 [M, r]).
int launch_lora_db(const LinearArgs& a, const WorkspaceLayout& L, const float* u32,
                   cudaStream_t stream) {
  side::QSrc qs{u32, a.r, 1, 1};  // Q(c = m, j) = U[m][j]
  side::Epi e = no_epi();
  e.out32 = a.dB;
  e.ld_row = a.r;
  e.ld_j = 1;
  e.scale32 = a.scale;
  if (fused_db(a)) {  // the partials come from the narrow V
    const int ntiles = static_cast<int>((a.M + side::TR - 1) / side::TR);
    const unsigned blocks = (unsigned)((a.N * 4 + 255) / 256);
    ProfileScope ps("side_db", stream);
    side::db_reduce<<<blocks, 256, 0, stream>>>(
        reinterpret_cast<const float*>(static_cast<uint8_t*>(a.ws) + L.dbpart), ntiles, a.N, a.r,
        a.scale, a.dB);
    return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
  }
  return run_side<true>("side_db", a.dY, a.N, a.M, a.N, qs, a.r, e, a, L, stream);
}

// dA = (X^T sV)^T  (rows k, contraction over m; sV already carries the scale).
int launch_lora_da(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  side::QSrc qs{ws + L.sV, L.rp, 1, 0};  // Q(c = m, j) = sV[m][j]
  side::Epi e = no_epi();
  e.out32 = a.dA;
  e.ld_row = 1;
  e.ld_j = a.K;
  return run_side<true>("side_da", a.X, a.K, a.M, a.K, qs, a.r, e, a, L, stream);
}

}  // namespace qlora
