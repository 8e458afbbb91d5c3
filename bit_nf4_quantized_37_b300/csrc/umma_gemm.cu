// umma_gemm.cu -- the fused NF4 + LoRA GEMMs on the 5th-generation tensor cores.
//
// infivelines.com "QLoRA": the base is dequantized to bf16 one block at a time inside the
// matrix multiply; addaly.com "QLoRA on one card": dequantized on the fly for each matrix
// multiply.  Here that "inside" is literal: warps expand the packed 4-bit codes of each
// 64-wide k-slice straight into the shared-memory operand tile of tcgen05.mma, so W' never
// exists in HBM.  The rank-r LoRA term rides in the same TMEM accumulator as extra
// contraction stages after the NF4 stages (so the GEMM can start, as a programmatic
// dependent launch, while the kernel producing sU / sV is still finishing):
//   forward          Y  = [X  | sU] . [W' | B]^T       (contract over K, then over r)
//   input gradient   dX = [dY | sV] . [W' ; A]         (contract over N, then over r)
//
// CTA tile 128 x 256 (UMMA M x N), k-slice 64, 4-stage ring.  Warp roles (384 threads):
//   warp 0      TMA producer: X/dY tiles, and for the LoRA stages both operands
//   warp 1      TMEM owner + single-thread UMMA issuer
//   warps 4-11  NF4 producers (one 64-weight block per thread per stage: codes and block
//               scale from global memory two stages ahead, byte-permute dequantization into
//               the swizzled operand layout), then the epilogue (TMEM -> bf16 -> TMA store)
// Every wait is bounded; on a time-out the CTA records the site and unwinds.
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "linear.h"
#include "profile.h"
#include "nf4_device.cuh"

namespace qlora {

// Device error word of the fused GEMMs (bounded waits that gave up).
__device__ int g_gemm_error = 0;

int read_and_clear_gemm_error(int* out) {
  int v = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int)) != cudaSuccess) return QLORA_ERR_CUDA;
  *out = v;
  return QLORA_OK;
}

namespace fused {

constexpr int UM = 128;  // rows of one UMMA (cta_group::1)
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int B_BYTES = BN * BK * 2;
constexpr int NUM_THREADS = 384;
constexpr int DEQ_WARP0 = 4;
constexpr int NUM_DEQ_WARPS = 8;

// kAcc TMEM accumulators of 128 x 256 per CTA share every dequantized W tile: the CTA tile
// is (128 kAcc) x 256, so each dequantized weight feeds 256 kAcc FLOPs.  The byte-permute
// dequantizer runs on the integer (ALU) pipe, which a 128-row tile saturates before the
// tensor pipe; two accumulators halve the ALU work per FLOP.
// The A tiles (X / dY, by TMA) and the B tiles (the dequantized W tile) sit in rings of their
// own (each stage is dequantized into registers before its B slot is free, so a freed slot
// only takes the stores).  The LoRA stages take an A and a B slot, by TMA.  Measured at
// M = 512 (4096 x 4096, two splits of 128 x 256 tiles): 4 A + 4 B stages 51.7 us per GEMM,
// 3 + 5 57.4 us, 5 + 4 59.5 us -- the 128-row tile dequantizes twice the weights per MMA of a
// pair and its dequant warps, not the rings, set the stage time.
template <int kAcc>
struct Tile {
  static constexpr int BM = UM * kAcc;
  static constexpr int SA = kAcc == 1 ? 4 : 3;  // A ring
  static constexpr int SB = 4;                  // B ring
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BASE = SA * A_BYTES;
  static constexpr int TMEM_COLS = 256 * kAcc;
  static constexpr int SMEM_BYTES = SA * A_BYTES + SB * B_BYTES + 1024;
};

struct Params {
  int64_t M;      // output rows (tokens)
  int64_t Nout;   // output columns
  int64_t Kc;     // NF4 contraction length (forward: K, input gradient: N)
  int64_t Kw;     // columns of W (K)
  int64_t Nw;     // rows of W (N)
  int n_lora;     // LoRA stages after the NF4 stages
  int lora_last_k16;
  const uint8_t* codes;
  const int8_t* qs;
  const float* steps;
  const float* mean;
  int dq;         // 1: double-quantized scales; 0: steps holds the fp32 absmax per block
  int fp8;        // second-level codes are E4M3 (else int8)
  // split contraction (single-CTA kernel): blockIdx.z takes NF4 stages
  // [z * split_stages, (z + 1) * split_stages); the last split also runs the LoRA stages.
  // With nsplit > 1 every CTA writes its fp32 tile to part[z] and the CTA that completes a
  // tile (arrival ticket) sums the splits in split order and stores the 16-bit output.
  int nsplit;
  int split_stages;
  float* part;    // [nsplit][M][Nout] fp32
  int* tickets;   // [output tiles] arrivals, zero at launch, zeroed again by the last CTA
  int64_t part_cap, ticket_cap;  // floats in part, ints in tickets (bounds checks)
  // staged base (single-CTA kernel): W' was dequantized into the workspace by the kernel
  // before this one; every NF4 stage takes its W tile by TMA (map tmW) like a LoRA stage
  int wstage;
  // single-CTA kernel, two splits: the splits of a tile form a cluster and exchange halves
  // of their accumulators in shared memory instead of going through part / tickets
  int csplit;
  // persistent CTA pairs: pers_clusters clusters share the 512 x 256 tiles; the cluster whose
  // leader draws ticket k from *pers_ctr (zero at launch) takes tiles k, k + G, k + 2G, ...;
  // its 16-bit output goes straight from registers to out (row pitch ld_out elements)
  int* pers_ctr;
  int pers_clusters;
  uint16_t* out;
  int64_t ld_out;
};

// One thread's share of an NF4 stage: 64 codes (32 bytes) and the block's scale code/step.
struct Slice {
  uint4 c0, c1;
  float step;
  float q;  // value of the block's second-level code
  bool valid;
};

__device__ __forceinline__ void load_slice(Slice& s, const Params& p, int64_t row, int64_t kcol) {
  s.valid = (row < p.Nw) && (kcol < p.Kw);
  if (s.valid) {
    const uint4* src = reinterpret_cast<const uint4*>(p.codes + row * (p.Kw / 2) + kcol / 2);
    s.c0 = __ldg(src);
    s.c1 = __ldg(src + 1);
    const int64_t b = row * (p.Kw / 64) + kcol / 64;
    if (p.dq) {
      s.q = nf4_second_level(static_cast<uint8_t>(__ldg(p.qs + b)), p.fp8);
      s.step = __ldg(p.steps + (b >> 8));
    } else {  // fmaf(1, absmax, 0) = absmax in the shared scale arithmetic
      s.q = 1.0f;
      s.step = __ldg(p.steps + b);
    }
  }
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* smem_src, int32_t x,
                                             int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(smem_u32(smem_src)), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ------------------------------------------------------------ split contraction epilogue
// With nsplit > 1 every CTA first writes its fp32 tile: one output row per thread (my_row),
// nchunk 32-column chunks read from TMEM at taddr + tcol0 + 32 c, for output columns
// gcol0 + 32 c (columns past Nout, a multiple of 64, skipped by whole float4).  Then the
// 256 epilogue threads (named barrier 1) take the tile's arrival ticket; the CTA completing
// the tile returns true and sums the splits chunk by chunk with split_sum.  Without a split
// it returns true at once.
__device__ __forceinline__ bool split_epilogue_partial(const Params& p, int split, uint32_t taddr,
                                                       int64_t my_row, int64_t gcol0, int nchunk,
                                                       int tcol0, bool ticket_thread, int tile,
                                                       int& s_last) {
  if (p.nsplit <= 1) return true;
  const size_t MN = static_cast<size_t>(p.M) * p.Nout;
  float* mine = p.part + split * MN;
  const bool in_part = QLORA_CHECK(static_cast<int64_t>(p.nsplit * MN) <= p.part_cap, &g_gemm_error,
                                   kBoundsPartial);
#pragma unroll 1
  for (int c = 0; c < nchunk; ++c) {
    const int64_t col = gcol0 + c * 32;
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + tcol0 + c * 32, v);
    tmem_ld_wait();
    if (my_row < p.M && in_part) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (col + 4 * j < p.Nout)
          __stcg(reinterpret_cast<float4*>(mine + my_row * p.Nout + col + 4 * j),
                 make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                             __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
    }
  }
  __threadfence();
  asm volatile("bar.sync 1, %0;" ::"n"(NUM_DEQ_WARPS * 32) : "memory");
  if (ticket_thread) {
    s_last = 0;
    if (QLORA_CHECK(tile < p.ticket_cap, &g_gemm_error, kBoundsTicket)) {
      const int before = atomicAdd(&p.tickets[tile], 1);
      (void)QLORA_CHECK(before < p.nsplit, &g_gemm_error, kBoundsTicket);
      s_last = before == p.nsplit - 1;
    }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(NUM_DEQ_WARPS * 32) : "memory");
  const bool last = s_last != 0;
  if (last) {
    __threadfence();
    if (ticket_thread) p.tickets[tile] = 0;  // ready for the next launch
  }
  return last;
}

// v: this CTA's 32 values of row my_row at output columns gcol .. gcol + 31 (from TMEM);
// becomes the sum over the splits in split order (the other splits' values from part).
__device__ __forceinline__ void split_sum(const Params& p, int split, int64_t my_row, int64_t gcol,
                                          uint32_t (&v)[32]) {
  if (p.nsplit <= 1 || my_row >= p.M) return;
  const size_t MN = static_cast<size_t>(p.M) * p.Nout;
  if (!QLORA_CHECK(static_cast<int64_t>(p.nsplit * MN) <= p.part_cap, &g_gemm_error, kBoundsPartial))
    return;
  // all loads of the chunk first (up to 4 splits x 8 float4 in flight), then the sums in
  // split order
  constexpr int kMaxSplit = 4;
  float4 t[kMaxSplit][8];
#pragma unroll
  for (int z = 0; z < kMaxSplit; ++z)
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (z < p.nsplit && z != split && gcol + 4 * j < p.Nout)
        t[z][j] = __ldcg(reinterpret_cast<const float4*>(p.part + z * MN + my_row * p.Nout + gcol + 4 * j));
      else
        t[z][j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                              __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
    }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float4 acc = t[0][j];
#pragma unroll
    for (int z = 1; z < kMaxSplit; ++z)
      if (z < p.nsplit) acc.x += t[z][j].x, acc.y += t[z][j].y, acc.z += t[z][j].z, acc.w += t[z][j].w;
    v[4 * j] = __float_as_uint(acc.x);
    v[4 * j + 1] = __float_as_uint(acc.y);
    v[4 * j + 2] = __float_as_uint(acc.z);
    v[4 * j + 3] = __float_as_uint(acc.w);
  }
}

// The 16-bit output of this warp's 32 TMEM lanes (row0 .. row0 + 31; my_row = row0 + lane):
// nchunk 32-column chunks, chunk c from TMEM columns tcol0 + 32 c to output columns
// gcol0 + 32 c.  Each chunk goes through a 2 KB buffer of its own (64-byte swizzle; the ring's
// shared memory is idle once the accumulator is complete) and one TMA store, so no store
// waits for an earlier one to release its buffer.
// recv (split clusters): the other split's values of this CTA's 128 columns, [128 rows] x
// [32 16-byte pieces] fp32, piece q of row rr at q ^ (rr & 7); the sum is split 0's value plus
// split 1's, as split_sum forms it.
template <bool H>
__device__ __forceinline__ void epilogue_store(const Params& p, const CUtensorMap* tmOut,
                                               uint32_t taddr, int tcol0, int64_t gcol0,
                                               int64_t row0, int64_t my_row, int split,
                                               int nchunk, uint8_t* buf0, int lane,
                                               const uint8_t* recv = nullptr, int rr = 0) {
#pragma unroll 1
  for (int c = 0; c < nchunk; ++c) {
    const int64_t col = gcol0 + c * 32;
    uint32_t v[32];
    tmem_ld_32x32b_x32(taddr + tcol0 + c * 32, v);
    tmem_ld_wait();
    if (recv) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 o = *reinterpret_cast<const float4*>(recv + rr * 512 + (((c * 8 + j) ^ (rr & 7)) << 4));
        const float ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float mine = __uint_as_float(v[4 * j + e]);
          v[4 * j + e] = __float_as_uint(split == 0 ? mine + ov[e] : ov[e] + mine);
        }
      }
    } else {
      split_sum(p, split, my_row, col, v);
    }
    uint8_t* buf = buf0 + c * 2048;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t phys = j ^ ((lane >> 1) & 3);  // 64-byte swizzle
      *reinterpret_cast<uint4*>(buf + lane * 64 + phys * 16) = make_uint4(
          pack_pair<H>(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
          pack_pair<H>(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
          pack_pair<H>(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
          pack_pair<H>(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (col < p.Nout && row0 < p.M) tma_store_2d(tmOut, buf, (int32_t)col, (int32_t)row0);
      bulk_commit();
    }
  }
  if (lane == 0) bulk_wait_all();
  __syncwarp();
}

// kMode 0: forward (W tile K-major), 1: input gradient (MN-major).  H: the fp16 compute type
// (operands, dequantized tiles and output in fp16), else bf16.
template <int kMode, int kAcc, bool H>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fused_nf4_lora_gemm(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmB2,
                        const __grid_constant__ CUtensorMap tmOut,
                        const __grid_constant__ CUtensorMap tmW, const Params p) {
  using T = Tile<kAcc>;
  constexpr int BM = T::BM, SA = T::SA, SB = T::SB, A_BYTES = T::A_BYTES, B_BASE = T::B_BASE;
  constexpr int TMEM_COLS = T::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t a_full[SA];
  __shared__ __align__(8) uint64_t a_empty[SA];
  __shared__ __align__(8) uint64_t bready_bar[SB];
  __shared__ __align__(8) uint64_t b_empty[SB];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ __align__(8) uint64_t peer_free, peer_data;  // split clusters (see csplit)
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  __shared__ int s_last;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n0 = (int64_t)blockIdx.x * BN;  // output-column tile
  const int64_t m0 = (int64_t)blockIdx.y * BM;  // token tile
  const int split = static_cast<int>(blockIdx.z);
  const int n_all = static_cast<int>(p.Kc / BK);
  const int kc0 = split * p.split_stages;  // first NF4 stage (global k-slice) of this split
  const int n_main = min(n_all, kc0 + p.split_stages) - kc0;
  const bool last_split = split == p.nsplit - 1;
  const int total = (last_split ? p.n_lora : 0) + n_main;
  volatile int* abort_p = &abort_flag;
  // the two splits of a tile as a cluster (rank = split): each finishes 128 of the 256 columns
  const bool cx = kAcc == 1 && p.csplit != 0 && p.nsplit == 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&bready_bar[i], NUM_DEQ_WARPS);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(&acc_bar, 1);
    mbar_init(&peer_free, 1);  // the peer: its B ring may take this CTA's half
    mbar_init(&peer_data, 4);  // the peer's four sending warps: their half has arrived
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc<1>(&tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  if (cx) cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one_sync()) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
      if (p.wstage) tma_prefetch_desc(&tmW);
      for (int s = 0; s < total; ++s) {
        const int as = s % SA, ar = s / SA;
        if (ar > 0 && !mbar_wait(&a_empty[as], (ar - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error)) break;
        uint8_t* a_dst = smem + as * A_BYTES;
        if (s < n_main && p.wstage) {
          // staged base: the W tile by TMA into the B slot, once that slot is free
          const int bs = s % SB, br = s / SB;
          if (br > 0 && !mbar_wait(&b_empty[bs], (br - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error)) break;
          uint8_t* b_dst = smem + B_BASE + bs * B_BYTES;
          if (s == 0) grid_dependency_wait();  // W' comes from the kernel before
          const int32_t k0 = (kc0 + s) * BK;
          mbar_arrive_expect_tx(&a_full[as], A_BYTES + B_BYTES);
          tma_load_2d(a_dst, &tmA, &a_full[as], k0, (int32_t)m0);
          if (kMode == 0) {
            tma_load_2d(b_dst, &tmW, &a_full[as], k0, (int32_t)n0);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              tma_load_2d(b_dst + i * 8192, &tmW, &a_full[as], (int32_t)(n0 + 64 * i), k0);
          }
        } else if (s >= n_main) {
          // a LoRA stage: its B tile comes by TMA into the B slot, once that slot is free
          const int bs = s % SB, br = s / SB;
          if (br > 0 && !mbar_wait(&b_empty[bs], (br - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error)) break;
          uint8_t* b_dst = smem + B_BASE + bs * B_BYTES;
          const int li = s - n_main;
          if (li == 0) grid_dependency_wait();  // sU / sV (and Bp) come from the kernel before
          mbar_arrive_expect_tx(&a_full[as], A_BYTES + B_BYTES);
          tma_load_2d(a_dst, &tmA2, &a_full[as], li * BK, (int32_t)m0);
          if (kMode == 0) {
            tma_load_2d(b_dst, &tmB2, &a_full[as], li * BK, (int32_t)n0);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              tma_load_2d(b_dst + i * 8192, &tmB2, &a_full[as], (int32_t)(n0 + 64 * i), li * BK);
          }
        } else {
          mbar_arrive_expect_tx(&a_full[as], A_BYTES);
          tma_load_2d(a_dst, &tmA, &a_full[as], (kc0 + s) * BK, (int32_t)m0);
        }
      }
      // never leave with a load in flight: the last issued stages must have landed
      for (int s = total - SA < 0 ? 0 : total - SA; s < total; ++s)
        mbar_wait(&a_full[s % SA], (s / SA) & 1, kWaitTmaFull, abort_p, &g_gemm_error);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    if (elect_one_sync()) {
      constexpr uint32_t idesc = idesc_bf16_f32(UM, BN, 0, kMode, H);
      bool ok = true;
      for (int s = 0; s < total && ok; ++s) {
        const int as = s % SA, ar = s / SA, bs = s % SB, br = s / SB;
        // the LoRA stages (the last ones), and every stage of a staged base, come entirely by
        // TMA: no dequantized tile to wait for
        ok = mbar_wait(&a_full[as], ar & 1, kWaitTmaFull, abort_p, &g_gemm_error) &&
             (s >= n_main || p.wstage ||
              mbar_wait(&bready_bar[bs], br & 1, kWaitBReady, abort_p, &g_gemm_error));
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + as * A_BYTES);
        const uint32_t b_addr = smem_u32(smem + B_BASE + bs * B_BYTES);
        const int ksteps = (s >= n_main && s == total - 1) ? p.lora_last_k16 : 4;
        for (int kk = 0; kk < ksteps; ++kk) {
          const uint64_t bdesc = (kMode == 0)
                                     ? smem_desc(b_addr + kk * 32, 16, 1024, Swizzle::B128)
                                     : smem_desc(b_addr + kk * 2048, 8192, 1024, Swizzle::B128);
#pragma unroll
          for (int acc = 0; acc < kAcc; ++acc) {
            // accumulator acc: A rows 128 acc .. 128 acc + 127 (16 KB apart), TMEM columns 256 acc
            const uint64_t adesc =
                smem_desc(a_addr + acc * (UM * BK * 2) + kk * 32, 16, 1024, Swizzle::B128);
            umma_bf16_ss<1>(tmem + acc * 256, adesc, bdesc, idesc, (s > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&a_empty[as]);
        umma_commit(&b_empty[bs]);
      }
      if (ok) umma_commit(&acc_bar);
    }
    __syncwarp();
  } else if (warp >= DEQ_WARP0) {
    // ------------------------------------------------------------ NF4 producers
    const int dt = threadIdx.x - DEQ_WARP0 * 32;  // 0..255
    const float mu = p.dq ? __ldg(p.mean) : 0.0f;
    int64_t row_base, kcol;
    uint32_t dst_off, swz;
    if (kMode == 0) {
      row_base = n0 + dt;  // one W row per thread, k-slice of the stage
      kcol = 0;
      dst_off = dt * 128;
      swz = dt & 7;
    } else {
      const int nl = (dt & 7) + 8 * ((dt >> 3) & 7);  // W row within the stage's 64
      const int blk = dt >> 6;                         // which 64 of the tile's 256 columns
      row_base = nl;
      kcol = n0 + blk * 64;
      dst_off = blk * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      swz = nl & 7;
    }
    auto slice_at = [&](int s, Slice& sl) {  // local NF4 stage s of this split
      sl.valid = false;
      if (s >= n_main) return;
      const int kc = kc0 + s;
      if (kMode == 0) load_slice(sl, p, row_base, (int64_t)kc * BK);
      else load_slice(sl, p, (int64_t)kc * BK + row_base, kcol);
    };
    // Slices four stages ahead in four register sets (set s & 3 holds stage s): a set is
    // refilled right after its stage was stored and signalled.  Each stage is dequantized into
    // registers before its B slot is free, so a freed slot only takes the stores.
    auto body = [&](int s, Slice& cur) -> bool {
      const int slot = s % SB, round = s / SB;
      uint4 rv[8];
      if (cur.valid) {
        const Nf4ByteTable tab = nf4_make_table<H>(__fmaf_rn(cur.q, cur.step, mu));
        const uint32_t words[8] = {cur.c0.x, cur.c0.y, cur.c0.z, cur.c0.w,
                                   cur.c1.x, cur.c1.y, cur.c1.z, cur.c1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[4];
          nf4_dequant8(tab, words[c], o);
          rv[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) rv[c] = make_uint4(0, 0, 0, 0);
      }
      if (round > 0 && !mbar_wait(&b_empty[slot], (round - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error))
        return false;
      uint8_t* dst = smem + B_BASE + slot * B_BYTES + dst_off;
#pragma unroll
      for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + ((c ^ swz) << 4)) = rv[c];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bready_bar[slot]);
      // the set just consumed takes the stage four ahead; its loads are issued after the
      // (release) arrive above, which therefore never waits for them
      slice_at(s + 4, cur);
      return true;
    };
    bool ok = true;
    if (!p.wstage) {  // (a staged base needs no dequantization here)
      Slice pf0, pf1, pf2, pf3;
      slice_at(0, pf0);
      slice_at(1, pf1);
      slice_at(2, pf2);
      slice_at(3, pf3);
      for (int s = 0; s < n_main && ok; s += 4) {  // the NF4 stages (the LoRA stages need nothing)
        ok = body(s, pf0);
        if (!ok || s + 1 >= n_main) break;
        ok = body(s + 1, pf1);
        if (!ok || s + 2 >= n_main) break;
        ok = body(s + 2, pf2);
        if (!ok || s + 3 >= n_main) break;
        ok = body(s + 3, pf3);
      }
    }

    // ------------------------------------------------------------ epilogue
    if (ok && mbar_wait(&acc_bar, 0, kWaitAccFull, abort_p, &g_gemm_error)) {
      tc_fence_after();
      const int lg = warp & 3;                     // TMEM lanes 32*lg .. 32*lg+31
      const int half = (warp - DEQ_WARP0) >> 2;    // kAcc 1: column half; kAcc 2: accumulator
      constexpr int NCHUNK = kAcc == 1 ? 4 : 8;    // 32-column chunks per warp
      const int col0 = kAcc == 1 ? half * 128 : 0;
      const uint32_t tbase = tmem + (kAcc == 1 ? 0u : static_cast<uint32_t>(half * 256));
      const int64_t row0 = m0 + (kAcc == 1 ? 0 : half * UM) + lg * 32;
      const int64_t my_row = row0 + lane;
      uint8_t* buf0 = smem + (warp - DEQ_WARP0) * (NCHUNK * 2048);
      const uint32_t taddr = tbase + (static_cast<uint32_t>(lg * 32) << 16);
      if (cx) {
        // This CTA's B ring is idle now (every stage consumed): the peer may write its half
        // there.  The warps of the column half the peer owns send their values to the peer's
        // ring (fp32, piece q of row rr at q ^ (rr & 7)); the others wait for the peer's half
        // and store the sums of their 128 columns.
        const uint32_t peer = static_cast<uint32_t>(split ^ 1);
        uint8_t* recv = smem + B_BASE;
        const int rr = lg * 32 + lane;
        if (warp == DEQ_WARP0 && lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&peer_free), peer));
        if (half != split) {
          if (mbar_wait<true>(&peer_free, 0, kWaitPeer, abort_p, &g_gemm_error)) {
            const uint32_t rbase = mapa_shared(smem_u32(recv), peer) + static_cast<uint32_t>(rr * 512);
#pragma unroll 1
            for (int c = 0; c < NCHUNK; ++c) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(taddr + col0 + c * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 8; ++j)
                asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                                 rbase + static_cast<uint32_t>(((c * 8 + j) ^ (rr & 7)) << 4)),
                             "r"(v[4 * j]), "r"(v[4 * j + 1]), "r"(v[4 * j + 2]), "r"(v[4 * j + 3])
                             : "memory");
            }
            asm volatile("fence.acq_rel.cluster;" ::: "memory");  // this lane's stores, cluster-wide
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&peer_data), peer));
          }
        } else if (mbar_wait<true>(&peer_data, 0, kWaitPeer, abort_p, &g_gemm_error)) {
          epilogue_store<H>(p, &tmOut, taddr, col0, n0 + col0, row0, my_row, split, NCHUNK, buf0,
                            lane, recv, rr);
        }
      } else {
        const bool store = split_epilogue_partial(p, split, taddr, my_row, n0 + col0, NCHUNK, col0,
                                                  warp == DEQ_WARP0 && lane == 0,
                                                  static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x), s_last);
        if (store)
          epilogue_store<H>(p, &tmOut, taddr, col0, n0 + col0, row0, my_row, split, NCHUNK, buf0, lane);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA of a split cluster leaves while the other may still write into it
  if (cx) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, TMEM_COLS);
  }
}

// ============================================================================ CTA pairs
// The same GEMMs on CTA pairs (cta_group::2).  A pair owns a 512 x 256 output tile: each CTA
// holds 256 rows of X/dY (two 128-row slabs) and half of the dequantized W tile (128 W rows
// for the forward, 128 output columns for the input gradient), the leader issues UMMAs of
// M = 256 (128 rows from each CTA) x N = 256 (128 columns from each CTA's W half) into two
// TMEM accumulators per CTA.  Each SM now dequantizes 8192 weights per stage for 4 x 128 x 256
// x 64 multiply-adds: twice the tensor work per integer-pipe instruction of the single-CTA
// 256 x 256 tile, and a quarter of its W tile in shared memory.
//   a_full     (leader) TMA bytes of both CTAs            waited by the leader's UMMA thread
//   a_empty    (each)   multicast tcgen05.commit          waited by each CTA's TMA thread
//   bready_bar (leader) the leader's 4 dequant warps + one peer relay lane, waited by the
//                       leader's UMMA thread
//   pready_bar (peer)   the peer's 4 dequant warps        waited by the peer's relay lane
// The dequant warps signal at CTA scope only; one lane of the peer per B slot forwards
// each stage to the leader with a single cluster-scope release (measured: a cluster-scope
// release costs ~0.6 us, more than the dequantization of a stage; one per warp and stage
// made the dequant warps the bottleneck, one thread for all stages made it the relay).
//   b_empty    (each)   multicast tcgen05.commit          waited by each CTA's dequant warps
//                                                         (and TMA thread, LoRA stages)
//   acc_bar    (each)   multicast tcgen05.commit          waited by each CTA's epilogue
// Two dequant groups of 4 warps take alternate stages (one 64-weight block per thread each).
// The A tiles (X / dY, by TMA) and the B tiles (dequantized W halves) sit in two rings of
// their own.  The B ring is the deeper one (six stages against four): a B slot goes round a
// longer loop -- the MMA's commit reaches both CTAs, the dequant warps store the stage they
// hold in registers, fence and signal, and the peer's relay forwards its half with a
// cluster-scope release -- measured at ~2 us on the 4096^2 step, so with one ring of four the
// MMA thread waited ~0.3 us for every stage's B tile while the A tiles were always there.  The
// LoRA stages take an A slot and a B slot, both by TMA.
namespace pairk {
constexpr int BM_CTA = 256;
constexpr int BN_CTA = 128;
constexpr int SA = 4;                      // A ring
constexpr int SB = 6;                      // B ring
constexpr int A_BYTES = BM_CTA * BK * 2;   // 32 KB
constexpr int B_BYTES = BN_CTA * BK * 2;   // 16 KB
constexpr int B_BASE = SA * A_BYTES;
constexpr int SMEM_BYTES = SA * A_BYTES + SB * B_BYTES + 1024;
constexpr int GROUP_WARPS = 4;
constexpr int TMEM_COLS = 512;
}  // namespace pairk

template <int kMode, bool H>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    fused_pair_gemm(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmA2,
                    const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmOut, const Params p) {
  using pairk::BM_CTA; using pairk::BN_CTA; using pairk::SA; using pairk::SB; using pairk::A_BYTES;
  using pairk::B_BASE; using pairk::GROUP_WARPS; using pairk::TMEM_COLS;
  constexpr int B_BYTES = pairk::B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t a_full[SA];    // (leader) TMA bytes of both CTAs
  __shared__ __align__(8) uint64_t a_empty[SA];   // (each) multicast commit of the stage's MMAs
  __shared__ __align__(8) uint64_t bready_bar[SB];
  __shared__ __align__(8) uint64_t pready_bar[SB];
  __shared__ __align__(8) uint64_t b_empty[SB];   // (each) multicast commit
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  __shared__ int s_last;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();           // 0: leader, 1: peer
  const int64_t m0 = (int64_t)(blockIdx.x >> 1) * 512 + rank * BM_CTA;  // this CTA's A rows
  const int64_t n0 = (int64_t)blockIdx.y * BN;                          // pair's columns
  const int64_t nb0 = n0 + rank * BN_CTA;                               // this CTA's W half
  const int split = static_cast<int>(blockIdx.z);
  const int n_all = static_cast<int>(p.Kc / BK);
  const int kc0 = split * p.split_stages;  // first NF4 stage (global k-slice) of this split
  const int n_main = min(n_all, kc0 + p.split_stages) - kc0;
  const int total = (split == p.nsplit - 1 ? p.n_lora : 0) + n_main;
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&bready_bar[i], GROUP_WARPS + 1);
      mbar_init(&pready_bar[i], GROUP_WARPS);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(&acc_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc<2>(&tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's barriers exist before the peer signals them
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (elect_one_sync()) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
      for (int s = 0; s < total; ++s) {
        const int as = s % SA, ar = s / SA;
        if (ar > 0 &&
            !mbar_wait<true>(&a_empty[as], (ar - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error))
          break;
        const uint32_t full_lead = mapa_shared(smem_u32(&a_full[as]), 0);
        uint8_t* a_dst = smem + as * A_BYTES;
        if (s >= n_main) {
          // a LoRA stage: its B tile comes by TMA into the B slot, once that slot is free
          const int bs = s % SB, br = s / SB;
          if (br > 0 &&
              !mbar_wait<true>(&b_empty[bs], (br - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error))
            break;
          uint8_t* b_dst = smem + B_BASE + bs * B_BYTES;
          const int li = s - n_main;
          if (li == 0) grid_dependency_wait();  // sU / sV (and Bp) come from the kernel before
          if (rank == 0) mbar_arrive_expect_tx(&a_full[as], 2 * (A_BYTES + B_BYTES));
          tma_load_2d_pair(a_dst, &tmA2, full_lead, li * BK, (int32_t)m0);
          if (kMode == 0) {
            tma_load_2d_pair(b_dst, &tmB2, full_lead, li * BK, (int32_t)nb0);
          } else {
#pragma unroll
            for (int i = 0; i < 2; ++i)
              tma_load_2d_pair(b_dst + i * 8192, &tmB2, full_lead, (int32_t)(nb0 + 64 * i), li * BK);
          }
        } else {
          if (rank == 0) mbar_arrive_expect_tx(&a_full[as], 2 * A_BYTES);
          tma_load_2d_pair(a_dst, &tmA, full_lead, (kc0 + s) * BK, (int32_t)m0);
        }
      }
      // the leader's full barriers count both CTAs' copies: the leader drains them
      if (rank == 0)
        for (int s = total - SA < 0 ? 0 : total - SA; s < total; ++s)
          mbar_drain(&a_full[s % SA], (s / SA) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer (leader)
    if (rank == 0 && elect_one_sync()) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * UM, BN, 0, kMode, H);
      bool ok = true;
      for (int s = 0; s < total && ok; ++s) {
        const int as = s % SA, ar = s / SA, bs = s % SB, br = s / SB;
        // the LoRA stages (the last ones) come entirely by TMA: no dequantized tile to wait for
        ok = mbar_wait<true>(&a_full[as], ar & 1, kWaitTmaFull, abort_p, &g_gemm_error) &&
             (s >= n_main ||
              mbar_wait<true>(&bready_bar[bs], br & 1, kWaitBReady, abort_p, &g_gemm_error));
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_addr = smem_u32(smem + as * A_BYTES);
        const uint32_t b_addr = smem_u32(smem + B_BASE + bs * B_BYTES);
        const int ksteps = (s >= n_main && s == total - 1) ? p.lora_last_k16 : 4;
        for (int kk = 0; kk < ksteps; ++kk) {
          const uint64_t bdesc = (kMode == 0)
                                     ? smem_desc(b_addr + kk * 32, 16, 1024, Swizzle::B128)
                                     : smem_desc(b_addr + kk * 2048, 8192, 1024, Swizzle::B128);
#pragma unroll
          for (int acc = 0; acc < 2; ++acc) {
            const uint64_t adesc =
                smem_desc(a_addr + acc * (UM * BK * 2) + kk * 32, 16, 1024, Swizzle::B128);
            umma_bf16_ss<2>(tmem + acc * 256, adesc, bdesc, idesc, (s > 0 || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit_pair(&a_empty[as], 0x3);
        umma_commit_pair(&b_empty[bs], 0x3);
      }
      if (ok) umma_commit_pair(&acc_bar, 0x3);
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ relay (peer)
    // each stage's dequantized half of the peer, forwarded to the leader's bready barrier;
    // one lane per B slot, so the (slow) cluster-scope releases of consecutive stages are in
    // flight together
    if (rank == 1 && lane < SB) {
      const uint32_t bready_lead = mapa_shared(smem_u32(&bready_bar[lane]), 0);
      for (int s = lane; s < n_main; s += SB) {
        if (!mbar_wait(&pready_bar[lane], (s / SB) & 1, kWaitBReady, abort_p, &g_gemm_error))
          break;
        mbar_arrive_cluster(bready_lead);
      }
    }
    __syncwarp();
  } else if (warp >= DEQ_WARP0) {
    // ------------------------------------------------------------ NF4 producers (both CTAs)
    const int group = (warp - DEQ_WARP0) / GROUP_WARPS;           // owns stages s % 2 == group
    const int t = ((warp - DEQ_WARP0) % GROUP_WARPS) * 32 + lane;  // 0..127
    const float mu = p.dq ? __ldg(p.mean) : 0.0f;
    int64_t row_base, kcol;
    uint32_t dst_off, swz;
    if (kMode == 0) {
      row_base = nb0 + t;  // one W row per thread, k-slice of the stage
      kcol = 0;
      dst_off = t * 128;
      swz = t & 7;
    } else {
      const int nl = (t & 7) + 8 * ((t >> 3) & 7);  // W row within the stage's 64
      const int blk = t >> 6;                        // which 64 of this CTA's 128 columns
      row_base = nl;
      kcol = nb0 + blk * 64;
      dst_off = blk * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      swz = nl & 7;
    }
    auto slice_at = [&](int s, Slice& sl) {  // local NF4 stage s of this split
      const int kc = kc0 + s;
      if (kMode == 0) load_slice(sl, p, row_base, (int64_t)kc * BK);
      else load_slice(sl, p, (int64_t)kc * BK + row_base, kcol);
    };
    // Each stage is dequantized into registers before its ring slot is free (while the group
    // waits for it), so a freed slot only takes the stores, the proxy fence and the signal.
    // The group's slices alternate between two register sets; a set is refilled right after
    // the stage it held was dequantized, one group iteration before it is needed again.
    uint4 rv[8];
    auto dequant = [&](const Slice& cur) {
      if (cur.valid) {
        const Nf4ByteTable tab = nf4_make_table<H>(__fmaf_rn(cur.q, cur.step, mu));
        const uint32_t words[8] = {cur.c0.x, cur.c0.y, cur.c0.z, cur.c0.w,
                                   cur.c1.x, cur.c1.y, cur.c1.z, cur.c1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[4];
          nf4_dequant8(tab, words[c], o);
          rv[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) rv[c] = make_uint4(0, 0, 0, 0);
      }
    };
    auto put = [&](int s) -> bool {  // NF4 stages only
      const int slot = s % SB, round = s / SB;
      {
        if (round > 0 &&
            !mbar_wait<true>(&b_empty[slot], (round - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error))
          return false;
        uint8_t* dst = smem + B_BASE + slot * B_BYTES + dst_off;
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + ((c ^ swz) << 4)) = rv[c];
        // this CTA's generic-proxy writes, ordered before the tensor core's (async-proxy)
        // reads; the leader sees them through the barriers below
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rank == 0 ? &bready_bar[slot] : &pready_bar[slot]);
      return true;
    };
    auto refill = [&](int s, Slice& sl) {
      sl.valid = false;
      if (s < n_main) slice_at(s, sl);
    };
    Slice sa, sb;
    refill(group, sa);
    refill(group + 2, sb);
    if (group < n_main) dequant(sa);
    bool ok = true;
    for (int s = group; s < n_main && ok; s += 4) {
      if (!(ok = put(s))) break;
      refill(s + 4, sa);
      if (s + 2 >= n_main) break;
      if (s + 2 < n_main) dequant(sb);
      if (!(ok = put(s + 2))) break;
      refill(s + 6, sb);
      if (s + 4 < n_main) dequant(sa);
    }

    // ------------------------------------------------------------ epilogue (both CTAs)
    if (ok && mbar_wait<true>(&acc_bar, 0, kWaitAccFull, abort_p, &g_gemm_error)) {
      tc_fence_after();
      const int lg = warp & 3;                           // TMEM lanes 32*lg .. 32*lg+31
      const int acc = (warp - DEQ_WARP0) >> 2;           // accumulator (128-row slab)
      const uint32_t tbase = tmem + static_cast<uint32_t>(acc * 256);
      const int64_t row0 = m0 + acc * UM + lg * 32;
      const int64_t my_row = row0 + lane;
      uint8_t* buf0 = smem + (warp - DEQ_WARP0) * (8 * 2048);
      const uint32_t taddr = tbase + (static_cast<uint32_t>(lg * 32) << 16);
      const bool store = split_epilogue_partial(p, split, taddr, my_row, n0, 8, 0,
                                                warp == DEQ_WARP0 && lane == 0,
                                                static_cast<int>(blockIdx.y * gridDim.x + blockIdx.x),
                                                s_last);
      if (store) epilogue_store<H>(p, &tmOut, taddr, 0, n0, row0, my_row, split, 8, buf0, lane);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its pair may still touch its barriers or smem
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<2>(tmem, TMEM_COLS);
  }
}


// ============================================================================ persistent pairs
// The pair GEMM with the tiles shared out among resident CTA pairs (one wave of clusters).
// Each cluster's leader draws an arrival ticket k and the cluster takes tiles k, k + G, ...
// (G clusters): the pairs that start first (the others may wait for SMs still held by the
// rank-r kernel before this one) take the second tiles.  The rings and their barrier phases
// run on across the tiles (global stage counter); between tiles the dequant warps first fill
// the B ring with the next tile's first stages, then drain the accumulators (tcgen05.ld ->
// 16-bit -> global stores straight from registers: the ring's shared memory is in use) and
// release TMEM to the MMA issuer (tmem_empty, all 16 epilogue warps of the pair), so the next
// tile starts on a full ring instead of a cold prologue.
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

template <int kMode, bool H>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    fused_pair_persistent(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmA2,
                          const __grid_constant__ CUtensorMap tmB2,
                          const __grid_constant__ CUtensorMap tmOut, const Params p) {
  using pairk::BM_CTA; using pairk::BN_CTA; using pairk::SA; using pairk::SB; using pairk::A_BYTES;
  using pairk::B_BASE; using pairk::GROUP_WARPS; using pairk::TMEM_COLS;
  constexpr int B_BYTES = pairk::B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t a_full[SA];    // (leader) TMA bytes of both CTAs
  __shared__ __align__(8) uint64_t a_empty[SA];   // (each) multicast commit of the stage's MMAs
  __shared__ __align__(8) uint64_t bready_bar[SB];
  __shared__ __align__(8) uint64_t pready_bar[SB];
  __shared__ __align__(8) uint64_t b_empty[SB];   // (each) multicast commit
  __shared__ __align__(8) uint64_t acc_bar;       // (each) multicast commit after a tile's MMAs
  __shared__ __align__(8) uint64_t tmem_empty;    // (leader) the pair's 16 epilogue warps
  __shared__ __align__(8) uint64_t staging_free;  // (each) its 8 epilogue warps' stores read
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int s_ticket;
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // 0: leader, 1: peer
  const int n_main = static_cast<int>(p.Kc / BK);
  const int total = p.n_lora + n_main;
  const int64_t row_blocks = (p.M + 511) / 512;
  const int64_t ntiles_all = row_blocks * ((p.Nout + BN - 1) / BN);
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&bready_bar[i], GROUP_WARPS + 1);
      mbar_init(&pready_bar[i], GROUP_WARPS);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(&acc_bar, 1);
    mbar_init(&tmem_empty, 2 * NUM_DEQ_WARPS);
    mbar_init(&staging_free, NUM_DEQ_WARPS);
    abort_flag = 0;
    if (rank == 0) s_ticket = atomicAdd(p.pers_ctr, 1);  // this cluster's place in arrival order
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc<2>(&tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's barriers and ticket exist before the peer uses them
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int ticket = rank == 0 ? s_ticket
                               : static_cast<int>(ld_shared_cluster_u32(mapa_shared(smem_u32(&s_ticket), 0)));
  const int G = p.pers_clusters;
  const int ntiles = ticket < ntiles_all ? static_cast<int>((ntiles_all - ticket + G - 1) / G) : 0;
  // tile i of this cluster: this CTA's A rows and W half
  const int rb = static_cast<int>(row_blocks);
  auto tile_m0 = [&](int i) -> int64_t {
    const int t = ticket + i * G;
    return (int64_t)(t % rb) * 512 + rank * BM_CTA;
  };
  auto tile_n0 = [&](int i) -> int64_t {
    const int t = ticket + i * G;
    return (int64_t)(t / rb) * BN;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (elect_one_sync()) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
      int g = 0;  // global stage
      bool ok = true;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int64_t m0 = tile_m0(i), nb0 = tile_n0(i) + rank * BN_CTA;
        for (int s = 0; s < total; ++s, ++g) {
          const int as = g % SA, ar = g / SA;
          if (ar > 0 &&
              !mbar_wait<true>(&a_empty[as], (ar - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error)) {
            ok = false;
            break;
          }
          const uint32_t full_lead = mapa_shared(smem_u32(&a_full[as]), 0);
          uint8_t* a_dst = smem + as * A_BYTES;
          if (s >= n_main) {
            const int bs = g % SB, br = g / SB;
            if (br > 0 &&
                !mbar_wait<true>(&b_empty[bs], (br - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error)) {
              ok = false;
              break;
            }
            uint8_t* b_dst = smem + B_BASE + bs * B_BYTES;
            const int li = s - n_main;
            if (i == 0 && li == 0) grid_dependency_wait();  // sU / sV (and Bp): the kernel before
            if (rank == 0) mbar_arrive_expect_tx(&a_full[as], 2 * (A_BYTES + B_BYTES));
            tma_load_2d_pair(a_dst, &tmA2, full_lead, li * BK, (int32_t)m0);
            if (kMode == 0) {
              tma_load_2d_pair(b_dst, &tmB2, full_lead, li * BK, (int32_t)nb0);
            } else {
#pragma unroll
              for (int h = 0; h < 2; ++h)
                tma_load_2d_pair(b_dst + h * 8192, &tmB2, full_lead, (int32_t)(nb0 + 64 * h), li * BK);
            }
          } else {
            if (rank == 0) mbar_arrive_expect_tx(&a_full[as], 2 * A_BYTES);
            tma_load_2d_pair(a_dst, &tmA, full_lead, s * BK, (int32_t)m0);
          }
        }
      }
      // the leader's full barriers count both CTAs' copies: the leader drains them
      if (rank == 0)
        for (int q = g - SA < 0 ? 0 : g - SA; q < g; ++q) mbar_drain(&a_full[q % SA], (q / SA) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer (leader)
    if (rank == 0 && elect_one_sync()) {
      constexpr uint32_t idesc = idesc_bf16_f32(2 * UM, BN, 0, kMode, H);
      bool ok = true;
      int g = 0;
      uint32_t nf4_parity = 0;  // bit j: parity of the NF4 stages through B slot j so far
      for (int i = 0; i < ntiles && ok; ++i) {
        if (i > 0) {  // the previous tile's accumulators drained by both CTAs' epilogues
          if (!(ok = mbar_wait<true>(&tmem_empty, (i - 1) & 1, kWaitAccFull, abort_p, &g_gemm_error)))
            break;
          tc_fence_after();
        }
        for (int s = 0; s < total; ++s, ++g) {
          const int as = g % SA, ar = g / SA, bs = g % SB;
          ok = mbar_wait<true>(&a_full[as], ar & 1, kWaitTmaFull, abort_p, &g_gemm_error);
          if (ok && s < n_main) {
            ok = mbar_wait<true>(&bready_bar[bs], (nf4_parity >> bs) & 1, kWaitBReady, abort_p,
                                 &g_gemm_error);
            nf4_parity ^= 1u << bs;
          }
          if (!ok) break;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + as * A_BYTES);
          const uint32_t b_addr = smem_u32(smem + B_BASE + bs * B_BYTES);
          const int ksteps = (s >= n_main && s == total - 1) ? p.lora_last_k16 : 4;
          for (int kk = 0; kk < ksteps; ++kk) {
            const uint64_t bdesc = (kMode == 0)
                                       ? smem_desc(b_addr + kk * 32, 16, 1024, Swizzle::B128)
                                       : smem_desc(b_addr + kk * 2048, 8192, 1024, Swizzle::B128);
#pragma unroll
            for (int acc = 0; acc < 2; ++acc) {
              const uint64_t adesc =
                  smem_desc(a_addr + acc * (UM * BK * 2) + kk * 32, 16, 1024, Swizzle::B128);
              umma_bf16_ss<2>(tmem + acc * 256, adesc, bdesc, idesc, (s > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit_pair(&a_empty[as], 0x3);
          umma_commit_pair(&b_empty[bs], 0x3);
        }
        if (ok) umma_commit_pair(&acc_bar, 0x3);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ------------------------------------------------------------ relay (peer)
    // each NF4 stage's dequantized half of the peer, forwarded to the leader's bready barrier;
    // lane j serves B slot j (the stages g with g % SB == j), so the cluster-scope releases of
    // consecutive stages are in flight together
    if (rank == 1 && lane < SB) {
      // each lane walks only its own stages (a loop over all stages would reconverge the warp
      // at every stage and serialise the lanes' waits)
      const uint32_t bready_lead = mapa_shared(smem_u32(&bready_bar[lane]), 0);
      uint32_t parity = 0;
      int s = lane;  // stage within the tile of global stage g
      for (int g = lane; g < ntiles * total; g += SB, s += SB) {
        while (s >= total) s -= total;
        if (s >= n_main) continue;  // a LoRA stage: by TMA, nothing to forward
        if (!mbar_wait(&pready_bar[lane], parity, kWaitBReady, abort_p, &g_gemm_error)) break;
        parity ^= 1;
        mbar_arrive_cluster(bready_lead);
      }
    }
    __syncwarp();
  } else if (warp >= DEQ_WARP0) {
    // ------------------------------------------------------------ NF4 producers + epilogue
    const int group = (warp - DEQ_WARP0) / GROUP_WARPS;           // stages s % 2 == group
    const int t = ((warp - DEQ_WARP0) % GROUP_WARPS) * 32 + lane;  // 0..127
    const float mu = p.dq ? __ldg(p.mean) : 0.0f;
    uint32_t dst_off, swz;
    int nl = 0, blk = 0;
    if (kMode == 0) {
      dst_off = t * 128;
      swz = t & 7;
    } else {
      nl = (t & 7) + 8 * ((t >> 3) & 7);  // W row within the stage's 64
      blk = t >> 6;                        // which 64 of this CTA's 128 columns
      dst_off = blk * 8192 + (nl >> 3) * 1024 + (nl & 7) * 128;
      swz = nl & 7;
    }
    // this group's items: (tile i, NF4 stage s = group + 2 j), tile-major, walked by two
    // cursors (the next item to store, and the item whose slice is loaded next) so that no
    // division runs per stage
    const int per = n_main > group ? (n_main - group + 1) / 2 : 0;
    const int nitems = ntiles * per;
    // A slice of NF4 stage s of a tile is 32 code bytes at cbase + s * cstride and the block
    // scale of block bbase + s * bstride (tile-constant bases, so no 64-bit index math per stage)
    struct Cursor {
      int i, j;              // tile of this cluster, item within the tile
      const uint8_t* cbase;  // this thread's code bytes in stage 0 of tile i
      int64_t bbase;         // its 64-block in stage 0
      bool valid;            // its W row / column lies inside W
    };
    const int64_t cstride = kMode == 0 ? BK / 2 : (int64_t)BK * (p.Kw / 2);
    const int64_t bstride = kMode == 0 ? 1 : (int64_t)BK * (p.Kw / 64);
    auto cursor_tile = [&](Cursor& c) {
      const int64_t nb0 = tile_n0(c.i) + rank * BN_CTA;
      const int64_t row = kMode == 0 ? nb0 + t : nl;         // W row in stage 0
      const int64_t kcol = kMode == 0 ? 0 : nb0 + blk * 64;  // W column in stage 0
      c.valid = row < p.Nw && kcol < p.Kw;
      c.cbase = p.codes + row * (p.Kw / 2) + kcol / 2;
      c.bbase = row * (p.Kw / 64) + kcol / 64;
    };
    auto advance = [&](Cursor& c) {
      if (++c.j == per) {
        c.j = 0;
        if (++c.i < ntiles) cursor_tile(c);
      }
    };
    Cursor ld{0, 0, nullptr, 0, false}, st{0, 0, nullptr, 0, false};
    if (ntiles > 0) {
      cursor_tile(ld);
      cursor_tile(st);
    }
    auto next_slice = [&](Slice& sl) {  // the slice of item `ld`, then advance it
      sl.valid = false;
      if (ld.i >= ntiles || per == 0) return;
      const int s = group + 2 * ld.j;
      if (ld.valid) {
        const uint4* src = reinterpret_cast<const uint4*>(ld.cbase + s * cstride);
        sl.c0 = __ldg(src);
        sl.c1 = __ldg(src + 1);
        const int64_t b = ld.bbase + s * bstride;
        if (p.dq) {
          sl.q = nf4_second_level(static_cast<uint8_t>(__ldg(p.qs + b)), p.fp8);
          sl.step = __ldg(p.steps + (b >> 8));
        } else {
          sl.q = 1.0f;
          sl.step = __ldg(p.steps + b);
        }
        sl.valid = true;
      }
      advance(ld);
    };
    uint4 rv[8];
    auto dequant = [&](const Slice& cur) {
      if (cur.valid) {
        const Nf4ByteTable tab = nf4_make_table<H>(__fmaf_rn(cur.q, cur.step, mu));
        const uint32_t words[8] = {cur.c0.x, cur.c0.y, cur.c0.z, cur.c0.w,
                                   cur.c1.x, cur.c1.y, cur.c1.z, cur.c1.w};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t o[4];
          nf4_dequant8(tab, words[c], o);
          rv[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) rv[c] = make_uint4(0, 0, 0, 0);
      }
    };
    auto put = [&]() -> bool {  // item `st`, then advance it
      const int g = st.i * total + group + 2 * st.j;
      advance(st);
      const int slot = g % SB, round = g / SB;
      if (round > 0 &&
          !mbar_wait<true>(&b_empty[slot], (round - 1) & 1, kWaitEmpty, abort_p, &g_gemm_error))
        return false;
      uint8_t* dst = smem + B_BASE + slot * B_BYTES + dst_off;
#pragma unroll
      for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(dst + ((c ^ swz) << 4)) = rv[c];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(rank == 0 ? &bready_bar[slot] : &pready_bar[slot]);
      return true;
    };
    // Epilogue of tile i: this warp's 32 TMEM lanes of its slab, 8 chunks of 32 columns (TMEM
    // -> 16-bit -> 64-byte-swizzled staging -> TMA store, two 2 KB buffers per warp).  The
    // staging lies in the two B slots that the next tile's stages 4 and 5 will take: the groups
    // fill only its first 4 stages before the epilogue, and every previous use of those two
    // slots was consumed before the accumulators were complete.  Then TMEM is released.
    const int lg = warp & 3;                  // TMEM lanes 32 lg .. 32 lg + 31
    const int acc = (warp - DEQ_WARP0) >> 2;  // accumulator (128-row slab)
    const uint32_t taddr = tmem + static_cast<uint32_t>(acc * 256) + (static_cast<uint32_t>(lg * 32) << 16);
    const uint32_t tmem_empty_lead = mapa_shared(smem_u32(&tmem_empty), 0);
    auto epilogue = [&](int i) -> bool {
      if (!mbar_wait<true>(&acc_bar, i & 1, kWaitAccFull, abort_p, &g_gemm_error)) return false;
      tc_fence_after();
      const int g0 = (i + 1) * total;  // the next tile's first stage (or one past the last)
      const int slot = (g0 + 4 + (warp - DEQ_WARP0) / 4) % SB;
      uint8_t* buf0 = smem + B_BASE + slot * B_BYTES + ((warp - DEQ_WARP0) % 4) * 4096;
      const int64_t row0 = tile_m0(i) + acc * UM + lg * 32;
      const int64_t n0 = tile_n0(i);
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(taddr + c * 32, v);
        tmem_ld_wait();
        uint8_t* buf = buf0 + (c & 1) * 2048;
        if (c >= 2) {
          if (lane == 0) bulk_wait_read1();
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t phys = j ^ ((lane >> 1) & 3);  // 64-byte swizzle
          *reinterpret_cast<uint4*>(buf + lane * 64 + phys * 16) = make_uint4(
              pack_pair<H>(__uint_as_float(v[8 * j + 0]), __uint_as_float(v[8 * j + 1])),
              pack_pair<H>(__uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3])),
              pack_pair<H>(__uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5])),
              pack_pair<H>(__uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7])));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (n0 + c * 32 < p.Nout && row0 < p.M)
            tma_store_2d(&tmOut, buf, (int32_t)(n0 + c * 32), (int32_t)row0);
          bulk_commit();
        }
      }
      if (lane == 0) bulk_wait_read0();  // the staging is read: the slots may be refilled
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(&tmem_empty);
        else mbar_arrive_cluster(tmem_empty_lead);
      }
      // every dequant warp's stores have left the staging before either slot is refilled
      // (a bounded wait: a warp that gave up never hangs the others)
      if (lane == 0) mbar_arrive(&staging_free);
      return mbar_wait(&staging_free, i & 1, kWaitAccFull, abort_p, &g_gemm_error);
    };
    // The item stream: `sa` / `sb` hold the slices of the next two items (by item parity);
    // step() stores the next item, starts the load of the one two ahead into the set it frees
    // and dequantizes the following one into registers.
    constexpr int kPre = 2;  // the next tile's stages per group filled before an epilogue
    const int pre = per < kPre ? per : kPre;
    // Two items per iteration with the two register sets in fixed roles, as in the one-tile
    // kernel: `sa` holds the next item (already dequantized into rv), `sb` the one after.
    Slice sa, sb;
    next_slice(sa);
    next_slice(sb);
    if (nitems > 0) dequant(sa);
    bool ok = true;
    int produced = 0;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int target = min((i + 1) * per + (i + 1 < ntiles ? pre : 0), nitems);
      while (ok && produced + 2 <= target) {
        if (!(ok = put())) break;
        next_slice(sa);
        dequant(sb);
        if (!(ok = put())) break;
        next_slice(sb);
        dequant(sa);
        produced += 2;
      }
      if (ok && produced < target) {  // an odd item: store it and let the sets trade roles
        if ((ok = put())) {
          next_slice(sa);
          dequant(sb);
          const Slice tmp = sa;
          sa = sb;
          sb = tmp;
          ++produced;
        }
      }
      if (ok) ok = epilogue(i);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while its pair may still touch its barriers or smem
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<2>(tmem, TMEM_COLS);
  }
}
}  // namespace fused

namespace {

// A 2-D map of 16-bit elements.  The copy is bitwise and the out-of-range fill is all-zero
// bits (+0 in bf16 and in fp16), so the same map serves the fp16 compute type.
bool map_bf16(CUtensorMap* m, const void* base, int64_t inner, int64_t outer, int64_t pitch_elems,
              uint32_t box_inner, uint32_t box_outer, MapSwizzle sw) {
  return make_tensor_map_2d(m, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)inner,
                            (uint64_t)outer, (uint64_t)pitch_elems * 2, box_inner, box_outer, sw);
}

template <int kMode, int kAcc, bool kPair, bool H>
int launch_fused(const LinearArgs& a, const WorkspaceLayout& L, const FusedPlan& plan,
                 cudaStream_t stream) {
  using namespace fused;
  constexpr int BM = kPair ? pairk::BM_CTA : Tile<kAcc>::BM;
  constexpr int SMEM_BYTES = kPair ? pairk::SMEM_BYTES : Tile<kAcc>::SMEM_BYTES;
  constexpr int BNB = kPair ? pairk::BN_CTA : BN;  // W-tile box of one CTA (forward)
  static DeviceCache<int> smem_attr;  // this instantiation's kernel, per device
  {
    const int st = kPair ? ensure_dynamic_smem(smem_attr, fused_pair_gemm<kMode, H>, SMEM_BYTES)
                         : ensure_dynamic_smem(smem_attr, fused_nf4_lora_gemm<kMode, kAcc, H>, SMEM_BYTES);
    if (st) return st;
  }
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const int64_t rp = L.rp;
  CUtensorMap tA, tA2, tB2, tOut;
  bool ok;
  Params p{};
  p.M = a.M;
  p.Kw = a.K;
  p.Nw = a.N;
  p.codes = a.q.codes;
  p.qs = a.q.scale_codes;
  p.steps = a.q.scale_steps;
  p.mean = a.q.scale_mean;
  p.dq = a.q.dq_block != 0 ? 1 : 0;
  p.fp8 = a.q.dq_type == NF4_DQ_FP8 ? 1 : 0;
  p.n_lora = static_cast<int>(rp / 64);
  p.lora_last_k16 = static_cast<int>((a.r - 64 * (p.n_lora - 1) + 15) / 16);
  p.nsplit = plan.nsplit;
  p.split_stages = plan.split_stages;
  // single-CTA tiles with two splits: the splits of a tile are a cluster (grid z)
  p.csplit = !kPair && kAcc == 1 && plan.nsplit == 2 ? 1 : 0;
  if (plan.nsplit > 1 &&  // the workspace layout must have made room for the split tiles
      (L.gpart_bytes < (uint64_t)plan.nsplit * a.M * p.Nout * 4 || L.ngtickets < (uint64_t)plan.tiles))
    return QLORA_ERR_WORKSPACE;
  p.part = plan.nsplit > 1 ? reinterpret_cast<float*>(ws + L.gpart) : nullptr;
  p.tickets = plan.nsplit > 1 ? reinterpret_cast<int*>(ws + L.gtickets) : nullptr;
  p.part_cap = static_cast<int64_t>(L.gpart_bytes / 4);
  p.ticket_cap = static_cast<int64_t>(L.ngtickets);
  if (kMode == 0) {
    p.Nout = a.N;
    p.Kc = a.K;
    ok = map_bf16(&tA, a.X, a.K, a.M, a.K, 64, BM, MapSwizzle::B128) &&
         map_bf16(&tA2, ws + L.sU, a.r, a.M, rp, 64, BM, MapSwizzle::B128) &&  // zeros past r
         (a.r % 8 == 0  // B [N, r] itself; TMA fills the columns past r with zeros
              ? map_bf16(&tB2, a.B, a.r, a.N, a.r, 64, BNB, MapSwizzle::B128)
              : map_bf16(&tB2, ws + L.Bp, rp, a.N, rp, 64, BNB, MapSwizzle::B128)) &&
         map_bf16(&tOut, a.Y, a.N, a.M, a.N, 32, 32, MapSwizzle::B64);
  } else {
    p.Nout = a.K;
    p.Kc = a.N;
    ok = map_bf16(&tA, a.dY, a.N, a.M, a.N, 64, BM, MapSwizzle::B128) &&
         map_bf16(&tA2, ws + L.sV, a.r, a.M, rp, 64, BM, MapSwizzle::B128) &&  // zeros past r
         map_bf16(&tB2, a.A, a.K, a.r, a.K, 64, 64, MapSwizzle::B128) &&  // rows past r: zeros
         map_bf16(&tOut, a.dX, a.K, a.M, a.K, 32, 32, MapSwizzle::B64);
  }
  if (!ok) return QLORA_ERR_CUDA;
  CUtensorMap tW = tB2;  // (not read without a staged base)
  p.wstage = plan.wstage && !kPair && kAcc == 1 ? 1 : 0;
  if (p.wstage) {
    if (L.Wd_bytes < (uint64_t)a.N * a.K * 2) return QLORA_ERR_WORKSPACE;
    // W' [N rows][K]: forward tiles are [64 k x 256 rows], input-gradient tiles four
    // [64 k x 64 rows] boxes (MN-major), as for the adapters of the LoRA stages
    if (!map_bf16(&tW, ws + L.Wd, a.K, a.N, a.K, 64, kMode == 0 ? BN : 64, MapSwizzle::B128))
      return QLORA_ERR_CUDA;
  }
  ProfileScope ps(kMode == 0 ? "fused_fwd_gemm" : "fused_dx_gemm", stream);
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  // programmatic dependent launch: the GEMM may start while the kernel before it (the
  // rank-r product it reads in its last stages) finishes; its TMA thread waits for that
  // kernel before the first LoRA-stage load
  cudaLaunchAttribute attr[3];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributePriority;
  attr[1].val.priority = a.gemm_priority;
  cfg.attrs = attr;
  cfg.numAttrs = a.gemm_priority ? 2 : 1;
  if (p.csplit) {
    attr[cfg.numAttrs].id = cudaLaunchAttributeClusterDimension;
    attr[cfg.numAttrs].val.clusterDim.x = 1;
    attr[cfg.numAttrs].val.clusterDim.y = 1;
    attr[cfg.numAttrs].val.clusterDim.z = 2;
    ++cfg.numAttrs;
  }
  cudaError_t e;
  // (the persistent kernel stages each epilogue in the B slots of the next tile's NF4 stages
  // 4 and 5, so it needs at least 6 NF4 stages)
  if (kPair && plan.nsplit == 1 && p.Kc / BK >= 6) {
    // persistent pairs: one wave of clusters sharing the tiles (the CTA pair is the kernel's
    // compile-time cluster shape)
    static DeviceCache<int> smem_attr_p;
    const int st = ensure_dynamic_smem(smem_attr_p, fused_pair_persistent<kMode, H>, SMEM_BYTES);
    if (st) return st;
    const int64_t tiles = ((a.M + 511) / 512) * ((p.Nout + BN - 1) / BN);
    const int clusters = static_cast<int>(std::min<int64_t>(tiles, num_sms() / 2));
    p.pers_ctr = reinterpret_cast<int*>(ws + L.pers_ctr);
    p.pers_clusters = clusters;
    p.out = kMode == 0 ? a.Y : a.dX;
    p.ld_out = p.Nout;
    cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
    e = cudaLaunchKernelEx(&cfg, fused_pair_persistent<kMode, H>, tA, tA2, tB2, tOut, p);
  } else if (kPair) {  // the CTA pair is the kernel's compile-time cluster shape
    cfg.gridDim = dim3((unsigned)(2 * ((a.M + 511) / 512)), (unsigned)((p.Nout + BN - 1) / BN),
                       (unsigned)plan.nsplit);
    e = cudaLaunchKernelEx(&cfg, fused_pair_gemm<kMode, H>, tA, tA2, tB2, tOut, p);
  } else {
    cfg.gridDim = dim3((unsigned)((p.Nout + BN - 1) / BN), (unsigned)((a.M + BM - 1) / BM),
                       (unsigned)plan.nsplit);
    e = cudaLaunchKernelEx(&cfg, fused_nf4_lora_gemm<kMode, kAcc, H>, tA, tA2, tB2, tOut, tW, p);
  }
  return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace

// Tile plan.  CTA pairs with 512 x 256 tiles when the tiles give at least half the pair
// slots work; single CTAs with 256 x 256 tiles when those fill the SMs; else 128 x 256
// tiles, with the contraction split (up to 4 splits of at least 8 stages of 64) so that
// tiles x splits fill the SMs once.  The pair kernel takes a split contraction too (blockIdx.z),
// which no plan selects at present.
namespace {
void split_into(FusedPlan& pl, int64_t n_all, int64_t want) {
  if (want > 4) want = 4;
  if (want > n_all / 8) want = n_all / 8;
  pl.nsplit = 1;
  pl.split_stages = static_cast<int>(n_all);
  if (want > 1) {
    const int64_t per = (n_all + want - 1) / want;
    pl.split_stages = static_cast<int>(per);
    pl.nsplit = static_cast<int>((n_all + per - 1) / per);  // every split has a stage
  }
}
}  // namespace

// Largest base that plans stage in the workspace: 128 MiB of bf16, about the L2.
constexpr int64_t kStagedBaseMaxWeights = 64LL << 20;

FusedPlan fused_plan(int64_t M, int64_t Nout, int64_t Kc) {
  FusedPlan pl{};
  const int64_t sms = num_sms();
  const int64_t pair_slots = sms / 2;
  const int64_t n_all = Kc / fused::BK;
  const int64_t pair_tiles = ((M + 511) / 512) * ((Nout + 255) / 256);
  // measured at M = 512 with 4096 output columns: 16 pair tiles x 4 splits ran at 255
  // TFLOP/s, 64 single-CTA tiles x 2 splits at 294 -- a pair's 256 KB fp32 tile per split
  // makes the sum of the splits long; pairs stay unsplit
  split_into(pl, n_all, 1);
  if (pair_tiles * 2 >= pair_slots) {
    pl.kind = 2;
    pl.tiles = 2 * pair_tiles;  // CTA tiles (each CTA of a pair takes its own ticket)
    return pl;
  }
  split_into(pl, n_all, 1);
  const int64_t tiles2 = ((M + 255) / 256) * ((Nout + 255) / 256);
  if (tiles2 >= sms) {
    pl.kind = 1;
    pl.tiles = tiles2;
    return pl;
  }
  pl.kind = 0;
  const int64_t tiles1 = ((M + 127) / 128) * ((Nout + 255) / 256);
  split_into(pl, n_all, sms / tiles1);
  pl.tiles = tiles1;
  // Past one row tile each weight would be dequantized once per row tile by the dequant
  // warps, which then set the stage time; dequantizing W' once into the workspace (it stays
  // in L2 at these sizes) and streaming it by TMA is faster.
  pl.wstage = M > 128 && Nout * Kc <= kStagedBaseMaxWeights ? 1 : 0;
  return pl;
}

uint64_t fused_partial_bytes(int64_t M, int64_t N, int64_t K, uint64_t* tickets) {
  const FusedPlan f = fused_plan(M, N, K), d = fused_plan(M, K, N);
  const uint64_t bf = f.nsplit > 1 ? (uint64_t)f.nsplit * M * N * 4 : 0;
  const uint64_t bd = d.nsplit > 1 ? (uint64_t)d.nsplit * M * K * 4 : 0;
  const uint64_t tf = f.nsplit > 1 ? (uint64_t)f.tiles : 0, td = d.nsplit > 1 ? (uint64_t)d.tiles : 0;
  if (tickets) *tickets = tf > td ? tf : td;
  return bf > bd ? bf : bd;
}

template <int kMode, bool H>
static int launch_fused_mode(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  const FusedPlan plan = kMode == 0 ? fused_plan(a.M, a.N, a.K) : fused_plan(a.M, a.K, a.N);
  switch (plan.kind) {
    case 2: return launch_fused<kMode, 2, true, H>(a, L, plan, stream);
    case 1: return launch_fused<kMode, 2, false, H>(a, L, plan, stream);
    default: return launch_fused<kMode, 1, false, H>(a, L, plan, stream);
  }
}

int launch_fused_fwd(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  return a.half ? launch_fused_mode<0, true>(a, L, stream)
                : launch_fused_mode<0, false>(a, L, stream);
}

int launch_fused_dx(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  return a.half ? launch_fused_mode<1, true>(a, L, stream)
                : launch_fused_mode<1, false>(a, L, stream);
}

}  // namespace qlora
