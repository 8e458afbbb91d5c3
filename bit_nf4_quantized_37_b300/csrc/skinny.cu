// skinny.cu -- the decode path: Y = X W'^T + s U B^T for M <= 16 tokens (junaidshaukat.com
// "QLoRA -- the democratization event": serve the 4-bit base plus a separate adapter;
// addaly.com "QLoRA on one card": keep the adapter separate and load it over the base).
// With so few tokens the layer is a stream over the packed weights: every weight byte is
// read once from HBM and nothing of W' is written anywhere.
//
// Arithmetic.  A weight is level[c] * a (a = the block's dequantized absmax), so a row's
// dot product with a token is  sum_b a_b * sum_{k in b} level[c_k] x_k.  The kernel forms
// the inner sums on the warp-level tensor cores from bf16(level[c]) and x (mma.sync
// m16n8k16, fp32 accumulate; weight rows are the MMA rows, tokens the MMA columns) and
// applies a_b to each 64-wide partial in fp32.  This is W' x up to the bf16 rounding of W'
// (the weight enters with its level rounded instead of its product with a), which is far
// inside the GEMM tolerance.  With the scale outside, the code -> operand step is one fixed
// table: byte v of the code stream (elements 2j, 2j+1 in its high and low nibble) maps to
// the bf16 pair (level[v >> 4], level[v & 15]), which is exactly one 32-bit MMA operand
// register.  The table sits in shared memory with one copy per lane (32 KB), so the
// lookups of a warp never collide on a bank: a byte costs one byte-extract, one multiply-
// add for the address and one shared load, instead of the ~10 integer-pipe operations of a
// per-block byte-permute table.
//
// Work split.  The packed codes are walked as stages of [128 rows x KSTEP k] (KSTEP = 512 for
// up to 8 tokens, 256 for up to 16; 128-byte TMA boxes with 128-byte swizzle) together with
// the tokens' [M x KSTEP] slice (64-wide boxes).  A stage reads 256 contiguous bytes of each
// weight row when KSTEP is 512: on B300 a TMA stream of 128-row x 128-byte boxes reached
// 3.9 TB/s, one of 128 x 256 bytes 4.8 TB/s.  The stages of all row blocks, k-fastest, are
// cut into one contiguous run per CTA (one CTA per SM): every SM streams the same number of
// bytes.  A row block whose stages fall to several CTAs ("pieces") is summed, in CTA order,
// by the CTA whose piece completes it (atomic stage count); the piece that starts a row block
// adds the LoRA term s U B^T (B rows by TMA) on the tensor cores as well.
// U = X A^T is formed inside the same launch: the producer warps of the first CTAs each take
// a 256-wide chunk of the contraction once the ring's first stages are on their way, and the
// last of them to finish sums the chunks in chunk order, publishes sU and raises a flag that
// the first LoRA flush of every CTA waits for (bounded).  No LoRA flush comes before a CTA has
// streamed a whole row block or its whole run, long after U is done.
// Inside a stage, warp w dequantizes 64-block (w % BPS) of GPW 16-row groups; the 16
// contraction slots of an MMA map to k = 16 q + 4 i + {0..3} of the block for lane class q
// and MMA i (the contraction order is free as long as the token operand uses the same map).
#include <algorithm>

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

constexpr int THREADS = 512;                     // 16 consumer warps
constexpr int PRODUCERS = 128;                   // one producer warpgroup (one thread per row)
constexpr int ROWS = 128;                        // weight rows per stage (8 groups of 16)
// Byte table: entry v at v * 256 bytes, lane l's copy of it at + 4 l (the upper half of each
// entry row is unused), so one byte_perm forms the address from the code word and 4 l.
constexpr int TABLE_BYTES = 256 * 256;
constexpr int LORA_BOX_BYTES = ROWS * 128;       // B rows [128 x 64 j] bf16, swizzled
constexpr int LORA_BYTES = 2 * LORA_BOX_BYTES;   // rank up to 128
constexpr int SU_PITCH = 128 + 8;                // bf16 per token row of the staged sU
constexpr int SU_BYTES = 16 * SU_PITCH * 2;
constexpr int SCALE_AHEAD = 4;                   // stages between a scale load and its use
constexpr int U_KC = 256;                        // contraction chunk of one U-computing CTA
// Fixed shared-window layout.  The byte table sits at a 64 KB boundary, so the window
// address of entry v, lane l's copy, is (0x02 << 16) | (v << 8) | 4 l: one byte_perm of the
// code word and a per-lane constant forms it, with no add.  The TMA ring and the staged sU
// lie below the table, the LoRA B-row tile (shared with the reduction) above it.
constexpr uint32_t kStageBase = 0x800;
constexpr uint32_t kTableBase = 0x20000;
constexpr uint32_t kLoraBase = kTableBase + TABLE_BYTES;

// NT token octets (M <= 8 NT).
template <int NT>
struct Cfg {
  static constexpr int KSTEP = 256;                       // k per stage
  static constexpr int BPS = KSTEP / 64;                  // 64-blocks per stage
  static constexpr int GPW = BPS / 2;                     // 16-row groups per consumer warp
  static constexpr int CODE_BYTES = ROWS * KSTEP / 2;     // 32 or 16 KB (128-byte boxes)
  static constexpr int XSLOT = NT * 8 * 128;              // [8 NT tokens x 64 k] bf16
  static constexpr int STAGE_BYTES = CODE_BYTES + BPS * XSLOT;
  static constexpr int STAGES = NT == 1 ? 6 : 5;
  static constexpr int TAB_ROWS = ROWS * BPS / 32;        // byte-table rows of a stage's scales
  static constexpr int ACC = GPW * NT * 4;                // accumulators per lane
  static constexpr int RED_BYTES = (THREADS / 32) * 32 * ACC * 4;
  // the B-row tile of the LoRA term and the cross-warp reduction share one region: the
  // tile is consumed before the reduction writes it
  static constexpr int LR_BYTES = LORA_BYTES > RED_BYTES ? LORA_BYTES : RED_BYTES;
  static constexpr uint32_t SU_BASE = kStageBase + STAGES * STAGE_BYTES;
  static constexpr uint32_t SMEM_END = kLoraBase + LR_BYTES;  // end of the used window
};
static_assert(Cfg<1>::SU_BASE + SU_BYTES <= kTableBase, "decode ring below the byte table");
static_assert(Cfg<2>::SU_BASE + SU_BYTES <= kTableBase, "decode ring below the byte table");
static_assert(Cfg<1>::SMEM_END <= 228 * 1024 && Cfg<2>::SMEM_END <= 228 * 1024,
              "decode kernel shared window");
static_assert(Cfg<1>::STAGES * Cfg<1>::TAB_ROWS <= 256 && Cfg<2>::STAGES * Cfg<2>::TAB_ROWS <= 256,
              "stage scale tables fit the byte-table holes");

// Row order inside a 16-row group: MMA row g (and g + 8) is weight row perm8(g) (and + 8),
// so the four rows a half-warp reads from one swizzled code tile hit eight distinct 16-byte
// bank groups.
__device__ __forceinline__ int perm8(int g) { return 2 * (g & 3) + (g >> 2); }
__device__ __forceinline__ int inv_perm8(int p) { return (p >> 1) + 4 * (p & 1); }

// One fp32 value rounded to the 16-bit type (bf16, or fp16 when H).
template <bool H>
__device__ __forceinline__ uint16_t round16(float v) {
  return static_cast<uint16_t>(pack_pair<H>(v, 0.0f) & 0xFFFFu);
}

// bf16 operands, or fp16 when H; fp32 accumulate
template <bool H>
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (H)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Same with a zero accumulator input.
template <bool H>
__device__ __forceinline__ void mma_16816_z(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (H)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
        " {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

struct Params {
  int64_t M, N, K;
  int64_t KB;   // 64-blocks per weight row
  int64_t KST;  // stages per row block
  int64_t T;    // stages in all
  const int8_t* qs;
  const float* steps;  // group steps, or without double quantization the block absmax
  const float* mean;
  int qs_words;        // scale codes of a row's stage are one aligned 32-bit word
  float* part;         // [CTAs][2][16][128] fp32 pieces of split row blocks
  int* tickets;        // [row blocks] stages summed so far
  int64_t part_cap;    // floats in part, ints in tickets, floats in part_u (bounds checks)
  int64_t ticket_cap;
  int64_t part_u_cap;
  int64_t rp;
  int r;
  uint16_t* Y;
  // [M][N] fp32 LoRA term computed outside (per-token adapters); when set, the kernel adds it
  // before the final rounding instead of forming s U B^T on the tensor cores
  const float* Z;
  // U = X A^T inside the launch (with the on-chip LoRA term): CTAs [0, nU) each take U chunks
  // c = blockIdx.x + k G of U_KC contraction columns
  int nU;
  const uint16_t* X;   // [M][K]
  const uint16_t* A;   // [r][K]
  float scale;
  float* U_out;        // [M][r] fp32, or null
  float* part_u;       // [chunks][16][rp] fp32 partial U
  int* u_ticket;       // arrivals of the U CTAs (zero at launch)
  int* u_ready;        // 1 once sU (in the workspace) is complete (zero at launch)
  uint16_t* sU_out;    // [M][rp] 16-bit scale * U, written by the last U CTA
  float levels[16];  // the NF4 levels (parameter space: no cold constant-cache miss)
};

// First stage of CTA c, and the CTA that owns stage s, for T stages over G CTAs.
__device__ __forceinline__ int64_t stage_begin(int64_t T, int64_t G, int64_t c) { return T * c / G; }
__device__ __forceinline__ int64_t owner_of(int64_t T, int64_t G, int64_t s) {
  return ((s + 1) * G + T - 1) / T - 1;
}

__device__ __forceinline__ uint32_t ld_s32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 ld_s64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 ld_s128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ float2 ld_sf2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}

// Consumer-warp barrier (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(THREADS) : "memory");
}

// Shared byte offset of stage-scale entry e (0 .. 128 BPS - 1) of ring slot sl: the scale
// tables live in the unused upper halves of the byte-table rows (128 bytes = 32 entries per
// row), TAB_ROWS rows per slot.
template <int TAB_ROWS>
__device__ __forceinline__ uint32_t scale_slot_off(int sl, int e) {
  return static_cast<uint32_t>(((sl * TAB_ROWS + (e >> 5)) * 256) + 128 + (e & 31) * 4);
}

// Bounded wait for a flag in global memory written by another CTA of the same launch.
// Returns false (and records kWaitLora) after the limit.
__device__ __forceinline__ bool wait_flag(const int* flag, volatile int* abort_flag, int* err) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
    if (v) return true;
    if ((it & 63u) == 63u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        atomicCAS(err, 0, kWaitLora);
        *abort_flag = 1;
        return false;
      }
    }
    __nanosleep(200);
  }
}

// Scale formats, a compile-time parameter so the producers' per-stage scale writes carry no
// format test: the int8 or E4M3 second level, or the fp32 block absmax (no double quant).
enum ScaleFormat : int { kScaleInt8 = 0, kScaleFp8 = 1, kScaleAbsmax = 2 };

// OWN_LORA: the LoRA term from sU and B on the tensor cores (else the fp32 term p.Z is added).
// H: fp16 tokens, adapters, output and level table (the fp16 compute type), else bf16.
template <int NT, int SCALE, bool OWN_LORA, bool H>
__global__ void __launch_bounds__(THREADS + PRODUCERS, 1)
    nf4_decode_gemv(const __grid_constant__ CUtensorMap tmCodes,
                    const __grid_constant__ CUtensorMap tmX,
                    const __grid_constant__ CUtensorMap tmB, const Params p) {
  using C = Cfg<NT>;
  constexpr int STAGES = C::STAGES;
  constexpr int KSTEP = C::KSTEP, BPS = C::BPS, GPW = C::GPW, CODE_BYTES = C::CODE_BYTES;
  constexpr bool kDq = SCALE != kScaleAbsmax;
  constexpr int kFp8 = SCALE == kScaleFp8 ? 1 : 0;
  static_assert(STAGES * 16 <= 256, "scale tables fit the byte-table holes");
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[STAGES];
  __shared__ __align__(8) uint64_t empty_bar[STAGES];
  __shared__ __align__(8) uint64_t lora_bar;
  __shared__ int abort_flag, s_last;
  volatile int* abort_p = &abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t G = gridDim.x;
  const int64_t s_begin = stage_begin(p.T, G, blockIdx.x);
  const int64_t s_end = stage_begin(p.T, G, blockIdx.x + 1);
  if (s_begin >= s_end) return;
  const int64_t rb_first = s_begin / p.KST;
  const int nst = static_cast<int>(s_end - s_begin);
  {
    // the fixed layout needs the dynamic window to start at or below the ring and reach
    // past the LoRA region (uniform over the CTA: nothing has been initialised yet)
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uint32_t base = smem_u32(smem_raw);
    if (base > kStageBase || base + dyn < C::SMEM_END) {
      if (tid == 0) atomicExch(&g_decode_error, kWaitLayout);
      return;
    }
  }
  uint8_t* const sWin = smem_raw - smem_u32(smem_raw);  // generic pointer of window offset 0
  uint8_t* sStage = sWin + kStageBase;
  uint8_t* sLora = sWin + kLoraBase;
  float* sRed = reinterpret_cast<float*>(sLora);  // shares the region (see Cfg)
  uint16_t* sUs = reinterpret_cast<uint16_t*>(sWin + C::SU_BASE);
  uint8_t* sTab = sWin + kTableBase;
  const uint32_t x_bytes = static_cast<uint32_t>(BPS) * 128u * static_cast<uint32_t>(p.M);
  auto issue_stage = [&](int slot, int64_t rb, int64_t ks) {
    uint8_t* d = sStage + slot * C::STAGE_BYTES;
    mbar_arrive_expect_tx(&full_bar[slot], CODE_BYTES + x_bytes);
#pragma unroll
    for (int h = 0; h < BPS / 4; ++h)  // 128-byte boxes of the rows' codes, k ascending
      tma_load_2d(d + h * (ROWS * 128), &tmCodes, &full_bar[slot],
                  static_cast<int32_t>(ks * (KSTEP / 2) + 128 * h), static_cast<int32_t>(rb * ROWS));
#pragma unroll
    for (int x = 0; x < BPS; ++x)
      tma_load_2d(d + CODE_BYTES + x * C::XSLOT, &tmX, &full_bar[slot],
                  static_cast<int32_t>(ks * KSTEP + 64 * x), 0);
  };
  const int pre = nst < STAGES ? nst : STAGES;  // stages issued before the table is built

  if (tid == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], PRODUCERS / 32 + 1);  // the TMA issuer + the scale writers
      mbar_init(&empty_bar[i], THREADS / 32);
    }
    mbar_init(&lora_bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == THREADS) {  // lane 0 of the first producer warp: fill the ring right away
    int64_t rb = rb_first, ks = s_begin % p.KST;
    for (int i = 0; i < pre; ++i) {
      issue_stage(i, rb, ks);
      if (++ks == p.KST) ks = 0, ++rb;
    }
  }
  static_assert(16 * (SU_PITCH / 8) <= THREADS, "one sU piece per consumer thread");
  for (int i = tid; i < 256 * 8; i += THREADS + PRODUCERS) {
    const int v = i >> 3;  // 8 threads per entry: 16 bytes (4 lane copies) each
    const uint32_t e = pack_pair<H>(p.levels[v >> 4], p.levels[v & 15]);
    *reinterpret_cast<uint4*>(sTab + v * 256 + (i & 7) * 16) = make_uint4(e, e, e, e);
  }
  __syncthreads();

  if (warp >= THREADS / 32) {
    // ============================================================ producer warpgroup
    // Per stage, lane 0 of the first producer warp issues the TMA of codes and token slice
    // (one arrival with the transaction bytes) as soon as the slot is free, and thread R of
    // the four producer warps writes the BPS block scales of weight row R into the stage's
    // slot table (one arrival per warp): the full barrier counts 1 + 4 arrivals.
    // A row's BPS scale codes of a stage are BPS / 4 aligned 32-bit words when the 64-blocks
    // per row are a multiple of BPS: those words and the dq step are loaded SCALE_AHEAD
    // stages early into rotating register sets; otherwise each code is read when needed.
    // In the first CTAs the warps form U = X A^T (see u_work) once the ring's first stages
    // have their scale tables.
    constexpr int SW = BPS / 4;
    struct ScaleSet {
      uint32_t w[SW];
      float st;
    };
    const int R = tid - THREADS;
    const int pw_idx = warp - THREADS / 32;
    const float mu = kDq ? __ldg(p.mean) : 0.0f;
    const bool word_path = p.qs_words != 0;
    const int e0 = 16 * (R >> 4) + 2 * inv_perm8(R & 7) + ((R >> 3) & 1);
    ScaleSet ps0, ps1, ps2, ps3;
    int64_t f_n = rb_first * ROWS + R, f_ks = s_begin % p.KST;  // next stage to fetch
    auto fetch = [&](ScaleSet& z) {
#pragma unroll
      for (int i = 0; i < SW; ++i) z.w[i] = 0u;
      z.st = 0.f;
      if (f_n < p.N) {
        const int64_t idx = f_n * p.KB + f_ks * BPS;
        if constexpr (SW == 2) {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(p.qs + idx));
          z.w[0] = v.x;
          z.w[SW - 1] = v.y;
        } else {
          z.w[0] = __ldg(reinterpret_cast<const uint32_t*>(p.qs + idx));
        }
        z.st = __ldg(p.steps + (idx >> 8));
      }
      if (++f_ks == p.KST) f_ks = 0, f_n += ROWS;
    };
    auto fetch_set = [&](int set) {
      switch (set) {
        case 0: fetch(ps0); break;
        case 1: fetch(ps1); break;
        case 2: fetch(ps2); break;
        default: fetch(ps3); break;
      }
    };
    auto write_set = [&](int slot, int64_t n, int64_t ks, const ScaleSet& z) {
#pragma unroll
      for (int b = 0; b < BPS; ++b) {
        const int64_t kb = ks * BPS + b;
        float v = 0.f;
        if (n < p.N && kb < p.KB) {
          if (word_path) {
            v = __fmaf_rn(nf4_second_level(z.w[b >> 2] >> (8 * (b & 3)), kFp8), z.st, mu);
          } else {
            const int64_t idx = n * p.KB + kb;
            v = kDq ? __fmaf_rn(nf4_second_level(static_cast<uint8_t>(__ldg(p.qs + idx)), kFp8),
                                __ldg(p.steps + (idx >> 8)), mu)
                    : __ldg(p.steps + idx);
          }
        }
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(kTableBase + scale_slot_off<C::TAB_ROWS>(slot, b * 128 + e0)),
                     "f"(v));
      }
    };
    // U = X A^T for the contraction chunks of this CTA (chunks c = blockIdx.x + k G of U_KC
    // columns): warp pw_idx takes the 8-row adapter tiles pw_idx, pw_idx + 4, ...; a lane
    // holds 16 consecutive k of its token rows and adapter row per 64-wide step (the same
    // contraction-slot map on both operands).  The partial sums go to part_u; the last CTA to
    // arrive sums the chunks in chunk order, writes sU (and U), and raises u_ready.
    auto u_work = [&]() {
      if (p.nU <= 0 || blockIdx.x >= p.nU) return;
      const int g = lane >> 2, q = lane & 3;
      const int ntiles = static_cast<int>(p.rp / 8);
      const int64_t nchunks = (p.K + U_KC - 1) / U_KC;
      auto ld16 = [&](const uint16_t* base, int64_t row, int64_t nrows, int64_t k) -> uint4 {
        return (row < nrows && k < p.K) ? __ldg(reinterpret_cast<const uint4*>(base + row * p.K + k))
                                        : make_uint4(0, 0, 0, 0);
      };
      for (int64_t c = blockIdx.x; c < nchunks; c += G) {
        float d[4][4];
#pragma unroll
        for (int t = 0; t < 4; ++t) d[t][0] = d[t][1] = d[t][2] = d[t][3] = 0.f;
#pragma unroll 1
        for (int kk = 0; kk < U_KC; kk += 64) {
          const int64_t k = c * U_KC + kk + 16 * q;
          const uint4 xa0 = ld16(p.X, g, p.M, k), xa1 = ld16(p.X, g, p.M, k + 8);
          const uint4 xb0 = NT > 1 ? ld16(p.X, g + 8, p.M, k) : make_uint4(0, 0, 0, 0);
          const uint4 xb1 = NT > 1 ? ld16(p.X, g + 8, p.M, k + 8) : make_uint4(0, 0, 0, 0);
          const uint32_t xw[8] = {xa0.x, xa0.y, xa0.z, xa0.w, xa1.x, xa1.y, xa1.z, xa1.w};
          const uint32_t yw[8] = {xb0.x, xb0.y, xb0.z, xb0.w, xb1.x, xb1.y, xb1.z, xb1.w};
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int j = pw_idx + 4 * t;
            if (j >= ntiles) continue;
            const uint4 a0 = ld16(p.A, 8 * j + g, p.r, k), a1 = ld16(p.A, 8 * j + g, p.r, k + 8);
            const uint32_t aw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
              mma_16816<H>(d[t], xw[2 * m], yw[2 * m], xw[2 * m + 1], yw[2 * m + 1], aw[2 * m],
                           aw[2 * m + 1]);
          }
        }
        // d[t]: [0] token g / adapter row 8j + 2q, [1] + 1, [2] token g + 8 / 8j + 2q, [3] + 1
        const int64_t base = c * 16 * p.rp;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int j = pw_idx + 4 * t;
          if (j >= ntiles) continue;
          const int64_t i0 = base + g * p.rp + 8 * j + 2 * q, i1 = i0 + 8 * p.rp;
          if (g < p.M && QLORA_CHECK(i0 + 2 <= p.part_u_cap, &g_decode_error, kBoundsPartial))
            __stcg(reinterpret_cast<float2*>(p.part_u + i0), make_float2(d[t][0], d[t][1]));
          if (g + 8 < p.M && QLORA_CHECK(i1 + 2 <= p.part_u_cap, &g_decode_error, kBoundsPartial))
            __stcg(reinterpret_cast<float2*>(p.part_u + i1), make_float2(d[t][2], d[t][3]));
        }
      }
      __threadfence();
      asm volatile("bar.sync 2, %0;" ::"n"(PRODUCERS) : "memory");
      if (R == 0) {
        const int before = atomicAdd(p.u_ticket, 1);
        (void)QLORA_CHECK(before < p.nU, &g_decode_error, kBoundsTicket);
        s_last = before == p.nU - 1;
      }
      asm volatile("bar.sync 2, %0;" ::"n"(PRODUCERS) : "memory");
      if (!s_last) return;
      __threadfence();
      const int rpi = static_cast<int>(p.rp);
      for (int i = R; i < static_cast<int>(p.M) * rpi; i += PRODUCERS) {
        const int t = i / rpi, j = i % rpi;
        const float* src = p.part_u + t * rpi + j;
        const int64_t cs = 16 * p.rp;  // stride between chunks
        float u = 0.f;
        int64_t c = 0;
        (void)QLORA_CHECK((nchunks - 1) * cs + t * rpi + j < p.part_u_cap, &g_decode_error, kBoundsPartial);
        for (; c + 8 <= nchunks; c += 8) {  // 8 loads in flight, summed in chunk order
          float a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) a[k] = __ldcg(src + (c + k) * cs);
#pragma unroll
          for (int k = 0; k < 8; ++k) u += a[k];
        }
        for (; c < nchunks; ++c) u += __ldcg(src + c * cs);
        p.sU_out[t * p.rp + j] = j < p.r ? round16<H>(u * p.scale) : 0;
        if (p.U_out && j < p.r) p.U_out[t * p.r + j] = u;
      }
      __threadfence();
      asm volatile("bar.sync 2, %0;" ::"n"(PRODUCERS) : "memory");
      if (R == 0) asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.u_ready), "r"(1) : "memory");
    };
    if (word_path)
      for (int d = 0; d < SCALE_AHEAD && d < nst; ++d) fetch_set(d);
    int64_t rb = rb_first, ks = s_begin % p.KST;
    int slot = 0, issued = 0;
    uint32_t phase = 0;
    bool u_done = false;
    for (int i = 0; i < nst; ++i) {
      if (i == pre && !u_done) {  // the prefilled stages have their tables
        u_work();
        u_done = true;
      }
      if (i >= STAGES &&
          !mbar_wait<false, true>(&empty_bar[slot], phase ^ 1u, kWaitEmpty, abort_p, &g_decode_error))
        break;
      if (pw_idx == 0 && lane == 0 && i >= pre) issue_stage(slot, rb, ks);
      const int set = i & (SCALE_AHEAD - 1);
      const int64_t n = rb * ROWS + R;
      switch (set) {
        case 0: write_set(slot, n, ks, ps0); break;
        case 1: write_set(slot, n, ks, ps1); break;
        case 2: write_set(slot, n, ks, ps2); break;
        default: write_set(slot, n, ks, ps3); break;
      }
      if (word_path && i + SCALE_AHEAD < nst) fetch_set(set);
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_bar[slot]);  // this warp's scales are written
      issued = i + 1;
      if (++ks == p.KST) ks = 0, ++rb;
      if (++slot == STAGES) slot = 0, phase ^= 1u;
    }
    if (!u_done) u_work();
    __syncthreads();  // with the consumers: everything issued has been consumed or aborted
    if (pw_idx == 0 && lane == 0 && *abort_p) {
      // never release shared memory with a copy still landing in it: only the last STAGES
      // issues can still be in flight (the first producer warp issued them all)
      for (int k = issued > STAGES ? issued - STAGES : 0; k < issued; ++k)
        mbar_drain(&full_bar[k % STAGES], static_cast<uint32_t>((k / STAGES) & 1));
    }
    return;
  }

  // ============================================================ consumer warps
  const int g = lane >> 2, q = lane & 3;
  const int blk = warp % BPS;             // the 64-block of each stage this warp dequantizes
  const int gi0 = (warp / BPS) * GPW;     // its first 16-row group (GPW per warp)
  const int lora_boxes = static_cast<int>(p.rp / 64);
  auto issue_lora = [&](int64_t rb) {
    mbar_arrive_expect_tx(&lora_bar, static_cast<uint32_t>(lora_boxes * LORA_BOX_BYTES));
    for (int i = 0; i < lora_boxes; ++i)
      tma_load_2d(sLora + i * LORA_BOX_BYTES, &tmB, &lora_bar, 64 * i, static_cast<int32_t>(rb * ROWS));
  };
  constexpr bool own_lora = OWN_LORA;
  if (tid == 0 && own_lora && s_begin % p.KST == 0) issue_lora(rb_first);
  bool lora_pending = own_lora && s_begin % p.KST == 0;  // a B-row tile in flight, not yet used

  const uint32_t lane_addr = kTableBase | (static_cast<uint32_t>(lane) * 4u);
  auto lut = [&](uint32_t word, uint32_t j) -> uint32_t {
    // byte j of the code word at bits 8..15; 4 * lane at bits 0..7 and the table's 64 KB
    // page at bits 16..31 from lane_addr: the entry's window address
    return ld_s32(__byte_perm(word, lane_addr, 0x7604u | (j << 4)));
  };

  float acc[GPW][NT][4];
#pragma unroll
  for (int j = 0; j < GPW; ++j)
#pragma unroll
    for (int o = 0; o < NT; ++o) acc[j][o][0] = acc[j][o][1] = acc[j][o][2] = acc[j][o][3] = 0.f;

  // ---------------------------------------------------------------- piece flush
  // Adds the LoRA term if the piece starts its row block, sums the BPS block-warps of each
  // row in a fixed order, and writes Y -- or the piece's partial sums, the last of which
  // sums all pieces of the row block in CTA order.  The first LoRA flush stages sU, once the
  // U flag of this launch is up.
  uint32_t lora_phase = 0;
  bool su_staged = false;
  const int nchunks = (p.r + 15) / 16;
  auto flush = [&](int64_t rb, int64_t ks_first, int64_t ks_last) -> bool {
    if (ks_first == 0 && own_lora) {
      if (!su_staged) {
        if (tid == 0) wait_flag(p.u_ready, abort_p, &g_decode_error);
        consumers_sync();
        if (*abort_p) return false;  // uniform after the barrier
        if (tid < 16 * (SU_PITCH / 8)) {
          const int t = tid / (SU_PITCH / 8), c8 = tid % (SU_PITCH / 8);
          uint4 v = make_uint4(0, 0, 0, 0);
          if (t < p.M && 8 * c8 < p.rp)
            v = __ldcg(reinterpret_cast<const uint4*>(p.sU_out + t * p.rp + 8 * c8));
          *reinterpret_cast<uint4*>(sUs + t * SU_PITCH + 8 * c8) = v;
        }
        consumers_sync();
        su_staged = true;
      }
      if (blk == 0 && mbar_wait(&lora_bar, lora_phase, kWaitLora, abort_p, &g_decode_error)) {
#pragma unroll
        for (int j = 0; j < GPW; ++j) {
          const int gi = gi0 + j;
          const int mat = lane >> 3, rr = lane & 7;
          const int R = 16 * gi + perm8(rr) + 8 * (mat & 1);
          for (int c = 0; c < nchunks; ++c) {
            const int jc8 = 2 * c + (mat >> 1);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(smem_u32(sLora + (jc8 >> 3) * LORA_BOX_BYTES + R * 128 +
                             (((jc8 & 7) ^ (R & 7)) << 4)),
                    a0, a1, a2, a3);
#pragma unroll
            for (int o = 0; o < NT; ++o) {
              const uint16_t* ur = sUs + (g + 8 * o) * SU_PITCH + 16 * c + 2 * q;
              const uint32_t b0 = *reinterpret_cast<const uint32_t*>(ur);
              const uint32_t b1 = *reinterpret_cast<const uint32_t*>(ur + 8);
              mma_16816<H>(acc[j][o], a0, a1, a2, a3, b0, b1);
            }
          }
        }
      }
      consumers_sync();  // the B-row tile is read before the reduction overwrites it
    }
    // every warp's accumulators to shared memory, lane-contiguous
#pragma unroll
    for (int j = 0; j < GPW; ++j)
#pragma unroll
      for (int o = 0; o < NT; ++o)
#pragma unroll
        for (int d = 0; d < 4; ++d)
          sRed[(warp * C::ACC + (j * NT + o) * 4 + d) * 32 + lane] = acc[j][o][d];
    consumers_sync();
    if (*abort_p) return false;  // uniform after the barrier; the B-row tile stays pending
    if (ks_first == 0 && own_lora) {
      lora_phase ^= 1u;
      lora_pending = false;
    }
    const bool whole = ks_first == 0 && ks_last == p.KST - 1;
    const int R = tid & (ROWS - 1);
    const int64_t n = rb * ROWS + R;
    const int gi = R >> 4, h = (R >> 3) & 1, gg = inv_perm8(R & 7);
    const int wb = BPS * (gi / GPW), jj = gi % GPW;
    const int64_t slot = rb == rb_first ? 0 : 1;
    const int64_t mine_at = (static_cast<int64_t>(blockIdx.x) * 2 + slot) * 16 * ROWS;
    float* mine = p.part + mine_at;
    for (int t = tid >> 7; t < p.M; t += THREADS / ROWS) {
      const int o = t >> 3, qq = (t & 7) >> 1, d = 2 * h + (t & 1);
      const int idx = ((jj * NT + o) * 4 + d) * 32 + 4 * gg + qq;
      float v = sRed[wb * C::ACC * 32 + idx];
#pragma unroll
      for (int b = 1; b < BPS; ++b) v += sRed[(wb + b) * C::ACC * 32 + idx];
      if (whole) {
        if (n < p.N) {
          if constexpr (!OWN_LORA) v += __ldg(p.Z + t * p.N + n);
          p.Y[t * p.N + n] = round16<H>(v);
        }
      } else if (QLORA_CHECK(mine_at + t * ROWS + R < p.part_cap, &g_decode_error, kBoundsPartial)) {
        __stcg(mine + t * ROWS + R, v);
      }
    }
    if (!whole) {
      __threadfence();
      consumers_sync();
      if (tid == 0) {
        const int add = static_cast<int>(ks_last - ks_first + 1);
        if (QLORA_CHECK(rb < p.ticket_cap, &g_decode_error, kBoundsTicket)) {
          const int after = atomicAdd(&p.tickets[rb], add) + add;
          (void)QLORA_CHECK(after <= p.KST, &g_decode_error, kBoundsTicket);
          s_last = after == p.KST;
        } else {
          s_last = 0;
        }
      }
      consumers_sync();
      if (s_last) {
        __threadfence();
        const int64_t c_lo = owner_of(p.T, G, rb * p.KST);
        const int64_t c_hi = owner_of(p.T, G, rb * p.KST + p.KST - 1);
        for (int t = tid >> 7; t < p.M; t += THREADS / ROWS) {
          float v = 0.f;
          for (int64_t c = c_lo; c <= c_hi; ++c) {
            const int64_t sl = rb == stage_begin(p.T, G, c) / p.KST ? 0 : 1;
            const int64_t at = (c * 2 + sl) * 16 * ROWS + t * ROWS + R;
            if (QLORA_CHECK(at < p.part_cap, &g_decode_error, kBoundsPartial)) v += __ldcg(p.part + at);
          }
          if (n < p.N) {
            if constexpr (!OWN_LORA) v += __ldg(p.Z + t * p.N + n);
            p.Y[t * p.N + n] = round16<H>(v);
          }
        }
        if (tid == 0) p.tickets[rb] = 0;  // ready for the next launch
      }
    }
    consumers_sync();  // the shared region is free again
#pragma unroll
    for (int j = 0; j < GPW; ++j)
#pragma unroll
      for (int o = 0; o < NT; ++o) acc[j][o][0] = acc[j][o][1] = acc[j][o][2] = acc[j][o][3] = 0.f;
    return true;
  };

  // ---------------------------------------------------------------- main loop
  // per-lane constant shared-memory offsets: code words of rows R0, R0 + 8 of the warp's
  // groups (block blk lies in the stage's 128-byte box blk / 4), the token fragments, and
  // the scale pairs
  uint32_t code_off[GPW], scale_e[GPW];
  {
    const int chunk = 2 * (blk & 3) + (q >> 1);
#pragma unroll
    for (int j = 0; j < GPW; ++j) {
      const int gi = gi0 + j;
      const int R0 = 16 * gi + perm8(g);  // MMA rows g, g + 8 -> weight rows R0, R0 + 8
      code_off[j] = (blk >> 2) * (ROWS * 128) + R0 * 128 + ((chunk ^ (R0 & 7)) << 4) + (q & 1) * 8;
      scale_e[j] = ((blk * 8 + gi) * 8 + g) * 2;
    }
  }
  uint32_t x_off[NT][2];
  bool x_live[NT];
#pragma unroll
  for (int o = 0; o < NT; ++o) {
    const int t = g + 8 * o;
    x_live[o] = t < p.M;
    x_off[o][0] = CODE_BYTES + blk * C::XSLOT + t * 128 + (((2 * q) ^ g) << 4);
    x_off[o][1] = CODE_BYTES + blk * C::XSLOT + t * 128 + (((2 * q + 1) ^ g) << 4);
  }
  const uint32_t stage_s = kStageBase;
  // the lane's fixed window offsets stay inside their regions: code words inside the stage's
  // code tile, token fragments inside the stage, scale pairs inside the upper halves of the
  // byte-table rows of their slot (a failed check skips the shared reads)
  bool window_ok = true;
#pragma unroll
  for (int j = 0; j < GPW; ++j) {
    window_ok &= QLORA_CHECK(code_off[j] + 8 * 128 + 8 <= static_cast<uint32_t>(CODE_BYTES),
                             &g_decode_error, kBoundsWindow);
    window_ok &= QLORA_CHECK(scale_e[j] + 1 < static_cast<uint32_t>(ROWS * BPS) &&
                                 (scale_slot_off<C::TAB_ROWS>(STAGES - 1, scale_e[j]) & 255u) >= 128u &&
                                 scale_slot_off<C::TAB_ROWS>(STAGES - 1, scale_e[j]) + 8 <= TABLE_BYTES,
                             &g_decode_error, kBoundsWindow);
  }
#pragma unroll
  for (int o = 0; o < NT; ++o)
    window_ok &= QLORA_CHECK(!x_live[o] || x_off[o][1] + 16 <= static_cast<uint32_t>(C::STAGE_BYTES),
                             &g_decode_error, kBoundsWindow);
  window_ok &= QLORA_CHECK(stage_s + STAGES * C::STAGE_BYTES <= C::SU_BASE, &g_decode_error, kBoundsWindow);

  bool ok = true;
  // 32-bit bookkeeping in the loop: stage counts per CTA and per row block are small
  const int KST = static_cast<int>(p.KST);
  int64_t rb = rb_first;
  int ks = static_cast<int>(s_begin % p.KST), ks_first = ks;
  int slot = 0;
  uint32_t phase = 0;
  for (int i = 0; i < nst; ++i) {
    if (ks == 0 && i != 0) {
      ks_first = 0;
      if (own_lora) {
        if (tid == 0) {
          fence_proxy_async_smem();  // the last flush's accesses to the region precede the refill
          issue_lora(rb);
        }
        lora_pending = true;
      }
    }
    const bool got =
        mbar_wait<false, true>(&full_bar[slot], phase, kWaitTmaFull, abort_p, &g_decode_error);
    if (got && window_ok) {
      const uint32_t cs = stage_s + slot * C::STAGE_BYTES;
      uint32_t xf[NT][8];
#pragma unroll
      for (int o = 0; o < NT; ++o) {
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (x_live[o]) {  // token rows past M hold no TMA data: zero operands, no loads
          lo = ld_s128(cs + x_off[o][0]);
          hi = ld_s128(cs + x_off[o][1]);
        }
        xf[o][0] = lo.x; xf[o][1] = lo.y; xf[o][2] = lo.z; xf[o][3] = lo.w;
        xf[o][4] = hi.x; xf[o][5] = hi.y; xf[o][6] = hi.z; xf[o][7] = hi.w;
      }
#pragma unroll
      for (int j = 0; j < GPW; ++j) {
        const uint2 c0 = ld_s64(cs + code_off[j]);
        const uint2 c1 = ld_s64(cs + code_off[j] + 8 * 128);
        const float2 sc = ld_sf2(kTableBase + scale_slot_off<C::TAB_ROWS>(slot, scale_e[j]));
        float d[NT][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const uint32_t w0 = m < 2 ? c0.x : c0.y, w1 = m < 2 ? c1.x : c1.y;
          const uint32_t by = (m & 1) * 2;
          const uint32_t a0 = lut(w0, by), a2 = lut(w0, by + 1);
          const uint32_t a1 = lut(w1, by), a3 = lut(w1, by + 1);
#pragma unroll
          for (int o = 0; o < NT; ++o) {
            if (m == 0)
              mma_16816_z<H>(d[o], a0, a1, a2, a3, xf[o][0], xf[o][1]);
            else
              mma_16816<H>(d[o], a0, a1, a2, a3, xf[o][2 * m], xf[o][2 * m + 1]);
          }
        }
#pragma unroll
        for (int o = 0; o < NT; ++o) {
          acc[j][o][0] = __fmaf_rn(sc.x, d[o][0], acc[j][o][0]);
          acc[j][o][1] = __fmaf_rn(sc.x, d[o][1], acc[j][o][1]);
          acc[j][o][2] = __fmaf_rn(sc.y, d[o][2], acc[j][o][2]);
          acc[j][o][3] = __fmaf_rn(sc.y, d[o][3], acc[j][o][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);  // this warp is done with the slot
    if (++slot == STAGES) slot = 0, phase ^= 1u;
    if (ks == KST - 1 || i == nst - 1) {
      if (!flush(rb, ks_first, ks)) ok = false;
      if (!ok) break;  // uniform: decided after a consumer barrier
    }
    if (++ks == KST) ks = 0, ++rb;
  }
  (void)ok;
  __syncthreads();  // with the producer warp
  if (tid == 0 && lora_pending && *abort_p) mbar_drain(&lora_bar, lora_phase);
}

}  // namespace skinny

namespace {

template <int NT>
int64_t skinny_stages(int64_t N, int64_t K) {
  return ((N + skinny::ROWS - 1) / skinny::ROWS) *
         ((K + skinny::Cfg<NT>::KSTEP - 1) / skinny::Cfg<NT>::KSTEP);
}

template <int NT>
int64_t skinny_ctas(int64_t N, int64_t K) {
  const int64_t T = skinny_stages<NT>(N, K);
  return T < num_sms() ? T : num_sms();
}

// The GEMV's split-row partial sums (two slots per CTA), then the U chunks' partials.
uint64_t gemv_partial_bytes(int64_t N, int64_t K) {
  const int64_t c = std::max(skinny_ctas<1>(N, K), skinny_ctas<2>(N, K));
  return (uint64_t)round_up(c * 2 * 16 * skinny::ROWS * 4, 256);
}

template <int NT, int SCALE, bool OWN_LORA, bool H = false>
int run_decode(const CUtensorMap& tmC, const CUtensorMap& tmX, const CUtensorMap& tmB,
               const skinny::Params& p, unsigned ctas, cudaStream_t stream) {
  using C = skinny::Cfg<NT>;
  // The kernel places its regions at fixed window offsets; it takes the whole opt-in
  // dynamic window, which starts after the reserved and static shared memory.
  static DeviceCache<int> window;  // this instantiation's dynamic window, per device
  int dyn = 0;
  const int st = window.get(device_context_key, &dyn, [](int* v) -> int {
    int dev = 0, optin = 0, reserved = 0;
    cudaFuncAttributes fa{};
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, skinny::nf4_decode_gemv<NT, SCALE, OWN_LORA, H>) != cudaSuccess) {
      cudaGetLastError();
      return QLORA_ERR_CUDA;
    }
    const int base = reserved + static_cast<int>(fa.sharedSizeBytes);
    const int size = optin - static_cast<int>(fa.sharedSizeBytes);
    if (base > static_cast<int>(skinny::kStageBase) ||
        base + size < static_cast<int>(C::SMEM_END))
      return QLORA_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(skinny::nf4_decode_gemv<NT, SCALE, OWN_LORA, H>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, size) != cudaSuccess) {
      cudaGetLastError();
      return QLORA_ERR_CUDA;
    }
    *v = size;
    return QLORA_OK;
  });
  if (st) return st == -1 ? QLORA_ERR_NO_DEVICE : st;
  skinny::nf4_decode_gemv<NT, SCALE, OWN_LORA, H><<<ctas, skinny::THREADS + skinny::PRODUCERS, dyn, stream>>>(tmC, tmX, tmB, p);
  return cudaGetLastError() == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace

uint64_t skinny_partial_bytes(int64_t M, int64_t N, int64_t K, int r) {
  if (M > kSkinnyMaxM) return 0;
  const uint64_t u = (uint64_t)((K + skinny::U_KC - 1) / skinny::U_KC) * 16 * round_up(r, 64) * 4;
  return gemv_partial_bytes(N, K) + u;
}

uint64_t skinny_ticket_count(int64_t M, int64_t N) {
  // a stage count per row block, then the U arrivals and the U flag
  return M > kSkinnyMaxM ? 0 : (uint64_t)((N + skinny::ROWS - 1) / skinny::ROWS) + 2;
}

int launch_decode_gemv(const LinearArgs& a, const WorkspaceLayout& L, const float* Z,
                       cudaStream_t stream) {
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  const bool own_lora = Z == nullptr;
  CUtensorMap tmC, tmX, tmB;
  const bool mapped =
      make_tensor_map_2d(&tmC, a.q.codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, (uint64_t)(a.K / 2),
                         (uint64_t)a.N, (uint64_t)(a.K / 2), 128, skinny::ROWS, MapSwizzle::B128) &&
      make_tensor_map_2d(&tmX, a.X, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)a.K,
                         (uint64_t)a.M, (uint64_t)a.K * 2, 64, (uint32_t)a.M, MapSwizzle::B128) &&
      (!own_lora || a.r % 8 == 0  // B [N, r] itself; TMA fills the columns past r with zeros
           ? make_tensor_map_2d(&tmB, a.B, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)a.r,
                                (uint64_t)a.N, (uint64_t)a.r * 2, 64, skinny::ROWS, MapSwizzle::B128)
           : make_tensor_map_2d(&tmB, ws + L.Bp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                (uint64_t)L.rp, (uint64_t)a.N, (uint64_t)L.rp * 2, 64, skinny::ROWS,
                                MapSwizzle::B128));
  if (!mapped) return QLORA_ERR_CUDA;
  skinny::Params p{};
  const bool wide = a.M <= 8;  // one token octet: 512-wide stages
  const int kstep = wide ? skinny::Cfg<1>::KSTEP : skinny::Cfg<2>::KSTEP;
  const int bps = kstep / 64;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.KB = a.K / 64;
  p.KST = (a.K + kstep - 1) / kstep;
  p.T = wide ? skinny_stages<1>(a.N, a.K) : skinny_stages<2>(a.N, a.K);
  p.qs = a.q.scale_codes;
  p.steps = a.q.scale_steps;
  p.mean = a.q.scale_mean;
  // a stage's scale codes of a row are whole aligned words when the blocks per row are a
  // multiple of the stage's blocks (the pointer is 16-byte aligned)
  p.qs_words = (a.q.dq_block != 0 && p.KB % bps == 0) ? 1 : 0;
  p.part = reinterpret_cast<float*>(ws + L.part);
  p.tickets = reinterpret_cast<int*>(ws + L.tickets);
  p.part_cap = static_cast<int64_t>(gemv_partial_bytes(a.N, a.K) / 4);
  p.ticket_cap = static_cast<int64_t>((a.N + skinny::ROWS - 1) / skinny::ROWS);
  p.rp = L.rp;
  p.r = a.r;
  p.Y = a.Y;
  p.Z = Z;
  {
    constexpr float Lv[16] = QLORA_NF4_LEVELS;
    for (int i = 0; i < 16; ++i) p.levels[i] = Lv[i];
  }
  const unsigned ctas = (unsigned)(wide ? skinny_ctas<1>(a.N, a.K) : skinny_ctas<2>(a.N, a.K));
  if (own_lora) {  // U inside the launch: the first CTAs take its contraction chunks
    const int64_t nrb = (a.N + skinny::ROWS - 1) / skinny::ROWS;
    const int64_t nchunks = (a.K + skinny::U_KC - 1) / skinny::U_KC;
    p.nU = static_cast<int>(nchunks < (int64_t)ctas ? nchunks : (int64_t)ctas);
    p.X = a.X;
    p.A = a.A;
    p.scale = a.scale;
    p.U_out = a.U;
    p.part_u = reinterpret_cast<float*>(ws + L.part + gemv_partial_bytes(a.N, a.K));
    p.part_u_cap = static_cast<int64_t>((L.part_bytes - gemv_partial_bytes(a.N, a.K)) / 4);
    p.u_ticket = p.tickets + nrb;
    p.u_ready = p.tickets + nrb + 1;
    p.sU_out = reinterpret_cast<uint16_t*>(ws + L.sU);
  }
  ProfileScope ps("decode_gemv", stream);
  const int fmt = a.q.dq_block == 0 ? skinny::kScaleAbsmax
                  : a.q.dq_type == NF4_DQ_FP8 ? skinny::kScaleFp8 : skinny::kScaleInt8;
  if (a.half)  // the fp16 compute type (with the LoRA term on chip)
    switch (fmt + 3 * (a.M > 8 ? 1 : 0)) {
      case 0: return run_decode<1, skinny::kScaleInt8, true, true>(tmC, tmX, tmB, p, ctas, stream);
      case 1: return run_decode<1, skinny::kScaleFp8, true, true>(tmC, tmX, tmB, p, ctas, stream);
      case 2: return run_decode<1, skinny::kScaleAbsmax, true, true>(tmC, tmX, tmB, p, ctas, stream);
      case 3: return run_decode<2, skinny::kScaleInt8, true, true>(tmC, tmX, tmB, p, ctas, stream);
      case 4: return run_decode<2, skinny::kScaleFp8, true, true>(tmC, tmX, tmB, p, ctas, stream);
      default: return run_decode<2, skinny::kScaleAbsmax, true, true>(tmC, tmX, tmB, p, ctas, stream);
    }
  if (!own_lora)  // per-token adapters: the int8 / fp8 / absmax formats without the LoRA MMA
    switch (fmt + 3 * (a.M > 8 ? 1 : 0)) {
      case 0: return run_decode<1, skinny::kScaleInt8, false>(tmC, tmX, tmB, p, ctas, stream);
      case 1: return run_decode<1, skinny::kScaleFp8, false>(tmC, tmX, tmB, p, ctas, stream);
      case 2: return run_decode<1, skinny::kScaleAbsmax, false>(tmC, tmX, tmB, p, ctas, stream);
      case 3: return run_decode<2, skinny::kScaleInt8, false>(tmC, tmX, tmB, p, ctas, stream);
      case 4: return run_decode<2, skinny::kScaleFp8, false>(tmC, tmX, tmB, p, ctas, stream);
      default: return run_decode<2, skinny::kScaleAbsmax, false>(tmC, tmX, tmB, p, ctas, stream);
    }
  switch (fmt + 3 * (a.M > 8 ? 1 : 0)) {
    case 0: return run_decode<1, skinny::kScaleInt8, true>(tmC, tmX, tmB, p, ctas, stream);
    case 1: return run_decode<1, skinny::kScaleFp8, true>(tmC, tmX, tmB, p, ctas, stream);
    case 2: return run_decode<1, skinny::kScaleAbsmax, true>(tmC, tmX, tmB, p, ctas, stream);
    case 3: return run_decode<2, skinny::kScaleInt8, true>(tmC, tmX, tmB, p, ctas, stream);
    case 4: return run_decode<2, skinny::kScaleFp8, true>(tmC, tmX, tmB, p, ctas, stream);
    default: return run_decode<2, skinny::kScaleAbsmax, true>(tmC, tmX, tmB, p, ctas, stream);
  }
}

int launch_skinny_fwd(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  int st;
  if (a.r % 8 && (st = launch_pad_b(a, L, stream))) return st;
  return launch_decode_gemv(a, L, nullptr, stream);
}

}  // namespace qlora
