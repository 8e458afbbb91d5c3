// nf4_device.cuh -- the NF4 data type on the device: the 16 fp32 levels, the 15 decision
// thresholds, level-index search, and the byte-permute dequantizer that turns packed codes
// plus one block scale into bf16 (infivelines.com "QLoRA": NF4 places its 16 levels at
// quantiles of a normal distribution; each block of 64 weights carries its own scale).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace qlora {

// Levels: the asymmetric normal-quantile construction (8 positive quantiles, 7 negative, an
// exact 0, normalised to +-1), rounded to fp32.  Thresholds: exact midpoints of adjacent
// fp32 levels rounded toward -inf, so "count thresholds strictly below x" is the nearest
// level with ties to the lower index.  Values written as exact hex floats.
#define QLORA_NF4_LEVELS                                                                   \
  {-0x1.000000p+0f, -0x1.647362p-1f, -0x1.0cd65cp-1f, -0x1.94653cp-2f, -0x1.234496p-2f,   \
   -0x1.7a6a7ap-3f, -0x1.74f0d2p-4f, 0x0.0p+0f,      0x1.45f602p-4f,  0x1.4995bep-3f,     \
   0x1.f809b4p-3f,  0x1.5a066cp-2f,  0x1.c3496ap-2f, 0x1.200f52p-1f,  0x1.722760p-1f,     \
   0x1.000000p+0f}
#define QLORA_NF4_THRESHOLDS                                                               \
  {-0x1.b239b2p-1f, -0x1.38a4e0p-1f, -0x1.d708fap-2f, -0x1.5bd4eap-2f, -0x1.e079d4p-3f,   \
   -0x1.1a7172p-3f, -0x1.74f0d2p-5f, 0x1.45f602p-5f,  0x1.ec90bep-4f,  0x1.a0cfb8p-3f,    \
   0x1.2b05a2p-2f,  0x1.8ea7eap-2f,  0x1.00da02p-1f,  0x1.491b58p-1f,  0x1.b913b0p-1f}

// Level index of x (already divided by its block absmax): a 4-step binary search over the
// thresholds with register selects.  Equals the count of thresholds strictly below x.
__device__ __forceinline__ uint32_t nf4_code(float x) {
  constexpr float T[15] = QLORA_NF4_THRESHOLDS;
  const bool b3 = x > T[7];
  const bool b2 = x > (b3 ? T[11] : T[3]);
  const float t1 = b3 ? (b2 ? T[13] : T[9]) : (b2 ? T[5] : T[1]);
  const bool b1 = x > t1;
  const float t0 = b3 ? (b2 ? (b1 ? T[14] : T[12]) : (b1 ? T[10] : T[8]))
                      : (b2 ? (b1 ? T[6] : T[4]) : (b1 ? T[2] : T[0]));
  const bool b0 = x > t0;
  return (b3 ? 8u : 0u) | (b2 ? 4u : 0u) | (b1 ? 2u : 0u) | (b0 ? 1u : 0u);
}

// Value of a second-level scale code (the low byte of `byte`): an int8 step count, or with
// fp8 an E4M3 number (widened exactly through half precision).
__device__ __forceinline__ float nf4_second_level(uint32_t byte, int fp8) {
  if (fp8) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte & 0xFFu), __NV_E4M3);
    return __half2float(__half(h));
  }
  return static_cast<float>(static_cast<int8_t>(byte & 0xFFu));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t lop_select(uint32_t a, uint32_t b, uint32_t m) {
  return (a & ~m) | (b & m);  // per bit: m ? b : a  (one LOP3)
}

// One block's 16 dequantized values T[c] = bf16_rne(level[c] * scale) (fp16 in the fp16
// compute type), kept as byte tables for prmt: lo[i] holds the low bytes of T[4i..4i+3],
// hi[i] their high bytes.
struct Nf4ByteTable {
  uint32_t lo[4];
  uint32_t hi[4];
};

// Two fp32 values rounded to nearest even as one 32-bit pair (lo in the low half): bf16, or
// fp16 when H (the fp16 compute type; fp16 subnormals kept).
template <bool H>
__device__ __forceinline__ uint32_t pack_pair(float lo, float hi) {
  if constexpr (H) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
}

// Value of one 16-bit element (the low half of `bits`): bf16, or fp16 when H.
template <bool H>
__device__ __forceinline__ float widen16(uint32_t bits) {
  if constexpr (H) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
  } else {
    return __uint_as_float(bits << 16);
  }
}

template <bool H = false>
__device__ __forceinline__ Nf4ByteTable nf4_make_table(float scale) {
  constexpr float L[16] = QLORA_NF4_LEVELS;
  uint32_t P[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    // one IEEE fp32 multiply per level, then round-to-nearest-even to the 16-bit type;
    // low half = T[2j], high half = T[2j+1]
    P[j] = pack_pair<H>(__fmul_rn(L[2 * j], scale), __fmul_rn(L[2 * j + 1], scale));
  }
  Nf4ByteTable t;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    t.lo[i] = prmt(P[2 * i], P[2 * i + 1], 0x6420u);
    t.hi[i] = prmt(P[2 * i], P[2 * i + 1], 0x7531u);
  }
  return t;
}

// Eight packed codes (one little-endian u32 of the code stream: byte j holds elements 2j in
// the high nibble and 2j+1 in the low nibble) -> eight 16-bit values in element order (the
// table's type), as four u32
// (element 2k in the low half of out[k]).
__device__ __forceinline__ void nf4_dequant8(const Nf4ByteTable& t, uint32_t q, uint32_t (&out)[4]) {
  const uint32_t q4 = q * 16u;  // a multiply (IMAD, FMA pipe) keeps the shift off the ALU pipe
  // byte masks from bit 3 of each index, via prmt's sign-replicate mode; nibble order of a
  // half-word is [e1, e0, e3, e2] (low nibble of byte 0 first)
  const uint32_t m_lo = prmt(q4, q, 0xD9C8u);
  const uint32_t m_hi = prmt(q4, q, 0xFBEAu);
  const uint32_t s_all = q & 0x77777777u;
  const uint32_t s_lo = s_all;                    // prmt reads only the low 16 selector bits
  const uint32_t s_hi = __umulhi(s_all, 0x10000u);  // s_all >> 16 as IMAD.HI (FMA pipe)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t s = h ? s_hi : s_lo;
    const uint32_t m = h ? m_hi : m_lo;
    const uint32_t lo = lop_select(prmt(t.lo[0], t.lo[1], s), prmt(t.lo[2], t.lo[3], s), m);
    const uint32_t hi = lop_select(prmt(t.hi[0], t.hi[1], s), prmt(t.hi[2], t.hi[3], s), m);
    // lo/hi bytes are ordered [e1, e0, e3, e2]; interleave into pairs (e0,e1),(e2,e3)
    out[2 * h + 0] = prmt(lo, hi, 0x4051u);
    out[2 * h + 1] = prmt(lo, hi, 0x6273u);
  }
}

}  // namespace qlora
