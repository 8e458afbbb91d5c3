// linear.h -- the LoRA-wrapped NF4 linear layer: argument bundle, workspace layout, and the
// forward / backward orchestration entry points (linear.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/qlora_nf4.h"

namespace qlora {

constexpr int kMaxRank = 128;
constexpr int64_t kSkinnyMaxM = 16;  // M at or below this takes the decode kernel

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct LinearArgs {
  int64_t M, N, K;
  int r;
  float scale;
  nf4_tensor q;
  const uint16_t* X;
  const uint16_t* A;
  const uint16_t* B;
  uint16_t* Y;
  float* U;             // forward: optional fp32 U output
  const float* U_in;    // backward: optional saved U
  const uint16_t* dY;
  uint16_t* dX;
  float* dA;
  float* dB;
  void* ws;
  uint64_t ws_bytes;
  int gemm_priority;    // launch priority of the fused GEMM (0: the stream's own)
  // per-token adapters (decode path only): A = [n_adapters, r, K], B = [n_adapters, N, r],
  // token t uses adapter adapter_idx[t] with scale scales[adapter_idx[t]] (both on the
  // device); an index outside [0, n_adapters) means no adapter for that token
  const int32_t* adapter_idx;
  int n_adapters;
  const float* scales;
  // fp16 compute type: X, A, B, dY, Y, dX, the staged sU / sV and the dequantized base in
  // fp16 (else bf16)
  bool half;
};

// Workspace regions (byte offsets, each 1024-aligned), for rank padded to rp = 64*ceil(r/64);
// the 16-bit regions hold bf16, or fp16 in the fp16 compute type.
struct WorkspaceLayout {
  int64_t rp;
  uint64_t sU;       // 16-bit [M, rp]  scale * U (columns past r: read as TMA zero fill)
  uint64_t sV;       // 16-bit [M, rp]  scale * V (the same)
  uint64_t U32;      // fp32 [M, r]   U recomputed by the backward when none is saved
  uint64_t dbpart;   // fp32 [ceil(M/128)][N][16] dB partials of the narrow V (rank <= 16)
  uint64_t dbpart_bytes;
  uint64_t Bp;       // 16-bit [N, rp]  B zero-padded (only for r not a multiple of 8)
  uint64_t part;     // fp32 split-contraction partial sums (side products, decode path)
  uint64_t part_bytes;
  uint64_t tickets;  // int [ntickets] arrival counters of the split reductions
  uint64_t ntickets;
  uint64_t gpart;    // fp32 [nsplit][M][Nout] split-contraction tiles of the fused GEMM
  uint64_t gpart_bytes;
  uint64_t gtickets; // int [ngtickets] its per-tile arrivals (right after the tickets above)
  uint64_t ngtickets;
  uint64_t pers_ctr; // int: the persistent pair GEMM's cluster tickets (right after those)
  uint64_t nticket_words;  // ints from `tickets` on, all zeroed at the start of a call
  uint64_t Z;        // fp32 [M, N] per-token LoRA term (decode path, per-token adapters)
  uint64_t Wd;       // 16-bit [N, K] W' dequantized once, for GEMM plans with a staged base
  uint64_t Wd_bytes;
  uint64_t total;
};

WorkspaceLayout workspace_layout(int64_t M, int64_t N, int64_t K, int r);
uint64_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int r);

// Tile plan of a fused GEMM with Nout output columns and contraction Kc: kind 2 = CTA pairs
// (512 x 256 tiles), 1 = single CTAs with 256 x 256 tiles, 0 = 128 x 256 tiles; the
// contraction is cut into nsplit runs of split_stages 64-wide stages (tiles: the output tiles).
// wstage: W' is dequantized once into the workspace beforehand and every stage's W tile
// comes by TMA (128-row tiles past one row tile, where each weight would otherwise be
// dequantized once per row tile).
struct FusedPlan {
  int kind;
  int nsplit;
  int split_stages;
  int64_t tiles;
  int wstage;
};
FusedPlan fused_plan(int64_t M, int64_t Nout, int64_t Kc);
// Workspace of the split contraction (the larger of the forward and the input gradient) and,
// in *tickets, its arrival counters.
uint64_t fused_partial_bytes(int64_t M, int64_t N, int64_t K, uint64_t* tickets);

int linear_forward(const LinearArgs& a, cudaStream_t stream);
int linear_backward(const LinearArgs& a, cudaStream_t stream);

// ---- kernels behind the orchestration (umma_gemm.cu, lora_side.cu, skinny.cu)
// Fused tcgen05 GEMMs.  Forward: Y = [X | sU] [W' | Bp]^T.  Input gradient:
// dX = [dY | sV] [W' ; Ap].  W' is dequantized inside the kernel, or read by TMA from the
// workspace for plans with a staged base.
int launch_fused_fwd(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream);
int launch_fused_dx(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream);
// W' = dequantize(q) into the workspace region Wd, for plans with a staged base.
int launch_stage_base(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream);
// Decode path (M <= 16): Y = X W'^T + sU Bp^T with the weights streamed once.
int launch_skinny_fwd(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream);
// The GEMV: forms U = X A^T inside the launch and the LoRA term from sU and B on the tensor
// cores, or adds a precomputed fp32 term Z when Z is not null.
int launch_decode_gemv(const LinearArgs& a, const WorkspaceLayout& L, const float* Z,
                       cudaStream_t stream);
// Decode path with per-token adapters (multi.cu): U_t = X_t A_{a(t)}^T, then
// Z_t = s_{a(t)} U_t B_{a(t)}^T, then the GEMV adding Z.
int launch_multi_fwd(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream);
// Rank-r side products on the tensor cores (mma.sync), split over the contraction, with the
// split reduction done by the last CTA of each row tile (lora_side.cu).
int launch_lora_u(const LinearArgs& a, const WorkspaceLayout& L, float* u32, cudaStream_t stream,
                  bool narrow_ok = true);
// Whether U / V take the narrow form (one CTA per 128-row tile beside a pair GEMM); that form
// also zeroes the call's arrival tickets, so the call needs no memset.
bool side_narrow_u(const LinearArgs& a);
bool side_narrow_v(const LinearArgs& a);
int launch_lora_v(const LinearArgs& a, const WorkspaceLayout& L, const float* u32,
                  cudaStream_t stream);
int launch_lora_db(const LinearArgs& a, const WorkspaceLayout& L, const float* u32,
                   cudaStream_t stream);
int launch_lora_da(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream);
int launch_pad_b(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream);
uint64_t side_partial_bytes(int64_t M, int64_t N, int64_t K, int r);
// Whether the backward's V forms the dB partials (and launch_lora_db only sums them).
bool fused_db(int64_t M, int64_t N, int64_t K, int r);
uint64_t side_ticket_count(int64_t M, int64_t N, int64_t K);
uint64_t skinny_partial_bytes(int64_t M, int64_t N, int64_t K, int r);
uint64_t skinny_ticket_count(int64_t M, int64_t N);

}  // namespace qlora
