// linear.cu -- orchestration of the LoRA-wrapped NF4 linear layer on one stream.
//
// forward   pad adapters -> U = X A^T (sU = bf16(s U)) -> fused GEMM (M > 16) or the decode
//           kernel (M <= 16)
// backward  pad adapters -> U^T (saved or recomputed) -> V = dY B (sV, sV^T)
//           -> dB = s dY^T U -> fused input-gradient GEMM -> dA = (X^T sV)^T
// The NF4 buffers are only read (junaidshaukat.com recipe item 3: the base never moves).
#include <algorithm>

#include "launch.h"
#include "linear.h"

namespace qlora {

WorkspaceLayout workspace_layout(int64_t M, int64_t N, int64_t K, int r) {
  WorkspaceLayout L{};
  L.rp = round_up(r, 64);
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t at = off;
    off = (uint64_t)round_up((int64_t)(off + bytes), 1024);
    return at;
  };
  L.sU = take((uint64_t)M * L.rp * 2);
  L.sV = take((uint64_t)M * L.rp * 2);
  L.U32 = take((uint64_t)M * r * 4);
  L.Bp = take(r % 8 ? (uint64_t)N * L.rp * 2 : 0);
  L.part_bytes = std::max(side_partial_bytes(M, N, K, r), skinny_partial_bytes(M, N, K, r));
  L.part = take(L.part_bytes);
  L.ntickets = side_ticket_count(M, N, K);
  L.tickets = take(L.ntickets * 4);
  L.total = off;
  return L;
}

uint64_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int r) {
  return workspace_layout(M, N, K, r).total;
}

static int clear_tickets(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  return cudaMemsetAsync(static_cast<uint8_t*>(a.ws) + L.tickets, 0, L.ntickets * 4, stream) ==
                 cudaSuccess
             ? QLORA_OK
             : QLORA_ERR_CUDA;
}

int linear_forward(const LinearArgs& a, cudaStream_t stream) {
  const WorkspaceLayout L = workspace_layout(a.M, a.N, a.K, a.r);
  int st = clear_tickets(a, L, stream);
  if (st) return st;
  if (a.M <= kSkinnyMaxM) return launch_skinny_fwd(a, L, stream);
  if ((st = launch_lora_u(a, L, a.U, stream))) return st;
  if (a.r % 8 && (st = launch_pad_b(a, L, stream))) return st;
  return launch_fused_fwd(a, L, stream);
}

int linear_backward(const LinearArgs& a, cudaStream_t stream) {
  const WorkspaceLayout L = workspace_layout(a.M, a.N, a.K, a.r);
  int st = clear_tickets(a, L, stream);
  if (st) return st;
  const float* u32 = a.U_in;
  if (!u32) {
    float* w = reinterpret_cast<float*>(static_cast<uint8_t*>(a.ws) + L.U32);
    if ((st = launch_lora_u(a, L, w, stream))) return st;
    u32 = w;
  }
  if ((st = launch_lora_v(a, L, stream))) return st;
  if ((st = launch_lora_db(a, L, u32, stream))) return st;
  if (a.dX && (st = launch_fused_dx(a, L, stream))) return st;
  return launch_lora_da(a, L, stream);
}

}  // namespace qlora
