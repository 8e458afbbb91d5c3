// linear.cu -- orchestration of the LoRA-wrapped NF4 linear layer.
//
// forward   pad adapters -> U = X A^T (sU = 16-bit(s U)) -> [W' dequantized once, for GEMM
//           plans with a staged base] -> fused GEMM (M > 16) or the decode kernel (M <= 16)
// backward  U (saved or recomputed) -> V = dY B (sV) -> fused input-gradient GEMM, with
//           dB = s dY^T U and dA = (X^T sV)^T on a side stream meanwhile
// The NF4 buffers are only read (junaidshaukat.com recipe item 3: the base never moves).
//
// The input-gradient GEMM leaves SMs idle in its last wave; the two rank-r side products
// of the backward do not depend on it, so they run on a low-priority side stream forked
// from the caller's stream (the GEMM is launched first, at the greatest priority) and the
// caller's stream waits for both before the call returns.  Fork and join are event-based,
// so the pattern is also captured into CUDA graphs.
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
  L.dbpart_bytes = fused_db(M, N, K, r) ? (uint64_t)((M + 127) / 128) * N * 64 : 0;
  L.dbpart = take(L.dbpart_bytes);
  L.Bp = take(r % 8 ? (uint64_t)N * L.rp * 2 : 0);
  L.part_bytes = std::max(side_partial_bytes(M, N, K, r), skinny_partial_bytes(M, N, K, r));
  L.part = take(L.part_bytes);
  // the split reductions' counters; at least one per token for the per-token adapter path
  L.ntickets = std::max<uint64_t>(std::max(side_ticket_count(M, N, K), skinny_ticket_count(M, N)),
                                  (uint64_t)kSkinnyMaxM);
  // the fused GEMMs' split contraction: the forward takes them above kSkinnyMaxM tokens, the
  // input gradient at every M
  const uint64_t gpart_bytes = fused_partial_bytes(M, N, K, &L.ngtickets);
  L.nticket_words = L.ntickets + L.ngtickets + 1;
  L.tickets = take(L.nticket_words * 4);
  L.gtickets = L.tickets + L.ntickets * 4;
  L.pers_ctr = L.gtickets + L.ngtickets * 4;
  L.gpart = take(gpart_bytes);
  L.gpart_bytes = gpart_bytes;
  L.Z = take(M <= kSkinnyMaxM ? (uint64_t)M * N * 4 : 0);
  L.Wd_bytes = (fused_plan(M, N, K).wstage || fused_plan(M, K, N).wstage) ? (uint64_t)N * K * 2 : 0;
  L.Wd = take(L.Wd_bytes);
  L.total = off;
  return L;
}

uint64_t linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int r) {
  return workspace_layout(M, N, K, r).total;
}

static int clear_tickets(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  return cudaMemsetAsync(static_cast<uint8_t*>(a.ws) + L.tickets, 0, L.nticket_words * 4,
                         stream) ==
                 cudaSuccess
             ? QLORA_OK
             : QLORA_ERR_CUDA;
}

int linear_forward(const LinearArgs& a, cudaStream_t stream) {
  const WorkspaceLayout L = workspace_layout(a.M, a.N, a.K, a.r);
  const bool small = a.adapter_idx || a.M <= kSkinnyMaxM;
  int st = QLORA_OK;
  // the narrow U zeroes the arrival tickets itself
  if ((small || !side_narrow_u(a)) && (st = clear_tickets(a, L, stream))) return st;
  if (a.adapter_idx) return launch_multi_fwd(a, L, stream);  // M <= 16, checked by the caller
  if (a.M <= kSkinnyMaxM) return launch_skinny_fwd(a, L, stream);
  if ((st = launch_lora_u(a, L, a.U, stream))) return st;
  if (a.r % 8 && (st = launch_pad_b(a, L, stream))) return st;
  if (fused_plan(a.M, a.N, a.K).wstage && (st = launch_stage_base(a, L, stream))) return st;
  return launch_fused_fwd(a, L, stream);
}

int launch_stage_base(const LinearArgs& a, const WorkspaceLayout& L, cudaStream_t stream) {
  if (L.Wd_bytes < (uint64_t)a.N * a.K * 2) return QLORA_ERR_WORKSPACE;
  // a programmatic dependent of the rank-r product before it: the two run side by side
  return launch_dequantize(a.q, a.N * a.K,
                           reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(a.ws) + L.Wd), a.half,
                           stream, /*dependent=*/true);
}

namespace {

// Side stream and fork / join events of the calling host thread on the current device
// (and its context: after a context is created again they are created again).
struct SideContext {
  int device = -1;
  uint64_t context = 0;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  int prio_hi = 0;
  ~SideContext() {
    if (side) cudaStreamDestroy(side);
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
  }
};

SideContext* side_context() {
  thread_local SideContext ctx[kMaxCachedDevices];
  const DeviceKey k = device_context_key();
  const int dev = k.device;
  if (dev < 0 || dev >= kMaxCachedDevices) return nullptr;
  SideContext& c = ctx[dev];
  if (c.device == dev && k.context != 0 && c.context == k.context) return &c;
  if (c.device == dev) {  // handles of a context that no longer exists: drop, do not destroy
    c.side = nullptr;
    c.fork = c.join = nullptr;
    c.device = -1;
  }
  int least = 0, greatest = 0;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&c.side, cudaStreamNonBlocking, least) != cudaSuccess ||
      cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  c.prio_hi = greatest;
  c.device = dev;
  c.context = device_context_key().context;  // the calls above created it if it was missing
  return &c;
}

}  // namespace

int linear_backward(const LinearArgs& a, cudaStream_t stream) {
  const WorkspaceLayout L = workspace_layout(a.M, a.N, a.K, a.r);
  int st = QLORA_OK;
  // the narrow V zeroes the arrival tickets itself, unless a recomputed U before it uses them
  if ((!a.U_in || !side_narrow_v(a)) && (st = clear_tickets(a, L, stream))) return st;
  const float* u32 = a.U_in;
  if (!u32) {
    float* w = reinterpret_cast<float*>(static_cast<uint8_t*>(a.ws) + L.U32);
    if ((st = launch_lora_u(a, L, w, stream, /*narrow_ok=*/false))) return st;
    u32 = w;
  }
  if ((st = launch_lora_v(a, L, u32, stream))) return st;
  SideContext* sc = a.dX ? side_context() : nullptr;
  const bool wstage = a.dX && fused_plan(a.M, a.K, a.N).wstage;
  if (!sc) {
    if ((st = launch_lora_db(a, L, u32, stream))) return st;
    if (wstage && (st = launch_stage_base(a, L, stream))) return st;
    if (a.dX && (st = launch_fused_dx(a, L, stream))) return st;
    return launch_lora_da(a, L, stream);
  }
  // fork: the GEMM first (greatest priority) on the caller's stream, then dB and dA on the
  // side stream; they share the split-reduction workspace only with each other
  if (cudaEventRecord(sc->fork, stream) != cudaSuccess) return QLORA_ERR_CUDA;
  LinearArgs hi = a;
  hi.gemm_priority = sc->prio_hi;
  if (wstage && (st = launch_stage_base(a, L, stream))) return st;
  if ((st = launch_fused_dx(hi, L, stream))) return st;
  if (cudaStreamWaitEvent(sc->side, sc->fork, 0) != cudaSuccess) return QLORA_ERR_CUDA;
  if ((st = launch_lora_db(a, L, u32, sc->side))) return st;
  if ((st = launch_lora_da(a, L, sc->side))) return st;
  if (cudaEventRecord(sc->join, sc->side) != cudaSuccess) return QLORA_ERR_CUDA;
  return cudaStreamWaitEvent(stream, sc->join, 0) == cudaSuccess ? QLORA_OK : QLORA_ERR_CUDA;
}

}  // namespace qlora
