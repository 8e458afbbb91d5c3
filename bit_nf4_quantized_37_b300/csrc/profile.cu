// profile.cu -- opt-in per-kernel device timing: while enabled, every launch of the library
// is bracketed by CUDA events on its own stream, and qlora_profile_stop sums the elapsed
// time per kernel.  Off by default; when off a scope costs one branch.
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "launch.h"
#include "profile.h"

namespace qlora {
namespace {

struct Rec {
  const char* name;
  cudaEvent_t a, b;
};

std::mutex g_mu;
bool g_on = false;
std::vector<Rec> g_recs;
std::vector<cudaEvent_t> g_pool;

// Inside a stream capture an event record must be "external" to become a real event-record
// node of the graph (a plain record only marks a capture dependency); outside a capture
// the plain record is the valid form.
void record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    cudaEventRecord(e, s);
}

cudaEvent_t take_event() {
  if (!g_pool.empty()) {
    cudaEvent_t e = g_pool.back();
    g_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

}  // namespace

bool profiling_enabled() { return g_on; }

ProfileScope::ProfileScope(const char* name, cudaStream_t stream) : name_(name), stream_(stream) {
  if (!g_on) return;
  std::lock_guard<std::mutex> lk(g_mu);
  start_ = take_event();
  if (start_) record(start_, stream_);
}

ProfileScope::~ProfileScope() {
  if (!g_on || !start_) return;
  std::lock_guard<std::mutex> lk(g_mu);
  cudaEvent_t stop = take_event();
  if (!stop) return;
  record(stop, stream_);
  g_recs.push_back({name_, start_, stop});
}

}  // namespace qlora

using namespace qlora;

extern "C" int qlora_profile_start(void) {
  std::lock_guard<std::mutex> lk(g_mu);
  for (auto& r : g_recs) {
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  g_on = true;
  return QLORA_OK;
}

extern "C" int qlora_profile_stop(qlora_kernel_time* out, int32_t capacity, int32_t* count) {
  if (!count || (capacity > 0 && !out)) return QLORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_mu);
  g_on = false;
  int st = QLORA_OK;
  std::vector<qlora_kernel_time> agg;
  for (auto& r : g_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) {
      st = QLORA_ERR_CUDA;
      continue;
    }
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
      st = QLORA_ERR_CUDA;
      continue;
    }
    qlora_kernel_time* slot = nullptr;
    for (auto& k : agg)
      if (std::strncmp(k.name, r.name, sizeof(k.name)) == 0) slot = &k;
    if (!slot) {
      qlora_kernel_time k{};
      std::strncpy(k.name, r.name, sizeof(k.name) - 1);
      agg.push_back(k);
      slot = &agg.back();
    }
    slot->launches += 1;
    slot->total_ms += ms;
  }
  for (auto& r : g_recs) {
    g_pool.push_back(r.a);
    g_pool.push_back(r.b);
  }
  g_recs.clear();
  *count = static_cast<int32_t>(agg.size());
  for (int i = 0; i < capacity && i < (int)agg.size(); ++i) out[i] = agg[i];
  return st;
}
