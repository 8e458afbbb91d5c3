// device_cache.h -- one-time set-up results kept per device: kernel attributes set with
// cudaFuncSetAttribute, occupancy figures, device addresses of __device__ symbols.
//
// Such results belong to one device's context, not to the process.  Each entry is keyed by
// the device ordinal and by the id of the context that was current when it was made, so a
// second device repeats the set-up for itself and a context destroyed and created again
// (cudaDeviceReset) does not reuse values from the old one.  A set-up that fails stores
// nothing: the next call tries again.  The lookup holds a mutex, so two host threads that
// meet the same first use run the set-up once.
//
// Plain C++ (no CUDA types): the caller passes the key (device_context_key() in
// tensormap.cu reads it from the runtime and driver).
#pragma once

#include <stdint.h>

#include <mutex>

namespace qlora {

constexpr int kMaxCachedDevices = 64;

struct DeviceKey {
  int device;       // ordinal; negative when it could not be read
  uint64_t context; // id of the device's current context; 0 before one exists
};

template <typename T>
class DeviceCache {
 public:
  // The value for the current key: the cached one, or compute(&v) (a status, 0 = success)
  // stored under the key read again after it ran (the set-up may itself create the
  // context).  key() returns the current DeviceKey.  Returns compute's status, or -1 for a
  // device ordinal out of range.
  template <typename KeyFn, typename ComputeFn>
  int get(KeyFn&& key, T* out, ComputeFn&& compute) {
    std::lock_guard<std::mutex> lk(mu_);
    DeviceKey k = key();
    if (k.device < 0 || k.device >= kMaxCachedDevices) return -1;
    Entry& e = entries_[k.device];
    if (e.valid && k.context != 0 && e.context == k.context) {
      *out = e.value;
      return 0;
    }
    T v{};
    const int st = compute(&v);
    if (st != 0) {
      e.valid = false;
      return st;
    }
    const DeviceKey after = key();
    e.context = after.device == k.device ? after.context : 0;
    e.value = v;
    e.valid = e.context != 0;  // without a context id the next call repeats the set-up
    *out = v;
    return 0;
  }

  // Forget the current device's entry (for instance after a launch with it failed).
  void invalidate(int device) {
    std::lock_guard<std::mutex> lk(mu_);
    if (device >= 0 && device < kMaxCachedDevices) entries_[device].valid = false;
  }

 private:
  struct Entry {
    bool valid = false;
    uint64_t context = 0;
    T value{};
  };
  std::mutex mu_;
  Entry entries_[kMaxCachedDevices];
};

}  // namespace qlora
