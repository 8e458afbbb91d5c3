// Host-only check of the per-device set-up cache (device_cache.h): built with g++ and run by
// tests/test_library_cpu.py.  The device / context key is faked, no CUDA is involved.
#include <cstdio>

#include "../bit_nf4_quantized_37_b300/csrc/device_cache.h"

using qlora::DeviceCache;
using qlora::DeviceKey;

static DeviceKey g_key{0, 0};
static int g_computes = 0;

static DeviceKey key() { return g_key; }

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      std::printf("FAILED line %d: %s\n", __LINE__, #c);      \
      return 1;                                               \
    }                                                         \
  } while (0)

int main() {
  DeviceCache<int> cache;
  int v = 0;
  auto compute = [](int* out) {
    ++g_computes;
    *out = 100 * g_key.device + static_cast<int>(g_key.context);
    return 0;
  };
  // first use on device 0, context 7: computed once, then served from the cache
  g_key = {0, 7};
  CHECK(cache.get(key, &v, compute) == 0 && v == 7 && g_computes == 1);
  CHECK(cache.get(key, &v, compute) == 0 && v == 7 && g_computes == 1);
  // another device: its own entry
  g_key = {1, 9};
  CHECK(cache.get(key, &v, compute) == 0 && v == 109 && g_computes == 2);
  g_key = {0, 7};
  CHECK(cache.get(key, &v, compute) == 0 && v == 7 && g_computes == 2);
  // device 0's context replaced (a reset): the set-up runs again
  g_key = {0, 8};
  CHECK(cache.get(key, &v, compute) == 0 && v == 8 && g_computes == 3);
  CHECK(cache.get(key, &v, compute) == 0 && v == 8 && g_computes == 3);
  // a failing set-up stores nothing and returns its status
  g_key = {2, 5};
  CHECK(cache.get(key, &v, [](int*) { return -5; }) == -5);
  CHECK(cache.get(key, &v, compute) == 0 && v == 205 && g_computes == 4);
  // no context yet before the set-up, one after it: stored under the context seen after
  g_key = {3, 0};
  CHECK(cache.get(key, &v, [](int* out) { g_key.context = 11; *out = 311; return 0; }) == 0);
  CHECK(cache.get(key, &v, compute) == 0 && v == 311 && g_computes == 4);
  // no context id at all: never cached
  g_key = {4, 0};
  CHECK(cache.get(key, &v, compute) == 0 && g_computes == 5);
  CHECK(cache.get(key, &v, compute) == 0 && g_computes == 6);
  // ordinals out of range are refused without running the set-up
  g_key = {-1, 1};
  CHECK(cache.get(key, &v, compute) == -1 && g_computes == 6);
  g_key = {qlora::kMaxCachedDevices, 1};
  CHECK(cache.get(key, &v, compute) == -1 && g_computes == 6);
  // invalidate forgets one device only
  g_key = {1, 9};
  cache.invalidate(1);
  CHECK(cache.get(key, &v, compute) == 0 && g_computes == 7);
  g_key = {0, 8};
  CHECK(cache.get(key, &v, compute) == 0 && v == 8 && g_computes == 7);
  std::printf("OK\n");
  return 0;
}
