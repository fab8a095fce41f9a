// Host-side failure injection for allocations (see alloc.h and mag_debug_fail_allocations).
#include "alloc.h"

#include <atomic>
#include <cstdint>

#include "mag.h"

namespace mag {
namespace {
std::atomic<int64_t> g_skip{0};  // allocations still to succeed before the failures
std::atomic<int64_t> g_fail{0};  // failures still to inject
}  // namespace

bool alloc_injected_failure() {
  if (g_fail.load(std::memory_order_relaxed) <= 0) return false;
  if (g_skip.fetch_sub(1, std::memory_order_relaxed) > 0) return false;
  g_skip.store(0, std::memory_order_relaxed);
  return g_fail.fetch_sub(1, std::memory_order_relaxed) > 0;
}

}  // namespace mag

extern "C" void mag_debug_fail_allocations(int32_t skip, int32_t count) {
  mag::g_skip.store(skip > 0 ? skip : 0);
  mag::g_fail.store(count > 0 ? count : 0);
}
