// Device error word set by kernels whose bounded waits give up; read and
// cleared by yr_sync_status().  The device addresses are looked up once per
// device and cached; the cache assumes the CUDA context of a device lives as
// long as the process (the library is not to be used across a device reset).
#include <atomic>
#include <mutex>

#include "internal.h"

namespace yr {

__device__ int g_status_word = 0;

int* device_status_word() {
  static std::mutex mu;
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

static std::atomic<unsigned long long> g_launches{0};
static std::atomic<long long> g_wait_limit{0};
static std::atomic<int> g_skip_unit{-1};

FaultInjection fault_injection() {
  const long long w = g_wait_limit.load(std::memory_order_relaxed);
  return {w > 0 ? w : 4000000000ll, g_skip_unit.load(std::memory_order_relaxed)};
}

cudaError_t launched(int n) {
  const cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed);
  return e;
}

}  // namespace yr

extern "C" yr_status yr_debug_inject_wait_fault(int64_t wait_limit_cycles, int32_t skip_unit) {
  yr::clear_error();
  if (wait_limit_cycles < 0 || skip_unit < -1)
    return yr::fail(YR_ERR_INVALID_ARG, "yr_debug_inject_wait_fault: wait_limit_cycles >= 0, skip_unit >= -1");
  yr::g_wait_limit.store(wait_limit_cycles, std::memory_order_relaxed);
  yr::g_skip_unit.store(skip_unit, std::memory_order_relaxed);
  return YR_OK;
}

extern "C" uint64_t yr_kernel_launch_count(void) { return yr::g_launches.load(std::memory_order_relaxed); }
