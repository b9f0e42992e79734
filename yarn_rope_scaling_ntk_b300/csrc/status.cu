// Device error word set by kernels whose bounded waits give up; read and
// cleared by yr_sync_status().
#include "internal.h"

namespace yr {

__device__ int g_status_word = 0;

int* device_status_word() {
  static int* cached[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

}  // namespace yr
