// kda_noalloc.cu -- the static device scratch behind kda_commit_noalloc.
//
// The commit kernel reads six per-layer tables (state, correction and
// key/gate base addresses and strides) through device pointers.  Callers that
// cannot allocate device memory get them from this file-scope array instead:
// the host entry copies its host tables into it, in stream order, and passes
// its address to the unchanged commit kernel.
#include <cuda_runtime.h>

#include <mutex>

#include "kda.h"

namespace kda {

// [6][KDA_NOALLOC_MAX_LAYERS] int64: state_base, state_slot_stride, corr_base,
// corr_row_stride, kg_base, kg_row_stride (3 KB).
static __device__ __align__(256) long long g_noalloc_tables[6 * KDA_NOALLOC_MAX_LAYERS];

// Device address of the scratch on the current device, resolved once per
// device (cudaGetSymbolAddress may load the module, so the first call is the
// set-up and must not happen inside a stream capture).
cudaError_t noalloc_tables(long long** out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static long long* cached[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_tables);
    if (e != cudaSuccess) return e;
    cached[dev] = static_cast<long long*>(ptr);
  }
  *out = cached[dev];
  return cudaSuccess;
}

}  // namespace kda
