// kda_noalloc.cu -- the static device scratch behind kda_commit_noalloc.
//
// The commit kernel reads six per-layer tables (state, correction and
// key/gate base addresses and strides) through device pointers.  Callers that
// cannot allocate device memory get them from this file-scope array instead:
// the host entry passes its host tables by value to fill_tables, which writes
// them into the array in stream order, and the unchanged commit kernel reads
// them from there.
#include <cuda_runtime.h>

#include <mutex>

#include "kda.h"

namespace kda {

// [6][KDA_NOALLOC_MAX_LAYERS] int64: state_base, state_slot_stride, corr_base,
// corr_row_stride, kg_base, kg_row_stride (3 KB).
static __device__ __align__(256) long long g_noalloc_tables[6 * KDA_NOALLOC_MAX_LAYERS];

struct NoallocTables {
  long long v[6 * KDA_NOALLOC_MAX_LAYERS];  // 3 KB of kernel parameters
};

// Copies the tables, passed by value in the launch parameters, into the scratch.
__global__ void fill_tables(const __grid_constant__ NoallocTables t) {
  for (int i = static_cast<int>(threadIdx.x); i < 6 * KDA_NOALLOC_MAX_LAYERS; i += static_cast<int>(blockDim.x))
    g_noalloc_tables[i] = t.v[i];
}

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

// Enqueues the fill of the scratch from six host tables of L entries (table
// j of layer l lands at [j * KDA_NOALLOC_MAX_LAYERS + l]; unused entries 0).
// The host arrays are read here, during the call, into the launch parameters.
cudaError_t noalloc_fill(const int64_t* const src[6], int L, cudaStream_t stream) {
  NoallocTables t;
  for (int j = 0; j < 6; ++j)
    for (int l = 0; l < KDA_NOALLOC_MAX_LAYERS; ++l)
      t.v[j * KDA_NOALLOC_MAX_LAYERS + l] = l < L ? static_cast<long long>(src[j][l]) : 0;
  fill_tables<<<1, 128, 0, stream>>>(t);
  return cudaGetLastError();
}

}  // namespace kda
