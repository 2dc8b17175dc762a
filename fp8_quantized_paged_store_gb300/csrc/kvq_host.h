// kvq_host.h — host-side helpers for the C ABI entry points: argument checks,
// launch-shape choice and launch-error mapping. Internal to the library.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Number of SMs of the current device (queried once per device). Internal
// linkage: as a plain inline function its cache would be one STB_GNU_UNIQUE
// object that the dynamic linker shares among every copy of the library
// loaded into a process; static keeps one per translation unit instead.
static inline int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

// Blocks of a kernel that fit on one SM at once (queried once per kernel and
// device through the occupancy calculator).
template <typename Kernel>
inline int resident_blocks_per_sm(Kernel kernel, int threads, size_t dynamic_smem, int* cache64) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache64[dev] == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, dynamic_smem) != cudaSuccess ||
        n <= 0)
      n = 1;
    cache64[dev] = n;
  }
  return cache64[dev];
}

// Grid for a grid-stride kernel: enough blocks to cover `work_blocks`, at
// most one full wave of resident blocks on every SM.
inline unsigned grid_for(int64_t work_blocks, int per_sm) {
  int64_t wave = (int64_t)sm_count() * per_sm;
  int64_t g = work_blocks < wave ? work_blocks : wave;
  return (unsigned)(g < 1 ? 1 : g);
}

// Status of the launch just issued. cudaGetLastError also resets the error, so
// a failed launch is reported once, here, and not again by the caller's next
// CUDA call.
inline int launch_status() {
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ECUDA;
}

}  // namespace kvq
