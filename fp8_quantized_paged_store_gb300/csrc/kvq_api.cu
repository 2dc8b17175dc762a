// kvq_api.cu — the small host-only entry points of the C ABI.
#include <cstdint>

#include <cuda_runtime.h>

#include "kvq.h"

extern "C" const char* kvq_strerror(int status) {
  switch (status) {
    case KVQ_OK:
      return "success";
    case KVQ_EINVAL:
      return "invalid argument (shape, range, null pointer or alignment); nothing was launched";
    case KVQ_ECUDA:
      return "CUDA kernel launch failed";
    case KVQ_ESCRATCH:
      return "the shapes need more scratch than the library's built-in array holds; nothing was "
             "launched";
    default:
      return "unknown status";
  }
}

// "vllm.v1.attention.ops.mxfp4_mla.store", module docstring: a packed row is
// d/2 code bytes followed by d/group scale bytes.
extern "C" int64_t kvq_row_bytes(int64_t latent_dim, int64_t group) {
  if (latent_dim <= 0 || group <= 0 || group % 2 != 0 || latent_dim % group != 0) return -1;
  return latent_dim / 2 + latent_dim / group;
}

// Where `ptr` lives, as far as a kernel launched on the current device can
// reach it under that same address.
extern "C" int kvq_pointer_kind(const void* ptr) {
  if (ptr == nullptr) return KVQ_EINVAL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ECUDA;
  }
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return KVQ_ECUDA;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
      return a.device == dev ? KVQ_PTR_DEVICE : KVQ_PTR_UNADDRESSABLE;
    case cudaMemoryTypeManaged:
      return KVQ_PTR_DEVICE;
    case cudaMemoryTypeHost:
      return a.devicePointer == ptr ? KVQ_PTR_HOST_MAPPED : KVQ_PTR_UNADDRESSABLE;
    default:
      return KVQ_PTR_UNADDRESSABLE;
  }
}
