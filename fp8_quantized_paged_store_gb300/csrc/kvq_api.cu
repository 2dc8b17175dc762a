// kvq_api.cu — the small host-only entry points of the C ABI.
#include <cstdint>

#include "kvq.h"

extern "C" const char* kvq_strerror(int status) {
  switch (status) {
    case KVQ_OK:
      return "success";
    case KVQ_EINVAL:
      return "invalid argument (shape, range, null pointer or alignment); nothing was launched";
    case KVQ_ECUDA:
      return "CUDA kernel launch failed";
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
