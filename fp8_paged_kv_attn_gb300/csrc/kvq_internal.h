// Host-side helpers shared by the kvq entry points.
#pragma once

#include <cmath>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "kvq.h"
#include "kvq_device.cuh"

namespace kvq {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// Number of SMs of the current device (cached per device).
kvq_status device_sm_count(int *sms);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda); null when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Self-tests of the bounded waits (kvq_selftest_wait): the split kernels'
// (decode_attn.cu) and the weight ring's (wq_gemm.cu).
kvq_status selftest_attn_wait(const uint32_t *src, uint32_t *err_word, uint32_t *landed,
                              cudaStream_t stream);
kvq_status selftest_ring_wait(const uint32_t *src, uint32_t *err_word, uint32_t *landed,
                              cudaStream_t stream);

// Launches `kernel` as a programmatic dependent of the work ahead of it on
// `stream`: its CTAs may be scheduled as soon as the previous kernel has let
// dependents go (or has finished), which hides the launch latency between
// the kernels of a decode step.  The kernel must call grid_dependency_wait()
// before it touches global memory, which keeps plain stream order for the
// data.  Captured into a CUDA graph, the launch becomes a programmatic edge.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Checks of the cache descriptor common to every entry point.
inline kvq_status validate_cache(const kvq_cache *c) {
  if (!c || !c->k_pool || !c->v_pool) return KVQ_ERR_INVALID_ARG;
  if (c->kv_dtype != KVQ_KV_E4M3 && c->kv_dtype != KVQ_KV_BF16) return KVQ_ERR_INVALID_ARG;
  if (c->num_pages <= 0 || c->num_kv_heads <= 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(c->k_pool) || !aligned16(c->v_pool)) return KVQ_ERR_INVALID_ARG;
  if (c->page_size != 16 && c->page_size != 32 && c->page_size != 64) return KVQ_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (c->kv_dtype == KVQ_KV_E4M3) {
    if (!(std::isfinite(c->k_scale) && c->k_scale > 0.f)) return KVQ_ERR_INVALID_ARG;
    if (!(std::isfinite(c->v_scale) && c->v_scale > 0.f)) return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

}  // namespace kvq
