// Host-side helpers shared by the kvq entry points.
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "kvq.h"
#include "kvq_device.cuh"

namespace kvq {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

// Number of SMs of the current device (cached per device).
kvq_status device_sm_count(int *sms);

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
