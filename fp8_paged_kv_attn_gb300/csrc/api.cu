// Entry points and host helpers that are not tied to one kernel.
#include <atomic>

#include "kvq_internal.h"

namespace kvq {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];  // 0 = not queried yet
}  // namespace

kvq_status device_sm_count(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KVQ_ERR_CUDA;
  if (dev < kMaxDevices) {
    const int cached = g_sm_count[dev].load(std::memory_order_relaxed);
    if (cached > 0) {
      *sms = cached;
      return KVQ_OK;
    }
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return KVQ_ERR_CUDA;
  if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  *sms = n;
  return KVQ_OK;
}

}  // namespace kvq

extern "C" const char *kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
  }
  return "KVQ_ERR_UNKNOWN";
}

extern "C" kvq_status kvq_selftest_wait(int32_t which, const void *src, uint32_t *err_word,
                                        uint32_t *landed, kvq_stream_t stream) {
  if (!src || !err_word || !landed || !kvq::aligned16(src)) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint32_t *w = static_cast<const uint32_t *>(src);
  if (which == 0) return kvq::selftest_attn_wait(w, err_word, landed, s);
  if (which == 1) return kvq::selftest_ring_wait(w, err_word, landed, s);
  return KVQ_ERR_INVALID_ARG;
}
