// kvq_decode_attn_static: decode attention for callers that cannot allocate
// device memory.
//
// kvq_decode_attn needs a caller-supplied workspace (the work plan and the
// split partials).  Some callers have no way to provide one: a serving
// runtime that reserves all device memory up front and hands it out only
// from its own pool has nothing to give a library on the decode hot path, a
// plugin host may forbid allocation inside its execute callback, and a
// latency-bound loop cannot afford cudaMalloc's implicit synchronisation.
// This entry point uses scratch that lives in this library's own device
// image instead: a file-scope device array of kStaticScratchBytes (64 MiB).
// Every GPU that loads this part of the library holds that array until the
// process exits.
//
// The array's host-side name is only a stand-in for the device symbol, so its
// device address is looked up with cudaGetSymbolAddress, with the caller's
// device current, on every call.  The lookup is a host-side query once the
// library's device code is loaded on that device; the first call on a device
// may load it, so that first call should come before any stream capture.
// Looking the address up each time (rather than caching it) keeps the call
// correct after the primary context is destroyed and re-created
// (cudaDeviceReset), when the array can move.  Every call shares the same
// array and it keeps the previous call's contents: the plan kernel rewrites
// everything the attention kernels read before they read it, so stale
// contents are harmless, but two calls whose kernels overlap on the GPU
// (different streams, or different host threads) race on the array and must
// not be issued.
#include "kvq_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = KVQ_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_kvq_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device.
kvq_status scratch_on_current_device(void **ptr) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_kvq_scratch) != cudaSuccess || !p) return KVQ_ERR_CUDA;
  *ptr = p;
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_decode_attn_static(const kvq_cache *cache, const void *q, int32_t B,
                                             int32_t Hq, const int32_t *block_table, int32_t MP,
                                             const int32_t *seq_lens, const uint8_t *abort_mask,
                                             float sm_scale, float *out, uint32_t *err_word,
                                             kvq_stream_t stream) {
  if (!cache || cache->num_kv_heads <= 0 || Hq <= 0 || B < 0) return KVQ_ERR_INVALID_ARG;
  const size_t need = kvq_decode_attn_workspace_size(B, Hq, cache->num_kv_heads, cache->head_dim);
  if (need == 0 && B > 0) return KVQ_ERR_INVALID_ARG;
  if (need > kStaticScratchBytes) return KVQ_ERR_WORKSPACE;  // batch too large for the array
  void *scratch = nullptr;
  const kvq_status st = scratch_on_current_device(&scratch);
  if (st != KVQ_OK) return st;
  return kvq_decode_attn(cache, q, B, Hq, block_table, MP, seq_lens, abort_mask, sm_scale, out,
                         scratch, kStaticScratchBytes, err_word, stream);
}
