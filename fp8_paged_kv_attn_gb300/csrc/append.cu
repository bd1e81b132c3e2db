// kvq_append: quantise-and-append of new K/V into physical cache pages.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "KV 缓存量化": the decode cache keeps K and V as e4m3 instead of BF16.  How
// the values are quantised is not stated; this kernel computes, per element,
// one IEEE fp32 division by the per-tensor scale and a round-to-nearest-even,
// saturating conversion to e4m3 (cvt.rn.satfinite).
//
// One thread owns one 16-byte chunk of the destination (16 e4m3 codes or
// 8 bf16 values) of one (token, kv head) row, so loads of the bf16 source
// (32 B) and stores to the page (16 B) are vectorised and coalesced.  The
// grid strides, so one launch handles a single decode token or a whole prompt.
// It is launched as a programmatic dependent of the work before it on the
// stream (launch_dependent), so it waits for that work before any access.
#include "kvq_internal.h"

namespace kvq {

struct AppendArgs {
  void *k_pool, *v_pool;
  const uint16_t *k_new, *v_new;
  const int32_t *req_idx, *pos, *block_table;
  uint32_t *err_word;
  int64_t n_tokens;
  int32_t num_pages, P, H, D, B, MP;
  float k_scale, v_scale;
};

template <bool kFp8>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  constexpr int kElems = kFp8 ? 16 : 8;  // elements per 16-byte output chunk
  const int64_t chunks_per_row = a.D / kElems;
  const int64_t per_token = static_cast<int64_t>(a.H) * chunks_per_row;
  const int64_t per_tensor = a.n_tokens * per_token;
  const int64_t total = 2 * per_tensor;
  const int64_t cap = static_cast<int64_t>(a.MP) * a.P;
  grid_dependency_wait();  // earlier work on the stream is complete and visible
  allow_dependents();

  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_v = idx >= per_tensor;
    const int64_t rem = is_v ? idx - per_tensor : idx;
    const int64_t t = rem / per_token;
    const int h = static_cast<int>((rem / chunks_per_row) % a.H);
    const int c = static_cast<int>(rem % chunks_per_row);
    const bool reporter = (rem % per_token) == 0 && !is_v;  // one report per bad token

    const int r = a.req_idx[t];
    const int p = a.pos[t];
    if (r < 0 || r >= a.B) {
      if (reporter) report(a.err_word, KVQ_ERRBIT_REQ);
      continue;
    }
    if (p < 0 || p >= cap) {
      if (reporter) report(a.err_word, KVQ_ERRBIT_POS);
      continue;
    }
    const int page = a.block_table[static_cast<int64_t>(r) * a.MP + p / a.P];
    if (page < 0 || page >= a.num_pages) {
      if (reporter) report(a.err_word, KVQ_ERRBIT_PAGE);
      continue;
    }
    const int slot = p % a.P;

    const uint16_t *src = (is_v ? a.v_new : a.k_new) +
                          (t * a.H + h) * static_cast<int64_t>(a.D) + c * kElems;
    const int64_t dst_elem =
        ((static_cast<int64_t>(page) * a.H + h) * a.P + slot) * a.D + c * kElems;

    if constexpr (kFp8) {
      const uint4 s0 = __ldg(reinterpret_cast<const uint4 *>(src));
      const uint4 s1 = __ldg(reinterpret_cast<const uint4 *>(src) + 1);
      const uint32_t w[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
      const float scale = is_v ? a.v_scale : a.k_scale;
      uint32_t o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float x[4];
        bf16x2_to_f32(w[2 * i], x);
        bf16x2_to_f32(w[2 * i + 1], x + 2);
        const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
        const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
        o[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      }
      uint8_t *dst = static_cast<uint8_t *>(is_v ? a.v_pool : a.k_pool) + dst_elem;
      *reinterpret_cast<uint4 *>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
      const uint4 s0 = __ldg(reinterpret_cast<const uint4 *>(src));
      uint16_t *dst = static_cast<uint16_t *>(is_v ? a.v_pool : a.k_pool) + dst_elem;
      *reinterpret_cast<uint4 *>(dst) = s0;
    }
  }
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_append(const kvq_cache *cache, const void *k_new, const void *v_new,
                                 const int32_t *req_idx, const int32_t *pos, int32_t n_tokens,
                                 const int32_t *block_table, int32_t B, int32_t MP,
                                 uint32_t *err_word, kvq_stream_t stream) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_tokens < 0 || B < 0 || MP <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_tokens == 0) return KVQ_OK;
  if (!k_new || !v_new || !req_idx || !pos || !block_table || B == 0)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(MP) * cache->page_size > INT32_MAX) return KVQ_ERR_INVALID_ARG;

  AppendArgs a;
  a.k_pool = cache->k_pool;
  a.v_pool = cache->v_pool;
  a.k_new = static_cast<const uint16_t *>(k_new);
  a.v_new = static_cast<const uint16_t *>(v_new);
  a.req_idx = req_idx;
  a.pos = pos;
  a.block_table = block_table;
  a.err_word = err_word;
  a.n_tokens = n_tokens;
  a.num_pages = cache->num_pages;
  a.P = cache->page_size;
  a.H = cache->num_kv_heads;
  a.D = cache->head_dim;
  a.B = B;
  a.MP = MP;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;

  const bool fp8 = cache->kv_dtype == KVQ_KV_E4M3;
  const int64_t chunk_elems = fp8 ? 16 : 8;
  const int64_t total = 2LL * n_tokens * a.H * (a.D / chunk_elems);
  const int threads = 256;
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const int64_t want = (total + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 16LL * sms ? want : 16LL * sms);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = fp8 ? launch_dependent(append_kernel<true>, blocks, threads, 0, s, a)
                            : launch_dependent(append_kernel<false>, blocks, threads, 0, s, a);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
