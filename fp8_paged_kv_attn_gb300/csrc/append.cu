// kvq_append: quantise-and-append of new K/V into physical cache pages.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "KV 缓存量化": the decode cache keeps K and V as e4m3 instead of BF16.  How
// the values are quantised is not stated; this kernel produces, per element,
// the e4m3 code of the correctly rounded fp32 quotient x / scale under
// round-to-nearest-even with saturation to +-448 (cvt.rn.satfinite).  The
// same call serves one decode token per request or whole prompts (the
// prefill -> decode handoff).
//
// Work layout: one warp per token.  The token's K and V (2 x H x D
// elements) are 16-byte output chunks (16 e4m3 codes or 8 bf16 values);
// lane l handles chunks l, l + 32, ... in batches of four, whose source words
// are loaded before anything else (their addresses need no lookup), so the
// token's request, position and block-table entry are looked up while the
// data is in flight.  D is a template parameter, so the chunk -> (head,
// dims) split is shifts and masks.
//
// The quantisation (a division-free bracket of the correctly rounded
// quotient, with the division as a fallback) is in quant_e4m3.cuh.
//
// It is launched as a programmatic dependent of the work before it on the
// stream (launch_dependent), so it waits for that work before any access.
#include <cfloat>

#include "check_body.cuh"
#include "kvq_internal.h"
#include "quant_e4m3.cuh"

namespace kvq {

struct AppendArgs {
  void *k_pool, *v_pool;
  const uint16_t *k_new, *v_new;
  const int32_t *req_idx, *pos, *block_table;
  uint32_t *err_word;
  int64_t n_tokens;
  int32_t num_pages, P, H, B, MP;
  QuantParams kq, vq;  // the quantiser's parameters for k_scale and v_scale
};

// The append of tokens warp, warp + nwarps, ... where warp counts the warps
// of CTAs cta, cta + nctas, ... (256 threads a CTA).
template <bool kFp8, int D>
__device__ __forceinline__ void append_tokens(const AppendArgs &a, int64_t cta, int64_t nctas) {
  constexpr int kElems = kFp8 ? 16 : 8;    // elements per 16-byte output chunk
  constexpr int kCpr = D / kElems;         // chunks per (token, head) row: a power of 2
  constexpr int kSrcWords = kFp8 ? 2 : 1;  // 16-byte source words per chunk
  constexpr int kPer = kFp8 ? 2 : 4;       // chunks per lane per batch
  const int64_t cap = static_cast<int64_t>(a.MP) * a.P;
  const int lane = threadIdx.x & 31;
  const int per_tensor = a.H * kCpr;  // chunks of one token's K (or V)
  const int total = 2 * per_tensor;
  const int64_t nwarps = (nctas * blockDim.x) >> 5;
  const int64_t head_stride = static_cast<int64_t>(a.P) * D;

  for (int64_t t = (cta * blockDim.x + threadIdx.x) >> 5; t < a.n_tokens; t += nwarps) {
    const uint4 *ksrc = reinterpret_cast<const uint4 *>(a.k_new + t * a.H * static_cast<int64_t>(D));
    const uint4 *vsrc = reinterpret_cast<const uint4 *>(a.v_new + t * a.H * static_cast<int64_t>(D));
    int req = 0, p = 0, page = 0, slot = 0;
    bool ok = false;
    for (int base = 0; base < total; base += 32 * kPer) {
      // the batch's source words first (their addresses need no lookup) ...
      uint4 s[kPer][kSrcWords];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int j = base + lane + 32 * k;
        if (j < total) {
          const uint4 *src = j < per_tensor ? ksrc + j * kSrcWords
                                            : vsrc + (j - per_tensor) * kSrcWords;
#pragma unroll
          for (int w = 0; w < kSrcWords; ++w) s[k][w] = __ldg(src + w);
        }
      }
      // ... then, once per token, where the token goes
      if (base == 0) {
        req = __ldg(a.req_idx + t);
        p = __ldg(a.pos + t);
        if (req < 0 || req >= a.B) {
          if (lane == 0) report(a.err_word, KVQ_ERRBIT_REQ);
        } else if (p < 0 || p >= cap) {
          if (lane == 0) report(a.err_word, KVQ_ERRBIT_POS);
        } else {
          page = __ldg(a.block_table + static_cast<int64_t>(req) * a.MP + p / a.P);
          if (page < 0 || page >= a.num_pages) {
            if (lane == 0) report(a.err_word, KVQ_ERRBIT_PAGE);
          } else {
            slot = p % a.P;
            ok = true;
          }
        }
        if (!ok) break;  // uniform over the warp
      }
      // element offset of (page, head 0, slot, dim 0); heads are P * D apart
      const int64_t dst0 = (static_cast<int64_t>(page) * a.H * a.P + slot) * D;
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int j = base + lane + 32 * k;
        if (j >= total) break;
        const bool is_v = j >= per_tensor;
        const int jj = is_v ? j - per_tensor : j;
        const int64_t dst = dst0 + (jj / kCpr) * head_stride + (jj % kCpr) * kElems;
        if constexpr (kFp8) {
          uint8_t *pool = static_cast<uint8_t *>(is_v ? a.v_pool : a.k_pool);
          *reinterpret_cast<uint4 *>(pool + dst) =
              quantise16(s[k][0], s[k][1], is_v ? a.vq : a.kq);
        } else {
          uint16_t *pool = static_cast<uint16_t *>(is_v ? a.v_pool : a.k_pool);
          *reinterpret_cast<uint4 *>(pool + dst) = s[k][0];
        }
      }
    }
  }
}

template <bool kFp8, int D>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  grid_dependency_wait();  // earlier work on the stream is complete and visible
  allow_dependents();
  append_tokens<kFp8, D>(a, blockIdx.x, gridDim.x);
}

// kvq_append_check: CTAs below n_append append, the rest check tags.  The
// two touch disjoint memory (the append writes pool pages; the check reads
// the tables, the lengths and the tags and writes the mask), so side by side
// they give what the two calls give in order, and the check no longer waits
// for the append on the critical path of a decode step.
template <bool kFp8, int D>
__global__ void __launch_bounds__(256) append_check_kernel(AppendArgs a, CheckArgs c,
                                                           int n_append) {
  grid_dependency_wait();
  allow_dependents();
  if (static_cast<int>(blockIdx.x) < n_append)
    append_tokens<kFp8, D>(a, blockIdx.x, n_append);
  else
    check_requests(c, blockIdx.x - n_append, gridDim.x - n_append);
}

using AppendFn = void (*)(AppendArgs);
using AppendCheckFn = void (*)(AppendArgs, CheckArgs, int);

inline AppendFn pick_append(bool fp8, int D) {
  if (D == 64) return fp8 ? append_kernel<true, 64> : append_kernel<false, 64>;
  if (D == 128) return fp8 ? append_kernel<true, 128> : append_kernel<false, 128>;
  return nullptr;
}

inline AppendCheckFn pick_append_check(bool fp8, int D) {
  if (D == 64) return fp8 ? append_check_kernel<true, 64> : append_check_kernel<false, 64>;
  if (D == 128) return fp8 ? append_check_kernel<true, 128> : append_check_kernel<false, 128>;
  return nullptr;
}

}  // namespace kvq

using namespace kvq;

namespace {

// Checks of kvq_append's arguments and its kernel arguments.
kvq_status append_args(const kvq_cache *cache, const void *k_new, const void *v_new,
                       const int32_t *req_idx, const int32_t *pos, int32_t n_tokens,
                       const int32_t *block_table, int32_t B, int32_t MP, uint32_t *err_word,
                       AppendArgs *a) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_tokens < 0 || B < 0 || MP <= 0) return KVQ_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!k_new || !v_new || !req_idx || !pos || !block_table || B == 0))
    return KVQ_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!aligned16(k_new) || !aligned16(v_new))) return KVQ_ERR_INVALID_ARG;
  if (n_tokens > 0 && static_cast<int64_t>(MP) * cache->page_size > INT32_MAX)
    return KVQ_ERR_INVALID_ARG;
  a->k_pool = cache->k_pool;
  a->v_pool = cache->v_pool;
  a->k_new = static_cast<const uint16_t *>(k_new);
  a->v_new = static_cast<const uint16_t *>(v_new);
  a->req_idx = req_idx;
  a->pos = pos;
  a->block_table = block_table;
  a->err_word = err_word;
  a->n_tokens = n_tokens;
  a->num_pages = cache->num_pages;
  a->P = cache->page_size;
  a->H = cache->num_kv_heads;
  a->B = B;
  a->MP = MP;
  a->kq = quant_params(cache->k_scale);
  a->vq = quant_params(cache->v_scale);
  return KVQ_OK;
}

constexpr int kAppendThreads = 256;

// CTAs for n tokens: a warp per token, at most 16 CTAs per SM.
int append_ctas(int64_t n_tokens, int sms) {
  const int64_t want = (n_tokens + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
  return static_cast<int>(want < 16LL * sms ? want : 16LL * sms);
}

}  // namespace

extern "C" kvq_status kvq_append(const kvq_cache *cache, const void *k_new, const void *v_new,
                                 const int32_t *req_idx, const int32_t *pos, int32_t n_tokens,
                                 const int32_t *block_table, int32_t B, int32_t MP,
                                 uint32_t *err_word, kvq_stream_t stream) {
  AppendArgs a;
  const kvq_status st =
      append_args(cache, k_new, v_new, req_idx, pos, n_tokens, block_table, B, MP, err_word, &a);
  if (st != KVQ_OK) return st;
  if (n_tokens == 0) return KVQ_OK;
  const AppendFn fn = pick_append(cache->kv_dtype == KVQ_KV_E4M3, cache->head_dim);
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const cudaError_t e = launch_dependent(fn, append_ctas(n_tokens, sms), kAppendThreads, 0,
                                         reinterpret_cast<cudaStream_t>(stream), a);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

extern "C" kvq_status kvq_append_check(const kvq_cache *cache, const void *k_new,
                                       const void *v_new, const int32_t *req_idx,
                                       const int32_t *pos, int32_t n_tokens,
                                       const int32_t *block_table, int32_t B, int32_t MP,
                                       const int32_t *seq_lens, const uint32_t *page_tags,
                                       const uint32_t *expected_tags, uint8_t *abort_mask,
                                       uint32_t *err_word, kvq_stream_t stream) {
  AppendArgs a;
  const kvq_status st =
      append_args(cache, k_new, v_new, req_idx, pos, n_tokens, block_table, B, MP, err_word, &a);
  if (st != KVQ_OK) return st;
  if (B > 0 && (!block_table || !seq_lens || !page_tags || !expected_tags || !abort_mask))
    return KVQ_ERR_INVALID_ARG;
  if (n_tokens == 0 && B == 0) return KVQ_OK;
  CheckArgs c{block_table, seq_lens, page_tags, expected_tags, abort_mask, B, MP,
              cache->page_size, cache->num_pages};
  const AppendCheckFn fn = pick_append_check(cache->kv_dtype == KVQ_KV_E4M3, cache->head_dim);
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const int n_append = n_tokens > 0 ? append_ctas(n_tokens, sms) : 0;
  const int n_check = B < 32 * sms ? B : 32 * sms;
  const cudaError_t e = launch_dependent(fn, n_append + n_check, kAppendThreads, 0,
                                         reinterpret_cast<cudaStream_t>(stream), a, c, n_append);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
