// The batched page-tag check's per-request work, shared by check_tags_kernel
// (kvq_check_tags) and append_check_kernel (kvq_append_check).
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "共享 KV 缓存保护": every physical page carries a tag that changes when the
// page is reallocated, the server records which (page, tag) each request
// expects, and the mappings are verified before decode reads the cache.
//
// A CTA takes requests cta, cta + nctas, ...: its threads stride over the
// request's logical pages, compare the recorded tag with the page's current
// tag, and a block-wide OR gives the request's abort flag.  Integer work
// only: the result is exact by construction.
#pragma once

#include "kvq_device.cuh"

namespace kvq {

struct CheckArgs {
  const int32_t *block_table, *seq_lens;
  const uint32_t *page_tags, *expected_tags;
  uint8_t *abort_mask;
  int32_t B, MP, P, num_pages;
};

// Every thread of the CTA calls it (a block-wide OR per request).
__device__ __forceinline__ void check_requests(const CheckArgs &a, int cta, int nctas) {
  const int64_t cap = static_cast<int64_t>(a.MP) * a.P;
  for (int b = cta; b < a.B; b += nctas) {
    const int L = a.seq_lens[b];
    int bad = (L < 0 || L > cap) ? 1 : 0;
    if (!bad) {
      const int n_pages = (L + a.P - 1) / a.P;
      const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.MP;
      const uint32_t *exp = a.expected_tags + static_cast<int64_t>(b) * a.MP;
#pragma unroll 4
      for (int i = threadIdx.x; i < n_pages; i += blockDim.x) {
        const int page = __ldg(bt + i);
        const uint32_t want = __ldg(exp + i);
        if (page < 0 || page >= a.num_pages) {
          bad = 1;
        } else if (__ldg(a.page_tags + page) != want) {
          bad = 1;
        }
      }
    }
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) a.abort_mask[b] = static_cast<uint8_t>(bad ? 1 : 0);
  }
}

}  // namespace kvq
