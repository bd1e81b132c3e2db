// kvq_check_tags: the batched page-tag integrity check.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "共享 KV 缓存保护": every physical page carries a tag that changes when the
// page is reallocated, the server records which (page, tag) each request
// expects, the mappings are verified before decode reads the cache, and a
// request with a mismatch is aborted.  The page states that the check runs as
// a separate batched pass and is not fused into the attention kernel (fusing
// it would race between thread groups).
//
// One CTA per request (grid-strided): its threads stride over the request's
// logical pages, compare the recorded tag with the page's current tag, and a
// block-wide OR gives the request's abort flag.  Integer work only: the
// result is exact by construction.  Launched as a programmatic dependent of
// the work before it on the stream, so in a decode step its launch overlaps
// the append kernel.
#include "kvq_internal.h"

namespace kvq {

struct CheckArgs {
  const int32_t *block_table, *seq_lens;
  const uint32_t *page_tags, *expected_tags;
  uint8_t *abort_mask;
  int32_t B, MP, P, num_pages;
};

__global__ void __launch_bounds__(256) check_tags_kernel(CheckArgs a) {
  const int64_t cap = static_cast<int64_t>(a.MP) * a.P;
  grid_dependency_wait();  // earlier work on the stream is complete and visible
  allow_dependents();
  for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
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

using namespace kvq;

extern "C" kvq_status kvq_check_tags(const int32_t *block_table, int32_t B, int32_t MP,
                                     const int32_t *seq_lens, int32_t page_size,
                                     const uint32_t *page_tags, int32_t num_pages,
                                     const uint32_t *expected_tags, uint8_t *abort_mask,
                                     kvq_stream_t stream) {
  if (B < 0 || MP <= 0 || page_size <= 0 || num_pages <= 0) return KVQ_ERR_INVALID_ARG;
  if (B == 0) return KVQ_OK;
  if (!block_table || !seq_lens || !page_tags || !expected_tags || !abort_mask)
    return KVQ_ERR_INVALID_ARG;
  CheckArgs a{block_table, seq_lens, page_tags, expected_tags, abort_mask, B, MP, page_size,
              num_pages};
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const int blocks = B < 32 * sms ? B : 32 * sms;
  const cudaError_t e = launch_dependent(check_tags_kernel, blocks, 256, 0,
                                         reinterpret_cast<cudaStream_t>(stream), a);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
