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
// One CTA per request (grid-strided; check_body.cuh).  Launched as a
// programmatic dependent of the work before it on the stream, so in a decode
// step its launch overlaps the append kernel; kvq_append_check (append.cu)
// runs the same work beside the append in one launch.
#include "check_body.cuh"
#include "kvq_internal.h"

namespace kvq {

__global__ void __launch_bounds__(256) check_tags_kernel(CheckArgs a) {
  grid_dependency_wait();  // earlier work on the stream is complete and visible
  allow_dependents();
  check_requests(a, blockIdx.x, gridDim.x);
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
