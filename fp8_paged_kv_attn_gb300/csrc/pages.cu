// kvq_pages_update: batched page release and acquisition with per-page tags.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "共享 KV 缓存保护": every physical page carries a tag that changes whenever
// the page is reallocated, and the server records the (page, tag) pairs each
// request was given, so that the batched check can refuse a request whose
// mapping went stale.  This is that allocator, on the GPU: free pages are a
// last-in-first-out stack, a batch releases before it acquires, and the tag
// of a page is incremented when the page is handed out.
//
// One CTA of 1024 threads runs the batch: its phases depend on one another
// (the releases decide which pages the acquisitions pop) and the work is
// small next to a decode step.  Lists are taken in rounds of 1024 entries
// with a carried prefix.  In a round, the entries' page counts are scanned
// (int64) in shared memory and the round's pages -- one entry may carry a
// whole prompt's -- are spread over the threads by a binary search of the
// scan.
//
// Acquisitions: entry i is served iff it is valid and
// (sum of the valid demands before it) + its demand <= free pages after the
// releases.  That is the sequential rule "serve in order until the first
// valid request that does not fit": once one fails, every later prefix is
// larger still.  Entry i's k-th page is stack[count - 1 - (prefix_i + k)].
#include "kvq_internal.h"

namespace kvq {

struct PagesArgs {
  int32_t *free_stack, *free_count;
  uint32_t *page_tags;
  int32_t *block_table;
  uint32_t *expected_tags;
  const int32_t *rel_req, *rel_npages, *acq_req, *acq_first, *acq_npages;
  uint8_t *acq_ok;
  uint32_t *err_word;
  int32_t num_pages, B, MP, n_rel, n_acq;
};

constexpr int kPagesThreads = 1024;

struct PagesSmem {
  long long pre[kPagesThreads];  // exclusive prefix of the round's page counts
  long long warp[33];            // scan scratch; [32] = round total
  int req[kPagesThreads];
  int first[kPagesThreads];
  uint8_t ok[kPagesThreads];
  unsigned int bits;
};

// Exclusive scan of v over the CTA; *total = the sum.
__device__ __forceinline__ long long cta_scan(long long v, PagesSmem &sm, long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) sm.warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const long long w = sm.warp[lane];  // kPagesThreads / 32 == 32 warps
    long long wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    sm.warp[lane] = wi - w;
    if (lane == 31) sm.warp[32] = wi;
  }
  __syncthreads();
  const long long r = sm.warp[warp] + incl - v;
  *total = sm.warp[32];
  __syncthreads();  // the scratch may be reused
  return r;
}

// The entry of a round (m entries) whose page range holds item e.
__device__ __forceinline__ int owner(const PagesSmem &sm, int m, long long e) {
  int lo = 0, hi = m - 1;
  while (lo < hi) {  // last entry with pre <= e
    const int mid = (lo + hi + 1) >> 1;
    if (sm.pre[mid] <= e)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kPagesThreads, 1) pages_kernel(PagesArgs a) {
  __shared__ PagesSmem sm;
  const int tid = threadIdx.x;
  grid_dependency_wait();  // earlier work on the stream is complete and visible
  allow_dependents();
  if (tid == 0) sm.bits = 0;
  const int count0 = *a.free_count;
  if (count0 < 0 || count0 > a.num_pages) {
    for (int i = tid; i < a.n_acq; i += kPagesThreads) a.acq_ok[i] = 0;
    if (tid == 0) report(a.err_word, KVQ_ERRBIT_PAGE);
    return;
  }
  __syncthreads();

  // ---- release, pass 1: validate the whole batch
  unsigned int rel_bits = 0;
  long long rel_total = 0;
  for (int base = 0; base < a.n_rel; base += kPagesThreads) {
    const int j = base + tid, m = min(kPagesThreads, a.n_rel - base);
    int b = 0;
    long long n = 0;
    if (j < a.n_rel) {
      b = a.rel_req[j];
      const int nn = a.rel_npages[j];
      if (b < 0 || b >= a.B)
        rel_bits |= KVQ_ERRBIT_REQ;
      else if (nn < 0 || nn > a.MP)
        rel_bits |= KVQ_ERRBIT_POS;
      else
        n = nn;
    }
    long long total;
    const long long pre = cta_scan(n, sm, &total);
    sm.pre[tid] = pre;
    sm.req[tid] = b;
    __syncthreads();
    for (long long e = tid; e < total; e += kPagesThreads) {
      const int o = owner(sm, m, e);
      const int page = a.block_table[static_cast<int64_t>(sm.req[o]) * a.MP + (e - sm.pre[o])];
      if (page < 0 || page >= a.num_pages) rel_bits |= KVQ_ERRBIT_PAGE;
    }
    rel_total += total;
    __syncthreads();
  }
  if (rel_bits) atomicOr(&sm.bits, rel_bits);
  __syncthreads();
  const bool release = sm.bits == 0 && count0 + rel_total <= a.num_pages;
  if (sm.bits == 0 && !release && tid == 0) atomicOr(&sm.bits, KVQ_ERRBIT_PAGE);

  // ---- release, pass 2: push in list order, unmap
  int count = count0;
  if (release) {
    long long carry = 0;
    for (int base = 0; base < a.n_rel; base += kPagesThreads) {
      const int j = base + tid, m = min(kPagesThreads, a.n_rel - base);
      int b = 0;
      long long n = 0;
      if (j < a.n_rel) {
        b = a.rel_req[j];
        n = a.rel_npages[j];
      }
      long long total;
      const long long pre = cta_scan(n, sm, &total);
      sm.pre[tid] = pre;
      sm.req[tid] = b;
      __syncthreads();
      for (long long e = tid; e < total; e += kPagesThreads) {
        const int o = owner(sm, m, e);
        int32_t *entry = a.block_table + static_cast<int64_t>(sm.req[o]) * a.MP + (e - sm.pre[o]);
        a.free_stack[count0 + carry + e] = *entry;
        *entry = -1;
      }
      carry += total;
      __syncthreads();
    }
    count = count0 + static_cast<int>(rel_total);
  }
  __syncthreads();  // the pushes are visible to every thread of the CTA

  // ---- acquire: served in order until the first valid request that does not fit
  unsigned int acq_bits = 0;
  long long carry = 0, served = 0;
  for (int base = 0; base < a.n_acq; base += kPagesThreads) {
    const int i = base + tid, m = min(kPagesThreads, a.n_acq - base);
    int b = 0, first = 0;
    bool valid = false;
    long long n = 0;
    if (i < a.n_acq) {
      b = a.acq_req[i];
      first = a.acq_first[i];
      const int nn = a.acq_npages[i];
      if (b < 0 || b >= a.B)
        acq_bits |= KVQ_ERRBIT_REQ;
      else if (first < 0 || nn < 0 || static_cast<long long>(first) + nn > a.MP)
        acq_bits |= KVQ_ERRBIT_POS;
      else {
        valid = true;
        n = nn;
      }
    }
    long long total;
    const long long pre = cta_scan(n, sm, &total);
    const bool ok = valid && carry + pre + n <= count;
    if (valid && !ok) acq_bits |= KVQ_ERRBIT_EXHAUSTED;
    if (i < a.n_acq) a.acq_ok[i] = ok ? 1 : 0;
    sm.pre[tid] = pre;
    sm.req[tid] = b;
    sm.first[tid] = first;
    sm.ok[tid] = ok ? 1 : 0;
    long long round_served;
    cta_scan(ok ? n : 0, sm, &round_served);  // also orders the writes above
    for (long long e = tid; e < total; e += kPagesThreads) {
      const int o = owner(sm, m, e);
      if (!sm.ok[o]) continue;
      const int page = a.free_stack[count - 1 - (carry + e)];
      if (page < 0 || page >= a.num_pages) {
        acq_bits |= KVQ_ERRBIT_PAGE;
        continue;
      }
      const uint32_t tag = a.page_tags[page] + 1u;
      a.page_tags[page] = tag;
      const int64_t at = static_cast<int64_t>(sm.req[o]) * a.MP + sm.first[o] + (e - sm.pre[o]);
      a.block_table[at] = page;
      a.expected_tags[at] = tag;
    }
    carry += total;
    served += round_served;
    __syncthreads();
  }
  if (acq_bits) atomicOr(&sm.bits, acq_bits);
  __syncthreads();
  if (tid == 0) {
    *a.free_count = count - static_cast<int>(served);
    if (sm.bits) report(a.err_word, sm.bits);
  }
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_pages_update(int32_t *free_stack, int32_t *free_count,
                                       uint32_t *page_tags, int32_t num_pages,
                                       int32_t *block_table, uint32_t *expected_tags, int32_t B,
                                       int32_t MP, const int32_t *rel_req,
                                       const int32_t *rel_npages, int32_t n_rel,
                                       const int32_t *acq_req, const int32_t *acq_first,
                                       const int32_t *acq_npages, int32_t n_acq, uint8_t *acq_ok,
                                       uint32_t *err_word, kvq_stream_t stream) {
  if (num_pages <= 0 || B <= 0 || MP <= 0 || n_rel < 0 || n_acq < 0) return KVQ_ERR_INVALID_ARG;
  if (!free_stack || !free_count || !page_tags || !block_table || !expected_tags)
    return KVQ_ERR_INVALID_ARG;
  if (n_rel > 0 && (!rel_req || !rel_npages)) return KVQ_ERR_INVALID_ARG;
  if (n_acq > 0 && (!acq_req || !acq_first || !acq_npages || !acq_ok)) return KVQ_ERR_INVALID_ARG;
  if (n_rel == 0 && n_acq == 0) return KVQ_OK;
  PagesArgs args{free_stack, free_count, page_tags,  block_table, expected_tags,
                 rel_req,    rel_npages, acq_req,    acq_first,   acq_npages,
                 acq_ok,     err_word,   num_pages,  B,           MP,
                 n_rel,      n_acq};
  const cudaError_t e = launch_dependent(pages_kernel, 1, kPagesThreads, 0,
                                         reinterpret_cast<cudaStream_t>(stream), args);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
