/*
 * kvq -- FP8 (e4m3) paged KV cache: quantise-and-append, the prefill -> decode
 * handoff of BF16 pages, batched page-tag integrity check, the page
 * allocator that sets the tags, single-query
 * paged decode attention, and the weight-only INT4 / FP8 decode matrix
 * product, for NVIDIA GB300 (sm_103a).  Plain C ABI: pointers,
 * sizes, a CUDA stream.  The library allocates no memory.
 *
 * Sources (web pages, cited by title and section):
 *   [KVQ]   "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全" (a translation
 *           of "Smaller, faster, safer: running Kimi and GLM at scale"), section
 *           "KV 缓存量化" (KV-cache quantisation): the decode cache holds K and V
 *           as 8-bit e4m3 instead of BF16 (half the bytes, twice the tokens);
 *           the FP8 attention kernel converts on read; prefill keeps BF16.  Its
 *           decode table compares a BF16-KV and an FP8-KV attention kernel.
 *   [GUARD] same page, section "共享 KV 缓存保护" (protecting the shared KV cache):
 *           each physical page has a tag that changes on every reallocation;
 *           the server records the page and tag each request expects; a
 *           separate batched check (not fused into attention) compares them
 *           before decode reads the cache, and a mismatching request is
 *           aborted instead of being served another request's data; the check
 *           is enabled per deployment, the default tracker does nothing.
 *   The e4m3 bit format is the OCP 8-bit floating point E4M3 format (bias 7,
 *   no infinities, S.1111.111 = NaN, largest finite 448).
 *
 * Conventions for every entry point
 *   - Pointers named *_host are host memory; every other pointer is DEVICE
 *     memory owned by the caller.  The library never allocates, frees or
 *     synchronises; all work is enqueued on `stream` (0 = legacy default).
 *   - Host-checkable argument errors return a status != KVQ_OK before any
 *     launch and enqueue nothing.  A failed launch returns KVQ_ERR_CUDA.
 *   - Data-dependent faults found on the device never trap: the kernel skips
 *     the access and ORs a KVQ_ERRBIT_* value into *err_word (device uint32,
 *     nullable; the caller zeroes it when it wants a fresh reading).
 *   - Layouts are row-major:
 *       pools        [num_pages][num_kv_heads][page_size][head_dim] elements
 *                    (uint8 e4m3 codes, or bf16);
 *       block_table  int32 [B][MP]: logical page i of request b lives in
 *                    physical page block_table[b*MP + i];
 *       q            bf16 [B][Hq][head_dim]; out fp32 [B][Hq][head_dim];
 *       k_new/v_new  bf16 [n_tokens][num_kv_heads][head_dim].
 *   - Query head h reads KV head h / (Hq / num_kv_heads).
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvq_stream_t; /* == cudaStream_t */

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer, bad scale */
    KVQ_ERR_WORKSPACE = 2,   /* workspace too small or misaligned */
    KVQ_ERR_CUDA = 3,        /* a kernel launch or device query failed */
    KVQ_ERR_UNSUPPORTED = 4  /* shape outside the compiled set (see each call) */
} kvq_status;

typedef enum { KVQ_KV_E4M3 = 0, KVQ_KV_BF16 = 1 } kvq_kv_dtype;
typedef enum { KVQ_W_INT4 = 0, KVQ_W_E4M3 = 1 } kvq_w_dtype;

/* Bits ORed into *err_word by the kernels. */
#define KVQ_ERRBIT_PAGE    (1u << 0) /* a block-table entry the call needs is outside [0, num_pages) */
#define KVQ_ERRBIT_SEQLEN  (1u << 1) /* seq_lens[b] < 0 or > MP * page_size */
#define KVQ_ERRBIT_POS     (1u << 2) /* append position outside [0, MP * page_size) */
#define KVQ_ERRBIT_REQ     (1u << 3) /* request index outside [0, B) (append, pages update) */
#define KVQ_ERRBIT_TIMEOUT (1u << 4) /* a bounded wait inside a kernel gave up (no result) */
#define KVQ_ERRBIT_EXHAUSTED (1u << 5) /* kvq_pages_update: an acquisition found too few free pages */

/* The paged cache ([KVQ]): two pools of identical shape, one for K, one for V.
 * Supported: page_size in {16, 32, 64}; head_dim in {64, 128};
 * k_scale/v_scale finite and > 0 (per-tensor; e4m3 only, ignored for bf16).
 * Pools must be 16-byte aligned. */
typedef struct {
    void *k_pool;
    void *v_pool;
    int32_t kv_dtype; /* kvq_kv_dtype */
    int32_t num_pages;
    int32_t page_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    float k_scale;
    float v_scale;
} kvq_cache;

/* Quantise-and-append ([KVQ]: the decode cache is stored as e4m3).
 * For each token t < n_tokens, request r = req_idx[t], position p = pos[t]:
 * page = block_table[r*MP + p/page_size], slot = p % page_size, and for every
 * kv head h and dim d
 *     k_pool[page][h][slot][d] = e4m3_rne_satfinite( float(k_new[t][h][d]) / k_scale )
 * (one IEEE fp32 division, round to nearest even, |x| > 448 and inf -> +-448,
 * NaN -> a NaN code), the same for V with v_scale.  For a bf16 cache the
 * bf16 values are copied unchanged.  Nothing else in the pools is written.
 * Invalid r, p or page: that token writes nothing and raises KVQ_ERRBIT_REQ,
 * _POS or _PAGE.  Two tokens must not target the same slot (unspecified).
 * n_tokens may be any size (a whole prompt in one call); n_tokens == 0 is a
 * no-op.  k_new/v_new 16-byte aligned. */
KVQ_API kvq_status kvq_append(const kvq_cache *cache, const void *k_new, const void *v_new,
                      const int32_t *req_idx, const int32_t *pos, int32_t n_tokens,
                      const int32_t *block_table, int32_t B, int32_t MP,
                      uint32_t *err_word, kvq_stream_t stream);

/* kvq_append and kvq_check_tags of one decode step in one launch: the same
 * effects, error bits and results as
 *     kvq_append(cache, k_new, v_new, req_idx, pos, n_tokens, block_table, B, MP,
 *                err_word, stream);
 *     kvq_check_tags(block_table, B, MP, seq_lens, cache->page_size, page_tags,
 *                    cache->num_pages, expected_tags, abort_mask, stream);
 * with every argument as documented there ([GUARD]: the check is a separate
 * batched pass before attention reads the cache; it stays one, running
 * beside the append instead of after it).  The append writes only pool
 * pages and the check only abort_mask, and neither reads what the other
 * writes, so the order of the two calls does not change either result; the
 * one launch takes the check off a decode step's critical path.  Argument
 * errors are those of the two calls (KVQ_ERR_INVALID_ARG for a null check
 * array when B > 0); n_tokens == 0 and B == 0 is a no-op. */
KVQ_API kvq_status kvq_append_check(const kvq_cache *cache, const void *k_new,
                                    const void *v_new, const int32_t *req_idx,
                                    const int32_t *pos, int32_t n_tokens,
                                    const int32_t *block_table, int32_t B, int32_t MP,
                                    const int32_t *seq_lens, const uint32_t *page_tags,
                                    const uint32_t *expected_tags, uint8_t *abort_mask,
                                    uint32_t *err_word, kvq_stream_t stream);

/* Prefill -> decode handoff of whole prompts ([KVQ]: the prefill side keeps
 * its KV cache in BF16, the decode side stores it as e4m3, so a prompt is
 * converted once when decode takes it over).  `src` is a paged BF16 cache
 * (kv_dtype KVQ_KV_BF16; its scales are ignored), `dst` the decode cache
 * (e4m3, or bf16 for a plain paged copy) with the same num_kv_heads and
 * head_dim; the two page sizes may differ.  For every request b < B and
 * logical position p in [first[b], first[b] + count[b]) (first may be NULL:
 * all zeros), the K/V of token p -- src page src_block_table[b*src_MP +
 * p/src->page_size], slot p % src->page_size -- are stored at dst page
 * dst_block_table[b*dst_MP + p/dst->page_size], slot p % dst->page_size,
 * exactly as kvq_append stores a token (same code for the same value, with
 * dst's k_scale / v_scale).  Nothing else in dst is written; src is only
 * read and must not overlap dst.
 * A request whose range is negative or reaches past either table's
 * capacity (MP * page_size) writes nothing and raises KVQ_ERRBIT_POS; a
 * token whose src or dst page is outside its pool writes nothing and raises
 * KVQ_ERRBIT_PAGE.  first and count are int32 [B] device arrays; pools
 * 16-byte aligned; num_kv_heads in {1, 2, 4, 8} (else KVQ_ERR_UNSUPPORTED). */
KVQ_API kvq_status kvq_handoff_pages(const kvq_cache *src, const int32_t *src_block_table,
                                     int32_t src_MP, const kvq_cache *dst,
                                     const int32_t *dst_block_table, int32_t dst_MP,
                                     const int32_t *first, const int32_t *count, int32_t B,
                                     uint32_t *err_word, kvq_stream_t stream);

/* Batched page-tag integrity check ([GUARD]), a separate pass before decode.
 * abort_mask[b] = 1 if, for some logical page i < ceil(seq_lens[b]/page_size),
 * block_table[b*MP+i] is outside [0, num_pages) or
 * page_tags[block_table[b*MP+i]] != expected_tags[b*MP+i]; also 1 when
 * seq_lens[b] is outside [0, MP*page_size]; else 0.  Block-table entries past
 * the request's length are not read.  page_tags uint32 [num_pages],
 * expected_tags uint32 [B][MP], abort_mask uint8 [B]. */
KVQ_API kvq_status kvq_check_tags(const int32_t *block_table, int32_t B, int32_t MP,
                          const int32_t *seq_lens, int32_t page_size,
                          const uint32_t *page_tags, int32_t num_pages,
                          const uint32_t *expected_tags, uint8_t *abort_mask,
                          kvq_stream_t stream);

/* Batched page release and acquisition with per-page tags: the allocator
 * side of the check ([GUARD]: a page's tag changes whenever the page is
 * reallocated, and the server records the (page, tag) pairs each request was
 * given).  The state is caller-owned device memory:
 *   free_stack   int32 [num_pages]: free page ids in free_stack[0 .. *free_count)
 *                (the top is the last one); free_count int32 [1];
 *   page_tags    uint32 [num_pages];
 *   block_table  int32 [B][MP] and expected_tags uint32 [B][MP] (the same
 *                tables kvq_check_tags reads).
 * One call is a batch of releases, then a batch of acquisitions:
 *  - Release: for j = 0 .. n_rel-1 in order, request rel_req[j] returns its
 *    logical pages 0 .. rel_npages[j]-1 in order: each page id is pushed on
 *    the stack and its block-table entry becomes -1; tags are unchanged.  All
 *    or nothing: if any request index is outside [0, B) (KVQ_ERRBIT_REQ), any
 *    count outside [0, MP] (_POS), any returned entry is not a page id
 *    (_PAGE), or the pushes would overfill the stack (_PAGE), nothing is
 *    released.
 *  - Acquire: for i = 0 .. n_acq-1 in order, request acq_req[i] asks for
 *    logical pages acq_first[i] .. acq_first[i] + acq_npages[i] - 1.  An
 *    invalid request index (_REQ) or range (_POS) gets nothing.  Valid
 *    requests are served in order: each pops its pages off the top of the
 *    stack in logical order; the popped page's tag is incremented (mod 2^32)
 *    and the request's block-table and expected-tag entries get the page and
 *    its new tag.  The first valid request that finds too few free pages,
 *    and every valid request after it, get nothing (KVQ_ERRBIT_EXHAUSTED).
 *    acq_ok[i] (uint8 [n_acq]) is 1 if request i was served, else 0.  A
 *    popped entry that is not a page id is consumed unmapped (_PAGE).
 * A *free_count outside [0, num_pages] changes nothing (_PAGE).
 * Preconditions (unchecked; the result is unspecified otherwise): a request
 * appears at most once in each list, releases exactly entries it holds, and
 * acquires only entries it does not hold.  Freshly set up state: free_stack
 * any permutation of the page ids, *free_count = num_pages, tags any values.
 * The lists may be empty (their pointers may then be NULL). */
KVQ_API kvq_status kvq_pages_update(int32_t *free_stack, int32_t *free_count, uint32_t *page_tags,
                                    int32_t num_pages, int32_t *block_table,
                                    uint32_t *expected_tags, int32_t B, int32_t MP,
                                    const int32_t *rel_req, const int32_t *rel_npages,
                                    int32_t n_rel, const int32_t *acq_req,
                                    const int32_t *acq_first, const int32_t *acq_npages,
                                    int32_t n_acq, uint8_t *acq_ok, uint32_t *err_word,
                                    kvq_stream_t stream);

/* Weight-only quantised matrix product for decode ([KVQ] section "模型权重压缩":
 * the decode pool keeps the weights as 4-bit integers instead of FP8; every
 * token reads all of them, so decode is bandwidth-bound; INT4 values are
 * widened before they are multiplied):
 *     y[m][n] = sum_k x[m][k] * W[n][k]
 * x bf16 [M][K] (row-major), y fp32 [M][N] (row-major, overwritten), and
 *   KVQ_W_INT4: w uint8 [N][K/2], two signed 4-bit values a byte (two's
 *     complement; k even in the low nibble); scales bf16 [N][K/128]:
 *     W[n][k] = int4(n, k) * scales[n][k/128];
 *   KVQ_W_E4M3: w uint8 e4m3 codes [N][K]; scales fp32 [N]:
 *     W[n][k] = e4m3(w[n][k]) * scales[n].
 * Products are exact and sums fp32.  Any bf16 x is accepted: each token's
 * values are scaled by a power of two for the products (exact for every
 * value down to 2^-32 of the token's largest finite |x| in a k range,
 * smaller ones are rounded to 2^-25 of it); NaN and inf propagate.
 * For one or two tokens (when a CTA's share of x fits its shared memory), and
 * for three to eight tokens where that share needs no k split past one wave
 * of CTAs, the weights stream through a shared-memory ring fed by the TMA
 * engine and a k split runs as a thread-block cluster whose partial sums are
 * added in a fixed order: every run gives the same bits.  Otherwise split-K partial
 * sums are added with fp32 atomics: their order varies from run to run, and
 * atomics flush subnormals, so a result below 2^-126 in magnitude can be off
 * by up to (2 K/128 + 1) * 2^-126.
 * w and scales are taken as constant model weights: the call starts reading
 * them before the work ahead of it on the stream has finished (programmatic
 * dependent launch), so they must not be written by the kernel launched just
 * before it on the same stream if that kernel lets its dependents start
 * early, as every kvq kernel does; x is read only once that work is done.
 * err_word (device uint32, nullable): KVQ_ERRBIT_TIMEOUT when a bounded wait
 * inside the kernel gave up (y is then undefined).
 * Supported: 1 <= M <= 64, K a multiple of 128.  w and x 16-byte aligned,
 * scales 4-byte aligned. */
KVQ_API kvq_status kvq_wq_gemm(int32_t w_dtype, const void *w, const void *scales, const void *x,
                               float *y, int32_t M, int32_t N, int32_t K, uint32_t *err_word,
                               kvq_stream_t stream);

/* Bytes of device workspace kvq_decode_attn needs for these sizes (split
 * partials and the per-call work plan).  Depends on B, Hq, num_kv_heads and
 * head_dim only, not on the sequence lengths. */
KVQ_API size_t kvq_decode_attn_workspace_size(int32_t B, int32_t Hq, int32_t num_kv_heads,
                                      int32_t head_dim);

/* Single-query paged decode attention over the cache ([KVQ]: e4m3 K/V are
 * converted on read; a bf16 cache is the comparison kernel).
 * For every request b and query head h, with L = seq_lens[b] tokens and
 * kv head g = h / (Hq/num_kv_heads), token j's K/V at
 * page block_table[b*MP + j/page_size], slot j % page_size:
 *     s_j = sm_scale * sum_d q[b][h][d] * k_scale * e4m3(k_code_j[d])
 *     out[b][h][:] = sum_j softmax(s)_j * v_scale * e4m3(v_code_j[:])
 * accumulated in fp32 (split over the sequence, merged by log-sum-exp).
 * abort_mask (uint8 [B], nullable; NULL = no check was run): a request with
 * abort_mask[b] != 0 reads none of its pages and gets out[b] = 0 ([GUARD]:
 * an aborted request is never served cache data).  L == 0 gives a zero row.
 * A page id outside the pool or an invalid L raises KVQ_ERRBIT_PAGE /
 * _SEQLEN and zeroes that request's rows without reading the bad page.
 * Supported: Hq/num_kv_heads in {1, 2, 4, 8}, head_dim in {64, 128},
 * page_size in {16, 32, 64}.  q 16-byte aligned; workspace 256-byte aligned
 * with at least kvq_decode_attn_workspace_size() bytes; the workspace must not
 * be shared by calls that can run at the same time. */
KVQ_API kvq_status kvq_decode_attn(const kvq_cache *cache, const void *q, int32_t B, int32_t Hq,
                           const int32_t *block_table, int32_t MP, const int32_t *seq_lens,
                           const uint8_t *abort_mask, float sm_scale, float *out,
                           void *workspace, size_t workspace_bytes, uint32_t *err_word,
                           kvq_stream_t stream);

/* kvq_decode_attn without a caller workspace.  The pages have no counterpart
 * to this call: it exists for callers that cannot allocate device memory (a
 * runtime that reserves all memory up front and serves it only from its own
 * pool, a plugin host that forbids allocation in its execute callback, a
 * latency-bound loop that cannot afford cudaMalloc).  It computes exactly what
 * kvq_decode_attn computes, with the workspace taken from a static device
 * array of KVQ_STATIC_SCRATCH_BYTES owned by the library (held on every GPU
 * that loads it, until exit).  It allocates nothing.
 * - Shapes whose kvq_decode_attn_workspace_size() exceeds
 *   KVQ_STATIC_SCRATCH_BYTES return KVQ_ERR_WORKSPACE before any launch.
 * - Every call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress), so the call stays valid after a device reset; the
 *   first call on a device may load the library's device code there, so make
 *   that first call before any stream capture.
 * - All calls share the one array: calls whose kernels can overlap on the GPU
 *   (different streams or host threads without ordering) race and must not be
 *   issued.  Stale contents from an earlier call are harmless. */
#define KVQ_STATIC_SCRATCH_BYTES (64u << 20)
KVQ_API kvq_status kvq_decode_attn_static(const kvq_cache *cache, const void *q, int32_t B,
                                          int32_t Hq, const int32_t *block_table, int32_t MP,
                                          const int32_t *seq_lens, const uint8_t *abort_mask,
                                          float sm_scale, float *out, uint32_t *err_word,
                                          kvq_stream_t stream);

/* Self-test of a kernel failure path (no fault, no hang): one CTA starts a
 * real bulk copy of 64 bytes from src (device, 16-byte aligned) into shared
 * memory, then waits on an mbarrier that nothing ever arrives at, with the
 * bounded wait of the split attention kernels (which = 0) or of the weight
 * ring of kvq_wq_gemm (which = 1).  The wait gives up after its bound (about
 * 2^31 SM cycles, ~1 s), ORs KVQ_ERRBIT_TIMEOUT into *err_word, then lets the
 * copy it started land before the CTA exits (the drain every such kernel runs
 * on this path) and stores the copy's first word in *landed (0 if the wait
 * or the drain did not behave).  The context stays usable afterwards.
 * err_word and landed: device uint32. */
KVQ_API kvq_status kvq_selftest_wait(int32_t which, const void *src, uint32_t *err_word,
                                     uint32_t *landed, kvq_stream_t stream);

/* Human-readable name of a status. */
KVQ_API const char *kvq_status_string(kvq_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
