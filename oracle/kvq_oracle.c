/*
 * CPU oracle for the FP8 paged-KV decode path.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, obviously-correct statement of what the GPU library
 * computes.  It shares no code, header, table or constant with the CUDA path,
 * and the product never links, loads or calls it: only the test suite, the
 * smoke check and the benchmark's CPU-baseline / reference arm do.
 *
 * Sources (web pages; cited by title and section):
 *   [KVQ]   "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全" (reed-read
 *           translation of "Smaller, faster, safer: running Kimi and GLM at
 *           scale"), section "KV 缓存量化" (KV-cache quantisation): keys and
 *           values are kept as 8-bit e4m3 instead of BF16, which halves the
 *           cache; the FP8 attention kernel converts the cache on read.
 *   [GUARD] same page, section "共享 KV 缓存保护" (protecting the shared KV
 *           cache): every physical page carries a tag that changes whenever the
 *           page is reallocated; the server records the (page, tag) pairs each
 *           request expects, compares them before the decode step reads the
 *           cache, and aborts a request on any mismatch.
 *   [OFP8]  OCP 8-bit floating point specification, format E4M3 (the pages only
 *           name "e4m3"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 *           bits, subnormals, no infinities, S.1111.111 is NaN, largest finite
 *           magnitude 448 (code 0x7E).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - quantisation is one IEEE fp32 division x/scale followed by
 *     round-to-nearest-even into e4m3 with saturation to +-448 (inf -> +-448,
 *     NaN -> 0x7F);
 *   - per-tensor scales, pool layout [page][kv_head][slot][dim];
 *   - query head h reads kv head h / (Hq/Hkv); logits scaled by sm_scale; no
 *     soft-cap, window or bias;
 *   - only logical pages i < ceil(L/P) of a request are read or checked;
 *   - an aborted, empty or invalid request gives an all-zero output row;
 *   - the page allocator (the step before the check): a page's tag is
 *     incremented when the page is handed to a new owner, free pages form a
 *     last-in-first-out stack, a batch releases before it acquires, and
 *     acquisitions are served in order until the first that does not fit.
 *
 * Every floating-point result of the attention is computed in fp64 and only
 * the final output is rounded to fp32.  Build with -ffp-contract=off and
 * without -ffast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Error bits reported by the oracle; the library documents the same meanings. */
#define ORACLE_ERR_PAGE   (1u << 0) /* a block-table entry the call needs is outside [0, num_pages) */
#define ORACLE_ERR_SEQLEN (1u << 1) /* seq_lens[b] < 0 or > MP * page_size */
#define ORACLE_ERR_POS    (1u << 2) /* append position outside [0, MP * page_size) */
#define ORACLE_ERR_REQ    (1u << 3) /* request index outside [0, B) */
#define ORACLE_ERR_EXHAUSTED (1u << 5) /* an acquisition found too few free pages */

#define ORACLE_KV_E4M3 0
#define ORACLE_KV_BF16 1

/* ------------------------------------------------------------------------ */
/* Scalar helpers                                                            */
/* ------------------------------------------------------------------------ */

/* Round a non-negative double holding a value with few significant bits to the
 * nearest integer, ties to the even integer. */
static double round_half_even(double x)
{
    double f = floor(x);
    double r = x - f;
    if (r > 0.5) return f + 1.0;
    if (r < 0.5) return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

static float bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* [OFP8] encode: round-to-nearest-even onto the e4m3 grid, saturating. */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a > 448.0) return (uint8_t)(sign | 0x7E); /* beyond the largest finite value, inf included */

    if (a < 0x1p-6) {
        /* Subnormal band: the grid is k * 2^-9, k = 0..7.  k == 8 rounds up
         * into the smallest normal 2^-6, whose code is 0x08 == 8. */
        double k = round_half_even(a * 0x1p9); /* scaling by 2^9 is exact */
        return (uint8_t)(sign | (uint8_t)k);
    }

    int e2;
    (void)frexp(a, &e2);       /* a = f * 2^e2 with f in [0.5, 1) */
    int E = e2 - 1;            /* unbiased exponent: a in [2^E, 2^(E+1)), -6 <= E <= 8 */
    double n = round_half_even(ldexp(a, 3 - E)); /* significand * 8, in [8, 16] */
    if (n == 16.0) {           /* rounding carried into the next binade */
        n = 8.0;
        E += 1;
    }
    /* a <= 448 = 1.75 * 2^8 keeps (E, n) at or below (8, 14): code 0x7E. */
    return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | ((int)n - 8)));
}

/* [OFP8] decode: exact value of a code (NaN for S.1111.111). */
double oracle_e4m3_decode(uint8_t c)
{
    int s = c >> 7;
    int E = (c >> 3) & 0xF;
    int M = c & 0x7;
    if (E == 0xF && M == 0x7) return NAN;
    double mag = (E == 0) ? ldexp((double)M, -9)        /* subnormal: M/8 * 2^-6 */
                          : ldexp(8.0 + M, E - 10);     /* (1 + M/8) * 2^(E-7) */
    return s ? -mag : mag;
}

void oracle_e4m3_encode_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const uint8_t *c, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}

/* [KVQ] the quantised value of one BF16 element: one fp32 division by the
 * per-tensor scale, then e4m3 encoding. */
uint8_t oracle_quantise(uint16_t bf16_bits, float scale)
{
    float x = bf16_to_float(bf16_bits);
    float y = x / scale; /* single IEEE fp32 division */
    return oracle_e4m3_encode(y);
}

void oracle_quantise_array(const uint16_t *bf16_bits, uint8_t *out, int64_t n, float scale)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_quantise(bf16_bits[i], scale);
}

/* ------------------------------------------------------------------------ */
/* Quantise-and-append                                                       */
/* ------------------------------------------------------------------------ */

/* [KVQ] Write the K/V of n new tokens into their physical slots.
 * Token t belongs to request req_idx[t] and sits at logical position pos[t];
 * its page is block_table[req * MP + pos / P] and its slot pos % P.  Pools
 * are [num_pages][Hkv][P][D] elements (1 byte each for e4m3, 2 for bf16).
 * A token whose request, position or page is invalid writes nothing and
 * raises the matching error bit.  Returns the error bits. */
uint32_t oracle_quant_append(int kv_dtype, void *k_pool, void *v_pool,
                             int num_pages, int page_size, int num_kv_heads, int head_dim,
                             float k_scale, float v_scale,
                             const uint16_t *k_new, const uint16_t *v_new,
                             const int32_t *req_idx, const int32_t *pos, int n,
                             const int32_t *block_table, int B, int MP)
{
    uint32_t err = 0;
    const int P = page_size, H = num_kv_heads, D = head_dim;
    for (int t = 0; t < n; ++t) {
        int r = req_idx[t];
        int p = pos[t];
        if (r < 0 || r >= B) { err |= ORACLE_ERR_REQ; continue; }
        if (p < 0 || (int64_t)p >= (int64_t)MP * P) { err |= ORACLE_ERR_POS; continue; }
        int page = block_table[(int64_t)r * MP + p / P];
        if (page < 0 || page >= num_pages) { err |= ORACLE_ERR_PAGE; continue; }
        int slot = p % P;
        for (int h = 0; h < H; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = ((int64_t)t * H + h) * D + d;
                int64_t dst = (((int64_t)page * H + h) * P + slot) * D + d;
                if (kv_dtype == ORACLE_KV_E4M3) {
                    ((uint8_t *)k_pool)[dst] = oracle_quantise(k_new[src], k_scale);
                    ((uint8_t *)v_pool)[dst] = oracle_quantise(v_new[src], v_scale);
                } else {
                    ((uint16_t *)k_pool)[dst] = k_new[src];
                    ((uint16_t *)v_pool)[dst] = v_new[src];
                }
            }
        }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Prefill -> decode handoff                                                 */
/* ------------------------------------------------------------------------ */

/* [KVQ] The prefill side keeps its KV cache in BF16 and the decode side stores
 * it as e4m3: a prompt is converted when decode takes it over.  For every
 * request b and logical position p in [first[b], first[b] + count[b])
 * (first may be NULL: zeros), token p's BF16 K and V [Hkv][D] are gathered
 * from the prefill pools (page src_bt[b * src_MP + p / src_P], slot
 * p % src_P) and written into the decode pools at the same logical position
 * of request b through dst_bt, by oracle_quant_append (the decode append's
 * own quantisation).  A request whose range is negative or reaches past
 * either table writes nothing (POS); a token whose prefill page is outside
 * the pool writes nothing (PAGE); the append reports a bad decode page
 * itself (PAGE).  Returns the error bits. */
uint32_t oracle_handoff_pages(const uint16_t *src_k, const uint16_t *src_v, int src_pages,
                              int src_P, const int32_t *src_bt, int src_MP,
                              int dst_dtype, void *dst_k, void *dst_v, int dst_pages, int dst_P,
                              const int32_t *dst_bt, int dst_MP, int num_kv_heads, int head_dim,
                              float k_scale, float v_scale, const int32_t *first,
                              const int32_t *count, int B, uint16_t *scratch)
{
    uint32_t err = 0;
    const int H = num_kv_heads, D = head_dim;
    uint16_t *tk = scratch, *tv = scratch + (int64_t)H * D; /* one token's K and V */
    for (int b = 0; b < B; ++b) {
        int64_t f = first ? first[b] : 0;
        int64_t n = count[b];
        if (f < 0 || n < 0 || f + n > (int64_t)src_MP * src_P || f + n > (int64_t)dst_MP * dst_P) {
            err |= ORACLE_ERR_POS;
            continue;
        }
        for (int64_t p = f; p < f + n; ++p) {
            int sp = src_bt[(int64_t)b * src_MP + p / src_P];
            if (sp < 0 || sp >= src_pages) { err |= ORACLE_ERR_PAGE; continue; }
            int slot = (int)(p % src_P);
            for (int h = 0; h < H; ++h) {
                for (int d = 0; d < D; ++d) {
                    int64_t at = (((int64_t)sp * H + h) * src_P + slot) * D + d;
                    tk[(int64_t)h * D + d] = src_k[at];
                    tv[(int64_t)h * D + d] = src_v[at];
                }
            }
            int32_t req = b, pos = (int32_t)p;
            err |= oracle_quant_append(dst_dtype, dst_k, dst_v, dst_pages, dst_P, H, D, k_scale,
                                       v_scale, tk, tv, &req, &pos, 1, dst_bt, B, dst_MP);
        }
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Page-tag integrity check                                                  */
/* ------------------------------------------------------------------------ */

/* [GUARD] For every request b, compare the tag it expects for each of its
 * pages with the page's current tag; any difference aborts the request.
 * Pages checked: logical i < ceil(L_b / P).  A page id outside the pool, or a
 * length outside [0, MP*P], also aborts.  abort_mask[b] is 1 or 0. */
void oracle_check_tags(const int32_t *block_table, int B, int MP, const int32_t *seq_lens,
                       int page_size, const uint32_t *page_tags, int num_pages,
                       const uint32_t *expected_tags, uint8_t *abort_mask)
{
    for (int b = 0; b < B; ++b) {
        int L = seq_lens[b];
        int bad = 0;
        if (L < 0 || (int64_t)L > (int64_t)MP * page_size) {
            bad = 1;
        } else {
            int n_pages = (L + page_size - 1) / page_size;
            for (int i = 0; i < n_pages; ++i) {
                int page = block_table[(int64_t)b * MP + i];
                if (page < 0 || page >= num_pages) { bad = 1; continue; }
                if (page_tags[page] != expected_tags[(int64_t)b * MP + i]) bad = 1;
            }
        }
        abort_mask[b] = (uint8_t)bad;
    }
}

/* ------------------------------------------------------------------------ */
/* Page allocator and tag tracker                                            */
/* ------------------------------------------------------------------------ */

/* [GUARD] The allocator side of the tag check: a page's tag changes every
 * time the page is handed to a new owner, and the server records, for each
 * request, the (page, tag) pairs it was given.
 *
 * State: a stack of free page ids free_stack[0 .. *free_count) (the top is
 * the last one), page_tags[num_pages], and for each request slot b its
 * block-table row and expected-tag row (MP entries each).
 *
 * One call is a batch of releases followed by a batch of acquisitions.
 *  Release: for j = 0, 1, ... in order, request rel_req[j] returns its
 *    logical pages k = 0 .. rel_npages[j]-1 in order; each page id is pushed
 *    on the stack and the block-table entry becomes -1 (tags are unchanged).
 *    All or nothing: if any request index is outside [0, B), any count is
 *    outside [0, MP], any returned entry is not a page id, or the pushes would
 *    overfill the stack, nothing is released and error bits are returned.
 *  Acquire: for i = 0, 1, ... in order, request acq_req[i] asks for logical
 *    pages acq_first[i] .. acq_first[i] + acq_npages[i] - 1.  A request with
 *    an invalid index (ERR_REQ) or range (ERR_POS) gets nothing.  Valid
 *    requests are served in order: each pops its pages off the top of the
 *    stack in logical order, increments the popped page's tag (mod 2^32) and
 *    records the page and its new tag in its block-table and expected-tag
 *    rows.  The first valid request that finds too few free pages, and every
 *    valid request after it, get nothing (ERR_EXHAUSTED).  acq_ok[i] says
 *    whether request i was served.  A popped entry that is not a page id is
 *    consumed without being mapped (ERR_PAGE).
 * A free count outside [0, num_pages] changes nothing (ERR_PAGE).
 * Returns the OR of the error bits. */
uint32_t oracle_pages_update(int32_t *free_stack, int32_t *free_count, uint32_t *page_tags,
                             int num_pages, int32_t *block_table, uint32_t *expected_tags,
                             int B, int MP, const int32_t *rel_req, const int32_t *rel_npages,
                             int n_rel, const int32_t *acq_req, const int32_t *acq_first,
                             const int32_t *acq_npages, int n_acq, uint8_t *acq_ok)
{
    uint32_t err = 0;
    int count = *free_count;
    for (int i = 0; i < n_acq; ++i) acq_ok[i] = 0;
    if (count < 0 || count > num_pages) return ORACLE_ERR_PAGE;

    /* release: validate the whole batch, then push */
    uint32_t rel_err = 0;
    int64_t pushes = 0;
    for (int j = 0; j < n_rel; ++j) {
        int b = rel_req[j], n = rel_npages[j];
        if (b < 0 || b >= B) { rel_err |= ORACLE_ERR_REQ; continue; }
        if (n < 0 || n > MP) { rel_err |= ORACLE_ERR_POS; continue; }
        for (int k = 0; k < n; ++k) {
            int page = block_table[(int64_t)b * MP + k];
            if (page < 0 || page >= num_pages) rel_err |= ORACLE_ERR_PAGE;
        }
        pushes += n;
    }
    if (rel_err == 0 && count + pushes > num_pages) rel_err |= ORACLE_ERR_PAGE;
    if (rel_err) {
        err |= rel_err;
    } else {
        for (int j = 0; j < n_rel; ++j) {
            int b = rel_req[j], n = rel_npages[j];
            for (int k = 0; k < n; ++k) {
                int32_t *entry = &block_table[(int64_t)b * MP + k];
                free_stack[count++] = *entry;
                *entry = -1;
            }
        }
    }

    /* acquire: in order, until the first valid request that does not fit */
    int stopped = 0;
    for (int i = 0; i < n_acq; ++i) {
        int b = acq_req[i], first = acq_first[i], n = acq_npages[i];
        if (b < 0 || b >= B) { err |= ORACLE_ERR_REQ; continue; }
        if (first < 0 || n < 0 || (int64_t)first + n > MP) { err |= ORACLE_ERR_POS; continue; }
        if (stopped || n > count) { stopped = 1; err |= ORACLE_ERR_EXHAUSTED; continue; }
        for (int k = 0; k < n; ++k) {
            int page = free_stack[--count];
            if (page < 0 || page >= num_pages) { err |= ORACLE_ERR_PAGE; continue; }
            page_tags[page] += 1u;
            block_table[(int64_t)b * MP + first + k] = page;
            expected_tags[(int64_t)b * MP + first + k] = page_tags[page];
        }
        acq_ok[i] = 1;
    }
    *free_count = count;
    return err;
}

/* ------------------------------------------------------------------------ */
/* Weight-only quantised matrix product (decode GEMV / skinny GEMM)          */
/* ------------------------------------------------------------------------ */

#define ORACLE_W_INT4 0
#define ORACLE_W_E4M3 1

/* The signed 4-bit value held in nibble k of a row of packed INT4 weights:
 * byte k/2, low nibble for even k, high nibble for odd k, two's complement
 * (0x8 .. 0xF are -8 .. -1). */
static int int4_value(const uint8_t *row, int64_t k)
{
    uint8_t byte = row[k / 2];
    int nib = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    return nib >= 8 ? nib - 16 : nib;
}

/* [KVQ] section "模型权重压缩" (weight compression): the decode pool keeps the
 * weights as 4-bit integers (from FP8); every generated token reads them all,
 * so decode is bound by memory bandwidth; INT4 weights are widened to a
 * higher precision before they take part in the computation.  The format is
 * not stated; read as weight-only, symmetric, per-group:
 *   INT4: w[n][k] = int4(n, k) * s[n][k / group]   (s bf16 [N][K/group])
 *   E4M3: w[n][k] = e4m3(code[n][k]) * s[n]         (s fp32 [N], the FP8 path
 *         the pages compare against)
 * and y[m][n] = sum_k x[m][k] * w[n][k] with x bf16 [M][K], summed in fp64
 * and rounded to fp32 once. */
void oracle_wq_gemm(int wdtype, const uint8_t *w, const void *scales, const uint16_t *x,
                    float *y, int M, int N, int K, int group)
{
    for (int n = 0; n < N; ++n) {
        const uint8_t *row = w + (int64_t)n * (wdtype == ORACLE_W_INT4 ? K / 2 : K);
        for (int m = 0; m < M; ++m) {
            const uint16_t *xm = x + (int64_t)m * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double wv;
                if (wdtype == ORACLE_W_INT4) {
                    const uint16_t *s = (const uint16_t *)scales + (int64_t)n * (K / group);
                    wv = (double)int4_value(row, k) * (double)bf16_to_float(s[k / group]);
                } else {
                    const float *s = (const float *)scales;
                    wv = oracle_e4m3_decode(row[k]) * (double)s[n];
                }
                acc += (double)bf16_to_float(xm[k]) * wv;
            }
            y[(int64_t)m * N + n] = (float)acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Single-query paged attention                                              */
/* ------------------------------------------------------------------------ */

/* Exact value of one cached element, before the per-tensor scale. */
static double cached_value(int kv_dtype, const void *pool, int64_t idx)
{
    if (kv_dtype == ORACLE_KV_E4M3) return oracle_e4m3_decode(((const uint8_t *)pool)[idx]);
    return (double)bf16_to_float(((const uint16_t *)pool)[idx]);
}

/* One output row o[b, h, :]: softmax over the L_b cached tokens of request b
 * of (q . k_j) * sm_scale, weights applied to v_j.  K and V are dequantised
 * on read ([KVQ]): value = code value * scale.  Two passes: the maximum
 * logit first, then the exponentials.  Returns error bits; the row is zero
 * on error, abort or an empty context. */
static uint32_t attend_row(int kv_dtype, const void *k_pool, const void *v_pool,
                           int num_pages, int P, int H, int D, double k_scale, double v_scale,
                           const uint16_t *q, int Hq, const int32_t *block_table, int MP,
                           const int32_t *seq_lens, const uint8_t *abort_mask, double sm_scale,
                           int b, int h, float *out, double *logits, double *acc)
{
    float *o = out + ((int64_t)b * Hq + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0f;
    if (abort_mask && abort_mask[b]) return 0;
    int L = seq_lens[b];
    if (L < 0 || (int64_t)L > (int64_t)MP * P) return ORACLE_ERR_SEQLEN;
    if (L == 0) return 0;
    int n_pages = (L + P - 1) / P;
    for (int i = 0; i < n_pages; ++i) {
        int page = block_table[(int64_t)b * MP + i];
        if (page < 0 || page >= num_pages) return ORACLE_ERR_PAGE;
    }

    int g = Hq / H;
    int kvh = h / g;
    const uint16_t *qrow = q + ((int64_t)b * Hq + h) * D;

    /* logits */
    double m = -INFINITY;
    for (int j = 0; j < L; ++j) {
        int page = block_table[(int64_t)b * MP + j / P];
        int64_t base = (((int64_t)page * H + kvh) * P + j % P) * D;
        double s = 0.0;
        for (int d = 0; d < D; ++d)
            s += (double)bf16_to_float(qrow[d]) * (cached_value(kv_dtype, k_pool, base + d) * k_scale);
        s *= sm_scale;
        logits[j] = s;
        if (s > m) m = s;
    }
    /* weights and weighted sum of V */
    double denom = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = 0; j < L; ++j) {
        double w = exp(logits[j] - m);
        denom += w;
        int page = block_table[(int64_t)b * MP + j / P];
        int64_t base = (((int64_t)page * H + kvh) * P + j % P) * D;
        for (int d = 0; d < D; ++d)
            acc[d] += w * (cached_value(kv_dtype, v_pool, base + d) * v_scale);
    }
    for (int d = 0; d < D; ++d) o[d] = (float)(acc[d] / denom);
    return 0;
}

/* [KVQ] Decode attention over the paged cache for all rows (b, h), or only for
 * the n_rows rows listed in rows[] as b * Hq + h (rows == NULL: all rows).
 * k_scale / v_scale apply to an e4m3 cache only; a bf16 cache is unscaled.
 * Rows not computed are left untouched.  scratch must hold
 * (max L + D) doubles per thread.  Returns the OR of the error bits. */
uint32_t oracle_decode_attn(int kv_dtype, const void *k_pool, const void *v_pool,
                            int num_pages, int page_size, int num_kv_heads, int head_dim,
                            float k_scale, float v_scale,
                            const uint16_t *q, int B, int Hq,
                            const int32_t *block_table, int MP, const int32_t *seq_lens,
                            const uint8_t *abort_mask, float sm_scale, float *out,
                            const int32_t *rows, int n_rows, int nthreads,
                            double *scratch, int64_t scratch_per_thread)
{
    uint32_t err = 0;
    int64_t total = rows ? n_rows : (int64_t)B * Hq;
    if (nthreads < 1) nthreads = 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : err)
#endif
    for (int64_t r = 0; r < total; ++r) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double *logits = scratch + (int64_t)tid * scratch_per_thread;
        double *acc = logits + (scratch_per_thread - head_dim);
        int64_t row = rows ? rows[r] : r;
        int b = (int)(row / Hq), h = (int)(row % Hq);
        /* a bf16 cache holds the values themselves: no scale applies */
        double ks = (kv_dtype == ORACLE_KV_E4M3) ? (double)k_scale : 1.0;
        double vs = (kv_dtype == ORACLE_KV_E4M3) ? (double)v_scale : 1.0;
        err |= attend_row(kv_dtype, k_pool, v_pool, num_pages, page_size, num_kv_heads,
                          head_dim, ks, vs, q, Hq, block_table, MP,
                          seq_lens, abort_mask, (double)sm_scale, b, h, out, logits, acc);
    }
    return err;
}

/* Reports whether the library was compiled with OpenMP (used to state the cores the CPU
 * baseline really ran on). */
int oracle_has_openmp(void)
{
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}
