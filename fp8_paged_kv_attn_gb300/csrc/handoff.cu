// kvq_handoff_pages: the prefill -> decode handoff of whole prompts, from a
// paged BF16 cache into the paged e4m3 decode cache.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "KV 缓存量化": the prefill side keeps its KV cache in BF16 and the decode
// side stores it as e4m3, so every prompt handed from prefill to decode is
// converted once.  The pages give no kernel for it; this one reads the
// prompt's BF16 K/V where the prefill cache holds them (through the prefill
// block table, with the prefill pool's own page size) and writes the codes
// where the decode cache wants them (through the decode block table), with
// the rounding kvq_append uses (quant_e4m3.cuh), so a token handed off and a
// token appended during decode are stored identically.
//
// Work layout: grid (token blocks, requests); a CTA of 8 warps takes 64
// consecutive tokens of one request, a warp 8 of them.  Lanes 0..7 of a warp
// look up the prefill and decode page of its 8 tokens at once (two loads
// each); then, token by token, the lanes take the token's 16-byte output
// chunks (16 codes; a head's row of D bf16 values is contiguous in the
// prefill page) in batches of two per lane, loading a batch's source words
// before converting and storing them.  Small register footprint: four CTAs
// (32 warps) per SM keep enough loads in flight.
// A request's token range is checked once; CTAs past the range exit at once.
//
// HBM-bound: per token and kv head 2 D (2 + s) bytes (read bf16 K and V,
// write s-byte codes), plus 4 bytes per prefill and per decode page.
#include <algorithm>

#include "kvq_internal.h"
#include "quant_e4m3.cuh"

namespace kvq {

struct HandoffArgs {
  const uint16_t *src_k, *src_v;  // bf16 [src_pages][H][Ps][D]
  void *dst_k, *dst_v;            // e4m3 or bf16 [dst_pages][H][Pd][D]
  const int32_t *src_bt, *dst_bt, *first, *count;
  uint32_t *err_word;
  int32_t src_pages, Ps, src_MP, dst_pages, Pd, dst_MP, H, B;
  float k_scale, v_scale;
  float k_rlo, k_rhi, v_rlo, v_rhi;
  int32_t k_fast, v_fast;
};

constexpr int kHoWarps = 8;
constexpr int kHoTokPerWarp = 8;
constexpr int kHoTokPerCta = kHoWarps * kHoTokPerWarp;

template <bool kFp8, int D>
__global__ void __launch_bounds__(32 * kHoWarps, 4) handoff_kernel(HandoffArgs a) {
  constexpr int kElems = kFp8 ? 16 : 8;  // elements per 16-byte output chunk
  constexpr int kCpr = D / kElems;       // chunks per (token, head) row
  constexpr int kSrcWords = kFp8 ? 2 : 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per_tensor = a.H * kCpr;
  const int total = 2 * per_tensor;
  constexpr int kPer = kFp8 ? 2 : 4;    // chunks per lane per batch
  grid_dependency_wait();
  allow_dependents();

  for (int b = blockIdx.y; b < a.B; b += gridDim.y) {
    const int64_t f = a.first ? __ldg(a.first + b) : 0;
    const int64_t n = __ldg(a.count + b);
    const int64_t src_cap = static_cast<int64_t>(a.src_MP) * a.Ps;
    const int64_t dst_cap = static_cast<int64_t>(a.dst_MP) * a.Pd;
    if (f < 0 || n < 0 || f + n > src_cap || f + n > dst_cap) {
      if (blockIdx.x == 0 && threadIdx.x == 0) report(a.err_word, KVQ_ERRBIT_POS);
      continue;
    }
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kHoTokPerCta + warp * kHoTokPerWarp;
    if (t0 >= n) continue;
    const int ntok = static_cast<int>(min(static_cast<int64_t>(kHoTokPerWarp), n - t0));
    // lanes 0..ntok-1: the prefill and decode pages of token f + t0 + lane
    int sp = -1, dp = -1;
    if (lane < ntok) {
      const int64_t p = f + t0 + lane;
      sp = __ldg(a.src_bt + static_cast<int64_t>(b) * a.src_MP + p / a.Ps);
      dp = __ldg(a.dst_bt + static_cast<int64_t>(b) * a.dst_MP + p / a.Pd);
    }
    for (int j = 0; j < ntok; ++j) {
      const int64_t p = f + t0 + j;
      const int spage = __shfl_sync(0xffffffffu, sp, j);
      const int dpage = __shfl_sync(0xffffffffu, dp, j);
      if (spage < 0 || spage >= a.src_pages || dpage < 0 || dpage >= a.dst_pages) {
        if (lane == 0) report(a.err_word, KVQ_ERRBIT_PAGE);
        continue;  // uniform over the warp
      }
      // element offsets of (page, head 0, slot, dim 0); heads are P * D apart
      const int64_t src0 = (static_cast<int64_t>(spage) * a.H * a.Ps + p % a.Ps) * D;
      const int64_t dst0 = (static_cast<int64_t>(dpage) * a.H * a.Pd + p % a.Pd) * D;
      const int64_t src_hs = static_cast<int64_t>(a.Ps) * D, dst_hs = static_cast<int64_t>(a.Pd) * D;
      // the lane's chunks in batches of kPer: the batch's source words first,
      // then its stores
      for (int base = 0; base < total; base += 32 * kPer) {
        uint4 s[kPer][kSrcWords];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int c = base + lane + 32 * k;
          if (c < total) {
            const bool is_v = c >= per_tensor;
            const int cc = is_v ? c - per_tensor : c;
            const uint4 *src = reinterpret_cast<const uint4 *>(
                (is_v ? a.src_v : a.src_k) + src0 + (cc / kCpr) * src_hs + (cc % kCpr) * kElems);
#pragma unroll
            for (int w = 0; w < kSrcWords; ++w) s[k][w] = __ldcs(src + w);
          }
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          const int c = base + lane + 32 * k;
          if (c >= total) break;
          const bool is_v = c >= per_tensor;
          const int cc = is_v ? c - per_tensor : c;
          const int64_t dst = dst0 + (cc / kCpr) * dst_hs + (cc % kCpr) * kElems;
          if constexpr (kFp8) {
            uint8_t *pool = static_cast<uint8_t *>(is_v ? a.dst_v : a.dst_k);
            *reinterpret_cast<uint4 *>(pool + dst) =
                quantise16(s[k][0], s[k][1], is_v ? a.v_scale : a.k_scale,
                           is_v ? a.v_rlo : a.k_rlo, is_v ? a.v_rhi : a.k_rhi,
                           is_v ? a.v_fast : a.k_fast);
          } else {
            uint16_t *pool = static_cast<uint16_t *>(is_v ? a.dst_v : a.dst_k);
            *reinterpret_cast<uint4 *>(pool + dst) = s[k][0];
          }
        }
      }
    }
  }
}

using HandoffFn = void (*)(HandoffArgs);

inline HandoffFn pick_handoff(bool fp8, int D) {
  if (D == 64) return fp8 ? handoff_kernel<true, 64> : handoff_kernel<false, 64>;
  if (D == 128) return fp8 ? handoff_kernel<true, 128> : handoff_kernel<false, 128>;
  return nullptr;
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_handoff_pages(const kvq_cache *src, const int32_t *src_block_table,
                                        int32_t src_MP, const kvq_cache *dst,
                                        const int32_t *dst_block_table, int32_t dst_MP,
                                        const int32_t *first, const int32_t *count, int32_t B,
                                        uint32_t *err_word, kvq_stream_t stream) {
  kvq_status st = validate_cache(src);
  if (st != KVQ_OK) return st;
  st = validate_cache(dst);
  if (st != KVQ_OK) return st;
  if (src->kv_dtype != KVQ_KV_BF16) return KVQ_ERR_INVALID_ARG;
  if (src->num_kv_heads != dst->num_kv_heads || src->head_dim != dst->head_dim)
    return KVQ_ERR_INVALID_ARG;
  if (src->num_kv_heads > 8) return KVQ_ERR_UNSUPPORTED;
  if (B < 0 || src_MP <= 0 || dst_MP <= 0) return KVQ_ERR_INVALID_ARG;
  if (B == 0) return KVQ_OK;
  if (!src_block_table || !dst_block_table || !count) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(src_MP) * src->page_size > INT32_MAX ||
      static_cast<int64_t>(dst_MP) * dst->page_size > INT32_MAX)
    return KVQ_ERR_INVALID_ARG;

  HandoffArgs a;
  a.src_k = static_cast<const uint16_t *>(src->k_pool);
  a.src_v = static_cast<const uint16_t *>(src->v_pool);
  a.dst_k = dst->k_pool;
  a.dst_v = dst->v_pool;
  a.src_bt = src_block_table;
  a.dst_bt = dst_block_table;
  a.first = first;
  a.count = count;
  a.err_word = err_word;
  a.src_pages = src->num_pages;
  a.Ps = src->page_size;
  a.src_MP = src_MP;
  a.dst_pages = dst->num_pages;
  a.Pd = dst->page_size;
  a.dst_MP = dst_MP;
  a.H = dst->num_kv_heads;
  a.B = B;
  a.k_scale = dst->k_scale;
  a.v_scale = dst->v_scale;
  reciprocals(a.k_scale, &a.k_rlo, &a.k_rhi, &a.k_fast);
  reciprocals(a.v_scale, &a.v_rlo, &a.v_rhi, &a.v_fast);

  const HandoffFn fn = pick_handoff(dst->kv_dtype == KVQ_KV_E4M3, dst->head_dim);
  if (!fn) return KVQ_ERR_UNSUPPORTED;
  // a request moves at most min(both capacities) tokens; token blocks past
  // its count exit at once
  const int64_t max_tok = std::min(static_cast<int64_t>(src_MP) * src->page_size,
                                   static_cast<int64_t>(dst_MP) * dst->page_size);
  const int64_t gx = (max_tok + kHoTokPerCta - 1) / kHoTokPerCta;
  if (gx > INT32_MAX) return KVQ_ERR_INVALID_ARG;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(B < 65535 ? B : 65535));
  const cudaError_t e = launch_dependent(fn, grid, 32 * kHoWarps, 0,
                                         reinterpret_cast<cudaStream_t>(stream), a);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
