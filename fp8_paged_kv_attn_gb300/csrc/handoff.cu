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
// each); then, token by token, the lanes take the token's K 16-byte output
// chunks (16 codes; a head's row of D bf16 values is contiguous in the
// prefill page), then its V chunks, each batch's source words loaded before
// any of them is converted and stored.  The kv-head count and D are template
// parameters, so every lane's chunk offsets are fixed before the token loop.
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

template <bool kFp8, int H, int D>
__global__ void __launch_bounds__(32 * kHoWarps, 6) handoff_kernel(HandoffArgs a) {
  constexpr int kElems = kFp8 ? 16 : 8;             // elements per 16-byte output chunk
  constexpr int kCpr = D / kElems;                  // chunks per (token, head) row
  constexpr int kChunks = H * kCpr;                 // chunks of one token's K (or V)
  constexpr int kPer = (kChunks + 31) / 32;         // chunks per lane per tensor
  constexpr int kSrcWords = kFp8 ? 2 : 1;           // 16-byte source words per chunk
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // this lane's chunks: element offsets inside a token's (page, head 0, slot)
  // block, the same for every token (heads are P * D elements apart)
  int soff[kPer], doff[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int c = lane + 32 * k;
    soff[k] = (c / kCpr) * a.Ps * D + (c % kCpr) * kElems;
    doff[k] = (c / kCpr) * a.Pd * D + (c % kCpr) * kElems;
  }
  grid_dependency_wait();
  allow_dependents();

  for (int b = blockIdx.y; b < a.B; b += gridDim.y) {
    const int f = a.first ? __ldg(a.first + b) : 0;
    const int n = __ldg(a.count + b);
    const long long end = static_cast<long long>(f) + n;
    if (f < 0 || n < 0 || end > static_cast<long long>(a.src_MP) * a.Ps ||
        end > static_cast<long long>(a.dst_MP) * a.Pd) {
      if (blockIdx.x == 0 && threadIdx.x == 0) report(a.err_word, KVQ_ERRBIT_POS);
      continue;
    }
    // positions fit in 32 bits from here on: both tables hold at most
    // INT32_MAX tokens (checked by the host)
    const long long t0l = static_cast<long long>(blockIdx.x) * kHoTokPerCta + warp * kHoTokPerWarp;
    if (t0l >= n) continue;
    const int t0 = static_cast<int>(t0l);
    const int ntok = min(kHoTokPerWarp, n - t0);
    // lanes 0..ntok-1: the prefill and decode pages of token f + t0 + lane
    int sp = -1, dp = -1;
    if (lane < ntok) {
      const int p = f + t0 + lane;
      sp = __ldg(a.src_bt + static_cast<int64_t>(b) * a.src_MP + p / a.Ps);
      dp = __ldg(a.dst_bt + static_cast<int64_t>(b) * a.dst_MP + p / a.Pd);
    }
    for (int j = 0; j < ntok; ++j) {
      const int p = f + t0 + j;
      const int spage = __shfl_sync(0xffffffffu, sp, j);
      const int dpage = __shfl_sync(0xffffffffu, dp, j);
      if (spage < 0 || spage >= a.src_pages || dpage < 0 || dpage >= a.dst_pages) {
        if (lane == 0) report(a.err_word, KVQ_ERRBIT_PAGE);
        continue;  // uniform over the warp
      }
      // element offsets of the token's (page, head 0, slot, dim 0)
      const int64_t src0 = (static_cast<int64_t>(spage) * H * a.Ps + p % a.Ps) * D;
      const int64_t dst0 = (static_cast<int64_t>(dpage) * H * a.Pd + p % a.Pd) * D;
      // K, then V: a batch's source words are all loaded before any is stored
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const uint16_t *src = (t ? a.src_v : a.src_k) + src0;
        uint4 s[kPer][kSrcWords];
#pragma unroll
        for (int k = 0; k < kPer; ++k)
          if (kChunks % 32 == 0 || lane + 32 * k < kChunks)
#pragma unroll
            for (int w = 0; w < kSrcWords; ++w)
              s[k][w] = __ldcs(reinterpret_cast<const uint4 *>(src + soff[k]) + w);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
          if (!(kChunks % 32 == 0 || lane + 32 * k < kChunks)) continue;
          if constexpr (kFp8) {
            uint8_t *dst = static_cast<uint8_t *>(t ? a.dst_v : a.dst_k) + dst0 + doff[k];
            *reinterpret_cast<uint4 *>(dst) =
                quantise16(s[k][0], s[k][1], t ? a.v_scale : a.k_scale, t ? a.v_rlo : a.k_rlo,
                           t ? a.v_rhi : a.k_rhi, t ? a.v_fast : a.k_fast);
          } else {
            uint16_t *dst = static_cast<uint16_t *>(t ? a.dst_v : a.dst_k) + dst0 + doff[k];
            *reinterpret_cast<uint4 *>(dst) = s[k][0];
          }
        }
      }
    }
  }
}

using HandoffFn = void (*)(HandoffArgs);

template <bool kFp8, int D>
HandoffFn pick_handoff_h(int H) {
  switch (H) {
    case 1: return handoff_kernel<kFp8, 1, D>;
    case 2: return handoff_kernel<kFp8, 2, D>;
    case 4: return handoff_kernel<kFp8, 4, D>;
    case 8: return handoff_kernel<kFp8, 8, D>;
  }
  return nullptr;
}

inline HandoffFn pick_handoff(bool fp8, int H, int D) {
  if (D == 64) return fp8 ? pick_handoff_h<true, 64>(H) : pick_handoff_h<false, 64>(H);
  if (D == 128) return fp8 ? pick_handoff_h<true, 128>(H) : pick_handoff_h<false, 128>(H);
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
  const int H = src->num_kv_heads;
  if (H != 1 && H != 2 && H != 4 && H != 8) return KVQ_ERR_UNSUPPORTED;
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

  const HandoffFn fn = pick_handoff(dst->kv_dtype == KVQ_KV_E4M3, dst->num_kv_heads, dst->head_dim);
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
