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
// Quantisation without a division per element.  Let u = 2^-24 (fp32 unit
// roundoff), y = RN(1 / scale), r_lo = RN(y (1 - 8u)) and r_hi =
// RN(y (1 + 8u)) (all three computed once on the host).  Then
// RN(x r_lo) = (x / scale)(1 + t) with t <= (1 + u)^3 (1 - 8u) - 1 < -u and
// RN(x r_hi) = (x / scale)(1 + t') with t' >= (1 - u)^3 (1 + 8u) - 1 > u,
// while RN(x / scale) = (x / scale)(1 + e) with |e| <= u: the correctly
// rounded quotient lies between lo = RN(x r_lo) and hi = RN(x r_hi) in
// magnitude.  Rounding to e4m3 with saturation is monotone in the magnitude,
// so when lo and hi give the same code that code is the code of
// RN(x / scale).  A 16-element chunk whose 16 pairs of codes all agree is
// stored at once; otherwise (some element within a few fp32 ulps of an e4m3
// rounding boundary) the chunk takes the correctly rounded division
// __fdiv_rn.  Underflow only moves values that all round to e4m3 zero;
// overflow and NaN give the same code at both ends and in the division.
// The bound needs y, r_lo and r_hi normal: for a scale whose reciprocal is
// not, every element takes the division.
//
// It is launched as a programmatic dependent of the work before it on the
// stream (launch_dependent), so it waits for that work before any access.
#include <cfloat>

#include "kvq_internal.h"

namespace kvq {

struct AppendArgs {
  void *k_pool, *v_pool;
  const uint16_t *k_new, *v_new;
  const int32_t *req_idx, *pos, *block_table;
  uint32_t *err_word;
  int64_t n_tokens;
  int32_t num_pages, P, H, B, MP;
  float k_scale, v_scale;
  float k_rlo, k_rhi, v_rlo, v_rhi;  // RN(RN(1 / scale) (1 -+ 8u))
  int32_t k_fast, v_fast;            // the reciprocals are normal floats
};

constexpr float kShrink = 1.0f - 0x1p-21f;  // 1 - 8u, exact in fp32
constexpr float kGrow = 1.0f + 0x1p-21f;    // 1 + 8u, exact in fp32

// two bf16 x bracketing reciprocals -> the e4m3 codes at both ends (low
// byte = element 0)
__device__ __forceinline__ void ends2(uint32_t w, float2 rlo, float2 rhi, uint16_t &lo,
                                      uint16_t &hi) {
  float x[2];
  bf16x2_to_f32(w, x);
  const float2 v = make_float2(x[0], x[1]);
  const float2 a = __fmul2_rn(v, rlo), b = __fmul2_rn(v, rhi);
  lo = f32x2_to_e4m3x2(a.x, a.y);
  hi = f32x2_to_e4m3x2(b.x, b.y);
}

// 16 bf16 (two 16-byte words) -> 16 e4m3 codes of RN(x / scale)
__device__ __forceinline__ uint4 quantise16(uint4 s0, uint4 s1, float scale, float rlo,
                                            float rhi, bool fast) {
  const uint32_t w[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t o[4];
  if (fast) {
    const float2 rl = make_float2(rlo, rlo), rh = make_float2(rhi, rhi);
    uint32_t diff = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint16_t l0, h0, l1, h1;
      ends2(w[2 * i], rl, rh, l0, h0);
      ends2(w[2 * i + 1], rl, rh, l1, h1);
      o[i] = static_cast<uint32_t>(l0) | (static_cast<uint32_t>(l1) << 16);
      diff |= o[i] ^ (static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16));
    }
    if (diff == 0) return make_uint4(o[0], o[1], o[2], o[3]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x[4];
    bf16x2_to_f32(w[2 * i], x);
    bf16x2_to_f32(w[2 * i + 1], x + 2);
    const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
    const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
    o[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <bool kFp8, int D>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  constexpr int kElems = kFp8 ? 16 : 8;    // elements per 16-byte output chunk
  constexpr int kCpr = D / kElems;         // chunks per (token, head) row: a power of 2
  constexpr int kSrcWords = kFp8 ? 2 : 1;  // 16-byte source words per chunk
  constexpr int kPer = kFp8 ? 2 : 4;       // chunks per lane per batch
  const int64_t cap = static_cast<int64_t>(a.MP) * a.P;
  const int lane = threadIdx.x & 31;
  const int per_tensor = a.H * kCpr;  // chunks of one token's K (or V)
  const int total = 2 * per_tensor;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t head_stride = static_cast<int64_t>(a.P) * D;
  grid_dependency_wait();  // earlier work on the stream is complete and visible
  allow_dependents();

  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       t < a.n_tokens; t += nwarps) {
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
              quantise16(s[k][0], s[k][1], is_v ? a.v_scale : a.k_scale,
                         is_v ? a.v_rlo : a.k_rlo, is_v ? a.v_rhi : a.k_rhi,
                         is_v ? a.v_fast : a.k_fast);
        } else {
          uint16_t *pool = static_cast<uint16_t *>(is_v ? a.v_pool : a.k_pool);
          *reinterpret_cast<uint4 *>(pool + dst) = s[k][0];
        }
      }
    }
  }
}

using AppendFn = void (*)(AppendArgs);

inline AppendFn pick_append(bool fp8, int D) {
  if (D == 64) return fp8 ? append_kernel<true, 64> : append_kernel<false, 64>;
  if (D == 128) return fp8 ? append_kernel<true, 128> : append_kernel<false, 128>;
  return nullptr;
}

// The bracketing reciprocals RN(RN(1 / scale) (1 -+ 8u)) (host IEEE fp32
// arithmetic) and whether all three are normal floats.
inline void reciprocals(float scale, float *rlo, float *rhi, int32_t *fast) {
  const float y = 1.0f / scale;
  const float lo = y * kShrink, hi = y * kGrow;
  *rlo = lo;
  *rhi = hi;
  *fast = std::isfinite(y) && std::isfinite(hi) && lo >= FLT_MIN ? 1 : 0;
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
  a.B = B;
  a.MP = MP;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  reciprocals(a.k_scale, &a.k_rlo, &a.k_rhi, &a.k_fast);
  reciprocals(a.v_scale, &a.v_rlo, &a.v_rhi, &a.v_fast);

  const bool fp8 = cache->kv_dtype == KVQ_KV_E4M3;
  const AppendFn fn = pick_append(fp8, cache->head_dim);
  if (!fn) return KVQ_ERR_UNSUPPORTED;
  constexpr int threads = 256, warps = threads / 32;
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const int64_t want = (static_cast<int64_t>(n_tokens) + warps - 1) / warps;  // warp per token
  const int blocks = static_cast<int>(want < 16LL * sms ? want : 16LL * sms);
  const cudaError_t e =
      launch_dependent(fn, blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream), a);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
