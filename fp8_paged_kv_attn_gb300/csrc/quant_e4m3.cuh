// e4m3 quantisation of bf16 values, shared by kvq_append and
// kvq_handoff_pages so that both store the same code for the same value:
// the code of the correctly rounded fp32 quotient x / scale under
// round-to-nearest-even with saturation to +-448 (cvt.rn.satfinite).
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
// RN(x / scale).  The bound needs y, r_lo and r_hi normal.
//
// Where the two codes differ, an e4m3 rounding boundary lies within a few
// fp32 ulps of the quotient.  On data whose scale is a power of two times a
// short odd number (amax / 448 with a round amax) this happens to about 6%
// of the elements, nearly all of them quotients that are exactly such a
// boundary (a bf16 times a short reciprocal is exact in fp32).  Those are
// settled without a division: q = RN(x y) and t = fma(-q, scale, x), the
// exact remainder rounded once.  t = 0 means x = q scale exactly (a nonzero
// remainder is a multiple of min(ulp(x), ulp(q) ulp(scale)) and so at least
// the smallest fp32 subnormal when q >= 2^-11, which a quotient next to a
// boundary is, and scale >= 2^-92), so x / scale = q is representable,
// RN(x / scale) = q and its code is cvt(q).  A boundary has at most 5
// significant bits and x at most 8, so x = q scale exactly needs a scale
// whose significand, trailing zeros dropped, has at most 8 bits: for any
// other scale the step could never fire and is skipped.  Elements left
// (a quotient a few ulps off a boundary) take the correctly rounded
// division __fdiv_rn one by one: a lane loops over its own undecided
// elements only, so a warp pays for the largest count among its lanes
// (usually one) rather than for a whole group.  Every element of a scale
// whose reciprocals are not normal is divided.
//
// A power-of-two scale (1.0, the usual uncalibrated one, among them) needs
// none of this: y = 1 / scale is exact, x y and x / scale are the same real
// number and round alike, so the code is that of RN(x y).
//
#pragma once

#include <cfloat>
#include <cmath>

#include "kvq_device.cuh"

namespace kvq {

constexpr float kShrink = 1.0f - 0x1p-21f;  // 1 - 8u, exact in fp32
constexpr float kGrow = 1.0f + 0x1p-21f;    // 1 + 8u, exact in fp32

// What the quantiser may use for one scale (host-computed, see quant_params).
constexpr int32_t kQuantBracket = 1;  // y, r_lo, r_hi normal: the two-code bracket holds
constexpr int32_t kQuantExact = 2;    // a short significand, scale >= 2^-92: the remainder step
constexpr int32_t kQuantPow2 = 4;     // scale a power of two with 1 / scale normal: x / scale = x y

struct QuantParams {
  float scale, rcp, rlo, rhi;  // scale, RN(1 / scale), RN(rcp (1 -+ 8u))
  int32_t mode;                // kQuantPow2, kQuantBracket [| kQuantExact], or 0 (divide)
};

// Two bf16 in a word -> the codes of RN(x r) for a bracketing reciprocal r.
__device__ __forceinline__ uint16_t scaled_codes2(uint32_t w, float2 r) {
  float x[2];
  bf16x2_to_f32(w, x);
  const float2 p = __fmul2_rn(make_float2(x[0], x[1]), r);
  return f32x2_to_e4m3x2(p.x, p.y);
}

// 2 N bf16 (N words, low half = lower element) -> their e4m3 codes (N / 2
// words, low byte = lowest element): the code of RN(x / scale) for each.
template <int N>
__device__ __forceinline__ void quantise_words(const uint32_t (&w)[N], const QuantParams &qp,
                                               uint32_t (&o)[N / 2]) {
  static_assert(N % 2 == 0, "whole words of codes");
  if (qp.mode & kQuantPow2) {
    const float2 y2 = make_float2(qp.rcp, qp.rcp);
#pragma unroll
    for (int i = 0; i < N / 2; ++i)
      o[i] = static_cast<uint32_t>(scaled_codes2(w[2 * i], y2)) |
             (static_cast<uint32_t>(scaled_codes2(w[2 * i + 1], y2)) << 16);
    return;
  }
  if (qp.mode & kQuantBracket) {
    const float2 rl = make_float2(qp.rlo, qp.rlo), rh = make_float2(qp.rhi, qp.rhi);
    uint32_t h[N / 2];
    uint32_t diff = 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      o[i] = static_cast<uint32_t>(scaled_codes2(w[2 * i], rl)) |
             (static_cast<uint32_t>(scaled_codes2(w[2 * i + 1], rl)) << 16);
      h[i] = static_cast<uint32_t>(scaled_codes2(w[2 * i], rh)) |
             (static_cast<uint32_t>(scaled_codes2(w[2 * i + 1], rh)) << 16);
      diff |= o[i] ^ h[i];
    }
    if (diff == 0) return;
    uint32_t left[N / 2];  // per word of 4 codes: 0xFF where the ends differ
#pragma unroll
    for (int i = 0; i < N / 2; ++i) left[i] = __vcmpne4(o[i], h[i]);
    if (qp.mode & kQuantExact) {
      // elements whose codes differ and whose quotient is exact take cvt(q)
      const float2 y2 = make_float2(qp.rcp, qp.rcp);
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        float x[4];
        bf16x2_to_f32(w[2 * i], x);
        bf16x2_to_f32(w[2 * i + 1], x + 2);
        const float2 q01 = __fmul2_rn(make_float2(x[0], x[1]), y2);
        const float2 q23 = __fmul2_rn(make_float2(x[2], x[3]), y2);
        const float q[4] = {q01.x, q01.y, q23.x, q23.y};
        uint32_t exact = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          exact |= (fmaf(-q[j], qp.scale, x[j]) == 0.0f ? 0xFFu : 0u) << (8 * j);
        const uint32_t c = static_cast<uint32_t>(f32x2_to_e4m3x2(q[0], q[1])) |
                           (static_cast<uint32_t>(f32x2_to_e4m3x2(q[2], q[3])) << 16);
        const uint32_t take = left[i] & exact;
        o[i] = (o[i] & ~take) | (c & take);
        left[i] &= ~exact;
      }
    }
    // what is left, one element at a time.  Word i of codes holds elements
    // 4i .. 4i + 3, from input words 2i and 2i + 1; one loop per 16-byte
    // source word (output words 2 i4 and 2 i4 + 1), bit 8j + h standing for
    // element j of output word 2 i4 + h.
#pragma unroll
    for (int i4 = 0; i4 < N / 4; ++i4) {
      uint32_t pw = (left[2 * i4] & 0x01010101u) | ((left[2 * i4 + 1] & 0x01010101u) << 1);
      while (pw) {
        const int bit = __ffs(pw) - 1;
        pw &= pw - 1;
        const int h = bit & 1, sh = bit & ~1;  // sh = 8 j
        const uint32_t ww = h ? ((sh & 16) ? w[4 * i4 + 3] : w[4 * i4 + 2])
                              : ((sh & 16) ? w[4 * i4 + 1] : w[4 * i4]);
        const float x = __uint_as_float((sh & 8) ? (ww & 0xFFFF0000u) : (ww << 16));
        const float d = __fdiv_rn(x, qp.scale);
        const uint32_t c = (static_cast<uint32_t>(f32x2_to_e4m3x2(d, d)) & 0xFFu) << sh;
        const uint32_t keep = ~(0xFFu << sh);
        if (h)
          o[2 * i4 + 1] = (o[2 * i4 + 1] & keep) | c;
        else
          o[2 * i4] = (o[2 * i4] & keep) | c;
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    float x[4];
    bf16x2_to_f32(w[2 * i], x);
    bf16x2_to_f32(w[2 * i + 1], x + 2);
    const uint16_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[0], qp.scale), __fdiv_rn(x[1], qp.scale));
    const uint16_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[2], qp.scale), __fdiv_rn(x[3], qp.scale));
    o[i] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
}

// 16 bf16 (two 16-byte words) -> 16 e4m3 codes
__device__ __forceinline__ uint4 quantise16(uint4 s0, uint4 s1, const QuantParams &qp) {
  const uint32_t w[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t o[4];
  quantise_words<8>(w, qp, o);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 8 bf16 (one 16-byte word) -> 8 e4m3 codes
__device__ __forceinline__ uint2 quantise8(uint4 s, const QuantParams &qp) {
  const uint32_t w[4] = {s.x, s.y, s.z, s.w};
  uint32_t o[2];
  quantise_words<4>(w, qp, o);
  return make_uint2(o[0], o[1]);
}

// The quantiser's parameters for one scale (host IEEE fp32 arithmetic): the
// bracketing reciprocals RN(RN(1 / scale) (1 -+ 8u)) and what may be used.
inline QuantParams quant_params(float scale) {
  QuantParams qp;
  const float y = 1.0f / scale;
  qp.scale = scale;
  qp.rcp = y;
  qp.rlo = y * kShrink;
  qp.rhi = y * kGrow;
  const bool bracket = std::isfinite(y) && std::isfinite(qp.rhi) && qp.rlo >= FLT_MIN;
  int exp2 = 0;
  const float m = std::frexp(scale, &exp2);  // scale = m 2^exp2, m in [0.5, 1)
  const bool pow2 = m == 0.5f && std::isfinite(y) && y >= FLT_MIN;
  uint32_t sig = static_cast<uint32_t>(std::ldexp(m, 24));  // the 24-bit significand
  while (sig != 0 && (sig & 1u) == 0) sig >>= 1;
  const bool short_sig = sig < 256u;
  qp.mode = pow2 ? kQuantPow2
                 : bracket ? (kQuantBracket | (short_sig && scale >= 0x1p-92f ? kQuantExact : 0))
                           : 0;
  return qp;
}

}  // namespace kvq
