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
// RN(x / scale).  A 16-element chunk whose 16 pairs of codes all agree is
// stored at once; otherwise (some element within a few fp32 ulps of an e4m3
// rounding boundary) the chunk takes the correctly rounded division
// __fdiv_rn.  Underflow only moves values that all round to e4m3 zero;
// overflow and NaN give the same code at both ends and in the division.
// The bound needs y, r_lo and r_hi normal: for a scale whose reciprocal is
// not, every element takes the division.
//
#pragma once

#include <cfloat>
#include <cmath>

#include "kvq_device.cuh"

namespace kvq {

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
