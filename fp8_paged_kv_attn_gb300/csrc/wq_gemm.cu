// kvq_wq_gemm: weight-only quantised matrix product for decode,
// y[m][n] = sum_k x[m][k] w[n][k], with INT4 or e4m3 weights widened in
// registers.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "模型权重压缩": the decode pool keeps the model's weights as 4-bit integers
// instead of FP8; each generated token reads every weight, so decode speed is
// set by memory bandwidth and the smaller weights make it faster, while the
// INT4 values must be widened before they take part in the computation.  The
// format is not stated; this library reads it as weight-only, symmetric and
// per-group (signed two's-complement nibbles, even k in the low nibble, bf16
// scales per 128-wide group of k), and the FP8 path it is compared with as
// e4m3 weights with an fp32 scale per output channel.
//
// Kernel: a CTA of 8 warps covers 128 output channels (16 per warp) and a
// range of 128-wide k groups (split-K over CTAs, partial sums added with
// atomics into a zeroed y).  The CTA first stages its slice of x in shared
// memory in MMA-fragment order (so each lane's B operand is one 8-byte
// load; a thread stages a 32-value chunk with four 16-byte loads and a
// permutation in registers); each lane then streams its weights straight
// from HBM as contiguous 16-byte runs (the k order inside a group is
// permuted consistently in the weights' fragments and in the staged x, which
// leaves the sum unchanged), with a register ring of the next 3 (INT4) or 2
// (e4m3) groups' loads in flight while the current one is computed.
//  x is scaled while staged, per token over the CTA's k range, by the power
//  of two 2^e that puts the token's largest finite |x| there in
//  [2^14, 2^15), then rounded to f16: exact for every bf16 value down to
//  2^-32 of that largest (f16 keeps 11 bits, bf16 has 8), whatever the
//  magnitude (bf16 reaches 2^128, f16 only 65504).  The products run on
//  mma.sync m16n8k16 f16 -> fp32 and the CTA's sums are multiplied by 2^-e
//  (exact) in the epilogue.
//  INT4: one LOP3 and one fma.f16x2 turn two signed nibbles into exact f16
//        values (magic number 1024; the high nibble of each byte needs no
//        shift, the upper byte pair one shift per word); a group's sum is
//        also multiplied by the group's bf16 scale.
//  e4m3: cvt.rn.f16x2.e4m3x2 widens two codes exactly; the channel scale is
//        applied at the end.
// Products are exact and the sums are fp32, so the result differs from the
// fp64 definition only by fp32 summation rounding (and, for x values more
// than 2^32 below their token's largest in the CTA's range, by the f16
// rounding of those).  The INT4 sums stay finite in the scaled domain for
// group scales below 2^97 in magnitude.
#include <atomic>

#include <cuda_fp16.h>

#include "kvq_internal.h"

namespace kvq {

struct WqArgs {
  const uint8_t *w;       // INT4 [N][K/2] or e4m3 [N][K]
  const void *scales;     // bf16 [N][K/128] or fp32 [N]
  const uint16_t *x;      // bf16 [M][K]
  float *y;               // fp32 [M][N]
  int32_t M, N, K;
  int32_t gpc;            // 128-wide k groups per CTA
  int32_t atomic;         // add into y (split-K) instead of storing
};

constexpr int kWqWarps = 8;
constexpr int kWqRows = 16 * kWqWarps;  // output channels per CTA
constexpr int kWqGroup = 128;

__device__ __forceinline__ void mma_f16_16816(float c[4], const uint32_t a[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Signed nibbles of v as exact f16 pairs, without a shift for the high
// nibble of a byte (f16 has a 10-bit mantissa):
//  lo: nibbles 0 and 4 (bits 0-3, 16-19): (nib ^ 8) | 0x6400 is the f16 value
//      1024 + (q + 8), and 1024 + (q + 8) - 1032 = q;
//  hi: nibbles 1 and 5 (bits 4-7, 20-23): ((nib ^ 8) << 4) | 0x6400 is
//      1024 + 16 (q + 8), and that / 16 - 72 = q.
// Every value on the way is an integer below 2048, exact in f16.
__device__ __forceinline__ uint32_t int4lo_to_f16x2(uint32_t v) {
  uint32_t t, r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(t) : "r"(v), "r"(0x000F000Fu), "r"(0x64086408u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(t), "r"(0x3C003C00u), "r"(0xE408E408u));
  return r;
}
__device__ __forceinline__ uint32_t int4hi_to_f16x2(uint32_t v) {
  uint32_t t, r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(t) : "r"(v), "r"(0x00F000F0u), "r"(0x64806480u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(t), "r"(0x2C002C00u), "r"(0xD480D480u));
  return r;
}

// The fragment order of a lane class's 32 k values in a group: slot i (0..3;
// slots 0-1 are the B register b0b1, 2-3 are b2b3) of step s (0..7) holds
// value j = frag_src(s, i).  INT4: step s uses nibbles (p, p + 4) and
// (p + 1, p + 5) of weight word q = s / 2 with p = 2 (s % 2), i.e. k offsets
// 8q + p + {0, 4, 1, 5}; e4m3: step s uses bytes 4s .. 4s + 3 in order.
template <bool kInt4>
__device__ __forceinline__ constexpr int frag_src(int s, int i) {
  if constexpr (kInt4) {
    const int q = s >> 1, p = 2 * (s & 1);
    const int d = (i == 0) ? 0 : (i == 1) ? 4 : (i == 2) ? 1 : 5;
    return 8 * q + p + d;
  } else {
    return 4 * s + i;
  }
}

// The exponent e of 2^e that puts a token's largest finite |x| (fp32 bits;
// 0 when all are zero) in [2^14, 2^15): in [-113, 147] for bf16 inputs.
__device__ __forceinline__ int x_exponent(uint32_t max_bits) {
  const float mx = __uint_as_float(max_bits);
  return mx > 0.f ? 14 - ilogbf(mx) : 0;
}

template <bool kInt4>
struct WqCfg {
  static constexpr int kWords = kInt4 ? 4 : 8;  // weight words per row half per lane per group
  static constexpr int kDepth = kInt4 ? 4 : 3;  // groups of weights held in registers per warp
};

// shared memory of a CTA: [group scales: kWqRows x gpc bf16][staged x]
// [largest finite |x| per staged token over the CTA's k range, fp32 bits]
__host__ __device__ constexpr int wq_staged_tokens(int nt, int M) { return nt == 1 ? M : 8 * nt; }
__host__ __device__ constexpr size_t wq_scale_bytes(int gpc) {
  return (size_t(kWqRows) * gpc * 2 + 15) / 16 * 16;
}
__host__ __device__ constexpr size_t wq_x_bytes(int gpc, int nt, int M) {
  return size_t(gpc) * kWqGroup * wq_staged_tokens(nt, M) * sizeof(uint16_t);
}
__host__ __device__ constexpr size_t wq_smem_bytes(int gpc, int nt, int M) {
  return wq_scale_bytes(gpc) + wq_x_bytes(gpc, nt, M) + size_t(wq_staged_tokens(nt, M)) * 4;
}

template <bool kInt4, int NT>
__global__ void __launch_bounds__(32 * kWqWarps) wq_gemm_kernel(WqArgs a) {
  using C = WqCfg<kInt4>;
  extern __shared__ __align__(16) uint8_t wq_smem[];
  uint16_t *sc_s = reinterpret_cast<uint16_t *>(wq_smem);  // [rows][gpc] bf16
  uint16_t *xs = reinterpret_cast<uint16_t *>(wq_smem + wq_scale_bytes(a.gpc));
  // tokens staged: 8 per tile, or just the M real ones when there is one
  // tile (lanes whose token is past M then use a zero operand)
  const int Mp = wq_staged_tokens(NT, a.M);
  uint32_t *xmax = reinterpret_cast<uint32_t *>(wq_smem + wq_scale_bytes(a.gpc) +
                                                wq_x_bytes(a.gpc, NT, a.M));  // [Mp]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, rr = lane >> 2;
  const int kc = a.gpc * kWqGroup;
  const int kb0 = blockIdx.y * kc;
  const int ng = min(a.gpc, (a.K - kb0) / kWqGroup);
  const int row_base = blockIdx.x * kWqRows;
  const int row0 = row_base + warp * 16 + rr;  // this lane's rows: row0, row0 + 8
  const bool ok0 = row0 < a.N, ok8 = row0 + 8 < a.N;
  const int64_t row_bytes = kInt4 ? a.K / 2 : a.K;
  constexpr int kGroupBytes = kInt4 ? kWqGroup / 2 : kWqGroup;
  const uint8_t *w0 = a.w + static_cast<int64_t>(row0) * row_bytes +
                      (kInt4 ? kb0 / 2 + c * 16 : kb0 + c * 32);
  const uint8_t *w8 = w0 + 8 * row_bytes;
  grid_dependency_wait();
  allow_dependents();

  // this lane's weights of group g (zeros for rows past N)
  auto load = [&](int g, uint32_t (&r0)[C::kWords], uint32_t (&r8)[C::kWords]) {
    if (g >= ng) return;
#pragma unroll
    for (int h = 0; h < C::kWords / 4; ++h) {
      const uint4 u0 = ok0 ? __ldcs(reinterpret_cast<const uint4 *>(w0 + g * kGroupBytes) + h)
                           : make_uint4(0, 0, 0, 0);
      const uint4 u8 = ok8 ? __ldcs(reinterpret_cast<const uint4 *>(w8 + g * kGroupBytes) + h)
                           : make_uint4(0, 0, 0, 0);
      r0[4 * h] = u0.x; r0[4 * h + 1] = u0.y; r0[4 * h + 2] = u0.z; r0[4 * h + 3] = u0.w;
      r8[4 * h] = u8.x; r8[4 * h + 1] = u8.y; r8[4 * h + 2] = u8.z; r8[4 * h + 3] = u8.w;
    }
  };
  // the first kDepth - 1 groups are in flight while x is staged
  uint32_t wr0[C::kDepth][C::kWords], wr8[C::kDepth][C::kWords];
#pragma unroll
  for (int d = 0; d < C::kDepth - 1; ++d) load(d, wr0[d], wr8[d]);

  // ---- stage x: one thread per (group, token, class) chunk of 32 k values,
  // in two passes.  The first finds each token's largest finite |x| over
  // the CTA's k range (non-negative floats order like their bit patterns).
  // The second loads the chunk again, one 16-byte load (8 values, which
  // feed exactly fragment steps 2h and 2h + 1 of either weight type) at a
  // time, scales it by 2^e, rounds it to f16 and stores the two steps'
  // 8-byte fragment words (a warp's stores for one step are 256 contiguous
  // bytes).
  const int nch = ng * Mp * 4;
  for (int m = tid; m < Mp; m += blockDim.x) xmax[m] = 0u;
  __syncthreads();
  auto chunk_src = [&](int ch) {
    const int cl = ch & 3, m = (ch >> 2) % Mp, g = (ch >> 2) / Mp;
    return reinterpret_cast<const uint4 *>(a.x + static_cast<int64_t>(m) * a.K + kb0 +
                                           g * kWqGroup + cl * 32);
  };
  for (int ch = tid; ch < nch; ch += blockDim.x) {
    const int m = (ch >> 2) % Mp;
    if (m >= a.M) continue;
    const uint4 *src = chunk_src(ch);
    float mx = 0.f;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 u = __ldg(src + h);
      float xf[8];
      bf16x2_to_f32(u.x, xf);
      bf16x2_to_f32(u.y, xf + 2);
      bf16x2_to_f32(u.z, xf + 4);
      bf16x2_to_f32(u.w, xf + 6);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float ax = fabsf(xf[e]);
        if (ax < INFINITY) mx = fmaxf(mx, ax);  // NaN and inf take no part
      }
    }
    if (mx > 0.f) atomicMax(xmax + m, __float_as_uint(mx));
  }
  __syncthreads();
  for (int ch = tid; ch < nch; ch += blockDim.x) {
    const int cl = ch & 3, m = (ch >> 2) % Mp, g = (ch >> 2) / Mp;
    const bool real = m < a.M;
    const uint4 *src = chunk_src(ch);
    float f1 = 0.f, f2 = 0.f;  // tokens past M: zeros
    if (real) {
      const int ex = x_exponent(xmax[m]);
      // x * 2^ex as two products by normal powers of two (2^ex alone is not
      // a float for ex > 127); each is exact for the values f16 can hold
      f1 = ldexpf(1.f, ex > 127 ? ex - 64 : ex);
      f2 = ex > 127 ? 18446744073709551616.f : 1.f;  // 2^64
    }
    uint2 *dst = reinterpret_cast<uint2 *>(xs) + (g * 8 * Mp + m) * 4 + cl;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const uint4 u = real ? __ldg(src + h) : make_uint4(0, 0, 0, 0);
      float xf[8];
      bf16x2_to_f32(u.x, xf);
      bf16x2_to_f32(u.y, xf + 2);
      bf16x2_to_f32(u.z, xf + 4);
      bf16x2_to_f32(u.w, xf + 6);
      auto h2 = [&](int i, int j) {  // f16 pair (value i low, value j high), scaled
        const __half2 r = __floats2half2_rn((xf[i] * f1) * f2, (xf[j] * f1) * f2);
        return *reinterpret_cast<const uint32_t *>(&r);
      };
#pragma unroll
      for (int st = 2 * h; st < 2 * h + 2; ++st)
        dst[st * Mp * 4] = make_uint2(h2(frag_src<kInt4>(st, 0) - 8 * h, frag_src<kInt4>(st, 1) - 8 * h),
                                      h2(frag_src<kInt4>(st, 2) - 8 * h, frag_src<kInt4>(st, 3) - 8 * h));
    }
  }
  // ---- group scales of the CTA's rows (INT4), bf16
  if constexpr (kInt4) {
    const uint16_t *sp = static_cast<const uint16_t *>(a.scales);
    const int64_t gs = a.K / kWqGroup;
    for (int e = tid; e < kWqRows * ng; e += blockDim.x) {
      const int r = e / ng, g = e % ng, row = row_base + r;
      sc_s[r * a.gpc + g] = row < a.N ? sp[row * gs + kb0 / kWqGroup + g] : uint16_t(0);
    }
  }
  __syncthreads();

  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  const uint2 *xb = reinterpret_cast<const uint2 *>(xs);
  const uint16_t *sc0 = sc_s + (warp * 16 + rr) * a.gpc, *sc8 = sc0 + 8 * a.gpc;

  for (int g0 = 0; g0 < ng; g0 += C::kDepth) {
#pragma unroll
    for (int d = 0; d < C::kDepth; ++d) {
      const int g = g0 + d;
      if (g >= ng) break;
      constexpr int kAhead = C::kDepth - 1;
      const int nd = (d + kAhead) % C::kDepth;  // register slot of group g + kDepth - 1
      load(g + kAhead, wr0[nd], wr8[nd]);
      float gacc[NT][4];
      if constexpr (kInt4) {
#pragma unroll
        for (int t = 0; t < NT; ++t) gacc[t][0] = gacc[t][1] = gacc[t][2] = gacc[t][3] = 0.f;
      }
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        uint32_t af[4];
        if constexpr (kInt4) {
          // step st: nibbles (p, p + 4), (p + 1, p + 5) of word st / 2, p = 2 (st % 2)
          const uint32_t v0 = (st & 1) ? wr0[d][st >> 1] >> 8 : wr0[d][st >> 1];
          const uint32_t v8 = (st & 1) ? wr8[d][st >> 1] >> 8 : wr8[d][st >> 1];
          af[0] = int4lo_to_f16x2(v0);
          af[1] = int4lo_to_f16x2(v8);
          af[2] = int4hi_to_f16x2(v0);
          af[3] = int4hi_to_f16x2(v8);
        } else {
          af[0] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr0[d][st] & 0xFFFFu));
          af[1] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr8[d][st] & 0xFFFFu));
          af[2] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr0[d][st] >> 16));
          af[3] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr8[d][st] >> 16));
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint2 b = (NT > 1 || rr < Mp) ? xb[((g * 8 + st) * Mp + t * 8 + rr) * 4 + c]
                                              : make_uint2(0u, 0u);
          mma_f16_16816(kInt4 ? gacc[t] : acc[t], af, b.x, b.y);
        }
      }
      if constexpr (kInt4) {
        const float s0 = __uint_as_float(uint32_t(sc0[g]) << 16);
        const float s8 = __uint_as_float(uint32_t(sc8[g]) << 16);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          acc[t][0] = fmaf(s0, gacc[t][0], acc[t][0]);
          acc[t][1] = fmaf(s0, gacc[t][1], acc[t][1]);
          acc[t][2] = fmaf(s8, gacc[t][2], acc[t][2]);
          acc[t][3] = fmaf(s8, gacc[t][3], acc[t][3]);
        }
      }
    }
  }

  // ---- epilogue: c0, c1 -> row0, tokens 2c, 2c + 1 of each tile; c2, c3 -> row0 + 8
  float f0 = 1.f, f8 = 1.f;
  if constexpr (!kInt4) {
    const float *sp = static_cast<const float *>(a.scales);
    f0 = ok0 ? sp[row0] : 0.f;
    f8 = ok8 ? sp[row0 + 8] : 0.f;
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = t * 8 + 2 * c + (e & 1);
      const int row = row0 + (e >> 1) * 8;
      if (n >= a.M || row >= a.N) continue;
      // the channel scale, then back to x's scale (exact unless the result
      // is below fp32's normal range; one rounding there)
      const float v = (acc[t][e] * ((e >> 1) ? f8 : f0)) * ldexpf(1.f, -x_exponent(xmax[n]));
      float *dst = a.y + static_cast<int64_t>(n) * a.N + row;
      if (a.atomic)
        atomicAdd(dst, v);
      else
        *dst = v;
    }
  }
}

using WqFn = void (*)(WqArgs);

template <bool kInt4>
WqFn pick_wq(int nt) {
  switch (nt) {
    case 1: return wq_gemm_kernel<kInt4, 1>;
    case 2: return wq_gemm_kernel<kInt4, 2>;
    case 3: return wq_gemm_kernel<kInt4, 3>;
    case 4: return wq_gemm_kernel<kInt4, 4>;
    case 5: return wq_gemm_kernel<kInt4, 5>;
    case 6: return wq_gemm_kernel<kInt4, 6>;
    case 7: return wq_gemm_kernel<kInt4, 7>;
    case 8: return wq_gemm_kernel<kInt4, 8>;
  }
  return nullptr;
}

constexpr size_t kWqSmemMax = 112 * 1024;

// Opt each kernel into the shared-memory budget once per device (slot =
// kernel variant), outside any stream capture after the first call.
bool wq_smem_opt_in(WqFn fn, int slot) {
  constexpr int kMaxDev = 64;
  static std::atomic<bool> done[kMaxDev][16];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  if (done[dev][slot].load(std::memory_order_acquire)) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kWqSmemMax)) != cudaSuccess)
    return false;
  done[dev][slot].store(true, std::memory_order_release);
  return true;
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_wq_gemm(int32_t w_dtype, const void *w, const void *scales,
                                  const void *x, float *y, int32_t M, int32_t N, int32_t K,
                                  kvq_stream_t stream) {
  if (w_dtype != KVQ_W_INT4 && w_dtype != KVQ_W_E4M3) return KVQ_ERR_INVALID_ARG;
  if (!w || !scales || !x || !y) return KVQ_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < kWqGroup) return KVQ_ERR_INVALID_ARG;
  if (M > 64 || K % kWqGroup) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(w) || !aligned16(x) ||
      (reinterpret_cast<uintptr_t>(y) & 3) || (reinterpret_cast<uintptr_t>(scales) & 3))
    return KVQ_ERR_INVALID_ARG;
  const bool int4 = w_dtype == KVQ_W_INT4;
  const int nt = (M + 7) / 8;
  const WqFn fn = int4 ? pick_wq<true>(nt) : pick_wq<false>(nt);
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;

  // split K so that the grid covers the GPU several times over; each CTA's
  // staged x must fit the shared-memory budget
  const int row_tiles = (N + kWqRows - 1) / kWqRows;
  const int groups = K / kWqGroup;
  auto smem_of = [&](int gpc) { return wq_smem_bytes(gpc, nt, M); };
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (!wq_smem_opt_in(fn, int4 ? nt - 1 : 8 + nt - 1)) return KVQ_ERR_CUDA;
  // k splits: as many as fill the GPU's resident CTAs once (at the occupancy
  // the staged x allows), fewer groups per CTA only when shared memory asks
  int gpc = groups;
  while (gpc > 1 && smem_of(gpc) > kWqSmemMax) --gpc;
  int ksplit = (groups + gpc - 1) / gpc;
  for (int pass = 0; pass < 2; ++pass) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, 32 * kWqWarps, smem_of(gpc)) !=
        cudaSuccess)
      return KVQ_ERR_CUDA;
    const int cap = (occ > 0 ? occ : 1) * sms;
    int want = cap / row_tiles;
    if (want < ksplit) want = ksplit;  // shared memory already needs this many
    if (want > groups) want = groups;
    gpc = (groups + want - 1) / want;
    ksplit = (groups + gpc - 1) / gpc;
  }
  const size_t smem = smem_of(gpc);

  if (ksplit > 1 &&
      cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * sizeof(float), s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  WqArgs args{static_cast<const uint8_t *>(w), scales, static_cast<const uint16_t *>(x), y,
              M, N, K, gpc, ksplit > 1 ? 1 : 0};
  const cudaError_t e = launch_dependent(fn, dim3(row_tiles, ksplit), 32 * kWqWarps, smem, s, args);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
