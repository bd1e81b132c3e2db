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
// memory in MMA-fragment order (so a lane's B registers for two MMA steps
// are one 16-byte load; a thread stages a 32-value chunk with four 16-byte
// loads and a permutation in registers) and, for INT4, its rows' group
// scales as fp32 pairs (rows r and r + 8: one 8-byte load per group; the
// scale loads are all issued before any is stored, so they cost one memory
// round trip, not one per element); each lane then streams its weights
// straight from HBM as contiguous 16-byte runs (the k order inside a group
// is permuted consistently in the weights' fragments and in the staged x,
// which leaves the sum unchanged), with a register ring of the next 3 (INT4)
// or 2 (e4m3) groups' loads in flight while the current one is computed.
// Rows past N and, with one token tile, token slots past M read a valid
// neighbour instead of branching (an output row depends only on its row of
// the A operand, an output token only on its column of B; neither is stored).
//  x is scaled while staged, per token and 128-wide k group, by the power of
//  two 2^e that puts the group's largest finite |x| in [2^14, 2^15), then
//  rounded to f16: exact for every bf16 value down to 2^-32 of that largest
//  (f16 keeps 11 bits, bf16 has 8), whatever the magnitude (bf16 reaches
//  2^128, f16 only 65504).  The products run on mma.sync m16n8k16 f16 ->
//  fp32; each group's sums are accumulated apart and multiplied by 2^-e
//  (exact) before they are added to the output.
//  INT4: one LOP3 and one fma.f16x2 turn two signed nibbles into exact f16
//        values (magic number 1024; the high nibble of each byte needs no
//        shift, the upper byte pair one shift per word); a group's sum is
//        also multiplied by the group's bf16 scale.
//  e4m3: cvt.rn.f16x2.e4m3x2 widens two codes exactly; the channel scale is
//        applied at the end.
// Products are exact and the sums are fp32, so the result differs from the
// fp64 definition only by fp32 summation rounding (and, for x values more
// than 2^32 below their group's largest, by the f16 rounding of those; and,
// for results below fp32's normal range, by the split-K atomics, since an
// fp32 atomic add flushes subnormal operands).
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

// The same with a zero accumulator in (the first step of a group's sum).
__device__ __forceinline__ void mma_f16_16816_zero(float c[4], const uint32_t a[4], uint32_t b0,
                                                   uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
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

// The exponent e of 2^e that puts a token's largest finite |x| (the bits of
// a non-negative fp32 value; 0 when all are zero) in [2^14, 2^15): 14 minus
// floor(log2 |x|), read off the bits (a subnormal m * 2^-149 has
// floor(log2) = -118 - clz(m)); in [-113, 149] for bf16 inputs.
__device__ __forceinline__ int x_exponent(uint32_t max_bits) {
  if (max_bits == 0u) return 0;
  const int field = static_cast<int>(max_bits >> 23);
  const int lg = field > 0 ? field - 127 : -118 - __clz(static_cast<int>(max_bits));
  return 14 - lg;
}

// 2^n as an fp32 bit pattern, n in [-126, 127] (exact, normal).
__device__ __forceinline__ float pow2i(int n) { return __int_as_float((n + 127) << 23); }

// 2^n for n in [-149, 127], a subnormal float below -126 (exact).
__device__ __forceinline__ float pow2_any(int n) {
  return n >= -126 ? pow2i(n) : __int_as_float(1 << (149 + n));
}

template <bool kInt4, int NT>
struct WqCfg {
  static constexpr int kWords = kInt4 ? 4 : 8;  // weight words per row half per lane per group
  // groups of weights held in registers per warp (fewer when more than four
  // token tiles need the registers; those products are bound by the MMAs)
  static constexpr int kDepth = NT > 4 ? 2 : kInt4 ? 4 : 3;
};

// shared memory of a CTA: [INT4 group scales: fp32 pairs for rows (r, r + 8),
// per pair and group][staged x][2^-e per (group, token slot of the tiles), fp32]
__host__ __device__ constexpr int wq_staged_tokens(int nt, int M) { return nt == 1 ? M : 8 * nt; }
__host__ __device__ constexpr size_t wq_scale_bytes(bool int4, int gpc) {
  return int4 ? size_t(kWqRows / 2) * gpc * 8 : 0;
}
__host__ __device__ constexpr size_t wq_x_bytes(int gpc, int nt, int M) {
  return size_t(gpc) * kWqGroup * wq_staged_tokens(nt, M) * sizeof(uint16_t);
}
__host__ __device__ constexpr size_t wq_smem_bytes(bool int4, int gpc, int nt, int M) {
  return wq_scale_bytes(int4, gpc) + wq_x_bytes(gpc, nt, M) + size_t(gpc) * 8 * nt * 4;
}

template <bool kInt4, int NT>
__global__ void __launch_bounds__(32 * kWqWarps, NT == 1 ? 3 : 2) wq_gemm_kernel(WqArgs a) {
  using C = WqCfg<kInt4, NT>;
  constexpr int kTok = 8 * NT;  // token slots of the MMA tiles
  extern __shared__ __align__(16) uint8_t wq_smem[];
  const size_t scb = wq_scale_bytes(kInt4, a.gpc);
  float2 *sc_s = reinterpret_cast<float2 *>(wq_smem);  // [kWqRows / 2][gpc]
  // staged x, one 16-byte word per (group, step pair, token, lane class):
  // the B registers of two consecutive MMA steps
  uint4 *xs = reinterpret_cast<uint4 *>(wq_smem + scb);
  // tokens staged: 8 per tile, or just the M real ones when there is one tile
  const int Mp = wq_staged_tokens(NT, a.M);
  float *xu = reinterpret_cast<float *>(wq_smem + scb + wq_x_bytes(a.gpc, NT, a.M));  // [gpc][kTok]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, rr = lane >> 2;
  const int kc = a.gpc * kWqGroup;
  const int kb0 = blockIdx.y * kc;
  const int ng = min(a.gpc, (a.K - kb0) / kWqGroup);
  const int row_base = blockIdx.x * kWqRows;
  const int row0 = row_base + warp * 16 + rr;  // this lane's rows: row0, row0 + 8
  // An output row depends only on its own row of A, an output token only on
  // its own column of B: rows past N read row N - 1 and, with one tile,
  // token slots past M read token M - 1; neither sum is ever stored.
  const int64_t row_bytes = kInt4 ? a.K / 2 : a.K;
  constexpr int kGroupBytes = kInt4 ? kWqGroup / 2 : kWqGroup;
  const int64_t lane_off = kInt4 ? kb0 / 2 + c * 16 : kb0 + c * 32;
  const uint8_t *w0 = a.w + static_cast<int64_t>(min(row0, a.N - 1)) * row_bytes + lane_off;
  const uint8_t *w8 = a.w + static_cast<int64_t>(min(row0 + 8, a.N - 1)) * row_bytes + lane_off;
  grid_dependency_wait();
  allow_dependents();

  // this lane's weights of group g
  auto load = [&](int g, uint32_t (&r0)[C::kWords], uint32_t (&r8)[C::kWords]) {
    if (g >= ng) return;
#pragma unroll
    for (int h = 0; h < C::kWords / 4; ++h) {
      const uint4 u0 = __ldcs(reinterpret_cast<const uint4 *>(w0 + g * kGroupBytes) + h);
      const uint4 u8 = __ldcs(reinterpret_cast<const uint4 *>(w8 + g * kGroupBytes) + h);
      r0[4 * h] = u0.x; r0[4 * h + 1] = u0.y; r0[4 * h + 2] = u0.z; r0[4 * h + 3] = u0.w;
      r8[4 * h] = u8.x; r8[4 * h + 1] = u8.y; r8[4 * h + 2] = u8.z; r8[4 * h + 3] = u8.w;
    }
  };
  // the first kDepth - 1 groups are in flight while x and the scales are staged
  uint32_t wr0[C::kDepth][C::kWords], wr8[C::kDepth][C::kWords];
#pragma unroll
  for (int d = 0; d < C::kDepth - 1; ++d) load(d, wr0[d], wr8[d]);

  // ---- INT4 group scales of the CTA's row pairs, fp32 in shared memory.
  // One item = (row pair p, group g): rows row_base + 16 (p / 8) + p % 8 and
  // 8 below.  Every load of a batch is issued before any is stored, and the
  // first batch's loads are in flight while x is staged
  constexpr int kScB = 5;  // items per thread per batch
  const int nsc = kInt4 ? (kWqRows / 2) * ng : 0;
  const uint16_t *sp = static_cast<const uint16_t *>(a.scales);
  const int64_t gs = a.K / kWqGroup;
  uint16_t scv[kScB][2];
  auto scale_loads = [&](int base) {
#pragma unroll
    for (int i = 0; i < kScB; ++i) {
      const int e = base + i * blockDim.x + tid;
      if (e < nsc) {
        const int p = e / ng, g = e - p * ng;
        const int r = row_base + (p >> 3) * 16 + (p & 7);
        const int64_t col = kb0 / kWqGroup + g;
        scv[i][0] = __ldg(sp + min(r, a.N - 1) * gs + col);
        scv[i][1] = __ldg(sp + min(r + 8, a.N - 1) * gs + col);
      }
    }
  };
  auto scale_stores = [&](int base) {
#pragma unroll
    for (int i = 0; i < kScB; ++i) {
      const int e = base + i * blockDim.x + tid;
      if (e < nsc) {
        const int p = e / ng, g = e - p * ng;
        sc_s[p * a.gpc + g] = make_float2(__uint_as_float(uint32_t(scv[i][0]) << 16),
                                          __uint_as_float(uint32_t(scv[i][1]) << 16));
      }
    }
  };
  // (with one token tile; with more, registers are short and x takes longer)
  constexpr bool kEarly = kInt4 && NT == 1;
  if constexpr (kEarly) scale_loads(0);

  // ---- stage x: one thread per (group, token, class) chunk of 32 k values:
  // four 16-byte loads; the chunk's largest finite |x| (a bf16 magnitude
  // below 0x7F80, compared as an integer), shared with the group's other
  // three chunks, which sit in lanes 4j .. 4j + 3 of the same warp (the
  // block size is a multiple of 4; every lane takes part in every pass);
  // the values times 2^e rounded to f16; the fragment permutation on whole
  // words (e4m3: the values' own order; INT4: two byte permutes per pair of
  // words); four 16-byte stores, one per step pair.
  const int nch = ng * Mp * 4;
  for (int base = 0; base < nch; base += blockDim.x) {
    const int ch = base + tid;
    const int cl = ch & 3, m = (ch >> 2) % Mp, g = (ch >> 2) / Mp;
    const bool real = ch < nch && m < a.M;
    uint32_t wv[16];  // bf16 pairs, value 2i in the low half of word i
    uint32_t mx = 0u;
    if (real) {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          a.x + static_cast<int64_t>(m) * a.K + kb0 + g * kWqGroup + cl * 32);
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 u = __ldg(src + h);
        wv[4 * h] = u.x;
        wv[4 * h + 1] = u.y;
        wv[4 * h + 2] = u.z;
        wv[4 * h + 3] = u.w;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t lo = wv[i] & 0x7FFFu, hi = (wv[i] >> 16) & 0x7FFFu;
        if (lo < 0x7F80u) mx = max(mx, lo);  // NaN and inf take no part
        if (hi < 0x7F80u) mx = max(mx, hi);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) wv[i] = 0u;
    }
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    if (ch < nch) {
      const int ex = x_exponent(mx << 16);
      if (cl == 0) xu[g * kTok + m] = pow2_any(-ex);
      // x * 2^ex as products by normal powers of two (2^ex alone is not a
      // float for ex > 127), each exact for the values f16 can hold
      const float f1 = pow2i(ex > 127 ? ex - 64 : ex);
      const float f2 = ex > 127 ? pow2i(64) : 1.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float xf[2];
        bf16x2_to_f32(wv[i], xf);
        const __half2 h = ex > 127 ? __floats2half2_rn((xf[0] * f1) * f2, (xf[1] * f1) * f2)
                                   : __floats2half2_rn(xf[0] * f1, xf[1] * f1);
        wv[i] = *reinterpret_cast<const uint32_t *>(&h);
      }
      uint4 *dst = xs + (g * 4 * Mp + m) * 4 + cl;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if constexpr (kInt4) {
          // step 2q + j: values 8q + 2j + {0, 4} and 8q + 2j + {1, 5}
          dst[q * Mp * 4] = make_uint4(__byte_perm(wv[4 * q], wv[4 * q + 2], 0x5410),
                                       __byte_perm(wv[4 * q], wv[4 * q + 2], 0x7632),
                                       __byte_perm(wv[4 * q + 1], wv[4 * q + 3], 0x5410),
                                       __byte_perm(wv[4 * q + 1], wv[4 * q + 3], 0x7632));
        } else {  // step 2q + j: values 8q + 4j .. 8q + 4j + 3
          dst[q * Mp * 4] = make_uint4(wv[4 * q], wv[4 * q + 1], wv[4 * q + 2], wv[4 * q + 3]);
        }
      }
    }
  }
  if constexpr (kInt4) {
    if constexpr (kEarly) scale_stores(0);
    for (int base = kEarly ? kScB * blockDim.x : 0; base < nsc; base += kScB * blockDim.x) {
      scale_loads(base);
      scale_stores(base);
    }
  }
  __syncthreads();

  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  // this lane's B words (token slot t * 8 + rr) and group scales
  const uint4 *xl = xs + (NT == 1 ? min(rr, Mp - 1) : rr) * 4 + c;
  const float2 *scl = sc_s + (warp * 8 + rr) * a.gpc;
  const float *xul = xu + 2 * c;

  for (int g0 = 0; g0 < ng; g0 += C::kDepth) {
#pragma unroll
    for (int d = 0; d < C::kDepth; ++d) {
      const int g = g0 + d;
      if (g >= ng) break;
      constexpr int kAhead = C::kDepth - 1;
      const int nd = (d + kAhead) % C::kDepth;  // register slot of group g + kDepth - 1
      load(g + kAhead, wr0[nd], wr8[nd]);
      float gacc[NT][4];  // the group's sums (the first step writes them)
      const uint4 *xg = xl + g * 4 * Mp * 4;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        // steps 2q and 2q + 1: with up to 4 tiles both A fragments, then per
        // tile one 16-byte load of both steps' B registers; with more, one
        // step at a time (registers) and 8-byte loads
        constexpr int kJ = 2;
#pragma unroll
        for (int j0 = 0; j0 < 2; j0 += kJ) {
          uint32_t af[kJ][4];
#pragma unroll
          for (int jj = 0; jj < kJ; ++jj) {
            const int j = j0 + jj;
            if constexpr (kInt4) {
              // step 2q + j: nibbles (p, p + 4), (p + 1, p + 5) of word q, p = 2 j
              const uint32_t v0 = j ? wr0[d][q] >> 8 : wr0[d][q];
              const uint32_t v8 = j ? wr8[d][q] >> 8 : wr8[d][q];
              af[jj][0] = int4lo_to_f16x2(v0);
              af[jj][1] = int4lo_to_f16x2(v8);
              af[jj][2] = int4hi_to_f16x2(v0);
              af[jj][3] = int4hi_to_f16x2(v8);
            } else {
              const int st = 2 * q + j;
              af[jj][0] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr0[d][st] & 0xFFFFu));
              af[jj][1] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr8[d][st] & 0xFFFFu));
              af[jj][2] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr0[d][st] >> 16));
              af[jj][3] = e4m3x2_to_f16x2(static_cast<uint16_t>(wr8[d][st] >> 16));
            }
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint4 *bp = xg + (q * Mp + t * 8) * 4;
            if constexpr (kJ == 2) {
              const uint4 bq = *bp;
              if (q == 0)
                mma_f16_16816_zero(gacc[t], af[0], bq.x, bq.y);
              else
                mma_f16_16816(gacc[t], af[0], bq.x, bq.y);
              mma_f16_16816(gacc[t], af[1], bq.z, bq.w);
            } else {
              const uint2 bh = reinterpret_cast<const uint2 *>(bp)[j0];
              if (q == 0 && j0 == 0)
                mma_f16_16816_zero(gacc[t], af[0], bh.x, bh.y);
              else
                mma_f16_16816(gacc[t], af[0], bh.x, bh.y);
            }
          }
        }
      }
      // the group's sums back to x's scale (2^-e of each token: exact unless
      // the sum is below fp32's normal range), times the INT4 group scale,
      // into the output
      float2 s = make_float2(1.f, 1.f);
      if constexpr (kInt4) s = scl[g];
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        // tokens t * 8 + 2c and + 1 (accumulator elements 0/2 and 1/3)
        const float2 u = *reinterpret_cast<const float2 *>(xul + g * kTok + t * 8);
        if constexpr (kInt4) {
          acc[t][0] = fmaf(s.x, gacc[t][0] * u.x, acc[t][0]);
          acc[t][1] = fmaf(s.x, gacc[t][1] * u.y, acc[t][1]);
          acc[t][2] = fmaf(s.y, gacc[t][2] * u.x, acc[t][2]);
          acc[t][3] = fmaf(s.y, gacc[t][3] * u.y, acc[t][3]);
        } else {
          acc[t][0] = fmaf(gacc[t][0], u.x, acc[t][0]);
          acc[t][1] = fmaf(gacc[t][1], u.y, acc[t][1]);
          acc[t][2] = fmaf(gacc[t][2], u.x, acc[t][2]);
          acc[t][3] = fmaf(gacc[t][3], u.y, acc[t][3]);
        }
      }
    }
  }

  // ---- epilogue: c0, c1 -> row0, tokens 2c, 2c + 1 of each tile; c2, c3 -> row0 + 8
  float f0 = 1.f, f8 = 1.f;
  if constexpr (!kInt4) {
    const float *fs = static_cast<const float *>(a.scales);
    f0 = fs[min(row0, a.N - 1)];
    f8 = fs[min(row0 + 8, a.N - 1)];
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = t * 8 + 2 * c + (e & 1);
      const int row = row0 + (e >> 1) * 8;
      if (n >= a.M || row >= a.N) continue;
      const float v = acc[t][e] * ((e >> 1) ? f8 : f0);
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
  auto smem_of = [&](int gpc) { return wq_smem_bytes(int4, gpc, nt, M); };
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
