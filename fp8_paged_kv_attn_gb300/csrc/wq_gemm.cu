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
// Two kernels, one per regime:
//  * the TMA-ring kernel (up to 8 tokens, see ring_plan): 64 output
//    channels per CTA; a producer warp streams the weights into a
//    shared-memory ring with the TMA engine, eight consumer warps read them
//    from there; a k split is a thread-block cluster whose partial sums are
//    added through distributed shared memory in rank order (details at the
//    kernel);
//  * the register-ring kernel (more tokens): a CTA of 8 warps covers 128
//    output channels (16 per warp) and a range of 128-wide k groups
//    (split-K over CTAs, partial sums added with atomics into a zeroed y);
//    each lane streams its weights straight from HBM as contiguous 16-byte
//    runs with a register ring of the next 3 (INT4) or 2 (e4m3) groups'
//    loads in flight while the current one is computed.
// Both first stage their slice of x in shared memory in MMA-fragment order
// (a lane's B registers for two MMA steps are one 16-byte load; the k order
// inside a group is permuted consistently in the weights' fragments and in
// the staged x, which leaves the sum unchanged) and, for INT4, their rows'
// group scales as fp32 pairs (rows r and r + 8: one 8-byte load per group;
// the scale loads are all issued before any is stored, so they cost one
// memory round trip).  The weights and scales are read before the kernel
// waits for the work ahead of it on the stream (they are constant); x after.
// Rows past N and, with one token tile, token slots past M read a valid
// neighbour instead of branching (an output row depends only on its row of
// the A operand, an output token only on its column of B; neither is stored).
// Arithmetic, both kernels:
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
// in the register-ring kernel, for results below fp32's normal range, by the
// split-K atomics, since an fp32 atomic add flushes subnormal operands).
#include <atomic>
#include <mutex>
#include <unordered_map>

#include <cuda_fp16.h>

#include "kvq_internal.h"

namespace kvq {

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

// ---------------------------------------------------------------------------
// Pieces shared by both kernels
// ---------------------------------------------------------------------------
//
// Fragment order.  mma.m16n8k16 pairs a lane's A slots with its own B slots:
// for lane class c (lane % 4), A registers 0/1 (rows r, r + 8) hold the k
// pair that B register 0 holds and A registers 2/3 the pair of B register 1.
// Which actual k sits in a slot is free, as long as A and B agree, so each
// lane class owns 32 k values of a 128-wide group and the B operand is
// staged in the order the weights arrive:
//  INT4: the class's 16 weight bytes per row, word q (8 nibbles) feeding
//        steps 2q (nibbles 0, 4 and 1, 5) and 2q + 1 (nibbles 2, 6 and 3, 7);
//  e4m3: the class's 32 code bytes per row, word st (4 codes) feeding step
//        st (codes 0, 1 and 2, 3).
// A lane's two B registers of steps 2q and 2q + 1 are one 16-byte word of
// the staged x: [group][step pair q][token slot][lane class].

// One group's products for NT token tiles: gacc[t] = the group's 4 step
// pairs (8 MMA steps) starting from zero.  w0 / w8: the lane's weight words
// of rows r and r + 8; xg: the lane's B word of the group's first step pair
// (token slot of tile 0), Mp token slots per step pair.
template <bool kInt4, int NT>
__device__ __forceinline__ void group_mma(float (&gacc)[NT][4],
                                          const uint32_t (&w0)[kInt4 ? 4 : 8],
                                          const uint32_t (&w8)[kInt4 ? 4 : 8], const uint4 *xg,
                                          int Mp) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t af[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      if constexpr (kInt4) {
        // step 2q + j: nibbles (p, p + 4), (p + 1, p + 5) of word q, p = 2 j
        const uint32_t v0 = j ? w0[q] >> 8 : w0[q];
        const uint32_t v8 = j ? w8[q] >> 8 : w8[q];
        af[j][0] = int4lo_to_f16x2(v0);
        af[j][1] = int4lo_to_f16x2(v8);
        af[j][2] = int4hi_to_f16x2(v0);
        af[j][3] = int4hi_to_f16x2(v8);
      } else {
        const int st = 2 * q + j;
        af[j][0] = e4m3x2_to_f16x2(static_cast<uint16_t>(w0[st] & 0xFFFFu));
        af[j][1] = e4m3x2_to_f16x2(static_cast<uint16_t>(w8[st] & 0xFFFFu));
        af[j][2] = e4m3x2_to_f16x2(static_cast<uint16_t>(w0[st] >> 16));
        af[j][3] = e4m3x2_to_f16x2(static_cast<uint16_t>(w8[st] >> 16));
      }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint4 bq = xg[(q * Mp + t * 8) * 4];
      if (q == 0)
        mma_f16_16816_zero(gacc[t], af[0], bq.x, bq.y);
      else
        mma_f16_16816(gacc[t], af[0], bq.x, bq.y);
      mma_f16_16816(gacc[t], af[1], bq.z, bq.w);
    }
  }
}

// The group's sums back to x's scale (2^-e of each token: exact unless the
// sum is below fp32's normal range), times the INT4 group scales s (rows r,
// r + 8), into the running sums.  xug: 2^-e of the group's token slots
// 2c, 2c + 1 of tile 0 (tiles 8 slots apart).  kOne (one token): only the
// sums of token slot 2c (elements 0 and 2) are kept, the others are never
// stored.
template <bool kInt4, int NT, bool kOne = false>
__device__ __forceinline__ void group_fold(float (&acc)[NT][4], const float (&gacc)[NT][4],
                                           float2 s, const float *xug) {
  if constexpr (kOne) {
    const float u = xug[0];
    acc[0][0] = kInt4 ? fmaf(s.x, gacc[0][0] * u, acc[0][0]) : fmaf(gacc[0][0], u, acc[0][0]);
    acc[0][2] = kInt4 ? fmaf(s.y, gacc[0][2] * u, acc[0][2]) : fmaf(gacc[0][2], u, acc[0][2]);
    return;
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const float2 u = *reinterpret_cast<const float2 *>(xug + t * 8);
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

// Stages x[m][kb0 .. kb0 + 128 ng) for Mp token slots (slots past M are
// zero) with threads tid = 0 .. nthr - 1 of whole warps, nthr a multiple of
// 32: one thread per (group, token, class) chunk of 32 k values: four
// 16-byte loads; the chunk's largest finite |x| (a bf16 magnitude below
// 0x7F80, compared as an integer), shared with the group's other three
// chunks, which sit in lanes 4j .. 4j + 3 of the same warp (every lane takes
// part in every pass); the values times 2^e (e puts the group's largest in
// [2^14, 2^15)) rounded to f16; 2^-e into xu[g * kTok + m]; the fragment
// permutation on whole words (e4m3: the values' own order; INT4: two byte
// permutes per pair of words); four 16-byte stores, one per step pair.
// A class's 32 values are x[32 cl ..] or, with kHalves (e4m3 weights that
// arrive as two 64-byte halves of a group), x[16 cl ..] and x[64 + 16 cl ..].
template <bool kInt4, bool kHalves>
__device__ __forceinline__ void stage_x(uint4 *xs, float *xu, int kTok, const uint16_t *x, int K,
                                        int M, int Mp, int kb0, int ng, int tid, int nthr) {
  const int nch = ng * Mp * 4;
  for (int base = 0; base < nch; base += nthr) {
    const int ch = base + tid;
    const int cl = ch & 3, m = (ch >> 2) % Mp, g = (ch >> 2) / Mp;
    const bool real = ch < nch && m < M;
    uint32_t wv[16];  // bf16 pairs, value 2i in the low half of word i
    uint32_t mx = 0u;
    if (real) {
      const uint16_t *row = x + static_cast<int64_t>(m) * K + kb0 + g * kWqGroup;
      const uint4 *s0 = reinterpret_cast<const uint4 *>(row + (kHalves ? 16 * cl : 32 * cl));
      const uint4 *s1 = kHalves ? reinterpret_cast<const uint4 *>(row + 64 + 16 * cl) : s0 + 2;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const uint4 u = __ldg(h < 2 ? s0 + h : s1 + (h - 2));
        wv[4 * h] = u.x;
        wv[4 * h + 1] = u.y;
        wv[4 * h + 2] = u.z;
        wv[4 * h + 3] = u.w;
      }
      // both halves of a word at once; NaN and inf (>= 0x7F80) take no part
      uint32_t mx2 = 0u;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t m = wv[i] & 0x7FFF7FFFu;
        mx2 = __vmaxu2(mx2, m & __vcmpltu2(m, 0x7F807F80u));
      }
      mx = max(mx2 & 0xFFFFu, mx2 >> 16);
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
}

// The row stride (in fp32 pairs) of the staged INT4 scales: gpc rounded up
// to an odd number, so that the eight row pairs a warp reads at once fall in
// eight different bank pairs.
__host__ __device__ constexpr int wq_scale_stride(int gpc) { return gpc | 1; }

// INT4 group scales of a CTA's row pairs as fp32 pairs, sc_s[p * stride + g]
// for pair p (rows row_base + 16 (p / 8) + p % 8 and 8 below, a row past N
// reads row N - 1) and group g < ng.  Items e = p * ng + g go to threads in
// order (a warp reads runs of consecutive scales), kScB per thread and
// batch: every load of a batch is issued before any is stored, so a batch
// costs one memory round trip.  p = e / ng is taken as trunc((e + 1/2)
// RN(1/ng)) in fp32, exact for every ng up to 2048 and e below 64 ng
// (checked exhaustively; ng is at most a few hundred here).
constexpr int kScB = 5;
struct ScaleStage {
  const uint16_t *sp;  // bf16 scales [N][K / 128], from the CTA's first group
  float2 *sc_s;
  int64_t gs;          // groups per row of the matrix
  int ng, gpc, N, row_base, n, tid, nthr;  // gpc: the row stride of sc_s
  float inv_ng;
  uint16_t v[kScB][2];
  __device__ __forceinline__ ScaleStage(const void *scales, float2 *sc_s_, int K, int N_,
                                        int kb0, int ng_, int stride, int row_base_, int pairs,
                                        int tid_, int nthr_) {
    gs = K / kWqGroup;
    sp = static_cast<const uint16_t *>(scales) + kb0 / kWqGroup;
    sc_s = sc_s_;
    ng = ng_;
    gpc = stride;
    N = N_;
    row_base = row_base_;
    n = pairs * ng_;
    tid = tid_;
    nthr = nthr_;
    inv_ng = 1.f / static_cast<float>(ng_);
  }
  __device__ __forceinline__ int batches() const {
    return (n + kScB * nthr - 1) / (kScB * nthr);
  }
  __device__ __forceinline__ void split(int e, int &p, int &g) const {
    p = static_cast<int>((static_cast<float>(e) + 0.5f) * inv_ng);
    g = e - p * ng;
  }
  __device__ __forceinline__ void load(int batch) {
#pragma unroll
    for (int i = 0; i < kScB; ++i) {
      const int e = (batch * kScB + i) * nthr + tid;
      if (e < n) {
        int p, g;
        split(e, p, g);
        const int r = row_base + (p >> 3) * 16 + (p & 7);
        v[i][0] = __ldg(sp + min(r, N - 1) * gs + g);
        v[i][1] = __ldg(sp + min(r + 8, N - 1) * gs + g);
      }
    }
  }
  __device__ __forceinline__ void store(int batch) {
#pragma unroll
    for (int i = 0; i < kScB; ++i) {
      const int e = (batch * kScB + i) * nthr + tid;
      if (e < n) {
        int p, g;
        split(e, p, g);
        sc_s[p * gpc + g] = make_float2(__uint_as_float(uint32_t(v[i][0]) << 16),
                                        __uint_as_float(uint32_t(v[i][1]) << 16));
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Register-ring kernel (any tile count; used for more tokens than the ring takes)
// ---------------------------------------------------------------------------

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
__host__ __device__ constexpr size_t wq_scale_bytes(bool int4, int pairs, int gpc) {
  return int4 ? size_t(pairs) * wq_scale_stride(gpc) * 8 : 0;
}
__host__ __device__ constexpr size_t wq_x_bytes(int gpc, int nt, int M) {
  return size_t(gpc) * kWqGroup * wq_staged_tokens(nt, M) * sizeof(uint16_t);
}
__host__ __device__ constexpr size_t wq_smem_bytes(bool int4, int gpc, int nt, int M) {
  return wq_scale_bytes(int4, kWqRows / 2, gpc) + wq_x_bytes(gpc, nt, M) + size_t(gpc) * 8 * nt * 4;
}

template <bool kInt4, int NT>
__global__ void __launch_bounds__(32 * kWqWarps, NT == 1 ? 3 : 2) wq_gemm_kernel(WqArgs a) {
  using C = WqCfg<kInt4, NT>;
  constexpr int kTok = 8 * NT;  // token slots of the MMA tiles
  extern __shared__ __align__(16) uint8_t wq_smem[];
  const size_t scb = wq_scale_bytes(kInt4, kWqRows / 2, a.gpc);
  float2 *sc_s = reinterpret_cast<float2 *>(wq_smem);  // [kWqRows / 2][stride]
  uint4 *xs = reinterpret_cast<uint4 *>(wq_smem + scb);
  // tokens staged: 8 per tile, or just the M real ones when there is one tile
  const int Mp = wq_staged_tokens(NT, a.M);
  float *xu = reinterpret_cast<float *>(wq_smem + scb + wq_x_bytes(a.gpc, NT, a.M));  // [gpc][kTok]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = lane & 3, rr = lane >> 2;
  const int kb0 = blockIdx.y * a.gpc * kWqGroup;
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

  // INT4 scales: with one token tile the first batch's loads are in flight
  // while x is staged (with more, registers are short and x takes longer)
  constexpr int nthr = 32 * kWqWarps;
  ScaleStage sst(a.scales, sc_s, a.K, a.N, kb0, ng, wq_scale_stride(a.gpc), row_base, kWqRows / 2,
                 tid, nthr);
  constexpr bool kEarly = kInt4 && NT == 1;
  if constexpr (kEarly) sst.load(0);
  // The weights and their scales are constant (see kvq_wq_gemm): only x
  // waits for the work ahead of this kernel on the stream.
  grid_dependency_wait();
  allow_dependents();
  stage_x<kInt4, false>(xs, xu, kTok, a.x, a.K, a.M, Mp, kb0, ng, tid, nthr);
  if constexpr (kInt4) {
    if constexpr (kEarly) sst.store(0);
    for (int b = kEarly ? 1 : 0; b < sst.batches(); ++b) {
      sst.load(b);
      sst.store(b);
    }
  }
  __syncthreads();

  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
  // this lane's B words (token slot t * 8 + rr) and group scales
  const uint4 *xl = xs + (NT == 1 ? min(rr, Mp - 1) : rr) * 4 + c;
  const float2 *scl = sc_s + (warp * 8 + rr) * wq_scale_stride(a.gpc);
  const float *xul = xu + 2 * c;

  for (int g0 = 0; g0 < ng; g0 += C::kDepth) {
#pragma unroll
    for (int d = 0; d < C::kDepth; ++d) {
      const int g = g0 + d;
      if (g >= ng) break;
      constexpr int kAhead = C::kDepth - 1;
      const int nd = (d + kAhead) % C::kDepth;  // register slot of group g + kDepth - 1
      load(g + kAhead, wr0[nd], wr8[nd]);
      float gacc[NT][4];
      group_mma<kInt4, NT>(gacc, wr0[d], wr8[d], xl + g * 4 * Mp * 4, Mp);
      group_fold<kInt4, NT>(acc, gacc, kInt4 ? scl[g] : make_float2(1.f, 1.f), xul + g * kTok);
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

// ---------------------------------------------------------------------------
// TMA-ring kernel (up to 8 tokens, one tile of token slots)
// ---------------------------------------------------------------------------
//
// A CTA covers 64 output channels and a range of k groups; a ninth warp's
// lane 0 streams the CTA's weights into a ring of shared-memory stages with
// the TMA engine, starting before the kernel's grid-dependency wait: one
// stage is 256 consecutive bytes of each of the 64 rows (four INT4 groups or
// two e4m3 groups), copied as four boxes of 64 bytes x 64 rows, each stored
// row after row (a warp's 16-byte reads of two adjacent rows fill all 32
// banks once).  Eight consumer warps: warp w takes rows 16 (w % 4) .. + 15
// of boxes 2 (w / 4) and 2 (w / 4) + 1 (INT4: groups 4k + 2 (w / 4) + {0, 1}
// of stage k; e4m3: both halves of group 2k + w / 4), so every SM keeps 24
// consumer warps busy; the two warps of a row block add their sums at the
// end.  The ring is as deep as three CTAs per SM allow (3 to 8 stages of
// 16 KB), so the bytes in flight do not depend on registers.  Rows past N
// are zero-filled by the copy.  Consumers wait for a stage, read their
// rows' words, compute, and release it; every wait is bounded.  Split-K
// runs as a thread-block cluster along k: every CTA but the first writes
// its partial sums into the first CTA's shared memory (distributed shared
// memory) and arrives on its mbarrier, and the first CTA adds them in rank
// order, so there is no memset, no atomic and the result does not vary
// from run to run.  One token (M == 1) has its own instantiation that keeps
// only the live accumulator elements.

constexpr int kRingWarps = 8;                          // consumer warps
constexpr int kRingRows = 64;                          // output channels per CTA
constexpr int kRingThreads = 32 * (kRingWarps + 1);    // + the producer warp
constexpr int kRingMaxStages = 8;
constexpr int kBoxBytes = 64;                          // a box: 64 bytes x kRingRows rows
constexpr int kStageBoxes = 4;                         // boxes per stage (2 per consumer warp)
constexpr int kStageBytes = kStageBoxes * kBoxBytes * kRingRows;  // 16 KB
constexpr int kRingMaxCluster = 8;
constexpr int kPartSlots = (kRingRows / 16) * 32;       // a float4 per row block and lane

struct RingArgs {
  const void *scales;     // bf16 [N][K/128] or fp32 [N]
  const uint16_t *x;      // bf16 [M][K]
  float *y;               // fp32 [M][N]
  uint32_t *err_word;
  int32_t M, N, K;
  int32_t gpc;            // 128-wide k groups per CTA
  int32_t stages;         // ring depth, 3 .. kRingMaxStages
};

struct RingCtl {
  uint64_t full[kRingMaxStages], empty[kRingMaxStages];
  uint64_t red;  // split K: the other CTAs' sums have arrived (cluster rank 0)
  int fail;
};

// Shared memory of a ring CTA (offsets from a 1024-byte aligned base).
struct RingLayout {
  size_t x, sc, xu, part, recv, ctl, total;
};
// recv: with split K, the cluster's first CTA receives the sums of the other
// ksplit - 1 CTAs there (a float4 per row block and lane each).
__host__ __device__ inline RingLayout ring_layout(bool int4, int stages, int gpc, int M,
                                                  int ksplit) {
  RingLayout L{};
  size_t o = size_t(stages) * kStageBytes;
  L.x = o;
  o += size_t(gpc) * kWqGroup * M * 2;
  L.sc = o;
  o += wq_scale_bytes(int4, kRingRows / 2, gpc);
  L.xu = o;
  o += size_t(gpc) * 8 * 4;
  L.part = o;
  o += size_t(kPartSlots) * 16;
  L.recv = o;
  o += size_t(ksplit > 1 ? ksplit - 1 : 0) * kPartSlots * 16;
  L.ctl = o;
  o += (sizeof(RingCtl) + 15) / 16 * 16;
  L.total = o + 1024;  // room to align the base
  return L;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// may sleep until it completes (or about 1 ms has passed) instead of
// returning at once, so waiting warps issue fewer polls.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return done != 0;
}

// Bounded wait (the bounds of mbar_wait: about 2^31 SM cycles or 2^24
// polls); on timeout the error bit is raised once and the CTA's fail flag
// tells every role to stop.
__device__ __forceinline__ bool ring_wait(RingCtl &ctl, uint64_t *bar, uint32_t parity,
                                          uint32_t *err_word) {
  volatile int *fail = &ctl.fail;
  if (*fail) return false;
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (clock64() - t0 > kWaitCycles) break;
  }
  if (atomicExch(&ctl.fail, 1) == 0) report(err_word, KVQ_ERRBIT_TIMEOUT);
  return false;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The address of `local` (this CTA's shared memory) in CTA `rank` of the
// cluster (every CTA of the kernel lays its shared memory out the same way).
__device__ __forceinline__ uint32_t cluster_addr(const void *local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  return remote;
}

__device__ __forceinline__ void st_cluster_f4(uint32_t remote, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

// Arrival on an mbarrier of another CTA of the cluster, ordered after this
// thread's earlier writes (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar)
               : "memory");
}

// Bounded wait (the bounds of mbar_wait) on a barrier that other CTAs of the
// cluster arrive at (acquire at cluster scope).
__device__ __forceinline__ bool ring_wait_cluster(RingCtl &ctl, uint64_t *bar, uint32_t parity,
                                                  uint32_t *err_word) {
  auto try_wait = [&]() {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
  };
  if (try_wait()) return true;
  const long long t0 = clock64();
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (try_wait()) return true;
    if (clock64() - t0 > kWaitCycles) break;
  }
  if (atomicExch(&ctl.fail, 1) == 0) report(err_word, KVQ_ERRBIT_TIMEOUT);
  return false;
}

template <bool kInt4, bool kOne>
__global__ void __launch_bounds__(kRingThreads, 3)
    wq_ring_kernel(const __grid_constant__ CUtensorMap wmap, RingArgs a) {
  extern __shared__ __align__(128) uint8_t ring_raw[];
  uint8_t *sm = ring_raw + ((1024 - (smem_addr(ring_raw) & 1023)) & 1023);
  const RingLayout L = ring_layout(kInt4, a.stages, a.gpc, a.M, gridDim.y);
  uint8_t *ring = sm;
  uint4 *xs = reinterpret_cast<uint4 *>(sm + L.x);
  float2 *sc_s = reinterpret_cast<float2 *>(sm + L.sc);
  float *xu = reinterpret_cast<float *>(sm + L.xu);
  float4 *part = reinterpret_cast<float4 *>(sm + L.part);
  RingCtl &ctl = *reinterpret_cast<RingCtl *>(sm + L.ctl);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = a.stages, Mp = kOne ? 1 : a.M;  // kOne: M == 1
  const int kb0 = blockIdx.y * a.gpc * kWqGroup;
  const int ng = min(a.gpc, (a.K - kb0) / kWqGroup);
  const int row_base = blockIdx.x * kRingRows;
  constexpr int kGroupBytes = kInt4 ? kWqGroup / 2 : kWqGroup;
  constexpr int kStageCols = kStageBoxes * kBoxBytes;  // bytes of each row per stage
  const int nst = (ng * kGroupBytes + kStageCols - 1) / kStageCols;  // stages

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kRingWarps);
    }
    // split K: every lane of the other CTAs' four lead warps arrives once
    if (gridDim.y > 1) mbar_init(&ctl.red, (gridDim.y - 1) * 32 * (kRingWarps / 2));
    ctl.fail = 0;
    fence_barrier_init();
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&wmap)) : "memory");
  }
  __syncthreads();
  // split K: no CTA may arrive on the first CTA's barrier before it exists
  if (gridDim.y > 1) cluster_sync_all();
  // The weights and their scales are constant (see kvq_wq_gemm): the
  // producer streams them and the consumers load the scales without waiting
  // for the work ahead of this kernel on the stream, so the first stages
  // arrive while that work finishes; only x (and y) wait for it.

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const int c = lane & 3, rr = lane >> 2;
  const int rb = warp & 3, h = warp >> 2;  // row block and box of a consumer warp
  const int rl = rb * 16 + rr;             // this lane's rows in the tile: rl, rl + 8
  if (warp == kRingWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      const int x0 = kInt4 ? kb0 / 2 : kb0;  // byte column of the first stage
      int k = 0, s = 0;
      uint32_t ph = 0;  // parity of the pass over the ring
      bool ok = true;
      for (; k < nst; ++k) {
        if (k >= S && !ring_wait(ctl, &ctl.empty[s], ph ^ 1u, a.err_word)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&ctl.full[s], kStageBytes);
        uint8_t *dst = ring + s * kStageBytes;
#pragma unroll
        for (int b = 0; b < kStageBoxes; ++b)
          tma_load_2d(dst + b * kBoxBytes * kRingRows, &wmap, x0 + k * kStageCols + b * kBoxBytes,
                      row_base, &ctl.full[s], pol);
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) {
        // A wait gave up: let the copies this CTA started land (bounded
        // waits) before it exits, so that none writes into shared memory the
        // SM may already have handed to another CTA.  Only the last S stages
        // can still be in flight.
        for (int j = k > S ? k - S : 0; j < k; ++j)
          mbar_wait(&ctl.full[j % S], static_cast<uint32_t>(j / S) & 1u);
      }
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------- consumers
    constexpr int nthr = 32 * kRingWarps;
    ScaleStage sst(a.scales, sc_s, a.K, a.N, kb0, ng, wq_scale_stride(a.gpc), row_base,
                   kRingRows / 2, tid, nthr);
    if constexpr (kInt4) sst.load(0);
    grid_dependency_wait();
    allow_dependents();
    stage_x<kInt4, !kInt4>(xs, xu, 8, a.x, a.K, a.M, Mp, kb0, ng, tid, nthr);
    if constexpr (kInt4) {
      sst.store(0);
      for (int b = 1; b < sst.batches(); ++b) {
        sst.load(b);
        sst.store(b);
      }
    }
    // the consumer warps only (named barrier 1): the producer is streaming
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kRingWarps) : "memory");

    const uint4 *xl = xs + min(rr, Mp - 1) * 4 + c;
    const float2 *scl = sc_s + (rb * 8 + rr) * wq_scale_stride(a.gpc);
    const float *xul = xu + 2 * c;
    float acc1[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    int s = 0;
    uint32_t ph = 0;
    // this warp's boxes of a stage: kHB = kStageBoxes / 2 of them, from box h kHB
    constexpr int kHB = kStageBoxes / 2;
    for (int k = 0; k < nst; ++k) {
      if (!ring_wait(ctl, &ctl.full[s], ph, a.err_word)) break;
      const uint8_t *st =
          ring + s * kStageBytes + h * kHB * kBoxBytes * kRingRows + rl * kBoxBytes + c * 16;
      uint4 u0[kHB], u8[kHB];
#pragma unroll
      for (int i = 0; i < kHB; ++i) {
        u0[i] = *reinterpret_cast<const uint4 *>(st + i * kBoxBytes * kRingRows);
        u8[i] = *reinterpret_cast<const uint4 *>(st + i * kBoxBytes * kRingRows + 8 * kBoxBytes);
      }
      float gacc[1][4];
      if constexpr (kInt4) {
        // box b of stage k = group kStageBoxes k + b
#pragma unroll
        for (int i = 0; i < kHB; ++i) {
          const int g = kStageBoxes * k + h * kHB + i;
          if (g < ng) {
            const uint32_t a0[4] = {u0[i].x, u0[i].y, u0[i].z, u0[i].w};
            const uint32_t a8[4] = {u8[i].x, u8[i].y, u8[i].z, u8[i].w};
            group_mma<true, 1>(gacc, a0, a8, xl + g * 4 * Mp * 4, Mp);
            group_fold<true, 1, kOne>(acc1, gacc, scl[g], xul + g * 8);
          }
        }
      } else {
        static_assert(kHB == 2, "an e4m3 warp takes both halves of a group");
        // boxes 2h, 2h + 1 = both halves of group 2k + h
        const int g = 2 * k + h;
        if (g < ng) {
          const uint32_t a0[8] = {u0[0].x, u0[0].y, u0[0].z, u0[0].w,
                                  u0[1].x, u0[1].y, u0[1].z, u0[1].w};
          const uint32_t a8[8] = {u8[0].x, u8[0].y, u8[0].z, u8[0].w,
                                  u8[1].x, u8[1].y, u8[1].z, u8[1].w};
          group_mma<false, 1>(gacc, a0, a8, xl + g * 4 * Mp * 4, Mp);
          group_fold<false, 1, kOne>(acc1, gacc, make_float2(1.f, 1.f), xul + g * 8);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.empty[s]);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] = acc1[0][e];
  }

  // ---- the CTA's sums: the two warps of a row block add theirs (box 1's
  // into box 0's); with split K every other CTA of the cluster writes them
  // into the first CTA's shared memory, arrives on its barrier and exits,
  // and the first CTA adds them in rank order and stores.  Every CTA sends,
  // whatever happened above, so the first CTA's wait ends.
  const bool consumer = warp < kRingWarps, lead = warp < kRingWarps / 2;
  if (consumer) {
    if (!lead) part[rb * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    asm volatile("bar.sync 2, %0;" ::"n"(32 * kRingWarps) : "memory");
    if (lead) {
      const float4 v = part[rb * 32 + lane];
      acc[0] += v.x;
      acc[1] += v.y;
      acc[2] += v.z;
      acc[3] += v.w;
    }
  }
  bool store = lead;
  if (gridDim.y > 1 && lead) {
    const uint32_t rank = cluster_rank();
    float4 *recv = reinterpret_cast<float4 *>(sm + L.recv);
    if (rank != 0) {
      st_cluster_f4(cluster_addr(recv + (rank - 1) * kPartSlots + rb * 32 + lane, 0),
                    make_float4(acc[0], acc[1], acc[2], acc[3]));
      mbar_arrive_cluster(cluster_addr(&ctl.red, 0));
      store = false;
    } else if (ring_wait_cluster(ctl, &ctl.red, 0, a.err_word)) {
      for (uint32_t r = 0; r + 1 < gridDim.y; ++r) {
        const float4 v = recv[r * kPartSlots + rb * 32 + lane];
        acc[0] += v.x;
        acc[1] += v.y;
        acc[2] += v.z;
        acc[3] += v.w;
      }
    }
  }
  if (store) {
    const int row0 = row_base + rl;
    float f0 = 1.f, f8 = 1.f;
    if constexpr (!kInt4) {
      const float *fs = static_cast<const float *>(a.scales);
      f0 = fs[min(row0, a.N - 1)];
      f8 = fs[min(row0 + 8, a.N - 1)];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int n = 2 * c + (e & 1);
      const int row = row0 + (e >> 1) * 8;
      if (n < a.M && row < a.N)
        a.y[static_cast<int64_t>(n) * a.N + row] = acc[e] * ((e >> 1) ? f8 : f0);
    }
  }
}

// Self-test of the ring kernel's failure path (kvq_selftest_wait, which = 1):
// as attn_wait_selftest_kernel, with the ring's wait (ring_wait, which sleeps
// between polls) on a barrier that nothing arrives at, then the drain of the
// bulk copy the CTA started.
__global__ void ring_wait_selftest_kernel(const uint32_t *src, uint32_t *err_word,
                                          uint32_t *landed) {
  __shared__ __align__(128) uint32_t buf[16];
  __shared__ RingCtl ctl;
  if (threadIdx.x == 0) {
    mbar_init(&ctl.full[0], 1);
    mbar_init(&ctl.full[1], 1);
    ctl.fail = 0;
    fence_barrier_init();
  }
  __syncthreads();
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&ctl.full[0], sizeof(buf));
    bulk_g2s(buf, src, sizeof(buf), &ctl.full[0]);
  }
  const bool ok = ring_wait(ctl, &ctl.full[1], 0, err_word);  // nothing arrives on full[1]
  if (threadIdx.x == 0) {
    const bool drained = mbar_wait(&ctl.full[0], 0);
    *landed = (!ok && drained) ? buf[0] : 0u;
  }
}

kvq_status selftest_ring_wait(const uint32_t *src, uint32_t *err_word, uint32_t *landed,
                              cudaStream_t stream) {
  const cudaError_t e =
      launch_dependent(ring_wait_selftest_kernel, dim3(1), dim3(64), 0, stream, src, err_word,
                       landed);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------

using WqFn = void (*)(WqArgs);
using RingFn = void (*)(CUtensorMap, RingArgs);

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

// Opt a kernel into a shared-memory budget once per device (slot = kernel
// variant), outside any stream capture after the first call.
bool wq_smem_opt_in(const void *fn, int slot, size_t bytes) {
  constexpr int kMaxDev = 64;
  static std::atomic<bool> done[kMaxDev][20];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  if (done[dev][slot].load(std::memory_order_acquire)) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return false;
  done[dev][slot].store(true, std::memory_order_release);
  return true;
}

// Resident CTAs per SM of a register-ring kernel variant at a dynamic
// shared-memory size (cached per device, variant and size: the split choice
// asks for several sizes on every call).
bool wq_occupancy(WqFn fn, int slot, size_t smem, int *occ) {
  static std::mutex mu;
  static std::unordered_map<uint64_t, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t key = (static_cast<uint64_t>(dev) << 40) | (static_cast<uint64_t>(slot) << 32) | smem;
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) {
      *occ = it->second;
      return true;
    }
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fn, 32 * kWqWarps, smem) != cudaSuccess)
    return false;
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = *occ;
  return true;
}

// Shared memory one CTA may use so that three of them fit on an SM (cached
// per device).
size_t smem_per_cta3() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int sm_bytes = 0, reserved = 0;
    if (cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess)
      return 0;
    v = sm_bytes / 3 - reserved;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return static_cast<size_t>(v);
}

// 2-D map over the weights [N rows][row_bytes bytes], boxes of 64 bytes x 64
// rows, no swizzle; rows past N read as zeros.
bool encode_weight_map(CUtensorMap *map, const void *w, int64_t row_bytes, int N) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(N)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[2] = {kBoxBytes, kRingRows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(w), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The ring kernel's plan for one call: k split (cluster size), groups per
// CTA, ring depth, shared memory.  False when the shape does not suit it.
struct RingPlan {
  int ksplit, gpc, stages;
  size_t smem;
};
bool ring_plan(bool int4, int M, int N, int K, int sms, RingPlan *p) {
  // one tile of 8 token slots; from three tokens on (below) only where the k
  // split that the staged x needs still fits one wave
  if (M > 8) return false;
  constexpr int kPerSm = 3;
  const size_t budget = smem_per_cta3();
  const int groups = K / kWqGroup;
  const int tiles = (N + kRingRows - 1) / kRingRows;
  const int slots = kPerSm * sms;
  // the staged x of a CTA stays small (<= 24 KB), and the grid fills the
  // GPU's slots once where it can, splitting k into clusters of up to 8
  constexpr size_t kXMax = 24 * 1024;
  auto x_bytes = [&](int g) { return size_t(g) * kWqGroup * M * 2; };
  auto gpc_of = [&](int k) { return (groups + k - 1) / k; };
  int ksplit = 1;
  while (ksplit <= kRingMaxCluster && x_bytes(gpc_of(ksplit)) > kXMax) ++ksplit;
  if (ksplit > kRingMaxCluster) return false;
  // measured: with three or more tokens, a split forced past one wave (the
  // 28672 x 5120 projection) loses to the register ring (INT4 153 -> 174 us
  // at three tokens), while the smaller projections of a layer gain 7-20%
  if (M > 2 && static_cast<int64_t>(tiles) * ksplit > slots) return false;
  // (a larger cluster also needs more room for the partial sums it sends:
  // grow only while three ring stages still fit)
  for (int k = ksplit + 1; k <= kRingMaxCluster && k <= groups; ++k)
    if (static_cast<int64_t>(tiles) * k <= slots &&
        ring_layout(int4, 3, gpc_of(k), M, k).total <= budget)
      ksplit = k;
  const int gpc = gpc_of(ksplit);
  ksplit = (groups + gpc - 1) / gpc;  // no CTA without groups
  int stages = kRingMaxStages;
  while (stages > 2 && ring_layout(int4, stages, gpc, M, ksplit).total > budget) --stages;
  const size_t smem = ring_layout(int4, stages, gpc, M, ksplit).total;
  if (smem > budget || stages < 3) return false;
  *p = RingPlan{ksplit, gpc, stages, smem};
  return true;
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_wq_gemm(int32_t w_dtype, const void *w, const void *scales,
                                  const void *x, float *y, int32_t M, int32_t N, int32_t K,
                                  uint32_t *err_word, kvq_stream_t stream) {
  if (w_dtype != KVQ_W_INT4 && w_dtype != KVQ_W_E4M3) return KVQ_ERR_INVALID_ARG;
  if (!w || !scales || !x || !y) return KVQ_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < kWqGroup) return KVQ_ERR_INVALID_ARG;
  if (M > 64 || K % kWqGroup) return KVQ_ERR_UNSUPPORTED;
  if (!aligned16(w) || !aligned16(x) ||
      (reinterpret_cast<uintptr_t>(y) & 3) || (reinterpret_cast<uintptr_t>(scales) & 3))
    return KVQ_ERR_INVALID_ARG;
  const bool int4 = w_dtype == KVQ_W_INT4;
  const int nt = (M + 7) / 8;
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int groups = K / kWqGroup;
  const int64_t row_bytes = int4 ? K / 2 : K;

  // one token tile: the TMA-ring kernel
  RingPlan rp;
  CUtensorMap wmap;
  if (ring_plan(int4, M, N, K, sms, &rp) && encode_weight_map(&wmap, w, row_bytes, N)) {
    const RingFn fn = int4 ? (M == 1 ? wq_ring_kernel<true, true> : wq_ring_kernel<true, false>)
                           : (M == 1 ? wq_ring_kernel<false, true> : wq_ring_kernel<false, false>);
    if (!wq_smem_opt_in(reinterpret_cast<const void *>(fn), 16 + (int4 ? 1 : 0) + (M == 1 ? 2 : 0),
                        smem_per_cta3()))
      return KVQ_ERR_CUDA;
    RingArgs ra{scales, static_cast<const uint16_t *>(x), y, err_word, M, N, K, rp.gpc, rp.stages};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kRingRows - 1) / kRingRows, rp.ksplit);
    cfg.blockDim = dim3(kRingThreads);
    cfg.dynamicSmemBytes = rp.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = rp.ksplit;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = rp.ksplit > 1 ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, fn, wmap, ra);
    return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
  }

  // otherwise the register-ring kernel.  Split K: shared memory sets the
  // most groups a CTA can stage x for; among the splits from there, take the
  // one with the least (waves of resident CTAs) x (groups per CTA), the
  // fewest splits on a tie (occupancy depends on the staged x).
  const WqFn fn = int4 ? pick_wq<true>(nt) : pick_wq<false>(nt);
  const int row_tiles = (N + kWqRows - 1) / kWqRows;
  auto smem_of = [&](int gpc) { return wq_smem_bytes(int4, gpc, nt, M); };
  const int slot = int4 ? nt - 1 : 8 + nt - 1;
  if (!wq_smem_opt_in(reinterpret_cast<const void *>(fn), slot, kWqSmemMax)) return KVQ_ERR_CUDA;
  int gpc_max = groups;
  while (gpc_max > 1 && smem_of(gpc_max) > kWqSmemMax) --gpc_max;
  const int ks_min = (groups + gpc_max - 1) / gpc_max;
  int gpc = gpc_max, ksplit = ks_min;
  int64_t best = -1;
  for (int ks = ks_min; ks <= groups && ks <= ks_min + 16; ++ks) {
    const int g = (groups + ks - 1) / ks;
    const int kse = (groups + g - 1) / g;  // no CTA without groups
    if (kse != ks) continue;
    int occ = 0;
    if (!wq_occupancy(fn, slot, smem_of(g), &occ)) return KVQ_ERR_CUDA;
    const int64_t slots = static_cast<int64_t>(occ > 0 ? occ : 1) * sms;
    const int64_t waves = (static_cast<int64_t>(row_tiles) * kse + slots - 1) / slots;
    const int64_t cost = waves * g;
    if (best < 0 || cost < best) {
      best = cost;
      gpc = g;
      ksplit = kse;
    }
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
