// Tensor-core split kernel for an e4m3 cache with head_dim 128 (included by
// decode_attn.cu; shares its plan and partial-merge conventions).
//
// A CTA works on rows of (request, group of HG kv heads).  One stage is 16
// cached tokens of all HG heads of the group: the pool layout
// [page][kv head][slot][dim] makes those 16 x HG x 128 bytes one contiguous
// block per page, so a single tiled TMA copy (cp.async.bulk.tensor, 4-D map,
// box [128 dims][16 slots][HG heads][1 page], 128-byte swizzle) stages all of
// K and one stages all of V.  Consumer warp w owns kv head w of the group:
// it keeps that head's G query rows, softmax state and output accumulators in
// registers, so no consumer warp ever waits for another except when a row
// split across CTAs is merged.  Warp HG is the producer.
//
// q.k and p.v run on the tensor cores with mma.sync m16n8k16 (f16 in, fp32
// accumulate).  Every e4m3 value is exactly representable in f16 and the
// query is bf16 scaled by a power of two into f16 range, so q.k is exact up
// to fp32 accumulation; the softmax weights are rounded to f16 (relative
// error 2^-11) for p.v.
//
// Fragment layout of one consumer warp (16 tokens, lane = 4g+t):
//   S[head][token]   = Q[head][dim] * K^T[dim][token]    (2 n-tiles of 8 tokens)
//       k-step s (16 dims): thread t supplies dims 32t+4s .. 32t+4s+3, so its
//       B operand is one 32-bit word of its K row (no shuffles, no permutes);
//   O^T[dim][head]  += V^T[dim][token] * P^T[token][head] (8 m-tiles of 16 dims)
//       the C fragment of S is the B operand P^T as is; thread (g,t) builds
//       V^T from rows 2t,2t+1,2t+8,2t+9 at dims 16g..16g+15 with byte permutes;
//       m-tile i, row g is dim 16g+2i and row g+8 is dim 16g+2i+1.
// Query heads occupy rows 0..G-1 of S (G <= 8) and columns 0..G-1 of O^T.
// A row r of the 16-token tile sits at byte r*128 of the head's 2 KB block
// with its 16-byte chunk c stored at chunk c ^ (r % 8) (TMA 128-byte swizzle).
//
// The bf16 variant (the comparison kernel for an uncompressed cache) stages
// each head as two such 128-byte-wide planes (dims 0-63 and 64-127, two TMA
// boxes), runs q.k as exact bf16 MMAs (thread t supplies dims 16t..16t+15 of
// each plane) and gets V^T straight from ldmatrix.trans (m-tile i is dims
// 16i..16i+15: row g is dim 16i+g, row g+8 is dim 16i+8+g).  The softmax
// weights are split into a bf16 head and a bf16 remainder, p = hi + lo, and
// p.v runs as two MMAs, so the weights keep about 16 significant bits.
#pragma once

namespace kvq {

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z,
                                            int w, uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar)),
      "l"(pol)
      : "memory");
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {  // low half -> .x
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const uint8_t *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(p)));
}

__device__ __forceinline__ uint32_t f32x2_to_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

constexpr int kTile = 16;  // tokens per stage of the tensor-core kernel
constexpr float kPScale = 128.f;  // scale of the e4m3 kernel's softmax weights
constexpr int kPlane = kTile * 128;  // 2 KB: 16 tokens x 128 bytes of one head

template <int G, int HG, bool kBf16>
struct HgCfg {
  static constexpr int D = 128;
  static constexpr int PLANES = kBf16 ? 2 : 1;          // 128-byte-wide planes per head
  static constexpr int PLANE = HG * kPlane;             // one plane of the head group
  static constexpr int TILES = 1;                       // 16-token tiles per stage
  static constexpr int TILE_BYTES = PLANES * PLANE;     // one tile of K (or V)
  static constexpr int KV_BYTES = TILES * TILE_BYTES;   // one stage of K (or V)
  // stages in the ring: 192 KB of K+V in flight per SM for 8-head groups
  static constexpr int NS = kBf16 ? 3 : ((HG * G >= 64) ? 5 : 6);
  static constexpr int Q_BYTES = HG * G * D * 2;        // the group's query rows (bf16)
  static constexpr int KPART = part_stride(G, D);       // floats per kv head in a slot
  static constexpr int PART = HG * KPART;               // floats per partial slot
  static constexpr size_t off_k = 0;                    // 1024-byte aligned
  static constexpr size_t off_v = off_k + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_q = off_v + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_ctl = off_q + 2ull * Q_BYTES;
  static constexpr size_t bytes = off_ctl + sizeof(Ctrl) + 1024;  // + alignment slack
  static_assert(G >= 1 && G <= 8 && HG >= 1 && HG <= 8, "group sizes");
  static_assert(KV_BYTES % 1024 == 0 && off_q % 1024 == 0 && off_ctl % 16 == 0, "alignment");
  static_assert(NS <= kMaxStages && TILES <= 2, "control block");
  static_assert(bytes <= 227 * 1024, "shared memory");
};

// One consumer warp's state for its kv head.
struct HeadState {
  uint32_t qa0[8], qa2[8];  // Q A-fragments (rows gq), per k-step
  float o[8][4];            // O^T accumulators, per 16-dim m-tile
  float m_run, l_run;       // softmax state of head gq (lanes with gq < G)
  float qk_scale;
};

// Rows of S and columns of O^T in the e4m3 kernel (the MMA's 8 query-head
// slots): slot h < G is query head h and carries the f16 weights p_hi; when
// 2G <= 8, slot G + h holds a copy of head h's query row, so the lanes of that
// row compute the same scores and weights and supply the remainders
// p_lo = f16(p - p_hi) to column G + h, which is added to column h at the
// segment's end.  G = 8 has no free slot and runs p_lo through a second MMA.
template <int G>
__device__ __forceinline__ int slot_head(int gq) {
  return gq < G ? gq : ((2 * G <= 8 && gq < 2 * G) ? gq - G : -1);
}

// q rows of this warp's kv head (bf16 in shared memory) -> f16 fragments,
// scaled by 2^e so that the largest |q| of the head group sits in [2^14, 2^15).
template <int G>
__device__ __forceinline__ void load_q(HeadState &st, const uint8_t *qhead, float q_scale, int gq,
                                       int tq) {
  float qf[32];
  float qmax = 0.f;
  const int hq = slot_head<G>(gq);
  if (hq >= 0) {
    const uint8_t *qs = qhead + (hq * 128 + 32 * tq) * 2;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 w4 = lds128(qs + 16 * c);
      bf16x2_to_f32(w4.x, qf + 8 * c);
      bf16x2_to_f32(w4.y, qf + 8 * c + 2);
      bf16x2_to_f32(w4.z, qf + 8 * c + 4);
      bf16x2_to_f32(w4.w, qf + 8 * c + 6);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) qmax = fmaxf(qmax, fabsf(qf[i]));
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) qf[i] = 0.f;
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o2));
  int e = (qmax > 0.f && qmax < INFINITY) ? 14 - ilogbf(qmax) : 0;
  e = max(-100, min(100, e));
  const float up = ldexpf(1.f, e);
  st.qk_scale = q_scale * ldexpf(1.f, -e);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    st.qa0[s] = f32x2_to_f16x2(qf[4 * s] * up, qf[4 * s + 1] * up);
    st.qa2[s] = f32x2_to_f16x2(qf[4 * s + 2] * up, qf[4 * s + 3] * up);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
  st.m_run = -INFINITY;
  st.l_run = 0.f;
}

// One 16-token tile of one kv head: ks / vs are the head's 2 KB swizzled
// blocks, ntok (1..16) the valid tokens.
template <int G>
__device__ __forceinline__ void tile_step(HeadState &st, const uint8_t *ks, const uint8_t *vs,
                                          int ntok, int gq, int tq) {
  // ---- S = Q K^T for tokens gq (n-tile 0) and 8+gq (n-tile 1); row % 8 == gq
  const uint8_t *k0 = ks + gq * 128;
  const uint8_t *k1 = k0 + 8 * 128;
  const int c0 = ((2 * tq) ^ gq) * 16, c1 = ((2 * tq + 1) ^ gq) * 16;
  const uint4 k0a = lds128(k0 + c0), k0b = lds128(k0 + c1);
  const uint4 k1a = lds128(k1 + c0), k1b = lds128(k1 + c1);
  const uint32_t kw0[8] = {k0a.x, k0a.y, k0a.z, k0a.w, k0b.x, k0b.y, k0b.z, k0b.w};
  const uint32_t kw1[8] = {k1a.x, k1a.y, k1a.z, k1a.w, k1b.x, k1b.y, k1b.z, k1b.w};
  // V^T rows 2t, 2t+1, 2t+8, 2t+9 at logical chunk gq, read with K so that
  // their latency hides under q.k
  const uint8_t *vr = vs + (2 * tq) * 128;
  uint4 va = lds128(vr + ((gq ^ (2 * tq)) * 16));
  uint4 vb = lds128(vr + 128 + ((gq ^ (2 * tq + 1)) * 16));
  uint4 vc = lds128(vr + 8 * 128 + ((gq ^ (2 * tq)) * 16));
  uint4 vd = lds128(vr + 9 * 128 + ((gq ^ (2 * tq + 1)) * 16));
  // even and odd k-steps accumulate apart: four independent chains of four
  // MMAs instead of two of eight (a consumer warp is bound by dependency
  // latency, not by issue), summed at the end
  float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
  float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int s = 0; s < 8; s += 2) {
    mma_16816(s0, st.qa0[s], 0u, st.qa2[s], 0u, e4m3x2_to_f16x2(kw0[s] & 0xFFFFu),
              e4m3x2_to_f16x2(kw0[s] >> 16));
    mma_16816(s1, st.qa0[s], 0u, st.qa2[s], 0u, e4m3x2_to_f16x2(kw1[s] & 0xFFFFu),
              e4m3x2_to_f16x2(kw1[s] >> 16));
    mma_16816(s2, st.qa0[s + 1], 0u, st.qa2[s + 1], 0u, e4m3x2_to_f16x2(kw0[s + 1] & 0xFFFFu),
              e4m3x2_to_f16x2(kw0[s + 1] >> 16));
    mma_16816(s3, st.qa0[s + 1], 0u, st.qa2[s + 1], 0u, e4m3x2_to_f16x2(kw1[s + 1] & 0xFFFFu),
              e4m3x2_to_f16x2(kw1[s + 1] >> 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s0[i] += s2[i];
    s1[i] += s3[i];
  }
  // ---- online softmax for head gq over the 16 tokens (log2 domain)
  const bool row_ok = slot_head<G>(gq) >= 0;
  const int t0 = 2 * tq, t1 = 8 + 2 * tq;
  const float x00 = (row_ok && t0 < ntok) ? s0[0] * st.qk_scale : -INFINITY;
  const float x01 = (row_ok && t0 + 1 < ntok) ? s0[1] * st.qk_scale : -INFINITY;
  const float x10 = (row_ok && t1 < ntok) ? s1[0] * st.qk_scale : -INFINITY;
  const float x11 = (row_ok && t1 + 1 < ntok) ? s1[1] * st.qk_scale : -INFINITY;
  float mx = fmaxf(fmaxf(x00, x01), fmaxf(x10, x11));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const bool grow = mx > st.m_run + kRescaleThreshold;
  if (__any_sync(0xffffffffu, grow)) {
    const float f = grow ? exp2f(st.m_run - mx) : 1.f;  // 0 when m_run is -inf
    if (grow) {
      st.m_run = mx;
      st.l_run *= f;
    }
    // O^T columns 2t and 2t+1 belong to the slots whose rows live in lanes 8t, 8t+4
    const float fa = __shfl_sync(0xffffffffu, f, 8 * tq);
    const float fb = __shfl_sync(0xffffffffu, f, 8 * tq + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.o[i][0] *= fa;
      st.o[i][1] *= fb;
      st.o[i][2] *= fa;
      st.o[i][3] *= fb;
    }
  }
  // The weights are 2^(x - m_run) * kPScale: the same factor is in l_run, so
  // it cancels (exactly: a power of two), and it puts the largest weight
  // (1..2^8 under lazy rescaling) high in f16's range.  p = hi + lo in f16
  // for p.v: one f16 alone leaves a relative error of 2^-11 per weight, which
  // a short context with a large V value turns into more than the 1e-3
  // tolerance; with the remainder the error is ~2^-22 relative (down to
  // weights 2^-10 below the largest, below which lo is subnormal and the
  // absolute error stays under 2^-25).
  const float p00 = x00 == -INFINITY ? 0.f : fast_exp2(x00 - st.m_run) * kPScale;
  const float p01 = x01 == -INFINITY ? 0.f : fast_exp2(x01 - st.m_run) * kPScale;
  const float p10 = x10 == -INFINITY ? 0.f : fast_exp2(x10 - st.m_run) * kPScale;
  const float p11 = x11 == -INFINITY ? 0.f : fast_exp2(x11 - st.m_run) * kPScale;
  st.l_run += (p00 + p01) + (p10 + p11);
  const uint32_t ph0 = f32x2_to_f16x2(p00, p01), ph1 = f32x2_to_f16x2(p10, p11);
  const float2 h0 = f16x2_to_f32x2(ph0), h1 = f16x2_to_f32x2(ph1);
  const uint32_t pl0 = f32x2_to_f16x2(p00 - h0.x, p01 - h0.y);
  const uint32_t pl1 = f32x2_to_f16x2(p10 - h1.x, p11 - h1.y);
  // B operand of p.v: lane (g, t) supplies column g, the remainders in the
  // copied slots (weights are 0 in slots without a head)
  const uint32_t b0 = gq < G ? ph0 : pl0, b1 = gq < G ? ph1 : pl1;

  // ---- O^T += V^T P^T
  if (ntok < kTile) {  // tail: cached bytes past the sequence may be anything
    const uint4 z = make_uint4(0, 0, 0, 0);
    if (t0 >= ntok) va = z;
    if (t0 + 1 >= ntok) vb = z;
    if (t1 >= ntok) vc = z;
    if (t1 + 1 >= ntok) vd = z;
  }
  const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
  const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;  // bytes (a.b, b.b, a.b+1, b.b+1)
    const uint32_t x = prmt(wa[i >> 1], wb[i >> 1], sel);
    const uint32_t y = prmt(wc[i >> 1], wd[i >> 1], sel);
    const uint32_t a0 = e4m3x2_to_f16x2(x & 0xFFFFu), a1 = e4m3x2_to_f16x2(x >> 16);
    const uint32_t a2 = e4m3x2_to_f16x2(y & 0xFFFFu), a3 = e4m3x2_to_f16x2(y >> 16);
    mma_16816(st.o[i], a0, a1, a2, a3, b0, b1);
    if constexpr (2 * G > 8) mma_16816(st.o[i], a0, a1, a2, a3, pl0, pl1);
  }
}


// Two consecutive 16-token tiles of one segment in one pass: tile a (ksa /
// vsa) is full, tile b holds ntok_b (1..16) valid tokens.  One softmax update
// covers the 32 tokens, and q.k runs as eight independent chains of four.
template <int G>
__device__ __forceinline__ void tile_step2(HeadState &st, const uint8_t *ksa, const uint8_t *vsa,
                                           const uint8_t *ksb, const uint8_t *vsb, int ntok_b,
                                           int gq, int tq) {
  const int c0 = ((2 * tq) ^ gq) * 16, c1 = ((2 * tq + 1) ^ gq) * 16;
  uint32_t kw[4][8];  // [2 * tile + n-tile][word]: rows gq (n-tile 0) and 8 + gq (n-tile 1)
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint8_t *kr = (j < 2 ? ksa : ksb) + (gq + 8 * (j & 1)) * 128;
    const uint4 x = lds128(kr + c0), y = lds128(kr + c1);
    kw[j][0] = x.x;
    kw[j][1] = x.y;
    kw[j][2] = x.z;
    kw[j][3] = x.w;
    kw[j][4] = y.x;
    kw[j][5] = y.y;
    kw[j][6] = y.z;
    kw[j][7] = y.w;
  }
  float sc[4][4], so[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) sc[j][i] = so[j][i] = 0.f;
#pragma unroll
  for (int s = 0; s < 8; s += 2) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      mma_16816(sc[j], st.qa0[s], 0u, st.qa2[s], 0u, e4m3x2_to_f16x2(kw[j][s] & 0xFFFFu),
                e4m3x2_to_f16x2(kw[j][s] >> 16));
      mma_16816(so[j], st.qa0[s + 1], 0u, st.qa2[s + 1], 0u,
                e4m3x2_to_f16x2(kw[j][s + 1] & 0xFFFFu), e4m3x2_to_f16x2(kw[j][s + 1] >> 16));
    }
  }
  // ---- online softmax over the 32 tokens
  const bool row_ok = slot_head<G>(gq) >= 0;
  float x[4][2];
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = 8 * (j & 1) + 2 * tq + e;  // token within its tile
      const bool ok = row_ok && (j < 2 || t < ntok_b);
      x[j][e] = ok ? (sc[j][e] + so[j][e]) * st.qk_scale : -INFINITY;
      mx = fmaxf(mx, x[j][e]);
    }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const bool grow = mx > st.m_run + kRescaleThreshold;
  if (__any_sync(0xffffffffu, grow)) {
    const float f = grow ? exp2f(st.m_run - mx) : 1.f;
    if (grow) {
      st.m_run = mx;
      st.l_run *= f;
    }
    const float fa = __shfl_sync(0xffffffffu, f, 8 * tq);
    const float fb = __shfl_sync(0xffffffffu, f, 8 * tq + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.o[i][0] *= fa;
      st.o[i][1] *= fb;
      st.o[i][2] *= fa;
      st.o[i][3] *= fb;
    }
  }
  uint32_t bw[4], lw[4];  // B-operand words (hi or, in the copied slots, lo) and lo
  float lsum = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float p0 = x[j][0] == -INFINITY ? 0.f : fast_exp2(x[j][0] - st.m_run) * kPScale;
    const float p1 = x[j][1] == -INFINITY ? 0.f : fast_exp2(x[j][1] - st.m_run) * kPScale;
    lsum += p0 + p1;
    const uint32_t ph = f32x2_to_f16x2(p0, p1);
    const float2 h = f16x2_to_f32x2(ph);
    const uint32_t pl = f32x2_to_f16x2(p0 - h.x, p1 - h.y);
    bw[j] = gq < G ? ph : pl;
    lw[j] = pl;
  }
  st.l_run += lsum;
  // ---- O^T += V^T P^T for each tile
#pragma unroll
  for (int tb = 0; tb < 2; ++tb) {
    const uint8_t *vr = (tb == 0 ? vsa : vsb) + (2 * tq) * 128;
    uint4 va = lds128(vr + ((gq ^ (2 * tq)) * 16));
    uint4 vb = lds128(vr + 128 + ((gq ^ (2 * tq + 1)) * 16));
    uint4 vc = lds128(vr + 8 * 128 + ((gq ^ (2 * tq)) * 16));
    uint4 vd = lds128(vr + 9 * 128 + ((gq ^ (2 * tq + 1)) * 16));
    if (tb == 1 && ntok_b < kTile) {
      const uint4 z = make_uint4(0, 0, 0, 0);
      const int t0 = 2 * tq, t1 = 8 + 2 * tq;
      if (t0 >= ntok_b) va = z;
      if (t0 + 1 >= ntok_b) vb = z;
      if (t1 >= ntok_b) vc = z;
      if (t1 + 1 >= ntok_b) vd = z;
    }
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
    const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
      const uint32_t xx = prmt(wa[i >> 1], wb[i >> 1], sel);
      const uint32_t yy = prmt(wc[i >> 1], wd[i >> 1], sel);
      const uint32_t a0 = e4m3x2_to_f16x2(xx & 0xFFFFu), a1 = e4m3x2_to_f16x2(xx >> 16);
      const uint32_t a2 = e4m3x2_to_f16x2(yy & 0xFFFFu), a3 = e4m3x2_to_f16x2(yy >> 16);
      mma_16816(st.o[i], a0, a1, a2, a3, bw[2 * tb], bw[2 * tb + 1]);
      if constexpr (2 * G > 8) mma_16816(st.o[i], a0, a1, a2, a3, lw[2 * tb], lw[2 * tb + 1]);
    }
  }
}

// bf16 query rows -> bf16 fragments (exact, no scaling); thread t supplies
// dims 16t+4s.. of plane 0 (k-steps 0-3) and 64+16t+4(s-4).. (k-steps 4-7).
template <int G>
__device__ __forceinline__ void load_q_bf16(HeadState &st, const uint8_t *qhead, float q_scale,
                                            int gq, int tq) {
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int dim = (s < 4) ? 16 * tq + 4 * s : 64 + 16 * tq + 4 * (s - 4);
    if (gq < G) {
      st.qa0[s] = *reinterpret_cast<const uint32_t *>(qhead + (gq * 128 + dim) * 2);
      st.qa2[s] = *reinterpret_cast<const uint32_t *>(qhead + (gq * 128 + dim + 2) * 2);
    } else {
      st.qa0[s] = st.qa2[s] = 0u;
    }
  }
  st.qk_scale = q_scale;
#pragma unroll
  for (int i = 0; i < 8; ++i) st.o[i][0] = st.o[i][1] = st.o[i][2] = st.o[i][3] = 0.f;
  st.m_run = -INFINITY;
  st.l_run = 0.f;
}

// One 16-token tile of one kv head with a bf16 cache: k0/k1 (v0/v1) are the
// head's two 2 KB planes (dims 0-63, 64-127).
template <int G>
__device__ __forceinline__ void tile_step_bf16(HeadState &st, const uint8_t *k0, const uint8_t *k1,
                                               const uint8_t *v0, const uint8_t *v1, int ntok,
                                               int gq, int tq, int lane) {
  float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int j = 0; j < 2; ++j) {  // n-tile j: token 8j+gq, row % 8 == gq
    const int r = 8 * j + gq;
    const int ca = ((2 * tq) ^ gq) * 16, cb = ((2 * tq + 1) ^ gq) * 16;
    const uint4 a = lds128(k0 + r * 128 + ca), b = lds128(k0 + r * 128 + cb);
    const uint4 c = lds128(k1 + r * 128 + ca), d = lds128(k1 + r * 128 + cb);
    const uint32_t w[16] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w,
                            c.x, c.y, c.z, c.w, d.x, d.y, d.z, d.w};
#pragma unroll
    for (int s = 0; s < 8; ++s) mma_16816_bf16(sc[j], st.qa0[s], 0u, st.qa2[s], 0u, w[2 * s], w[2 * s + 1]);
  }
  const bool row_ok = gq < G;
  const int t0 = 2 * tq, t1 = 8 + 2 * tq;
  const float x00 = (row_ok && t0 < ntok) ? sc[0][0] * st.qk_scale : -INFINITY;
  const float x01 = (row_ok && t0 + 1 < ntok) ? sc[0][1] * st.qk_scale : -INFINITY;
  const float x10 = (row_ok && t1 < ntok) ? sc[1][0] * st.qk_scale : -INFINITY;
  const float x11 = (row_ok && t1 + 1 < ntok) ? sc[1][1] * st.qk_scale : -INFINITY;
  float mx = fmaxf(fmaxf(x00, x01), fmaxf(x10, x11));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const bool grow = mx > st.m_run + kRescaleThreshold;
  if (__any_sync(0xffffffffu, grow)) {
    const float f = grow ? exp2f(st.m_run - mx) : 1.f;
    if (grow) {
      st.m_run = mx;
      st.l_run *= f;
    }
    const float fa = __shfl_sync(0xffffffffu, f, 8 * tq);
    const float fb = __shfl_sync(0xffffffffu, f, 8 * tq + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      st.o[i][0] *= fa;
      st.o[i][1] *= fb;
      st.o[i][2] *= fa;
      st.o[i][3] *= fb;
    }
  }
  const float p00 = x00 == -INFINITY ? 0.f : fast_exp2(x00 - st.m_run);
  const float p01 = x01 == -INFINITY ? 0.f : fast_exp2(x01 - st.m_run);
  const float p10 = x10 == -INFINITY ? 0.f : fast_exp2(x10 - st.m_run);
  const float p11 = x11 == -INFINITY ? 0.f : fast_exp2(x11 - st.m_run);
  st.l_run += (p00 + p01) + (p10 + p11);
  // p = hi + lo, both bf16
  const uint32_t h0 = f32x2_to_bf16x2(p00, p01), h1 = f32x2_to_bf16x2(p10, p11);
  const uint32_t l0 = f32x2_to_bf16x2(p00 - __uint_as_float(h0 << 16),
                                      p01 - __uint_as_float(h0 & 0xFFFF0000u));
  const uint32_t l1 = f32x2_to_bf16x2(p10 - __uint_as_float(h1 << 16),
                                      p11 - __uint_as_float(h1 & 0xFFFF0000u));

  // ---- O^T += V^T P^T; ldmatrix.trans lane l addresses row (l%8) + 8*(l>=16)
  // of 16-byte chunk 2(i%4) + ((l/8)&1) in plane i/4
  const int lrow = (lane & 7) + ((lane >> 4) << 3);
  const int lchunk = (lane >> 3) & 1;
  const bool tail = ntok < kTile;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint8_t *vp = (i < 4 ? v0 : v1) + lrow * 128 + (((2 * (i & 3) + lchunk) ^ (lrow & 7)) * 16);
    uint32_t a[4];
    ldsm_x4_trans(a, vp);
    if (tail) {  // cached values past the sequence may be anything: zero them
      const uint32_t m0 = (t0 < ntok ? 0xFFFFu : 0u) | (t0 + 1 < ntok ? 0xFFFF0000u : 0u);
      const uint32_t m1 = (t1 < ntok ? 0xFFFFu : 0u) | (t1 + 1 < ntok ? 0xFFFF0000u : 0u);
      a[0] &= m0;
      a[1] &= m0;
      a[2] &= m1;
      a[3] &= m1;
    }
    mma_16816_bf16(st.o[i], a[0], a[1], a[2], a[3], h0, h1);
    mma_16816_bf16(st.o[i], a[0], a[1], a[2], a[3], l0, l1);
  }
}

// Output dims held by thread (g,t) in m-tile i: rows g and g+8 of O^T.
template <bool kBf16>
__device__ __forceinline__ int dim_lo(int i, int gq) { return kBf16 ? 16 * i + gq : 16 * gq + 2 * i; }
template <bool kBf16>
__device__ __forceinline__ int dim_hi(int i, int gq) {
  return kBf16 ? 16 * i + 8 + gq : 16 * gq + 2 * i + 1;
}

template <int G, int HG, bool kBf16>
__global__ void __launch_bounds__(32 * (HG + 1))
    split_hg_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, SplitArgs a) {
  using C = HgCfg<G, HG, kBf16>;
  constexpr int NS = C::NS;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // TMA 128-byte swizzle needs 1024-byte aligned destinations
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint8_t *kbuf = smem + C::off_k;
  uint8_t *vbuf = smem + C::off_v;
  uint8_t *qbuf = smem + C::off_q;
  Ctrl &ctl = *reinterpret_cast<Ctrl *>(smem + C::off_ctl);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    ctrl_init(ctl, NS, HG);
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
  }
  __syncthreads();

  // Where this CTA starts.  Everything ahead of this kernel on the stream
  // (the tag check that wrote the abort mask, whatever wrote the lengths;
  // for a large batch the plan) is complete and visible once
  // grid_dependency_wait() returns.  For up to 32 x (HG + 1) x kSelfSchedPer
  // requests there is no plan kernel: every CTA works out the schedule
  // itself and does the plan's other work for the requests without work that
  // fall to it (zeroed rows, their descriptors, length errors).  Larger
  // batches read the plan's schedule.
  const int c = blockIdx.x;
  const int groups = a.Hkv / HG;  // rows per request
  SchedStart sc;
  grid_dependency_wait();
  if (self_schedule<32 * (HG + 1), kSelfSchedPer>(a, groups, kTile, ctl, sc))
    zero_requests<C::D>(a, groups, ctl);
  else
    sc = plan_schedule(a, groups);
  allow_dependents();  // the combine grid may become resident and wait
  const int S = sc.S, U = sc.U;

  if (warp == HG) {
    // ------------------------------------------------------------- producer
    const long long cap = static_cast<long long>(a.MP) * a.P;
    long long u = static_cast<long long>(c) * U;
    const long long u_end = min(u + U, static_cast<long long>(S));
    // request b: p0 units before it, length L, units_b units in each of its rows
    int b = sc.b, p0 = sc.p0, L = sc.L, units_b = sc.ub, grp = 0, s = 0;
    if (u < u_end && units_b > 0) {
      const int r = static_cast<int>(u - p0);
      grp = r / units_b;
      s = r % units_b;
    } else {
      u = u_end;  // no work (the owner of a unit always has units)
    }
    const uint64_t pol = policy_evict_first();
    // block-table window of the current request: lane i holds logical page
    // win+i (cur) and win+32+i (nxt, loaded one window ahead)
    int win_b = -1, win = 0, cur = -1, nxt = -1;
    const int32_t *bt_row = a.block_table;
    auto bt_load = [&](int lp) -> int { return lp < a.MP ? __ldg(bt_row + lp) : -1; };
    uint32_t g = 0, nseg = 0, nq = 0;  // stages, segments and query copies issued
    bool ok = true;
    while (ok && u < u_end && b < a.B) {
      const int row = b * groups + grp;
      const long long ur = static_cast<long long>(p0) + static_cast<long long>(grp) * units_b;
      const int c_lo = static_cast<int>(ur / U);
      const int nparts = static_cast<int>((ur + units_b - 1) / U) - c_lo + 1;
      const int seg_units = static_cast<int>(min(static_cast<long long>(units_b - s), u_end - u));
      const int t_begin = s * kTile;
      const int t_end = min((s + seg_units) * kTile, L);
      constexpr int kStageTok = kTile * C::TILES;
      const int nstages = (t_end - t_begin + kStageTok - 1) / kStageTok;
      const int lp0 = t_begin / a.P;
      if (b != win_b || lp0 < win || lp0 >= win + 32) {
        win_b = b;
        win = lp0;
        bt_row = a.block_table + static_cast<int64_t>(b) * a.MP;
        cur = bt_load(win + lane);
        nxt = bt_load(win + 32 + lane);
      }
      // the CTA that holds the row's first unit writes the row's descriptor
      if (lane == 0 && s == 0) a.desc[row] = make_int4(c_lo, nparts, b, 0);
      // the group's query rows, double-buffered per segment
      const int qs = nseg & 1;
      if (lane == 0) {
        bool w_ok = true;
        if (nseg >= 2) w_ok = ctl_wait(ctl, &ctl.qempty[qs], ((nseg >> 1) - 1) & 1, a.err_word);
        if (w_ok) {
          mbar_arrive_expect_tx(&ctl.qfull[qs], C::Q_BYTES);
          bulk_g2s(qbuf + qs * C::Q_BYTES,
                   a.q + (static_cast<int64_t>(b) * a.Hq + grp * HG * G) * C::D, C::Q_BYTES,
                   &ctl.qfull[qs]);
          ++nq;
        }
      }
      for (int st = 0; st < nstages; ++st, ++g) {
        const int slot = g % NS;
        bool waited = true;
        if (lane == 0 && g >= NS)
          waited = ctl_wait(ctl, &ctl.empty[slot], ((g / NS) - 1) & 1, a.err_word);
        ok = __shfl_sync(0xffffffffu, waited ? 1 : 0, 0) != 0 &&
             !*reinterpret_cast<volatile int *>(&ctl.fail);
        if (!ok) break;
        const int tok0 = t_begin + st * kStageTok;
        const int ntok = min(kStageTok, t_end - tok0);
        const int lp_first = tok0 / a.P;
        while (lp_first >= win + 32) {  // slide the window by 32 pages
          win += 32;
          cur = nxt;
          nxt = bt_load(win + 32 + lane);
        }
        if constexpr (C::TILES == 1) {
          const int page = __shfl_sync(0xffffffffu, cur, lp_first - win);
          const bool bad_page = page < 0 || page >= a.num_pages;
          if (lane == 0) {
            if (bad_page) report(a.err_word, KVQ_ERRBIT_PAGE);
            ctl.desc[slot][0] = make_int4(
                row, tok0,
                ntok | (st == 0 ? kFirst : 0) | (st == nstages - 1 ? kLast : 0) |
                    (bad_page ? kBad : 0),
                nparts);
            ctl.desc[slot][1] = make_int4(row + c, c_lo, b, grp | (qs << 16));
            mbar_arrive_expect_tx(&ctl.full[slot], bad_page ? 0u : 2u * C::KV_BYTES);
            if (!bad_page) {
              const int y = tok0 % a.P;
#pragma unroll
              for (int pl = 0; pl < C::PLANES; ++pl) {  // plane pl: 128 bytes from x = 64*pl
                const uint32_t off = slot * C::KV_BYTES + pl * C::PLANE;
                tma_load_4d(kbuf + off, &kmap, 64 * pl, y, grp * HG, page, &ctl.full[slot], pol);
                tma_load_4d(vbuf + off, &vmap, 64 * pl, y, grp * HG, page, &ctl.full[slot], pol);
              }
            }
          }
        } else {
          // tile k of the stage: tokens tok0+16k.., logical page (tok0+16k)/P,
          // which lies in [win, win+64): cur or nxt
          int tile_page[C::TILES];
          int bad_bits = 0;
#pragma unroll
          for (int k = 0; k < C::TILES; ++k) {
            const int lpk = (tok0 + kTile * k) / a.P - win;
            const int from_cur = __shfl_sync(0xffffffffu, cur, lpk & 31);
            const int from_nxt = __shfl_sync(0xffffffffu, nxt, lpk & 31);
            tile_page[k] = -1;
            if (kTile * k < ntok) {
              const int page = lpk < 32 ? from_cur : from_nxt;
              if (page < 0 || page >= a.num_pages)
                bad_bits |= kBad << k;
              else
                tile_page[k] = page;
            }
          }
          if (lane == 0) {
            if (bad_bits) report(a.err_word, KVQ_ERRBIT_PAGE);
            ctl.desc[slot][0] = make_int4(
                row, tok0,
                ntok | (st == 0 ? kFirst : 0) | (st == nstages - 1 ? kLast : 0) | bad_bits,
                nparts);
            ctl.desc[slot][1] = make_int4(row + c, c_lo, b, grp | (qs << 16));
            uint32_t tx = 0;
#pragma unroll
            for (int k = 0; k < C::TILES; ++k)
              if (tile_page[k] >= 0) tx += 2u * C::TILE_BYTES;
            mbar_arrive_expect_tx(&ctl.full[slot], tx);
#pragma unroll
            for (int k = 0; k < C::TILES; ++k) {
              if (tile_page[k] < 0) continue;
              const int y = (tok0 + kTile * k) % a.P;
#pragma unroll
              for (int pl = 0; pl < C::PLANES; ++pl) {
                const uint32_t off = slot * C::KV_BYTES + k * C::TILE_BYTES + pl * C::PLANE;
                tma_load_4d(kbuf + off, &kmap, 64 * pl, y, grp * HG, tile_page[k],
                            &ctl.full[slot], pol);
                tma_load_4d(vbuf + off, &vmap, 64 * pl, y, grp * HG, tile_page[k],
                            &ctl.full[slot], pol);
              }
            }
          }
        }
        __syncwarp();
      }
      ++nseg;
      u += seg_units;
      s = 0;
      if (++grp == groups) {
        grp = 0;
        p0 += units_b * groups;
        // the next request with work (aborted, empty or invalid ones own no units)
        units_b = 0;
        while (units_b == 0 && ++b < a.B) units_b = request_units(a, b, cap, kTile, L);
      }
    }
    // tell the consumers there is nothing more
    if (ok) {
      const int slot = g % NS;
      bool waited = true;
      if (lane == 0 && g >= NS)
        waited = ctl_wait(ctl, &ctl.empty[slot], ((g / NS) - 1) & 1, a.err_word);
      if (lane == 0 && waited) {
        ctl.desc[slot][0] = make_int4(-1, 0, 0, 0);
        mbar_arrive(&ctl.full[slot]);
      }
    } else if (lane == 0) {
      // A wait gave up: before the CTA exits, let the copies it started land
      // (bounded waits), so that none writes into shared memory the SM may
      // already have handed to another CTA.  Only the last NS stages and the
      // last two query copies can still be in flight (a slot is reused only
      // after its previous copy completed and was consumed).
      drain_copies(ctl.full, NS, g, ctl.qfull, nq);
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  const int gq = lane >> 2;  // fragment row group
  const int tq = lane & 3;   // thread in group
  HeadState hs;
  uint32_t g = 0, nseg = 0;
  bool seg_bad = false;

  while (true) {
    const int slot = g % NS;
    if (!ctl_wait(ctl, &ctl.full[slot], (g / NS) & 1, a.err_word)) break;
    int4 d0 = ctl.desc[slot][0];
    if (d0.x < 0) break;
    int4 d1 = ctl.desc[slot][1];
    const int ntok = d0.z & 0xFFFF;
    if (d0.z & kFirst) {
      const int qs = (d1.w >> 16) & 1;
      if (!ctl_wait(ctl, &ctl.qfull[qs], (nseg >> 1) & 1, a.err_word)) break;
      if constexpr (kBf16)
        load_q_bf16<G>(hs, qbuf + qs * C::Q_BYTES + warp * G * C::D * 2, a.q_scale, gq, tq);
      else
        load_q<G>(hs, qbuf + qs * C::Q_BYTES + warp * G * C::D * 2, a.q_scale, gq, tq);
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.qempty[qs]);
      seg_bad = false;
    }
    bool paired = false;
    if constexpr (!kBf16 && C::TILES == 1 && 2 * G > 8) {
      // a stage that does not end its segment is full and followed by one of
      // the same segment: take the two together when neither has a bad page
      // (G = 8 only: its p.v runs two MMAs per tile, and the pair's shared
      // softmax pays for them; for G <= 4 it measured 0-2% slower)
      if (!(d0.z & (kLast | kBad))) {
        const int slot2 = (g + 1) % NS;
        if (!ctl_wait(ctl, &ctl.full[slot2], ((g + 1) / NS) & 1, a.err_word)) break;
        const int4 e0 = ctl.desc[slot2][0];
        if (!(e0.z & kBad)) {
          tile_step2<G>(hs, kbuf + slot * C::KV_BYTES + warp * kPlane,
                        vbuf + slot * C::KV_BYTES + warp * kPlane,
                        kbuf + slot2 * C::KV_BYTES + warp * kPlane,
                        vbuf + slot2 * C::KV_BYTES + warp * kPlane, e0.z & 0xFFFF, gq, tq);
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&ctl.empty[slot]);
            mbar_arrive(&ctl.empty[slot2]);
          }
          d0 = e0;
          d1 = ctl.desc[slot2][1];
          ++g;
          paired = true;
        }
      }
    }
    if (paired) {
      // both stages done (and released) above
    } else if constexpr (C::TILES == 1) {
      seg_bad |= (d0.z & kBad) != 0;
      if (!(d0.z & kBad)) {
        const uint8_t *kt = kbuf + slot * C::KV_BYTES + warp * kPlane;
        const uint8_t *vt = vbuf + slot * C::KV_BYTES + warp * kPlane;
        if constexpr (kBf16)
          tile_step_bf16<G>(hs, kt, kt + C::PLANE, vt, vt + C::PLANE, ntok, gq, tq, lane);
        else
          tile_step<G>(hs, kt, vt, ntok, gq, tq);
      }
    } else {
#pragma unroll
      for (int k = 0; k < C::TILES; ++k) {
        const int nt = ntok - kTile * k;
        if (nt <= 0) break;
        if (d0.z & (kBad << k)) {
          seg_bad = true;
          continue;
        }
        const uint8_t *kt = kbuf + slot * C::KV_BYTES + k * C::TILE_BYTES + warp * kPlane;
        const uint8_t *vt = vbuf + slot * C::KV_BYTES + k * C::TILE_BYTES + warp * kPlane;
        if constexpr (kBf16)
          tile_step_bf16<G>(hs, kt, kt + C::PLANE, vt, vt + C::PLANE, min(nt, kTile), gq, tq,
                            lane);
        else
          tile_step<G>(hs, kt, vt, min(nt, kTile), gq, tq);
      }
    }
    if (!paired) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.empty[slot]);
    }

    if (d0.z & kLast) {
      const int nparts = d0.w, pslot = d1.x, b = d1.z;
      const int kvh = (d1.w & 0xFFFF) * HG + warp;
      if constexpr (!kBf16 && 2 * G <= 8) {  // add the p_lo columns G.. to columns 0..
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if constexpr (G == 1) {
            hs.o[i][0] += hs.o[i][1];
            hs.o[i][2] += hs.o[i][3];
          } else {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              hs.o[i][k] += __shfl_down_sync(0xffffffffu, hs.o[i][k], G / 2);
          }
        }
      }
      hs.l_run += __shfl_xor_sync(0xffffffffu, hs.l_run, 1);
      hs.l_run += __shfl_xor_sync(0xffffffffu, hs.l_run, 2);
      // heads 2t and 2t+1 of the O^T columns: their m, l live in lanes 8t, 8t+4
      const float la = __shfl_sync(0xffffffffu, hs.l_run, 8 * tq);
      const float lb = __shfl_sync(0xffffffffu, hs.l_run, 8 * tq + 4);
      const float ma = __shfl_sync(0xffffffffu, hs.m_run, 8 * tq);
      const float mb = __shfl_sync(0xffffffffu, hs.m_run, 8 * tq + 4);
      const int ha = 2 * tq, hb = 2 * tq + 1;
      float *out = a.out + (static_cast<int64_t>(b) * a.Hq + kvh * G) * C::D;
      if (nparts == 1) {
        // a row with a page outside the pool is stored as zeros, selected
        // rather than scaled by 0: its other pages may hold NaN codes
        const float sa = seg_bad ? 0.f : a.v_scale / la;
        const float sb = seg_bad ? 0.f : a.v_scale / lb;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int dl = dim_lo<kBf16>(i, gq), dh = dim_hi<kBf16>(i, gq);
          if constexpr (!kBf16) {  // dims dl, dl+1: one 8-byte store
            if (ha < G)
              *reinterpret_cast<float2 *>(out + ha * C::D + dl) =
                  seg_bad ? make_float2(0.f, 0.f) : make_float2(hs.o[i][0] * sa, hs.o[i][2] * sa);
            if (hb < G)
              *reinterpret_cast<float2 *>(out + hb * C::D + dl) =
                  seg_bad ? make_float2(0.f, 0.f) : make_float2(hs.o[i][1] * sb, hs.o[i][3] * sb);
          } else {
            if (ha < G) {
              out[ha * C::D + dl] = seg_bad ? 0.f : hs.o[i][0] * sa;
              out[ha * C::D + dh] = seg_bad ? 0.f : hs.o[i][2] * sa;
            }
            if (hb < G) {
              out[hb * C::D + dl] = seg_bad ? 0.f : hs.o[i][1] * sb;
              out[hb * C::D + dh] = seg_bad ? 0.f : hs.o[i][3] * sb;
            }
          }
        }
      } else {
        // partial of this head: acc[G][D], then m[G], l[G]
        float *mine = a.part + static_cast<int64_t>(pslot) * C::PART +
                      static_cast<int64_t>(warp) * C::KPART;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int dl = dim_lo<kBf16>(i, gq), dh = dim_hi<kBf16>(i, gq);
          if constexpr (!kBf16) {  // dims dl, dl+1: one 8-byte store
            if (ha < G)
              *reinterpret_cast<float2 *>(mine + ha * C::D + dl) =
                  make_float2(hs.o[i][0], hs.o[i][2]);
            if (hb < G)
              *reinterpret_cast<float2 *>(mine + hb * C::D + dl) =
                  make_float2(hs.o[i][1], hs.o[i][3]);
          } else {
            if (ha < G) {
              mine[ha * C::D + dl] = hs.o[i][0];
              mine[ha * C::D + dh] = hs.o[i][2];
            }
            if (hb < G) {
              mine[hb * C::D + dl] = hs.o[i][1];
              mine[hb * C::D + dh] = hs.o[i][3];
            }
          }
        }
        if (gq == 0) {  // l = -1 marks a part that met a page outside the pool
          if (ha < G) {
            mine[G * C::D + ha] = ma;
            mine[G * C::D + G + ha] = seg_bad ? -1.f : la;
          }
          if (hb < G) {
            mine[G * C::D + hb] = mb;
            mine[G * C::D + G + hb] = seg_bad ? -1.f : lb;
          }
        }
      }
      ++nseg;
    }
    ++g;
  }
}

}  // namespace kvq
