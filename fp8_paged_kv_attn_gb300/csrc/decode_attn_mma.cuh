// Tensor-core split kernel for an e4m3 cache with head_dim 128 (included by
// decode_attn.cu; shares its plan, workspace, partial format and combine).
//
// Same producer/consumer structure as the CUDA-core kernel, but:
//  * pages are staged with tiled TMA copies (cp.async.bulk.tensor, 4-D map
//    over the pool [page][kv head][slot][dim], 128-byte swizzle), so the
//    fragment loads below are free of shared-memory bank conflicts;
//  * q.k and p.v run on the tensor cores with mma.sync m16n8k16 (f16 in,
//    fp32 accumulate).  Every e4m3 value is exactly representable in f16 and
//    the query is bf16 scaled by a power of two into f16 range, so q.k is
//    exact up to fp32 accumulation; the softmax weights are rounded to f16
//    (relative error 2^-11) for p.v.
//
// Fragment layout of one consumer warp (16 tokens of the stage, lane = 4g+t):
//   S[head][token]   = Q[head][dim] * K^T[dim][token]    (2 n-tiles of 8 tokens)
//       k-step s (16 dims): thread t supplies dims 32t+4s .. 32t+4s+3, so its
//       B operand is one 32-bit word of its K row (no shuffles, no permutes);
//   O^T[dim][head]  += V^T[dim][token] * P^T[token][head] (8 m-tiles of 16 dims)
//       the C fragment of S is the B operand P^T as is; thread (g,t) builds
//       V^T from rows 2t,2t+1,2t+8,2t+9 at dims 16g..16g+15 with byte permutes;
//       m-tile i, row g is dim 16g+2i and row g+8 is dim 16g+2i+1.
// Query heads occupy rows 0..G-1 of S (G <= 8) and columns 0..G-1 of O^T.
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

__device__ __forceinline__ uint4 lds128(const uint8_t *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

template <int G>
struct MmaCfg {
  static constexpr int D = 128;
  static constexpr int TS = 64;  // tokens per stage: 4 consumer warps x 16
  static constexpr int NS = kStages;
  static constexpr int NCW = kConsumerWarps;
  static constexpr int KV_BYTES = TS * D;  // one stage of K (or V), e4m3
  static constexpr int Q_BYTES = G * D * 2;
  static constexpr int RED = G * D + (2 * G + 3) / 4 * 4;
  static constexpr int PART = G * (D + 2);
  static constexpr size_t off_k = 0;  // 1024-byte aligned (128-byte swizzle atoms)
  static constexpr size_t off_v = off_k + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_q = off_v + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_red = off_q + static_cast<size_t>(NS) * Q_BYTES;
  static constexpr size_t off_desc = off_red + 2ull * NCW * RED * sizeof(float);
  static constexpr size_t off_bar = off_desc + NS * sizeof(int4);
  static constexpr size_t bytes = off_bar + (2 * NS + 2) * sizeof(uint64_t) + 16 + 1024;
  static_assert(G >= 1 && G <= 8, "query heads per kv head");
  static_assert(KV_BYTES % 1024 == 0 && off_red % 16 == 0 && off_desc % 16 == 0, "alignment");
  static_assert(TS == NCW * 16 && kTokQuant % TS == 0, "stage mapping");
};

template <int G>
__global__ void __launch_bounds__(32 * (kConsumerWarps + 1), 2)
    split_mma_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, SplitArgs a) {
  using C = MmaCfg<G>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  // TMA 128-byte swizzle needs 1024-byte aligned destinations
  uint8_t *smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint8_t *kbuf = smem + C::off_k;
  uint8_t *vbuf = smem + C::off_v;
  uint8_t *qbuf = smem + C::off_q;
  float *red = reinterpret_cast<float *>(smem + C::off_red);
  int4 *desc = reinterpret_cast<int4 *>(smem + C::off_desc);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::off_bar);
  uint64_t *empty = full + C::NS;
  uint64_t *fin = empty + C::NS;
  volatile int *fail = reinterpret_cast<volatile int *>(fin + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NCW);
    }
    mbar_init(&fin[0], C::NCW);
    mbar_init(&fin[1], C::NCW);
    *fail = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == C::NCW) {
    // ------------------------------------------------------------- producer
    const int total_items = a.hdr[1];
    const uint32_t page_box = static_cast<uint32_t>(a.P) * C::D;  // bytes of one page box
    const uint64_t pol = policy_evict_first();
    uint32_t g = 0;
    bool ok = true;
    while (ok) {
      int item = 0;
      if (lane == 0) item = atomicAdd(a.hdr_counter, 1);
      item = __shfl_sync(0xffffffffu, item, 0);
      const bool done = item >= total_items;
      int4 it = make_int4(0, 0, 0, 0);
      if (!done) it = a.items[item];
      const int nstages = done ? 1 : (it.w - it.z + C::TS - 1) / C::TS;
      for (int st = 0; st < nstages; ++st, ++g) {
        const int slot = g % C::NS;
        if (lane == 0 && g >= C::NS) {
          if (*fail || !mbar_wait(&empty[slot], ((g / C::NS) - 1) & 1)) {
            if (!*fail) report(a.err_word, KVQ_ERRBIT_TIMEOUT);
            *fail = 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, *fail, 0) == 0;
        if (!ok) break;
        if (done) {
          if (lane == 0) {
            desc[slot] = make_int4(-1, 0, 0, 0);
            mbar_arrive(&full[slot]);
          }
          ok = false;
          break;
        }
        const int b = it.x, kvh = it.y;
        const int tok0 = it.z + st * C::TS;
        const int ntok = min(C::TS, it.w - tok0);
        const int npages = (ntok + a.P - 1) / a.P;  // page_size <= TS
        int page = -1;
        if (lane < npages) {
          page = __ldg(a.block_table + static_cast<int64_t>(b) * a.MP + tok0 / a.P + lane);
          if (page < 0 || page >= a.num_pages) {
            atomicOr(a.bad + b, 1);
            report(a.err_word, KVQ_ERRBIT_PAGE);
            page = -1;
          }
        }
        const unsigned valid_mask = __ballot_sync(0xffffffffu, page >= 0);
        const bool first = st == 0, last = st == nstages - 1;
        if (lane == 0) {
          desc[slot] = make_int4(item, b * a.Hkv + kvh, tok0,
                                 ntok | (first ? kFirst : 0) | (last ? kLast : 0));
          const uint32_t tx = 2u * __popc(valid_mask) * page_box + (first ? C::Q_BYTES : 0u);
          mbar_arrive_expect_tx(&full[slot], tx);
          if (first)
            bulk_g2s(qbuf + slot * C::Q_BYTES,
                     a.q + (static_cast<int64_t>(b) * a.Hq + kvh * G) * C::D, C::Q_BYTES,
                     &full[slot]);
        }
        __syncwarp();  // the transaction count is armed before any page copy is issued
        if (page >= 0) {
          const uint32_t dst = lane * page_box;
          tma_load_4d(kbuf + slot * C::KV_BYTES + dst, &kmap, 0, 0, kvh, page, &full[slot], pol);
          tma_load_4d(vbuf + slot * C::KV_BYTES + dst, &vmap, 0, 0, kvh, page, &full[slot], pol);
        }
        __syncwarp();
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  const int gq = lane >> 2;  // fragment row group
  const int tq = lane & 3;   // thread in group
  uint32_t qa0[8], qa2[8];   // Q A-fragments (rows gq), per k-step
  float o[8][4];             // O^T accumulators, per 16-dim m-tile
  float m_run = -INFINITY, l_run = 0.f;  // softmax state of head gq (lanes with gq < G)
  float qk_scale = 0.f;
  uint32_t g = 0, n_items_done = 0;
  int cur_item = 0;

  while (true) {
    const int slot = g % C::NS;
    if (*fail || !mbar_wait(&full[slot], (g / C::NS) & 1)) {
      if (!*fail) report(a.err_word, KVQ_ERRBIT_TIMEOUT);
      *fail = 1;
      break;
    }
    const int4 d = desc[slot];
    if (d.x < 0) break;
    const int ntok = d.w & 0xFFFF;
    if (d.w & kFirst) {
      cur_item = d.x;
      // query rows gq < G, dims 32t..32t+31 (bf16) -> f16 scaled by 2^e so the
      // largest |q| of the group sits in [2^14, 2^15)
      float qf[32];
      float qmax = 0.f;
      if (gq < G) {
        const uint8_t *qs = qbuf + slot * C::Q_BYTES + (gq * C::D + 32 * tq) * 2;
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
      qk_scale = a.q_scale * ldexpf(1.f, -e);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        qa0[s] = f32x2_to_f16x2(qf[4 * s] * up, qf[4 * s + 1] * up);
        qa2[s] = f32x2_to_f16x2(qf[4 * s + 2] * up, qf[4 * s + 3] * up);
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      m_run = -INFINITY;
      l_run = 0.f;
    }

    const int tl0 = warp * 16;  // this warp's first token in the stage
    if (tl0 < ntok) {
      const uint8_t *ks = kbuf + slot * C::KV_BYTES;
      const uint8_t *vs = vbuf + slot * C::KV_BYTES;
      // ---- S = Q K^T for tokens tl0+gq (n-tile 0) and tl0+8+gq (n-tile 1);
      // swizzled 16-byte chunk c of row r sits at chunk c ^ (r % 8), r % 8 == gq
      const uint8_t *k0 = ks + (tl0 + gq) * C::D;
      const uint8_t *k1 = k0 + 8 * C::D;
      const int c0 = ((2 * tq) ^ gq) * 16, c1 = ((2 * tq + 1) ^ gq) * 16;
      const uint4 k0a = lds128(k0 + c0), k0b = lds128(k0 + c1);
      const uint4 k1a = lds128(k1 + c0), k1b = lds128(k1 + c1);
      const uint32_t kw0[8] = {k0a.x, k0a.y, k0a.z, k0a.w, k0b.x, k0b.y, k0b.z, k0b.w};
      const uint32_t kw1[8] = {k1a.x, k1a.y, k1a.z, k1a.w, k1b.x, k1b.y, k1b.z, k1b.w};
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        mma_16816(s0, qa0[s], 0u, qa2[s], 0u, e4m3x2_to_f16x2(kw0[s] & 0xFFFFu),
                  e4m3x2_to_f16x2(kw0[s] >> 16));
        mma_16816(s1, qa0[s], 0u, qa2[s], 0u, e4m3x2_to_f16x2(kw1[s] & 0xFFFFu),
                  e4m3x2_to_f16x2(kw1[s] >> 16));
      }
      // ---- online softmax for head gq over this warp's 16 tokens (log2 domain)
      const bool row_ok = gq < G;
      const int t0 = tl0 + 2 * tq, t1 = tl0 + 8 + 2 * tq;
      const float x00 = (row_ok && t0 < ntok) ? s0[0] * qk_scale : -INFINITY;
      const float x01 = (row_ok && t0 + 1 < ntok) ? s0[1] * qk_scale : -INFINITY;
      const float x10 = (row_ok && t1 < ntok) ? s1[0] * qk_scale : -INFINITY;
      const float x11 = (row_ok && t1 + 1 < ntok) ? s1[1] * qk_scale : -INFINITY;
      float mx = fmaxf(fmaxf(x00, x01), fmaxf(x10, x11));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const bool grow = mx > m_run + kRescaleThreshold;
      if (__any_sync(0xffffffffu, grow)) {
        const float f = grow ? exp2f(m_run - mx) : 1.f;  // 0 when m_run is -inf
        if (grow) {
          m_run = mx;
          l_run *= f;
        }
        // O^T columns 2t and 2t+1 belong to heads whose rows live in lanes 8t, 8t+4
        const float fa = __shfl_sync(0xffffffffu, f, 8 * tq);
        const float fb = __shfl_sync(0xffffffffu, f, 8 * tq + 4);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[i][0] *= fa;
          o[i][1] *= fb;
          o[i][2] *= fa;
          o[i][3] *= fb;
        }
      }
      const float p00 = x00 == -INFINITY ? 0.f : fast_exp2(x00 - m_run);
      const float p01 = x01 == -INFINITY ? 0.f : fast_exp2(x01 - m_run);
      const float p10 = x10 == -INFINITY ? 0.f : fast_exp2(x10 - m_run);
      const float p11 = x11 == -INFINITY ? 0.f : fast_exp2(x11 - m_run);
      l_run += (p00 + p01) + (p10 + p11);
      const uint32_t pb0 = f32x2_to_f16x2(p00, p01);
      const uint32_t pb1 = f32x2_to_f16x2(p10, p11);

      // ---- O^T += V^T P^T: rows tl0+2t, +1, +8, +9 at logical chunk gq
      const uint8_t *vr = vs + (tl0 + 2 * tq) * C::D;
      uint4 va = lds128(vr + ((gq ^ (2 * tq)) * 16));
      uint4 vb = lds128(vr + C::D + ((gq ^ (2 * tq + 1)) * 16));
      uint4 vc = lds128(vr + 8 * C::D + ((gq ^ (2 * tq)) * 16));
      uint4 vd = lds128(vr + 9 * C::D + ((gq ^ (2 * tq + 1)) * 16));
      if (tl0 + 16 > ntok) {  // tail: cached bytes past the sequence may be anything
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
        mma_16816(o[i], e4m3x2_to_f16x2(x & 0xFFFFu), e4m3x2_to_f16x2(x >> 16),
                  e4m3x2_to_f16x2(y & 0xFFFFu), e4m3x2_to_f16x2(y >> 16), pb0, pb1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);

    if (d.w & kLast) {
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
      l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
      const int rb = n_items_done & 1;
      float *my = red + (rb * C::NCW + warp) * C::RED;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int dim = 16 * gq + 2 * i;
        if (2 * tq < G)
          *reinterpret_cast<float2 *>(my + (2 * tq) * C::D + dim) = make_float2(o[i][0], o[i][2]);
        if (2 * tq + 1 < G)
          *reinterpret_cast<float2 *>(my + (2 * tq + 1) * C::D + dim) =
              make_float2(o[i][1], o[i][3]);
      }
      if (tq == 0 && gq < G) {
        my[G * C::D + gq] = m_run;
        my[G * C::D + G + gq] = l_run;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&fin[rb]);
      if (*fail || !mbar_wait(&fin[rb], (n_items_done >> 1) & 1)) {
        if (!*fail) report(a.err_word, KVQ_ERRBIT_TIMEOUT);
        *fail = 1;
        break;
      }
      const float *rr = red + rb * C::NCW * C::RED;
      float *out = a.part + static_cast<int64_t>(cur_item) * C::PART;
      const int ctid = warp * 32 + lane;
      for (int idx = ctid; idx < G * C::D + G; idx += C::NCW * 32) {
        const int h = idx < G * C::D ? idx / C::D : idx - G * C::D;
        float mstar = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) mstar = fmaxf(mstar, rr[w * C::RED + G * C::D + h]);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) {
          const float mw = rr[w * C::RED + G * C::D + h];
          const float f = mw == -INFINITY ? 0.f : exp2f(mw - mstar);
          const float v = idx < G * C::D ? rr[w * C::RED + idx] : rr[w * C::RED + G * C::D + G + h];
          sum = fmaf(f, v, sum);
        }
        if (idx < G * C::D) {
          out[idx] = sum;
        } else {
          out[G * C::D + h] = mstar;
          out[G * C::D + G + h] = sum;
        }
      }
      ++n_items_done;
    }
    ++g;
  }
}

}  // namespace kvq
