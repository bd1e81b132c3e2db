// kvq_decode_attn: single-query paged decode attention over an e4m3 (or bf16)
// KV cache, converting the cache on read.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "KV 缓存量化": the decode pool's cache is e4m3; its FP8 attention kernel
// converts the cache while reading it (the reason FP8 is a little slower per
// token than the BF16 kernel it is compared with in the section's table).
// The pages give no kernel design; this one is written for GB300:
//
//   plan     1 CTA: per-request split counts so that the whole batch becomes
//            about kItemTarget equal work items of T tokens (T a multiple of
//            64), plus a flat item list (b, kv head, token range).
//   split    persistent, (#SMs x resident CTAs) CTAs of 5 warps.  Warp 4 is a
//            producer: it takes items from an atomic counter, reads the block
//            table and issues 1-D bulk copies (TMA engine) of each page's
//            contiguous [slot][dim] chunk for this kv head into a 4-stage
//            shared-memory ring (mbarrier-tracked, L2 evict-first).  Warps 0-3
//            consume the ring: e4m3 -> fp32 in registers, q.k for the G query
//            heads that share the kv head (each cached element is converted
//            once and used G times), online softmax in the log2 domain with
//            lazy rescaling, p.v accumulation; at the end of an item the four
//            warps merge and write one partial (acc[G][D], m[G], l[G]).
//   combine  1 CTA per (request, kv head): log-sum-exp merge of the request's
//            partials, times v_scale; aborted / empty / invalid rows are 0.
//
// Every wait is bounded (see mbar_wait); a wait that gives up raises
// KVQ_ERRBIT_TIMEOUT and the CTA leaves its loop.
#include <cfloat>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kvq_internal.h"

namespace kvq {

constexpr int kItemTarget = 4096;  // work items a call aims for
constexpr int kTokQuant = 64;      // item boundaries are multiples of this
constexpr int kConsumerWarps = 4;
constexpr int kStages = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------

struct WsLayout {
  size_t hdr, n_items, base, bad, items, part, total;
  int64_t max_items;
};

inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline WsLayout ws_layout(int B, int Hq, int Hkv, int D) {
  WsLayout w;
  const int G = Hq / Hkv;
  w.max_items = kItemTarget + static_cast<int64_t>(B) * Hkv;
  size_t off = 0;
  w.hdr = off;
  off = round256(off + 64 * sizeof(int32_t));
  w.n_items = off;
  off = round256(off + static_cast<size_t>(B) * sizeof(int32_t));
  w.base = off;
  off = round256(off + static_cast<size_t>(B) * sizeof(int32_t));
  w.bad = off;
  off = round256(off + static_cast<size_t>(B) * sizeof(int32_t));
  w.items = off;
  off = round256(off + static_cast<size_t>(w.max_items) * sizeof(int4));
  w.part = off;
  off = round256(off + static_cast<size_t>(w.max_items) * G * (D + 2) * sizeof(float));
  w.total = off;
  return w;
}

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------

struct PlanArgs {
  const int32_t *seq_lens;
  const uint8_t *abort_mask;
  int32_t *hdr, *n_items, *base, *bad;
  int4 *items;
  uint32_t *err_word;
  int32_t B, Hkv, MP, P;
};

__global__ void __launch_bounds__(1024) plan_kernel(PlanArgs a) {
  __shared__ long long s_sum[32];
  __shared__ int s_scan[32];
  __shared__ int s_carry;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = nt >> 5;
  const long long cap = static_cast<long long>(a.MP) * a.P;

  // tokens of every request that will be read
  long long sum = 0;
  for (int b = tid; b < a.B; b += nt) {
    const int L = a.seq_lens[b];
    const bool aborted = a.abort_mask && a.abort_mask[b];
    if (!aborted) {
      if (L < 0 || L > cap)
        report(a.err_word, KVQ_ERRBIT_SEQLEN);
      else
        sum += L;
    }
  }
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane == 0) s_sum[warp] = sum;
  if (tid == 0) s_carry = 0;
  __syncthreads();
  long long total_tokens = 0;
  for (int w = 0; w < nwarps; ++w) total_tokens += s_sum[w];

  // tokens per item: the batch's kv-head work spread over ~kItemTarget items
  const long long work = total_tokens * a.Hkv;
  long long T = (work + kItemTarget - 1) / kItemTarget;
  T = (T + kTokQuant - 1) / kTokQuant * kTokQuant;
  if (T < kTokQuant) T = kTokQuant;

  // per-request split counts and an exclusive scan of their item counts
  for (int b0 = 0; b0 < a.B; b0 += nt) {
    const int b = b0 + tid;
    int n = 0;
    if (b < a.B) {
      const int L = a.seq_lens[b];
      const bool aborted = a.abort_mask && a.abort_mask[b];
      if (!aborted && L > 0 && L <= cap) n = static_cast<int>((L + T - 1) / T);
    }
    const int cnt = n * a.Hkv;
    int incl = cnt;
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    int warp_off = 0;
    for (int w = 0; w < warp; ++w) warp_off += s_scan[w];
    const int base = s_carry + warp_off + incl - cnt;
    if (b < a.B) {
      a.n_items[b] = n;
      a.base[b] = base;
      a.bad[b] = 0;
    }
    __syncthreads();
    if (tid == nt - 1) s_carry = base + cnt;
    __syncthreads();
  }
  const int total_items = s_carry;

  // flat item list: item i belongs to the last request whose base is <= i
  for (int i = tid; i < total_items; i += nt) {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldcg(a.base + mid) <= i)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int b = lo;
    const int n = __ldcg(a.n_items + b);
    const int r = i - __ldcg(a.base + b);
    const int kvh = r / n, s = r % n;
    const long long t0 = static_cast<long long>(s) * T;
    const long long t1 = min(t0 + T, static_cast<long long>(a.seq_lens[b]));
    a.items[i] = make_int4(b, kvh, static_cast<int>(t0), static_cast<int>(t1));
  }
  if (tid == 0) {
    a.hdr[0] = 0;  // work counter for the split kernel
    a.hdr[1] = total_items;
    a.hdr[2] = static_cast<int>(T);
  }
}

// ---------------------------------------------------------------------------
// split
// ---------------------------------------------------------------------------

template <int D, int G, bool kFp8>
struct Cfg {
  static constexpr int ES = kFp8 ? 1 : 2;                 // bytes per cached element
  static constexpr int TS = kFp8 ? 64 : 32;               // tokens per stage
  static constexpr int NS = kStages;
  static constexpr int NCW = kConsumerWarps;
  static constexpr int EPL = (kFp8 && G < 8) ? 16 : 8;    // elements per lane per token
  static constexpr int LPT = D / EPL;                     // lanes per token
  static constexpr int TPW = 32 / LPT;                    // tokens per warp per iteration
  static constexpr int TPI = TPW * NCW;                   // tokens per CTA per iteration
  static constexpr int ITERS = TS / TPI;                  // iterations per stage
  static constexpr int CI = (16 / G < ITERS) ? 16 / G : ITERS;  // iterations per softmax chunk
  static constexpr int KV_BYTES = TS * D * ES;            // one stage of K (or V)
  static constexpr int Q_BYTES = G * D * 2;
  // floats per warp in the merge area: acc[G][D], m[G], l[G], padded so that
  // every warp's area starts on a 16-byte boundary (float4 stores)
  static constexpr int RED = G * D + (2 * G + 3) / 4 * 4;
  static constexpr int PART = G * (D + 2);                // floats per partial

  static constexpr size_t off_k = 0;
  static constexpr size_t off_v = off_k + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_q = off_v + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_red = off_q + static_cast<size_t>(NS) * Q_BYTES;
  static constexpr size_t off_desc = off_red + 2ull * NCW * RED * sizeof(float);
  static constexpr size_t off_bar = off_desc + NS * sizeof(int4);
  static constexpr size_t bytes = off_bar + (2 * NS + 2) * sizeof(uint64_t) + 16;

  static_assert(D % EPL == 0 && 32 % LPT == 0, "lane mapping");
  static_assert(TS % TPI == 0 && ITERS % CI == 0, "stage mapping");
  static_assert(kTokQuant % TS == 0, "items must hold whole stages");
  static_assert(off_q % 16 == 0 && off_red % 16 == 0 && off_desc % 16 == 0, "alignment");
  static_assert(RED % 4 == 0 && (G * D) % 4 == 0 && (EPL * ES) % 8 == 0, "vector alignment");
};

struct SplitArgs {
  const uint8_t *k_pool, *v_pool;
  const uint16_t *q;
  const int32_t *block_table;
  const int32_t *hdr;
  int32_t *hdr_counter;
  const int4 *items;
  int32_t *bad;
  float *part;
  uint32_t *err_word;
  int32_t num_pages, P, Hkv, Hq, MP;
  float q_scale;  // sm_scale * k_scale * log2(e)
};

// desc.w packs the number of valid tokens (low 16 bits) and flags
constexpr int kFirst = 1 << 16;
constexpr int kLast = 1 << 17;

// 2^x on the SFU (relative error ~2^-22; exactly 1 at x = 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D, int G, bool kFp8, int EPL>
__device__ __forceinline__ void load_row(const uint8_t *p, float *x) {
  if constexpr (kFp8) {
    if constexpr (EPL == 16) {
      const uint4 w = *reinterpret_cast<const uint4 *>(p);
      e4m3x4_to_f32(w.x, x);
      e4m3x4_to_f32(w.y, x + 4);
      e4m3x4_to_f32(w.z, x + 8);
      e4m3x4_to_f32(w.w, x + 12);
    } else {
      const uint2 w = *reinterpret_cast<const uint2 *>(p);
      e4m3x4_to_f32(w.x, x);
      e4m3x4_to_f32(w.y, x + 4);
    }
  } else {
    const uint4 w = *reinterpret_cast<const uint4 *>(p);
    bf16x2_to_f32(w.x, x);
    bf16x2_to_f32(w.y, x + 2);
    bf16x2_to_f32(w.z, x + 4);
    bf16x2_to_f32(w.w, x + 6);
  }
}

template <int D, int G, bool kFp8>
__global__ void __launch_bounds__(32 * (kConsumerWarps + 1), 2) split_kernel(SplitArgs a) {
  using C = Cfg<D, G, kFp8>;
  extern __shared__ __align__(128) uint8_t smem[];
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
    const uint32_t copy_tokens = C::TS > a.P ? a.P : C::TS;
    const uint32_t copy_bytes = copy_tokens * D * C::ES;
    const uint64_t pol = policy_evict_first();
    uint32_t g = 0;  // stages issued by this CTA
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
        const int npages = C::TS > a.P ? (ntok + a.P - 1) / a.P : 1;
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
          const uint32_t tx = 2u * __popc(valid_mask) * copy_bytes + (first ? C::Q_BYTES : 0u);
          mbar_arrive_expect_tx(&full[slot], tx);
          if (first)
            bulk_g2s(qbuf + slot * C::Q_BYTES,
                     a.q + (static_cast<int64_t>(b) * a.Hq + kvh * G) * D, C::Q_BYTES,
                     &full[slot]);
        }
        __syncwarp();  // the transaction count is armed before any page copy is issued
        // lanes holding a valid page issue its K and V copies
        if (page >= 0) {
          const int64_t in_page = C::TS > a.P ? 0 : (tok0 % a.P);
          const int64_t src = ((static_cast<int64_t>(page) * a.Hkv + kvh) * a.P + in_page) * D *
                              C::ES;
          const uint32_t dst = lane * copy_bytes;
          bulk_g2s_hint(kbuf + slot * C::KV_BYTES + dst, a.k_pool + src, copy_bytes,
                        &full[slot], pol);
          bulk_g2s_hint(vbuf + slot * C::KV_BYTES + dst, a.v_pool + src, copy_bytes,
                        &full[slot], pol);
        }
        __syncwarp();
      }
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  const int grp = lane / C::LPT;    // token within the warp's iteration
  const int chunk = lane % C::LPT;  // which EPL-element slice of the row
  float q[G][C::EPL];
  float acc[G][C::EPL];
  float m_run[G], l_run[G];
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
      const uint16_t *qs = reinterpret_cast<const uint16_t *>(qbuf + slot * C::Q_BYTES);
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int e = 0; e < C::EPL; e += 2) {
          float x[2];
          bf16x2_to_f32(*reinterpret_cast<const uint32_t *>(qs + h * D + chunk * C::EPL + e), x);
          q[h][e] = x[0] * a.q_scale;
          q[h][e + 1] = x[1] * a.q_scale;
          acc[h][e] = 0.f;
          acc[h][e + 1] = 0.f;
        }
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
      }
    }

    const uint8_t *ks = kbuf + slot * C::KV_BYTES;
    const uint8_t *vs = vbuf + slot * C::KV_BYTES;
#pragma unroll
    for (int c0 = 0; c0 < C::ITERS; c0 += C::CI) {
      float sc[C::CI][G];
#pragma unroll
      for (int ci = 0; ci < C::CI; ++ci) {
        const int tl = (c0 + ci) * C::TPI + warp * C::TPW + grp;
        float kx[C::EPL];
        load_row<D, G, kFp8, C::EPL>(ks + (tl * D + chunk * C::EPL) * C::ES, kx);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float s = 0.f;
#pragma unroll
          for (int e = 0; e < C::EPL; ++e) s = fmaf(q[h][e], kx[e], s);
#pragma unroll
          for (int o = 1; o < C::LPT; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
          sc[ci][h] = tl < ntok ? s : -INFINITY;
        }
      }
      // chunk maximum per head over the warp; rescale only when it grew a lot
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = sc[0][h];
#pragma unroll
        for (int ci = 1; ci < C::CI; ++ci) mx = fmaxf(mx, sc[ci][h]);
#pragma unroll
        for (int o = C::LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (mx > m_run[h] + kRescaleThreshold) {
          const float f = exp2f(m_run[h] - mx);  // 0 when m_run is -inf
          l_run[h] *= f;
#pragma unroll
          for (int e = 0; e < C::EPL; ++e) acc[h][e] *= f;
          m_run[h] = mx;
        }
      }
#pragma unroll
      for (int ci = 0; ci < C::CI; ++ci) {
        const int tl = (c0 + ci) * C::TPI + warp * C::TPW + grp;
        if (tl < ntok) {
          float vx[C::EPL];
          load_row<D, G, kFp8, C::EPL>(vs + (tl * D + chunk * C::EPL) * C::ES, vx);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float p = fast_exp2(sc[ci][h] - m_run[h]);
            l_run[h] += p;
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) acc[h][e] = fmaf(p, vx[e], acc[h][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);

    if (d.w & kLast) {
      // merge the warp's token groups
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int o = C::LPT; o < 32; o <<= 1) {
          l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], o);
#pragma unroll
          for (int e = 0; e < C::EPL; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
        }
      }
      const int rb = n_items_done & 1;
      float *my = red + (rb * C::NCW + warp) * C::RED;
      if (lane < C::LPT) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < C::EPL; e += 4)
            *reinterpret_cast<float4 *>(my + h * D + chunk * C::EPL + e) =
                make_float4(acc[h][e], acc[h][e + 1], acc[h][e + 2], acc[h][e + 3]);
      }
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          my[G * D + h] = m_run[h];
          my[G * D + G + h] = l_run[h];
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&fin[rb]);
      if (*fail || !mbar_wait(&fin[rb], (n_items_done >> 1) & 1)) {
        if (!*fail) report(a.err_word, KVQ_ERRBIT_TIMEOUT);
        *fail = 1;
        break;
      }
      // merge the four warps and write the item's partial
      const float *rr = red + rb * C::NCW * C::RED;
      float *out = a.part + static_cast<int64_t>(cur_item) * C::PART;
      const int ctid = warp * 32 + lane;
      for (int idx = ctid; idx < G * D + G; idx += C::NCW * 32) {
        const int h = idx < G * D ? idx / D : idx - G * D;
        float mstar = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) mstar = fmaxf(mstar, rr[w * C::RED + G * D + h]);
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < C::NCW; ++w) {
          const float mw = rr[w * C::RED + G * D + h];
          const float f = mw == -INFINITY ? 0.f : exp2f(mw - mstar);
          const float v = idx < G * D ? rr[w * C::RED + idx] : rr[w * C::RED + G * D + G + h];
          sum = fmaf(f, v, sum);
        }
        if (idx < G * D) {
          out[idx] = sum;
        } else {
          out[G * D + h] = mstar;
          out[G * D + G + h] = sum;
        }
      }
      ++n_items_done;
    }
    ++g;
  }
}

}  // namespace kvq

#include "decode_attn_mma.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// combine
// ---------------------------------------------------------------------------

struct CombineArgs {
  const int32_t *n_items, *base, *bad;
  const float *part;
  float *out;
  int32_t Hq, Hkv, G, D;
  float v_scale;
};

__global__ void __launch_bounds__(256) combine_kernel(CombineArgs a) {
  const int b = blockIdx.x / a.Hkv, kvh = blockIdx.x % a.Hkv;
  const int n = a.n_items[b];
  const bool zero = n == 0 || a.bad[b] != 0;
  const int GD = a.G * a.D;
  const int stride = a.G * (a.D + 2);
  float *out = a.out + (static_cast<int64_t>(b) * a.Hq + kvh * a.G) * a.D;
  const float *p0 = a.part + static_cast<int64_t>(a.base[b] + kvh * n) * stride;
  for (int idx = threadIdx.x; idx < GD; idx += blockDim.x) {
    if (zero) {
      out[idx] = 0.f;
      continue;
    }
    const int h = idx / a.D;
    float mstar = -INFINITY;
    for (int s = 0; s < n; ++s) mstar = fmaxf(mstar, p0[s * stride + GD + h]);
    float num = 0.f, den = 0.f;
    for (int s = 0; s < n; ++s) {
      const float ms = p0[s * stride + GD + h];
      const float f = ms == -INFINITY ? 0.f : exp2f(ms - mstar);
      num = fmaf(f, p0[s * stride + idx], num);
      den = fmaf(f, p0[s * stride + GD + a.G + h], den);
    }
    out[idx] = num / den * a.v_scale;
  }
}

// ---------------------------------------------------------------------------
// host dispatch
// ---------------------------------------------------------------------------

using SplitFn = void (*)(SplitArgs);
using SplitTmaFn = void (*)(CUtensorMap, CUtensorMap, SplitArgs);

struct SplitKernel {
  SplitFn fn = nullptr;      // CUDA-core kernel (bulk copies)
  SplitTmaFn tma = nullptr;  // tensor-core kernel (tiled TMA); used when set
  size_t smem = 0;
  const void *ptr() const {
    return tma ? reinterpret_cast<const void *>(tma) : reinterpret_cast<const void *>(fn);
  }
};

template <int D, int G, bool kFp8>
SplitKernel make_split() {
  SplitKernel k;
  k.fn = split_kernel<D, G, kFp8>;
  k.smem = Cfg<D, G, kFp8>::bytes;
  return k;
}

template <int G>
SplitKernel make_split_mma() {
  SplitKernel k;
  k.tma = split_mma_kernel<G>;
  k.smem = MmaCfg<G>::bytes;
  return k;
}

template <int D, bool kFp8>
bool pick_g(int G, SplitKernel *k) {
  switch (G) {
    case 1: *k = make_split<D, 1, kFp8>(); return true;
    case 2: *k = make_split<D, 2, kFp8>(); return true;
    case 4: *k = make_split<D, 4, kFp8>(); return true;
    case 8: *k = make_split<D, 8, kFp8>(); return true;
  }
  return false;
}

bool pick_split(int D, int G, bool fp8, SplitKernel *k) {
  if (fp8 && D == 128) {
    switch (G) {
      case 1: *k = make_split_mma<1>(); return true;
      case 2: *k = make_split_mma<2>(); return true;
      case 4: *k = make_split_mma<4>(); return true;
      case 8: *k = make_split_mma<8>(); return true;
    }
    return false;
  }
  if (D == 64) return fp8 ? pick_g<64, true>(G, k) : pick_g<64, false>(G, k);
  if (D == 128) return fp8 ? pick_g<128, true>(G, k) : pick_g<128, false>(G, k);
  return false;
}

// Per (device, kernel) launch set-up: opt into the dynamic shared memory and
// read back how many CTAs fit on one SM.
int split_ctas_per_sm(const SplitKernel &k) {
  constexpr int kMaxDev = 64, kMaxFn = 64;
  static int cache_dev_fn[kMaxDev][kMaxFn];
  static const void *fns[kMaxFn];
  static int nfns = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  const void *f = k.ptr();
  int fi = -1;
  for (int i = 0; i < nfns; ++i)
    if (fns[i] == f) fi = i;
  if (fi < 0) {
    if (nfns >= kMaxFn) return 0;
    fi = nfns;
    fns[nfns++] = f;
  }
  if (cache_dev_fn[dev][fi] > 0) return cache_dev_fn[dev][fi];
  if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(k.smem)) != cudaSuccess)
    return 0;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, f, 32 * (kConsumerWarps + 1), k.smem) !=
      cudaSuccess)
    return 0;
  cache_dev_fn[dev][fi] = occ;
  return occ;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 4-D map over an e4m3 pool [num_pages][Hkv][P][D] (D = 128 bytes innermost);
// one box is one page of one kv head, 128-byte swizzled.
bool encode_pool_map(CUtensorMap *map, const void *pool, const kvq_cache &c) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t D = c.head_dim, P = c.page_size, H = c.num_kv_heads, NP = c.num_pages;
  const cuuint64_t dims[4] = {D, P, H, NP};
  const cuuint64_t strides[3] = {D, P * D, H * P * D};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(P), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(pool), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kvq

using namespace kvq;

extern "C" size_t kvq_decode_attn_workspace_size(int32_t B, int32_t Hq, int32_t num_kv_heads,
                                                 int32_t head_dim) {
  if (B < 0 || Hq <= 0 || num_kv_heads <= 0 || head_dim <= 0 || Hq % num_kv_heads) return 0;
  return ws_layout(B, Hq, num_kv_heads, head_dim).total;
}

extern "C" kvq_status kvq_decode_attn(const kvq_cache *cache, const void *q, int32_t B,
                                      int32_t Hq, const int32_t *block_table, int32_t MP,
                                      const int32_t *seq_lens, const uint8_t *abort_mask,
                                      float sm_scale, float *out, void *workspace,
                                      size_t workspace_bytes, uint32_t *err_word,
                                      kvq_stream_t stream) {
  kvq_status st = validate_cache(cache);
  if (st != KVQ_OK) return st;
  if (B < 0 || Hq <= 0 || MP <= 0) return KVQ_ERR_INVALID_ARG;
  if (B == 0) return KVQ_OK;
  const int Hkv = cache->num_kv_heads, D = cache->head_dim;
  if (Hq % Hkv) return KVQ_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (!q || !block_table || !seq_lens || !out || !workspace) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q)) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(MP) * cache->page_size > INT32_MAX) return KVQ_ERR_INVALID_ARG;
  SplitKernel sk;
  if (!pick_split(D, G, cache->kv_dtype == KVQ_KV_E4M3, &sk)) return KVQ_ERR_UNSUPPORTED;
  const WsLayout ws = ws_layout(B, Hq, Hkv, D);
  if (!aligned256(workspace) || workspace_bytes < ws.total) return KVQ_ERR_WORKSPACE;

  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const int occ = split_ctas_per_sm(sk);
  if (occ <= 0) return KVQ_ERR_CUDA;

  uint8_t *w = static_cast<uint8_t *>(workspace);
  int32_t *hdr = reinterpret_cast<int32_t *>(w + ws.hdr);
  int32_t *n_items = reinterpret_cast<int32_t *>(w + ws.n_items);
  int32_t *base = reinterpret_cast<int32_t *>(w + ws.base);
  int32_t *bad = reinterpret_cast<int32_t *>(w + ws.bad);
  int4 *items = reinterpret_cast<int4 *>(w + ws.items);
  float *part = reinterpret_cast<float *>(w + ws.part);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool fp8 = cache->kv_dtype == KVQ_KV_E4M3;

  PlanArgs pa{seq_lens, abort_mask, hdr, n_items, base, bad, items, err_word,
              B, Hkv, MP, cache->page_size};
  plan_kernel<<<1, 1024, 0, s>>>(pa);

  SplitArgs sa;
  sa.k_pool = static_cast<const uint8_t *>(cache->k_pool);
  sa.v_pool = static_cast<const uint8_t *>(cache->v_pool);
  sa.q = static_cast<const uint16_t *>(q);
  sa.block_table = block_table;
  sa.hdr = hdr;
  sa.hdr_counter = hdr;
  sa.items = items;
  sa.bad = bad;
  sa.part = part;
  sa.err_word = err_word;
  sa.num_pages = cache->num_pages;
  sa.P = cache->page_size;
  sa.Hkv = Hkv;
  sa.Hq = Hq;
  sa.MP = MP;
  sa.q_scale = sm_scale * (fp8 ? cache->k_scale : 1.0f) * kLog2e;
  if (sk.tma) {
    CUtensorMap kmap, vmap;
    if (!encode_pool_map(&kmap, cache->k_pool, *cache) ||
        !encode_pool_map(&vmap, cache->v_pool, *cache))
      return KVQ_ERR_CUDA;
    sk.tma<<<sms * occ, 32 * (kConsumerWarps + 1), sk.smem, s>>>(kmap, vmap, sa);
  } else {
    sk.fn<<<sms * occ, 32 * (kConsumerWarps + 1), sk.smem, s>>>(sa);
  }

  CombineArgs ca{n_items, base, bad, part, out, Hq, Hkv, G, D, fp8 ? cache->v_scale : 1.0f};
  combine_kernel<<<B * Hkv, 256, 0, s>>>(ca);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
