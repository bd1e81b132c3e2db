// kvq_decode_attn: single-query paged decode attention over an e4m3 (or bf16)
// KV cache, converting the cache on read.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "KV 缓存量化": the decode pool's cache is e4m3; its FP8 attention kernel
// converts the cache while reading it (the reason FP8 is a little slower per
// token than the BF16 kernel it is compared with in the section's table).
// The pages give no kernel design; this one is written for GB300:
//
//   Every kernel of the call is launched as a programmatic dependent of the
//   one before it (the first of them of whatever precedes the call on the
//   stream, e.g. the tag check), so launch latency overlaps the previous
//   kernel's tail; each waits for its predecessor before touching memory.
//
//   plan   (only for batches the split kernel cannot schedule itself, and
//          for the head_dim-64 kernel) 1 CTA: per-request unit counts, their
//          prefix sum, where each persistent CTA starts; rows of aborted /
//          empty / invalid requests are written as zeros with a descriptor
//          of 0 parts.
//   split  persistent grid of (#SMs x resident CTAs).  The tensor-core
//          kernel works out its own start from the lengths and the abort
//          mask for up to 4,608 requests, so then it is the call's first
//          kernel.  Each CTA owns an equal run of units (see
//          decode_common.cuh).  A producer warp reads the block table and
//          stages the pages with TMA-engine copies into a shared-memory ring
//          (mbarrier-tracked, L2 evict-first); consumer warps convert, run
//          q.k for the query heads sharing a kv head (each cached element
//          converted once, used G times), the online softmax in the log2
//          domain with lazy rescaling, and p.v; at the end of a segment they
//          write the output row or, for a row split across CTAs, a partial.
//   combine merges the partials of every split row once the split grid has
//          finished (a warp per output row for rows of a few parts, a CTA
//          per output row for rows of many), reading each row's descriptor.
//   Two split kernels exist: a tensor-core one for head_dim 128, e4m3 or
//   bf16 (decode_attn_mma.cuh: rows are groups of up to 8 kv heads, 16-token
//   units, one consumer warp per kv head) and a CUDA-core one for head_dim 64
//   (rows are single kv heads, 64-token units, four consumer warps per row).
//
// Every wait is bounded (see mbar_wait); a wait that gives up raises
// KVQ_ERRBIT_TIMEOUT and the CTA leaves its loop.
#include <cfloat>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "kvq_internal.h"
#include "decode_common.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// workspace layout
// ---------------------------------------------------------------------------

struct WsLayout {
  size_t hdr, prefix, start, desc, part, total;
};

inline size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

inline WsLayout ws_layout(int B, int Hq, int Hkv, int D) {
  WsLayout w;
  const int G = Hq / Hkv;
  const size_t rows = static_cast<size_t>(B) * Hkv;
  size_t off = 0;
  w.hdr = off;
  off = round256(off + 16 * sizeof(int32_t));
  w.prefix = off;
  off = round256(off + (static_cast<size_t>(B) + 1) * sizeof(int32_t));
  w.start = off;
  off = round256(off + static_cast<size_t>(kMaxCtas) * sizeof(int4));
  // a descriptor per row (first CTA, parts, request): rows are kv heads or
  // groups of kv heads, at most B * Hkv
  w.desc = off;
  off = round256(off + rows * sizeof(int4));
  // partial slots: row + CTA for every row split across CTAs; a tensor-core
  // row holds up to 8 kv heads, a CUDA-core row one
  w.part = off;
  off = round256(off + (rows + 8ull * kMaxCtas) * part_stride(G, D) * sizeof(float));
  w.total = off;
  return w;
}

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------

// The plan runs beside a split CTA on its SM (the split grid launches while
// the plan is still running): 256 threads and 8 KB of shared memory leave
// room for a split CTA's registers and ring.
constexpr int kPlanThreads = 256;
constexpr int kPlanSmemPrefix = 2048;

struct PlanArgs {
  const int32_t *seq_lens;
  const uint8_t *abort_mask;
  int32_t *hdr, *prefix;
  int4 *start;
  int4 *desc;
  float *out;
  uint32_t *err_word;
  int32_t B, Hq, D, MP, P, nctas;
  int32_t rows_per_req;  // rows of work per request (kv heads or kv-head groups)
  int32_t unit;          // tokens per scheduling unit
};

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  grid_dependency_wait();  // e.g. the tag check's abort mask is visible from here on
  allow_dependents();      // the split grid may launch; it waits for this grid
  __shared__ int s_scan[32];
  __shared__ int s_carry;
  __shared__ int s_prefix[kPlanSmemPrefix];
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const long long cap = static_cast<long long>(a.MP) * a.P;
  if (tid == 0) s_carry = 0;
  __syncthreads();

  for (int b0 = 0; b0 < a.B; b0 += nt) {
    const int b = b0 + tid;
    int units = 0;
    if (b < a.B) {
      const int L = a.seq_lens[b];
      const bool aborted = a.abort_mask && a.abort_mask[b];
      const bool in_range = L >= 0 && L <= cap;
      if (!aborted && !in_range) report(a.err_word, KVQ_ERRBIT_SEQLEN);
      if (!aborted && in_range) units = (L + a.unit - 1) / a.unit;
    }
    const int cnt = units * a.rows_per_req;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    int warp_off = 0;
    for (int w = 0; w < warp; ++w) warp_off += s_scan[w];
    const int pre = s_carry + warp_off + incl - cnt;
    if (b < a.B) {
      a.prefix[b] = pre;
      if (b < kPlanSmemPrefix) s_prefix[b] = pre;
      if (units == 0) {  // aborted, empty or invalid: the rows are zero, with no parts
        float4 *o = reinterpret_cast<float4 *>(a.out + static_cast<int64_t>(b) * a.Hq * a.D);
        for (int i = 0; i < a.Hq * a.D / 4; ++i) o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r = 0; r < a.rows_per_req; ++r)
          a.desc[b * a.rows_per_req + r] = make_int4(0, 0, b, 0);
      }
    }
    __syncthreads();
    if (tid == nt - 1) s_carry = pre + cnt;
    __syncthreads();
  }
  const int S = s_carry;
  const int U = S > 0 ? (S + a.nctas - 1) / a.nctas : 1;
  if (tid == 0) {
    a.prefix[a.B] = S;
    if (a.B < kPlanSmemPrefix) s_prefix[a.B] = S;
  }
  __syncthreads();

  // where each CTA starts: the request whose units contain u = c * U
  const bool in_smem = a.B < kPlanSmemPrefix;
  for (int c = tid; c < a.nctas; c += nt) {
    const long long u = static_cast<long long>(c) * U;
    if (u >= S) {
      a.start[c] = make_int4(-1, 0, 0, 0);
      continue;
    }
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {  // last b with prefix[b] <= u (it owns unit u)
      const int mid = (lo + hi + 1) >> 1;
      const int pm = in_smem ? s_prefix[mid] : __ldcg(a.prefix + mid);
      if (pm <= u)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int p0 = in_smem ? s_prefix[lo] : __ldcg(a.prefix + lo);
    const int p1 = in_smem ? s_prefix[lo + 1] : __ldcg(a.prefix + lo + 1);
    const int units_b = (p1 - p0) / a.rows_per_req;
    const int r = static_cast<int>(u - p0);
    a.start[c] = make_int4(lo, r / units_b, r % units_b, 0);
  }
  if (tid == 0) {
    a.hdr[0] = S;
    a.hdr[1] = U;
  }
}

// ---------------------------------------------------------------------------
// CUDA-core split kernel (head_dim 64)
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

  static constexpr size_t off_k = 0;
  static constexpr size_t off_v = off_k + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_q = off_v + static_cast<size_t>(NS) * KV_BYTES;
  static constexpr size_t off_red = off_q + static_cast<size_t>(NS) * Q_BYTES;
  static constexpr size_t off_ctl = off_red + 2ull * NCW * RED * sizeof(float);
  static constexpr size_t bytes = off_ctl + sizeof(Ctrl);

  static_assert(D % EPL == 0 && 32 % LPT == 0, "lane mapping");
  static_assert(TS % TPI == 0 && ITERS % CI == 0, "stage mapping");
  static_assert(off_q % 16 == 0 && off_red % 16 == 0 && off_ctl % 16 == 0, "alignment");
  static_assert(RED % 4 == 0 && (G * D) % 4 == 0 && (EPL * ES) % 8 == 0, "vector alignment");
};

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
  Ctrl &ctl = *reinterpret_cast<Ctrl *>(smem + C::off_ctl);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) ctrl_init(ctl, C::NS, C::NCW);
  __syncthreads();
  grid_dependency_wait();  // the plan's outputs are visible from here on
  allow_dependents();      // the combine grid may become resident and wait

  if (warp == C::NCW) {
    const uint32_t copy_tokens = C::TS > a.P ? a.P : C::TS;
    const uint32_t copy_bytes = copy_tokens * D * C::ES;
    const uint64_t pol = policy_evict_first();
    producer_loop<C::TS, C::Q_BYTES, G, D>(
        a, ctl, qbuf, lane, copy_bytes, [&](int slot, int l, int page, int kvh, int tok0) {
          const int64_t in_page = C::TS > a.P ? 0 : (tok0 % a.P);
          const int64_t src =
              ((static_cast<int64_t>(page) * a.Hkv + kvh) * a.P + in_page) * D * C::ES;
          const uint32_t dst = l * copy_bytes;
          bulk_g2s_hint(kbuf + slot * C::KV_BYTES + dst, a.k_pool + src, copy_bytes,
                        &ctl.full[slot], pol);
          bulk_g2s_hint(vbuf + slot * C::KV_BYTES + dst, a.v_pool + src, copy_bytes,
                        &ctl.full[slot], pol);
        });
    return;
  }

  // --------------------------------------------------------------- consumers
  const int grp = lane / C::LPT;    // token within the warp's iteration
  const int chunk = lane % C::LPT;  // which EPL-element slice of the row
  float q[G][C::EPL];
  float acc[G][C::EPL];
  float m_run[G], l_run[G];
  uint32_t g = 0, segs = 0;
  bool seg_bad = false;

  while (true) {
    const int slot = g % C::NS;
    if (!ctl_wait(ctl, &ctl.full[slot], (g / C::NS) & 1, a.err_word)) break;
    const int4 d0 = ctl.desc[slot][0];
    if (d0.x < 0) break;
    const int4 d1 = ctl.desc[slot][1];
    const int ntok = d0.z & 0xFFFF;
    if (d0.z & kFirst) {
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
      seg_bad = false;
    }
    seg_bad |= (d0.z & kBad) != 0;

    const uint8_t *ks = kbuf + slot * C::KV_BYTES;
    const uint8_t *vs = vbuf + slot * C::KV_BYTES;
    // a stage with a page outside the pool holds stale bytes where that page
    // would be: its row is written as zeros, so its math is skipped
    const int c_end = (d0.z & kBad) ? 0 : C::ITERS;
#pragma unroll
    for (int c0 = 0; c0 < c_end; c0 += C::CI) {
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
    if (lane == 0) mbar_arrive(&ctl.empty[slot]);

    if (d0.z & kLast) {
      // merge the warp's token groups, then the four warps
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int o = C::LPT; o < 32; o <<= 1) {
          l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], o);
#pragma unroll
          for (int e = 0; e < C::EPL; ++e) acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
        }
      }
      const int rb = segs & 1;
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
      if (lane == 0) mbar_arrive(&ctl.fin[rb]);
      if (!ctl_wait(ctl, &ctl.fin[rb], (segs >> 1) & 1, a.err_word)) break;
      finish_segment<G, D, C::RED>(a, red + rb * C::NCW * C::RED, d0, d1, seg_bad, lane);
      ++segs;
    }
    ++g;
  }
}

// ---------------------------------------------------------------------------
// combine: every row split across CTAs
// ---------------------------------------------------------------------------

struct CombineArgs {
  const int4 *desc;
  const float *part;
  float *out;
  int32_t B, Hq, Hkv, G, D, hg, rows_per_req;
  float v_scale;
};

constexpr int kWarpBatch = 4;  // parts loaded at once by a warp-merged row

// One output row (query head hr of a row) and where its parts live.
struct CombineItem {
  float *out;         // D floats
  const float *base;  // part 0 of this query head's kv head
  int nparts, hq;
};

// d: the row's descriptor (first CTA, parts, request, 0).
__device__ __forceinline__ CombineItem combine_item(const CombineArgs &a, int row, int4 d, int hr,
                                                    int64_t slot_floats, int64_t kpart) {
  CombineItem it;
  it.nparts = d.y;
  const int c_lo = d.x, b = d.z;
  const int rin = row % a.rows_per_req;
  const int kvh_in = hr / a.G;
  it.hq = hr % a.G;
  it.out = a.out + (static_cast<int64_t>(b) * a.Hq + (rin * a.hg + kvh_in) * a.G + it.hq) * a.D;
  it.base = a.part + static_cast<int64_t>(row + c_lo) * slot_floats + kvh_in * kpart;
  return it;
}

// Folds parts p0, p0 + step, ... (< nparts) of one output row into a running
// maximum M, denominator den and accumulator acc (dims 4*lane..+3): the
// parts are loaded NB at a time, every load of a batch issued together.  A
// part whose l is negative met a page outside the pool: `bad` is set.
template <int NB>
__device__ __forceinline__ void merge_parts(const CombineItem &it, int p0, int step, int slot32,
                                            int GD, int G, int D, int lane, bool active,
                                            float &M, float &den, float4 &acc, bool &bad) {
  for (int pb = p0; pb < it.nparts; pb += NB * step) {
    float m[NB], l[NB];
    float4 v[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int p = pb + j * step;
      const bool in = p < it.nparts;
      const float *pp = it.base + p * slot32;
      m[j] = in ? __ldcg(pp + GD + it.hq) : -INFINITY;
      l[j] = in ? __ldcg(pp + GD + G + it.hq) : 0.f;
      v[j] = in && active ? __ldcg(reinterpret_cast<const float4 *>(pp + it.hq * D) + lane)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) bad |= l[j] < 0.f;
    float Mb = M;
#pragma unroll
    for (int j = 0; j < NB; ++j) Mb = fmaxf(Mb, m[j]);
    if (Mb == -INFINITY) continue;  // no part with a weight yet
    const float f = M == -INFINITY ? 0.f : exp2f(M - Mb);
    den *= f;
    acc = make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const float wp = m[j] == -INFINITY ? 0.f : exp2f(m[j] - Mb);
      if (wp != 0.f) den = fmaf(wp, l[j], den);
      acc.x = fmaf(wp, v[j].x, acc.x);
      acc.y = fmaf(wp, v[j].y, acc.y);
      acc.z = fmaf(wp, v[j].z, acc.z);
      acc.w = fmaf(wp, v[j].w, acc.w);
    }
    M = Mb;
  }
}

// Launched as a programmatic dependent of the split kernel; it waits for the
// whole split grid, then merges by log-sum-exp every row that grid left in
// parts (part p of a row is the slot of CTA c_lo + p, holding acc[G][D],
// m[G], l[G] per kv head, m in the log2 domain):
//   out = v_scale * sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,  M = max_p m_p.
// A part whose maximum is -inf carries no weight and its values are not used;
// a row with a part that met a page outside the pool (l < 0) is written as
// zeros.  The work items are all output rows (row, query head); a CTA takes
// items blockIdx, blockIdx + grid, ... in passes of 32.  In a pass lane j of
// warp 0 loads item j's row descriptor (one round trip for the pass) and
// sorts the item into one of two lists: rows in more than kWarpMergeMax
// parts (a row of a short batch can have hundreds), merged by the whole CTA
// one item at a time, its kSubsets warps folding every kSubsets-th part and
// warp 0 folding their results from shared memory; and rows in 2 to
// kWarpMergeMax parts, a warp each.  Two builds: kSubsets = 16 warps uncapped
// (more of a long row's loads in flight) for grids of at most #SMs CTAs, and
// 8 warps capped at 64 registers (4 CTAs per SM) otherwise, small enough
// that one CTA becomes resident beside a running split CTA and is waiting
// when the split grid ends.
template <int kMinBlocks, int kSubsets>
__global__ void __launch_bounds__(32 * kSubsets, kMinBlocks) combine_kernel(CombineArgs a) {
  __shared__ float s_m[kSubsets], s_den[kSubsets];
  __shared__ float4 s_acc[kSubsets][32];
  __shared__ int s_bad[kSubsets];
  __shared__ int4 s_items[32];  // (item, first CTA, parts, request): CTA-merged
  __shared__ int4 s_witems[32];  // the same for warp-merged items
  __shared__ int s_n, s_nw;
  grid_dependency_wait();
  allow_dependents();  // e.g. the next step's append may be scheduled
  const int tid = threadIdx.x, sub = tid >> 5, lane = tid & 31;
  const int heads_per_row = a.hg * a.G;
  const int nout = a.B * a.Hq;  // output rows: row-major over (row, query head in row)
  const int64_t kpart = part_stride(a.G, a.D);  // 16-byte multiple
  const int64_t slot_floats = a.hg * kpart;
  const int slot32 = static_cast<int>(slot_floats);  // at most 8 x 1040 floats
  const int GD = a.G * a.D;
  const bool active = 4 * lane < a.D;

  for (int64_t base = 0; blockIdx.x + base * gridDim.x < nout; base += 32) {
    if (sub == 0) {
      const int64_t item = blockIdx.x + (base + lane) * gridDim.x;
      int4 d = make_int4(0, 0, 0, 0);
      if (item < nout) d = __ldcg(a.desc + item / heads_per_row);
      const int4 li = make_int4(static_cast<int>(item), d.x, d.y, d.z);
      const bool big = d.y > kWarpMergeMax, small = d.y >= 2 && d.y <= kWarpMergeMax;
      const unsigned bb = __ballot_sync(0xffffffffu, big);
      const unsigned bs = __ballot_sync(0xffffffffu, small);
      const unsigned below = (1u << lane) - 1;
      if (big) s_items[__popc(bb & below)] = li;
      if (small) s_witems[__popc(bs & below)] = li;
      if (lane == 0) {
        s_n = __popc(bb);
        s_nw = __popc(bs);
      }
    }
    __syncthreads();
    const int n = s_n, nw = s_nw;

    // ---- rows of many parts: the whole CTA per output row
    for (int k = 0; k < n; ++k) {
      const int4 li = s_items[k];
      const int row = li.x / heads_per_row;
      const CombineItem it = combine_item(a, row, make_int4(li.y, li.z, li.w, 0),
                                          li.x % heads_per_row, slot_floats, kpart);
      // subset `sub` folds parts sub, sub + kSubsets, ...; then the subsets are folded
      float M = -INFINITY, den = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      bool bad = false;
      merge_parts<kMinBlocks == 1 ? 8 : kWarpBatch>(it, sub, kSubsets, slot32, GD, a.G, a.D, lane,
                                                    active, M, den, acc, bad);
      s_acc[sub][lane] = acc;
      bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) {
        s_m[sub] = M;
        s_den[sub] = den;
        s_bad[sub] = bad;
      }
      __syncthreads();
      if (sub == 0 && active) {
        float Mr = -INFINITY;
        bool row_bad = false;
#pragma unroll
        for (int i = 0; i < kSubsets; ++i) {
          Mr = fmaxf(Mr, s_m[i]);
          row_bad |= s_bad[i] != 0;
        }
        float d = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kSubsets; ++i) {
          const float wi = s_m[i] == -INFINITY ? 0.f : exp2f(s_m[i] - Mr);
          const float4 v = s_acc[i][lane];
          d = fmaf(wi, s_den[i], d);
          o.x = fmaf(wi, v.x, o.x);
          o.y = fmaf(wi, v.y, o.y);
          o.z = fmaf(wi, v.z, o.z);
          o.w = fmaf(wi, v.w, o.w);
        }
        const float sc = a.v_scale / d;
        // a bad row is stored as zeros, not scaled by 0: its parts may hold
        // values computed from a stage whose page was never copied
        reinterpret_cast<float4 *>(it.out)[lane] =
            row_bad ? make_float4(0.f, 0.f, 0.f, 0.f)
                    : make_float4(o.x * sc, o.y * sc, o.z * sc, o.w * sc);
      }
      __syncthreads();  // s_acc, s_m, s_den, s_bad are reused by the next item
    }

    // ---- rows of 2..kWarpMergeMax parts: a warp per output row
    for (int k = sub; k < nw; k += kSubsets) {
      const int4 li = s_witems[k];
      const int row = li.x / heads_per_row;
      const CombineItem it = combine_item(a, row, make_int4(li.y, li.z, li.w, 0),
                                          li.x % heads_per_row, slot_floats, kpart);
      float M = -INFINITY, den = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      bool bad = false;
      merge_parts<kWarpBatch>(it, 0, 1, slot32, GD, a.G, a.D, lane, active, M, den, acc, bad);
      bad = __any_sync(0xffffffffu, bad);
      if (active) {
        const float sc = a.v_scale / den;
        reinterpret_cast<float4 *>(it.out)[lane] =
            bad ? make_float4(0.f, 0.f, 0.f, 0.f)
                : make_float4(acc.x * sc, acc.y * sc, acc.z * sc, acc.w * sc);
      }
    }
    __syncthreads();  // the lists are rewritten by the next pass
  }
}

}  // namespace kvq

#include "decode_attn_mma.cuh"

namespace kvq {

// ---------------------------------------------------------------------------
// host dispatch
// ---------------------------------------------------------------------------

using SplitFn = void (*)(SplitArgs);
using SplitTmaFn = void (*)(CUtensorMap, CUtensorMap, SplitArgs);

struct SplitKernel {
  SplitFn fn = nullptr;      // CUDA-core kernel (bulk copies)
  SplitTmaFn tma = nullptr;  // tensor-core kernel (tiled TMA); used when set
  size_t smem = 0;
  int threads = 0;
  int hg = 1;        // kv heads per row
  int unit = kUnit;  // tokens per scheduling unit
  const void *ptr() const {
    return tma ? reinterpret_cast<const void *>(tma) : reinterpret_cast<const void *>(fn);
  }
};

template <int D, int G, bool kFp8>
SplitKernel make_split() {
  SplitKernel k;
  k.fn = split_kernel<D, G, kFp8>;
  k.smem = Cfg<D, G, kFp8>::bytes;
  k.threads = 32 * (kConsumerWarps + 1);
  return k;
}

template <int G, int HG, bool kBf16>
SplitKernel make_split_hg() {
  SplitKernel k;
  k.tma = split_hg_kernel<G, HG, kBf16>;
  k.smem = HgCfg<G, HG, kBf16>::bytes;
  k.threads = 32 * (HG + 1);
  k.hg = HG;
  k.unit = kTile;
  return k;
}

template <int G, bool kBf16>
bool pick_hg(int Hkv, SplitKernel *k) {
  if (Hkv % 8 == 0) { *k = make_split_hg<G, 8, kBf16>(); return true; }
  if (Hkv % 4 == 0) { *k = make_split_hg<G, 4, kBf16>(); return true; }
  if (Hkv % 2 == 0) { *k = make_split_hg<G, 2, kBf16>(); return true; }
  *k = make_split_hg<G, 1, kBf16>();
  return true;
}

template <bool kBf16>
bool pick_hg_g(int G, int Hkv, SplitKernel *k) {
  switch (G) {
    case 1: return pick_hg<1, kBf16>(Hkv, k);
    case 2: return pick_hg<2, kBf16>(Hkv, k);
    case 4: return pick_hg<4, kBf16>(Hkv, k);
    case 8: return pick_hg<8, kBf16>(Hkv, k);
  }
  return false;
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

bool pick_split(int D, int G, int Hkv, bool fp8, SplitKernel *k) {
  if (D == 128) return fp8 ? pick_hg_g<false>(G, Hkv, k) : pick_hg_g<true>(G, Hkv, k);
  if (D == 64) return fp8 ? pick_g<64, true>(G, k) : pick_g<64, false>(G, k);
  return false;
}

// Per (device, kernel) launch set-up: opt into the dynamic shared memory and
// read back how many CTAs fit on one SM.
int split_ctas_per_sm(const SplitKernel &k) {
  constexpr int kMaxDev = 64, kMaxFn = 64;
  static int cache_dev_fn[kMaxDev][kMaxFn];
  static const void *fns[kMaxFn];
  static int nfns = 0;
  static std::mutex mu;  // calls may come from several host threads
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  std::lock_guard<std::mutex> lock(mu);
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
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, f, k.threads, k.smem) != cudaSuccess)
    return 0;
  // The split grid launches while the plan is still running.  An SM takes
  // its shared-memory carveout from the first CTA placed on it, so the plan's
  // SM would otherwise be configured too small for a split CTA, and that
  // CTA would start only after the plan had exited.
  if (cudaFuncSetAttribute(plan_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    return 0;
  cache_dev_fn[dev][fi] = occ;
  return occ;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  // looked up once, thread-safely (a function-local static's initialiser)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// 4-D map over a pool [num_pages][Hkv][P][D] (D innermost); one box is 128
// bytes of dims x 16 slots x `hg` consecutive kv heads of one page, 128-byte
// swizzled (all of D for e4m3, half of it for bf16).
bool encode_pool_map(CUtensorMap *map, const void *pool, const kvq_cache &c, int hg) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const bool bf16 = c.kv_dtype == KVQ_KV_BF16;
  const cuuint64_t es = bf16 ? 2 : 1;
  const cuuint64_t D = c.head_dim, P = c.page_size, H = c.num_kv_heads, NP = c.num_pages;
  const cuuint64_t dims[4] = {D, P, H, NP};
  const cuuint64_t strides[3] = {D * es, P * D * es, H * P * D * es};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(kTile),
                             static_cast<cuuint32_t>(hg), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
             const_cast<void *>(pool), dims, strides, box,
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
  if (!aligned16(q) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(MP) * cache->page_size > INT32_MAX) return KVQ_ERR_INVALID_ARG;
  SplitKernel sk;
  if (!pick_split(D, G, Hkv, cache->kv_dtype == KVQ_KV_E4M3, &sk)) return KVQ_ERR_UNSUPPORTED;
  const WsLayout ws = ws_layout(B, Hq, Hkv, D);
  if (!aligned256(workspace) || workspace_bytes < ws.total) return KVQ_ERR_WORKSPACE;

  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const int occ = split_ctas_per_sm(sk);
  if (occ <= 0) return KVQ_ERR_CUDA;
  const int nctas = sms * occ < kMaxCtas ? sms * occ : kMaxCtas;

  uint8_t *w = static_cast<uint8_t *>(workspace);
  int32_t *hdr = reinterpret_cast<int32_t *>(w + ws.hdr);
  int32_t *prefix = reinterpret_cast<int32_t *>(w + ws.prefix);
  int4 *start = reinterpret_cast<int4 *>(w + ws.start);
  int4 *desc = reinterpret_cast<int4 *>(w + ws.desc);
  float *part = reinterpret_cast<float *>(w + ws.part);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool fp8 = cache->kv_dtype == KVQ_KV_E4M3;

  // The tensor-core kernel schedules batches of up to 4,608 requests itself
  // (the same test as its self_schedule): then there is no plan kernel and
  // the split grid is the call's first kernel.
  const bool self = sk.tma && self_schedulable(B, sk.threads, kSelfSchedPer, nctas);
  if (!self) {
    PlanArgs pa{seq_lens, abort_mask, hdr, prefix, start, desc, out, err_word,
                B, Hq, D, MP, cache->page_size, nctas, Hkv / sk.hg, sk.unit};
    if (launch_dependent(plan_kernel, 1, kPlanThreads, 0, s, pa) != cudaSuccess)
      return KVQ_ERR_CUDA;
  }

  SplitArgs sa;
  sa.k_pool = static_cast<const uint8_t *>(cache->k_pool);
  sa.v_pool = static_cast<const uint8_t *>(cache->v_pool);
  sa.q = static_cast<const uint16_t *>(q);
  sa.block_table = block_table;
  sa.seq_lens = seq_lens;
  sa.abort_mask = abort_mask;
  sa.hdr = hdr;
  sa.prefix = prefix;
  sa.start = start;
  sa.desc = desc;
  sa.part = part;
  sa.out = out;
  sa.err_word = err_word;
  sa.num_pages = cache->num_pages;
  sa.P = cache->page_size;
  sa.Hkv = Hkv;
  sa.Hq = Hq;
  sa.MP = MP;
  sa.B = B;
  sa.q_scale = sm_scale * (fp8 ? cache->k_scale : 1.0f) * kLog2e;
  sa.v_scale = fp8 ? cache->v_scale : 1.0f;

  // the split grid is a programmatic dependent of the work before it (the
  // plan, or whatever precedes the call): its CTAs start (shared-memory and
  // barrier set-up) while that work finishes, and wait for it with
  // griddepcontrol.wait
  cudaError_t e;
  if (sk.tma) {
    CUtensorMap kmap, vmap;
    if (!encode_pool_map(&kmap, cache->k_pool, *cache, sk.hg) ||
        !encode_pool_map(&vmap, cache->v_pool, *cache, sk.hg))
      return KVQ_ERR_CUDA;
    e = launch_dependent(sk.tma, nctas, sk.threads, sk.smem, s, kmap, vmap, sa);
  } else {
    e = launch_dependent(sk.fn, nctas, sk.threads, sk.smem, s, sa);
  }
  if (e != cudaSuccess) return KVQ_ERR_CUDA;

  // rows split across CTAs are merged by combine_kernel, a programmatic
  // dependent of the split grid; with no such rows it exits after reading
  // the descriptors
  CombineArgs ca{desc, part, out, B, Hq, Hkv, G, D, sk.hg, Hkv / sk.hg,
                 fp8 ? cache->v_scale : 1.0f};
  const int crows = B * Hq;
  cudaError_t ce;
  if (crows <= sms)
    ce = launch_dependent(combine_kernel<1, 16>, crows, 512, 0, s, ca);
  else
    ce = launch_dependent(combine_kernel<4, 8>, crows < 4 * sms ? crows : 4 * sms, 256, 0, s, ca);
  if (ce != cudaSuccess) return KVQ_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
