// Scheduling, staging and merge code shared by the two decode-attention split
// kernels (CUDA-core and tensor-core).  Included by decode_attn.cu.
//
// Work split ("stream-K" over the sequence): every request is cut into
// rows (its kv heads, or groups of kv heads), each a run of units of a fixed
// number of tokens.  The rows are laid end to end and each of the C
// persistent CTAs takes the same number U of consecutive units, so the load
// is balanced to within one unit whatever the length mix.  A CTA's range cuts
// rows into segments; a row owned by one CTA is normalised and written
// directly, otherwise every CTA writes a partial (acc[G][D], m[G], l[G] per
// kv head; l = -1 marks a part that met a page outside the pool) and the
// combine kernel merges the row by log-sum-exp once the split grid has
// finished: one warp per output row when the row has few parts, a whole CTA
// per output row when it has many.  The CTA that holds a row's first unit
// writes the row's merge descriptor (first CTA, parts, request); rows of
// requests without work get a descriptor of 0 parts from whoever zeroes
// their output.  No split CTA ever waits for another, so the grid ends when
// the last CTA's stream does.
#pragma once

namespace kvq {

constexpr int kUnit = 64;           // tokens per scheduling unit (CUDA-core kernel)
constexpr int kMaxCtas = 1024;      // upper bound on the persistent grid
constexpr int kConsumerWarps = 4;   // consumer warps of the CUDA-core kernel
constexpr int kStages = 4;          // ring stages of the CUDA-core kernel
constexpr int kMaxStages = 6;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when the max grows by > 2^8

// stage descriptor flags (packed above the 16-bit token count)
constexpr int kFirst = 1 << 16;  // first stage of a segment
constexpr int kLast = 1 << 17;   // last stage of a segment
constexpr int kBad = 1 << 18;    // a page of this stage (of its tile k: kBad << k) was outside the pool

struct SplitArgs {
  const uint8_t *k_pool, *v_pool;
  const uint16_t *q;
  const int32_t *block_table, *seq_lens;
  const uint8_t *abort_mask;  // [B] or null
  const int32_t *hdr;     // [0] total units S, [1] units per CTA U (plan)
  const int32_t *prefix;  // [B+1]: units before request b, over all its kv heads (plan)
  const int4 *start;      // [C]: (b, kv head, unit in row) where CTA c begins (plan)
  int4 *desc;             // [rows]: (first CTA, parts, request, 0) of every row
  float *part;            // [B*Hkv + C][G][D+2] partials
  float *out;             // [B][Hq][D]
  uint32_t *err_word;
  int32_t num_pages, P, Hkv, Hq, MP, B;
  float q_scale;  // sm_scale * k_scale * log2(e)
  float v_scale;
};

// Floats of one kv head's partial: acc[G][D], m[G], l[G], padded to a
// multiple of four floats so every head's block is 16-byte aligned.
__host__ __device__ constexpr int part_stride(int G, int D) { return G * D + (2 * G + 3) / 4 * 4; }

// Requests without work (aborted, empty or of invalid length) that one CTA
// zeroes in a call whose schedule the split kernel works out itself: request
// b goes to CTA b % grid, and that schedule covers at most 4,608 requests
// over at least 152 CTAs.
constexpr int kZeroMax = 32;

// Requests per thread in a CTA's own schedule scan (tensor-core kernel):
// 32 x (HG + 1) threads x 16 = 4,608 requests for 8-kv-head groups.
constexpr int kSelfSchedPer = 16;

// Rows split over at most this many CTAs are merged by one warp per output
// row in the combine kernel (all parts' loads issued at once); rows split
// further by a whole combine CTA per output row.
constexpr int kWarpMergeMax = 8;

// Shared-memory control block.
struct Ctrl {
  int4 desc[kMaxStages][2];  // {row, tok0, ntok|flags, nparts}, {slot, c_lo, b, kvh or group}
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t qfull[2], qempty[2];  // double-buffered query rows (tensor-core kernel)
  uint64_t fin[2];               // per-segment merge of the consumer warps (CUDA-core kernel)
  int fail;
  int scan[16];                  // per-warp sums of the CTA's own schedule scan
  int sched[4];                  // where the CTA starts: request, its prefix, length, units
  int nzero;                     // requests without work this CTA zeroes (own schedule)
  int zero[kZeroMax];
};

// 2^x on the SFU (relative error ~2^-22; exactly 1 at x = 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ns ring stages, nc consumer warps (each consumer warp arrives once per phase)
__device__ __forceinline__ void ctrl_init(Ctrl &ctl, int ns, int nc) {
  for (int s = 0; s < ns; ++s) {
    mbar_init(&ctl.full[s], 1);
    mbar_init(&ctl.empty[s], nc);
  }
  for (int i = 0; i < 2; ++i) {
    mbar_init(&ctl.qfull[i], 1);
    mbar_init(&ctl.qempty[i], nc);
    mbar_init(&ctl.fin[i], nc);
  }
  ctl.fail = 0;
  fence_barrier_init();
}

// Bounded wait shared by every role: on timeout the error bit is raised once
// and the CTA's fail flag tells everybody to leave.
__device__ __forceinline__ bool ctl_wait(Ctrl &ctl, uint64_t *bar, uint32_t parity,
                                         uint32_t *err_word) {
  volatile int *fail = &ctl.fail;
  if (*fail) return false;
  if (mbar_wait(bar, parity)) return true;
  if (atomicExch(&ctl.fail, 1) == 0) report(err_word, KVQ_ERRBIT_TIMEOUT);
  return false;
}

// ---------------------------------------------------------------------------
// a CTA's own copy of the plan's schedule
// ---------------------------------------------------------------------------

// Units per row of request b, counted as the plan counts them: ceil(L / unit),
// or 0 for an aborted request or a length outside [0, cap].  L is returned.
// The read-only path is safe even before this grid's dependency wait: both
// arrays were written before the grid launched (see self_schedule), and the
// lines it leaves in L1 make the producer's later visits to neighbouring
// requests hits.
__device__ __forceinline__ int request_units(const SplitArgs &a, int b, long long cap, int unit,
                                             int &L) {
  L = __ldg(a.seq_lens + b);
  const bool aborted = a.abort_mask && __ldg(a.abort_mask + b) != 0;
  return (aborted || L < 0 || L > cap) ? 0 : (L + unit - 1) / unit;
}

// Whether a CTA of NT threads can work out the schedule of B requests
// itself (PER requests a thread) and hold the list of requests without work
// that fall to it (B / grid of them at most).  The host takes the same
// decision when it leaves out the plan kernel.
__host__ __device__ constexpr bool self_schedulable(int B, int NT, int PER, int grid) {
  return B <= NT * PER && B <= kZeroMax * grid;
}

// Where this CTA starts, as the plan would place it.
struct SchedStart {
  int S, U;   // total units, units per CTA
  int b, p0;  // first request and the units before it (all of its rows)
  int L, ub;  // that request's length and units per row
};

// The CTA works out its own start from seq_lens and the abort mask with the
// plan's arithmetic (rows of ceil(L / unit) units, U = ceil(S / grid)), one
// request set of PER consecutive requests per thread, so that it need not
// wait for the plan kernel before it starts copying pages.  Reading those two
// arrays before grid_dependency_wait() is safe because the plan kernel lets
// this grid launch only after its own wait: by then everything ahead of the
// plan on the stream (the tag check that wrote the mask, whatever wrote the
// lengths) has completed.  Only what the plan itself writes (bad-page flags,
// the merge lists, zeroed rows) needs the wait.  Returns false, with nothing read,
// when the batch is larger than NT x PER requests; the caller then waits and
// takes the plan's schedule.  Every thread of the CTA calls it.
template <int NT, int PER>
__device__ __forceinline__ bool self_schedule(const SplitArgs &a, int rows_per_req, int unit,
                                              Ctrl &ctl, SchedStart &sc) {
  static_assert(NT % 32 == 0 && NT / 32 <= 16, "CTA size");
  if (!self_schedulable(a.B, NT, PER, gridDim.x)) return false;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long cap = static_cast<long long>(a.MP) * a.P;
  const int base = tid * PER;
  int cnt[PER], len[PER];
  // every length and abort byte of the thread's requests is loaded before
  // any is used, so that both arrays' lines are fetched in one round trip
#pragma unroll
  for (int i = 0; i < PER; ++i) len[i] = base + i < a.B ? __ldg(a.seq_lens + base + i) : 0;
  uint32_t aborted = 0;  // bit i: request base + i was aborted
  if (a.abort_mask) {
#pragma unroll
    for (int i = 0; i < PER; ++i)
      if (base + i < a.B && __ldg(a.abort_mask + base + i) != 0) aborted |= 1u << i;
  }
  int sum = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    // units of request base + i, as request_units counts them
    const int L = len[i];
    cnt[i] = (base + i >= a.B || ((aborted >> i) & 1u) || L < 0 || L > cap)
                 ? 0 : (L + unit - 1) / unit;
    sum += cnt[i] * rows_per_req;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) ctl.scan[warp] = incl;
  if (tid == 0) ctl.sched[0] = ctl.sched[1] = ctl.sched[2] = ctl.sched[3] = 0;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const int t = ctl.scan[w];
    if (w < warp) before += t;
    total += t;
  }
  sc.S = total;
  sc.U = total > 0 ? (total + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x) : 1;
  const long long u0 = static_cast<long long>(blockIdx.x) * sc.U;
  int pre = before + incl - sum;  // units before this thread's first request
  if (tid == 0) ctl.nzero = 0;
  __syncthreads();
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int n = cnt[i] * rows_per_req;
    if (n > 0 && u0 >= pre && u0 < pre + n) {  // at most one request of the batch owns u0
      ctl.sched[0] = base + i;
      ctl.sched[1] = pre;
      ctl.sched[2] = len[i];
      ctl.sched[3] = cnt[i];
    }
    // a request without work is this CTA's to zero when b % grid == CTA
    if (base + i < a.B && n == 0 && (base + i) % static_cast<int>(gridDim.x) == blockIdx.x) {
      const int k = atomicAdd(&ctl.nzero, 1);
      if (k < kZeroMax) ctl.zero[k] = base + i;  // at most ceil(B / grid) <= kZeroMax
    }
    pre += n;
  }
  __syncthreads();
  sc.b = ctl.sched[0];  // meaningful only when u0 < S
  sc.p0 = ctl.sched[1];
  sc.L = ctl.sched[2];
  sc.ub = ctl.sched[3];
  return true;
}

// With its own schedule, the CTA also stands in for the plan on the requests
// without work that fall to it: their output rows are zeroed, their rows get
// a descriptor of 0 parts, and a length outside [0, MP * P] (of a request
// that was not aborted) raises KVQ_ERRBIT_SEQLEN.  Every thread calls it.
template <int D>
__device__ __forceinline__ void zero_requests(const SplitArgs &a, int rows_per_req,
                                              const Ctrl &ctl) {
  const int n = min(ctl.nzero, kZeroMax);
  const long long cap = static_cast<long long>(a.MP) * a.P;
  for (int i = 0; i < n; ++i) {
    const int b = ctl.zero[i];
    float4 *o = reinterpret_cast<float4 *>(a.out + static_cast<int64_t>(b) * a.Hq * D);
    for (int k = threadIdx.x; k < a.Hq * D / 4; k += blockDim.x)
      o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x < rows_per_req) a.desc[b * rows_per_req + threadIdx.x] = make_int4(0, 0, b, 0);
    if (threadIdx.x == 0) {
      const int L = __ldg(a.seq_lens + b);
      const bool aborted = a.abort_mask && __ldg(a.abort_mask + b) != 0;
      if (!aborted && (L < 0 || L > cap)) report(a.err_word, KVQ_ERRBIT_SEQLEN);
    }
  }
}

// The same start read from the plan's results (after grid_dependency_wait()).
__device__ __forceinline__ SchedStart plan_schedule(const SplitArgs &a, int rows_per_req) {
  SchedStart sc;
  sc.S = a.hdr[0];
  sc.U = a.hdr[1];
  sc.b = sc.p0 = sc.L = sc.ub = 0;
  if (static_cast<long long>(blockIdx.x) * sc.U < sc.S) {
    sc.b = a.start[blockIdx.x].x;
    sc.p0 = a.prefix[sc.b];
    sc.ub = (a.prefix[sc.b + 1] - sc.p0) / rows_per_req;
    sc.L = a.seq_lens[sc.b];
  }
  return sc;
}

// ---------------------------------------------------------------------------
// producer: walk this CTA's units, one stage (TS tokens of one row) at a time
// ---------------------------------------------------------------------------

// CopyPages(slot, lane, page, kvh, tok0) issues the K and V copies of page
// `page` (the lane-th page of the stage) into the stage's buffers; each copy
// moves `copy_bytes`.
template <int TS, int QBYTES, int G, int D, typename CopyPages>
__device__ __forceinline__ void producer_loop(const SplitArgs &a, Ctrl &ctl, uint8_t *qbuf,
                                              int lane, uint32_t copy_bytes, CopyPages copy) {
  static_assert(kUnit % TS == 0, "a unit holds whole stages");
  const int S = a.hdr[0], U = a.hdr[1];
  const int c = blockIdx.x;
  long long u = static_cast<long long>(c) * U;
  const long long u_end = min(u + U, static_cast<long long>(S));
  int b = 0, kvh = 0, s = 0;
  if (u < u_end) {
    const int4 st = a.start[c];
    b = st.x;
    kvh = st.y;
    s = st.z;
  }
  uint32_t g = 0;  // stages issued
  // Block-table window of the current request: lane i holds logical page
  // win+i in `cur` and win+32+i in `nxt`; `nxt` is loaded one window ahead so
  // the page ids of a stage never wait on memory.
  int win_b = -1, win = 0, cur = -1, nxt = -1;
  const int32_t *bt_row = a.block_table;
  auto bt_load = [&](int lp) -> int { return lp < a.MP ? __ldg(bt_row + lp) : -1; };
  bool ok = true;
  while (ok) {
    const bool done = u >= u_end;
    int units_b = 0, L = 0, row = 0, nparts = 1, c_lo = c;
    if (!done) {
      const int p0 = __ldg(a.prefix + b), p1 = __ldg(a.prefix + b + 1);
      units_b = (p1 - p0) / a.Hkv;
      L = __ldg(a.seq_lens + b);
      row = b * a.Hkv + kvh;
      const long long ur = static_cast<long long>(p0) + static_cast<long long>(kvh) * units_b;
      c_lo = static_cast<int>(ur / U);
      nparts = static_cast<int>((ur + units_b - 1) / U) - c_lo + 1;
      const int lp0 = s * kUnit / a.P;
      if (b != win_b || lp0 < win || lp0 >= win + 32) {
        win_b = b;
        win = lp0;
        bt_row = a.block_table + static_cast<int64_t>(b) * a.MP;
        cur = bt_load(win + lane);
        nxt = bt_load(win + 32 + lane);
      }
    }
    const int seg_units = done ? 0 : static_cast<int>(min(static_cast<long long>(units_b - s),
                                                          u_end - u));
    const int t_begin = s * kUnit;
    const int t_end = done ? 0 : min((s + seg_units) * kUnit, L);
    const int nstages = done ? 1 : (t_end - t_begin + TS - 1) / TS;
    for (int st = 0; st < nstages; ++st, ++g) {
      const int slot = g % kStages;
      bool waited = true;
      if (lane == 0 && g >= kStages)
        waited = ctl_wait(ctl, &ctl.empty[slot], ((g / kStages) - 1) & 1, a.err_word);
      ok = __shfl_sync(0xffffffffu, waited ? 1 : 0, 0) != 0;
      if (!ok) break;
      if (done) {
        if (lane == 0) {
          ctl.desc[slot][0] = make_int4(-1, 0, 0, 0);
          mbar_arrive(&ctl.full[slot]);
        }
        ok = false;
        break;
      }
      const int tok0 = t_begin + st * TS;
      const int ntok = min(TS, t_end - tok0);
      const int npages = TS > a.P ? (ntok + a.P - 1) / a.P : 1;
      const int lp = tok0 / a.P;  // first logical page of the stage
      while (lp + npages > win + 32) {  // slide the window by 32 pages
        win += 32;
        cur = nxt;
        nxt = bt_load(win + 32 + lane);
      }
      const int idx = lp - win + lane;  // < 64 for lane < npages
      const int from_cur = __shfl_sync(0xffffffffu, cur, idx & 31);
      const int from_nxt = __shfl_sync(0xffffffffu, nxt, idx & 31);
      int page = -1;
      bool bad_page = false;
      if (lane < npages) {
        page = idx < 32 ? from_cur : from_nxt;
        if (page < 0 || page >= a.num_pages) {
          bad_page = true;
          page = -1;
          report(a.err_word, KVQ_ERRBIT_PAGE);
        }
      }
      const unsigned valid_mask = __ballot_sync(0xffffffffu, page >= 0);
      const bool any_bad = __any_sync(0xffffffffu, bad_page);
      const bool first = st == 0, last = st == nstages - 1;
      if (lane == 0 && first && s == 0)  // this CTA holds the row's first unit
        a.desc[row] = make_int4(c_lo, nparts, b, 0);
      if (lane == 0) {
        ctl.desc[slot][0] = make_int4(row, tok0,
                                      ntok | (first ? kFirst : 0) | (last ? kLast : 0) |
                                          (any_bad ? kBad : 0),
                                      nparts);
        ctl.desc[slot][1] = make_int4(row + c, c_lo, b, kvh);
        const uint32_t tx = 2u * __popc(valid_mask) * copy_bytes + (first ? QBYTES : 0u);
        mbar_arrive_expect_tx(&ctl.full[slot], tx);
        if (first)
          bulk_g2s(qbuf + slot * QBYTES, a.q + (static_cast<int64_t>(b) * a.Hq + kvh * G) * D,
                   QBYTES, &ctl.full[slot]);
      }
      __syncwarp();  // the transaction count is armed before any page copy is issued
      if (page >= 0) copy(slot, lane, page, kvh, tok0);
      __syncwarp();
    }
    if (!done) {
      u += seg_units;
      s = 0;
      if (++kvh == a.Hkv) {
        kvh = 0;
        ++b;
        // requests without work (aborted, empty or invalid) own no units
        while (b < a.B && __ldg(a.prefix + b + 1) == __ldg(a.prefix + b)) ++b;
      }
    }
  }
  // A wait gave up (not the normal end, which arrives with the end marker):
  // before the CTA exits, let the copies it started land (bounded waits), so
  // that none writes into shared memory the SM may already have handed to
  // another CTA.  Only the last kStages stages can still be in flight.
  if (lane == 0 && *reinterpret_cast<volatile int *>(&ctl.fail))
    for (uint32_t k = g > kStages ? g - kStages : 0; k < g; ++k)
      mbar_wait(&ctl.full[k % kStages], (k / kStages) & 1);
}

// ---------------------------------------------------------------------------
// consumers: finish a segment from the warps' merge areas
// red: [kConsumerWarps][RED] floats, each acc[G][D] then m[G], l[G]
// ---------------------------------------------------------------------------

template <int G, int D, int RED>
__device__ __forceinline__ void finish_segment(const SplitArgs &a, const float *red, int4 d0,
                                               int4 d1, bool seg_bad, int lane) {
  const int ctid = (threadIdx.x >> 5) * 32 + lane;
  const int nparts = d0.w, slot = d1.x, b = d1.z, kvh = d1.w;
  constexpr int GD = G * D;
  constexpr int PART = part_stride(G, D);
  float *out = a.out + (static_cast<int64_t>(b) * a.Hq + kvh * G) * D;
  float *mine = a.part + static_cast<int64_t>(slot) * PART;
  for (int idx = ctid; idx < GD; idx += kConsumerWarps * 32) {
    const int h = idx / D;
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) mstar = fmaxf(mstar, red[w * RED + GD + h]);
    float acc = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = red[w * RED + GD + h];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - mstar);
      acc = fmaf(f, red[w * RED + idx], acc);
      l = fmaf(f, red[w * RED + GD + G + h], l);
    }
    if (nparts == 1) {
      out[idx] = seg_bad ? 0.f : acc / l * a.v_scale;
    } else {
      mine[idx] = acc;
      if (idx % D == 0) {
        mine[GD + h] = mstar;
        mine[GD + G + h] = seg_bad ? -1.f : l;  // -1: this part met a bad page
      }
    }
  }
}

}  // namespace kvq
