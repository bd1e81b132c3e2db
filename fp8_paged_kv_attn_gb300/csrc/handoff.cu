// kvq_handoff_pages: the prefill -> decode handoff of whole prompts, from a
// paged BF16 cache into the paged e4m3 decode cache.
//
// Source: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全", section
// "KV 缓存量化": the prefill side keeps its KV cache in BF16 and the decode
// side stores it as e4m3, so every prompt handed from prefill to decode is
// converted once.  The pages give no kernel for it; this one reads the
// prompt's BF16 K/V where the prefill cache holds them (through the prefill
// block table, with the prefill pool's own page size) and writes the codes
// where the decode cache wants them (through the decode block table), with
// the rounding kvq_append uses (quant_e4m3.cuh), so a token handed off and a
// token appended during decode are stored identically.
//
// Work layout: grid (block groups, requests).  A request's positions are
// cut into 64-aligned blocks of 64; a CTA takes kHoBlocksPerCta consecutive
// blocks of one request, and a stage of its shared-memory ring is one
// (block, kv head): the block's K rows and V rows of that head.  In a
// prefill page a head's rows are contiguous, so a stage is filled by one
// 1-D bulk copy (TMA engine) per prefill page the block touches and tensor
// (page sizes 16..64 divide 64: one to four pages).  A producer warp looks up
// both block tables once per block (two positions per lane), writes each
// position's decode-pool offset into the stage's header and issues the
// copies; sixteen consumer warps convert 8 values a thread (one 16-byte
// shared-memory load, one 8-byte store; a warp stores 256 contiguous bytes)
// and release the stage.  Two CTAs per SM keep up to six stages (~192 KB)
// of reads in flight per SM, and 32 consumer warps per SM hide the latency
// of the quantiser's rare division.
// HBM-bound: per token and kv head 2 D (2 + s) bytes (read bf16 K and V,
// write s-byte codes), plus 4 bytes per prefill and per decode page.
#include <algorithm>
#include <atomic>

#include "kvq_internal.h"
#include "quant_e4m3.cuh"

namespace kvq {

struct HandoffArgs {
  const uint16_t *src_k, *src_v;  // bf16 [src_pages][H][Ps][D]
  void *dst_k, *dst_v;            // e4m3 or bf16 [dst_pages][H][Pd][D]
  const int32_t *src_bt, *dst_bt, *first, *count;
  uint32_t *err_word;
  int32_t src_pages, Ps, src_MP, dst_pages, Pd, dst_MP, H, B;
  QuantParams kq, vq;
};

constexpr int kHoBlock = 64;          // positions per stage: one 64-aligned block
constexpr int kHoConsumers = 16;      // consumer warps
constexpr int kHoThreads = 32 * (kHoConsumers + 1);
constexpr int kHoBlocksPerCta = 2;
constexpr int kHoMaxStages = 6;

template <int D>
struct HoCfg {
  static constexpr int ROW = 2 * D;             // bytes of one bf16 (token, head) row
  static constexpr int TILE = kHoBlock * ROW;   // one tensor's rows of a stage
  static constexpr int STAGE = 2 * TILE;        // K, then V
  static constexpr int NS = D == 128 ? 3 : 6;   // ring depth: 96 KB of rows
  static constexpr int GROUPS = kHoBlock * D / 8 / (32 * kHoConsumers);  // per thread and tensor
  static_assert(NS <= kHoMaxStages, "ring depth");
};

struct HoCtl {
  uint64_t full[kHoMaxStages], empty[kHoMaxStages];
  int32_t live[kHoMaxStages];  // 1: the stage holds a (block, head); 0: nothing follows
  int32_t fail;
};

template <int D>
constexpr size_t ho_smem_bytes() {
  return static_cast<size_t>(HoCfg<D>::NS) * HoCfg<D>::STAGE +
         static_cast<size_t>(HoCfg<D>::NS) * kHoBlock * sizeof(int64_t) + sizeof(HoCtl);
}

// Bounded wait of either role: on timeout the error bit is raised once and
// the fail flag tells the other role to leave.
__device__ __forceinline__ bool ho_wait(HoCtl &ctl, uint64_t *bar, uint32_t parity,
                                        uint32_t *err_word) {
  if (*reinterpret_cast<volatile int32_t *>(&ctl.fail)) return false;
  if (mbar_wait(bar, parity)) return true;
  if (atomicExch(&ctl.fail, 1) == 0) report(err_word, KVQ_ERRBIT_TIMEOUT);
  return false;
}

template <bool kFp8, int D>
__global__ void __launch_bounds__(kHoThreads, 2) handoff_kernel(HandoffArgs a) {
  using C = HoCfg<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *rows = smem;  // [NS][K rows | V rows], row r of a stage = position blk*64 + r
  int64_t *hdr = reinterpret_cast<int64_t *>(smem + C::NS * C::STAGE);  // [NS][64]
  HoCtl &ctl = *reinterpret_cast<HoCtl *>(smem + C::NS * C::STAGE + C::NS * kHoBlock * 8);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&ctl.full[i], 1);
      mbar_init(&ctl.empty[i], kHoConsumers);
    }
    ctl.fail = 0;
    fence_barrier_init();
  }
  __syncthreads();
  grid_dependency_wait();
  allow_dependents();
  // The grid's x extent comes from the tables' capacity, not the prompts'
  // lengths: a CTA with no block group of any of its requests leaves here,
  // all of it at once (the producer below reports bad ranges, so a CTA of
  // group 0 always stays).
  if (blockIdx.x > 0) {
    bool any = false;
    for (int b = blockIdx.y; !any && b < a.B; b += gridDim.y) {
      const int f = a.first ? __ldg(a.first + b) : 0;
      const int n = __ldg(a.count + b);
      any = n > 0 && f >= 0 &&
            f / kHoBlock + static_cast<long long>(blockIdx.x) * kHoBlocksPerCta <=
                (static_cast<long long>(f) + n - 1) / kHoBlock;
    }
    if (!any) return;
  }

  if (warp == kHoConsumers) {
    // ---------------------------------------------------------- producer
    const int64_t src_head = static_cast<int64_t>(a.Ps) * D;  // elements between heads
    const int64_t dst_head = static_cast<int64_t>(a.Pd) * D;
    const uint64_t pol = policy_evict_first();
    uint32_t g = 0;
    bool ok = true;
    for (int b = blockIdx.y; ok && b < a.B; b += gridDim.y) {
      const int f = a.first ? __ldg(a.first + b) : 0;
      const int n = __ldg(a.count + b);
      const long long end = static_cast<long long>(f) + n;
      if (f < 0 || n < 0 || end > static_cast<long long>(a.src_MP) * a.Ps ||
          end > static_cast<long long>(a.dst_MP) * a.Pd) {
        if (blockIdx.x == 0 && lane == 0) report(a.err_word, KVQ_ERRBIT_POS);
        continue;
      }
      if (n == 0) continue;
      // positions fit in 32 bits from here on: both tables hold at most
      // INT32_MAX tokens (checked by the host).  Block groups blockIdx.x,
      // blockIdx.x + gridDim.x, ... of the request are this CTA's.
      const int blk_first = f / kHoBlock, blk_last = (f + n - 1) / kHoBlock;
      for (int x = blockIdx.x; ok && blk_first + x * kHoBlocksPerCta <= blk_last;
           x += gridDim.x) {
        const int blk_end = min(blk_first + (x + 1) * kHoBlocksPerCta - 1, blk_last);
        for (int blk = blk_first + x * kHoBlocksPerCta; ok && blk <= blk_end; ++blk) {
          const int lo = max(blk * kHoBlock, f), hi = min(blk * kHoBlock + kHoBlock, f + n);
          // positions blk*64 + lane and + 32: the decode-pool offset (head 0;
          // -1: not stored) and, where a prefill page's piece starts, the copy
          int64_t doff[2], soff[2];
          int run[2];
          uint32_t tx = 0;
  #pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int p = blk * kHoBlock + lane + 32 * r;
            doff[r] = -1;
            soff[r] = 0;
            run[r] = 0;
            if (p >= lo && p < hi) {
              const int sp = __ldg(a.src_bt + static_cast<int64_t>(b) * a.src_MP + p / a.Ps);
              const int dp = __ldg(a.dst_bt + static_cast<int64_t>(b) * a.dst_MP + p / a.Pd);
              const bool src_ok = sp >= 0 && sp < a.src_pages;
              if (!src_ok || dp < 0 || dp >= a.dst_pages) report(a.err_word, KVQ_ERRBIT_PAGE);
              else doff[r] = (static_cast<int64_t>(dp) * a.H * a.Pd + p % a.Pd) * D;
              if (src_ok && (p == lo || p % a.Ps == 0)) {
                run[r] = min(hi, (p / a.Ps + 1) * a.Ps) - p;
                soff[r] = (static_cast<int64_t>(sp) * a.H * a.Ps + p % a.Ps) * D;
                tx += 2u * run[r] * C::ROW;
              }
            }
          }
          tx = __reduce_add_sync(0xffffffffu, tx);
          for (int h = 0; h < a.H; ++h, ++g) {
            const int slot = g % C::NS;
            bool waited = true;
            if (lane == 0 && g >= C::NS)
              waited = ho_wait(ctl, &ctl.empty[slot], ((g / C::NS) - 1) & 1, a.err_word);
            ok = __shfl_sync(0xffffffffu, waited ? 1 : 0, 0) != 0 &&
                 !*reinterpret_cast<volatile int32_t *>(&ctl.fail);
            if (!ok) break;
            int64_t *hd = hdr + slot * kHoBlock;
            hd[lane] = doff[0] < 0 ? -1 : doff[0] + h * dst_head;
            hd[lane + 32] = doff[1] < 0 ? -1 : doff[1] + h * dst_head;
            __syncwarp();
            if (lane == 0) {
              ctl.live[slot] = 1;
              mbar_arrive_expect_tx(&ctl.full[slot], tx);
            }
            __syncwarp();
  #pragma unroll
            for (int r = 0; r < 2; ++r) {
              if (run[r] == 0) continue;
              uint8_t *kdst = rows + slot * C::STAGE + (lane + 32 * r) * C::ROW;
              const int64_t src = soff[r] + h * src_head;
              const uint32_t bytes = static_cast<uint32_t>(run[r]) * C::ROW;
              bulk_g2s_hint(kdst, a.src_k + src, bytes, &ctl.full[slot], pol);
              bulk_g2s_hint(kdst + C::TILE, a.src_v + src, bytes, &ctl.full[slot], pol);
            }
          }
        }
      }
    }
    if (lane == 0) {
      if (ok) {
        // tell the consumers there is nothing more
        const int slot = g % C::NS;
        if (g < C::NS || ho_wait(ctl, &ctl.empty[slot], ((g / C::NS) - 1) & 1, a.err_word)) {
          ctl.live[slot] = 0;
          mbar_arrive(&ctl.full[slot]);
        }
      } else {
        // A wait gave up: before the CTA exits, let the copies it started
        // land (bounded waits), so that none writes into shared memory the
        // SM may already have handed to another CTA.  Only the last NS
        // stages can still be in flight.
        for (uint32_t s = g > C::NS ? g - C::NS : 0; s < g; ++s)
          mbar_wait(&ctl.full[s % C::NS], (s / C::NS) & 1);
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  uint32_t g = 0;
  while (true) {
    const int slot = g % C::NS;
    if (!ho_wait(ctl, &ctl.full[slot], (g / C::NS) & 1, a.err_word)) break;
    if (!ctl.live[slot]) break;
    const int64_t *hd = hdr + slot * kHoBlock;
    const uint8_t *st = rows + slot * C::STAGE;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
#pragma unroll
      for (int j = 0; j < C::GROUPS; ++j) {
        const int e = threadIdx.x + 32 * kHoConsumers * j;  // 8-value group of the tile
        const int row = e / (D / 8), col = (e % (D / 8)) * 8;
        const int64_t off = hd[row];
        if (off < 0) continue;
        const uint4 s = *reinterpret_cast<const uint4 *>(st + t * C::TILE + row * C::ROW + col * 2);
        if constexpr (kFp8) {
          uint8_t *dst = static_cast<uint8_t *>(t ? a.dst_v : a.dst_k) + off + col;
          *reinterpret_cast<uint2 *>(dst) = quantise8(s, t ? a.vq : a.kq);
        } else {
          uint16_t *dst = static_cast<uint16_t *>(t ? a.dst_v : a.dst_k) + off + col;
          *reinterpret_cast<uint4 *>(dst) = s;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl.empty[slot]);
    ++g;
  }
}

using HandoffFn = void (*)(HandoffArgs);

// Opt each variant into its shared-memory size once per device.
bool ho_smem_opt_in(HandoffFn fn, int variant, size_t bytes) {
  constexpr int kMaxDev = 64;
  static std::atomic<bool> done[kMaxDev][4];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  if (done[dev][variant].load(std::memory_order_acquire)) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes)) != cudaSuccess)
    return false;
  done[dev][variant].store(true, std::memory_order_release);
  return true;
}

}  // namespace kvq

using namespace kvq;

extern "C" kvq_status kvq_handoff_pages(const kvq_cache *src, const int32_t *src_block_table,
                                        int32_t src_MP, const kvq_cache *dst,
                                        const int32_t *dst_block_table, int32_t dst_MP,
                                        const int32_t *first, const int32_t *count, int32_t B,
                                        uint32_t *err_word, kvq_stream_t stream) {
  kvq_status st = validate_cache(src);
  if (st != KVQ_OK) return st;
  st = validate_cache(dst);
  if (st != KVQ_OK) return st;
  if (src->kv_dtype != KVQ_KV_BF16) return KVQ_ERR_INVALID_ARG;
  if (src->num_kv_heads != dst->num_kv_heads || src->head_dim != dst->head_dim)
    return KVQ_ERR_INVALID_ARG;
  const int H = src->num_kv_heads;
  if (H != 1 && H != 2 && H != 4 && H != 8) return KVQ_ERR_UNSUPPORTED;
  if (B < 0 || src_MP <= 0 || dst_MP <= 0) return KVQ_ERR_INVALID_ARG;
  if (B == 0) return KVQ_OK;
  if (!src_block_table || !dst_block_table || !count) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(src_MP) * src->page_size > INT32_MAX ||
      static_cast<int64_t>(dst_MP) * dst->page_size > INT32_MAX)
    return KVQ_ERR_INVALID_ARG;

  HandoffArgs a;
  a.src_k = static_cast<const uint16_t *>(src->k_pool);
  a.src_v = static_cast<const uint16_t *>(src->v_pool);
  a.dst_k = dst->k_pool;
  a.dst_v = dst->v_pool;
  a.src_bt = src_block_table;
  a.dst_bt = dst_block_table;
  a.first = first;
  a.count = count;
  a.err_word = err_word;
  a.src_pages = src->num_pages;
  a.Ps = src->page_size;
  a.src_MP = src_MP;
  a.dst_pages = dst->num_pages;
  a.Pd = dst->page_size;
  a.dst_MP = dst_MP;
  a.H = H;
  a.B = B;
  a.kq = quant_params(dst->k_scale);
  a.vq = quant_params(dst->v_scale);

  const bool fp8 = dst->kv_dtype == KVQ_KV_E4M3;
  const bool d128 = dst->head_dim == 128;
  const HandoffFn fn = d128 ? (fp8 ? handoff_kernel<true, 128> : handoff_kernel<false, 128>)
                            : (fp8 ? handoff_kernel<true, 64> : handoff_kernel<false, 64>);
  const size_t smem = d128 ? ho_smem_bytes<128>() : ho_smem_bytes<64>();
  if (!ho_smem_opt_in(fn, (d128 ? 2 : 0) + (fp8 ? 1 : 0), smem)) return KVQ_ERR_CUDA;
  // A request moves at most min(both capacities) tokens, which span at most
  // ceil(that / 64) blocks, so that many block groups a request cover any
  // prompt.  Tables sized for long contexts would make that grid mostly CTAs
  // with nothing to do; the x extent is capped so that the grid holds about
  // 16 waves of CTAs, and a CTA takes block groups x, x + gridDim.x, ...
  int sms = 0;
  if (device_sm_count(&sms) != KVQ_OK) return KVQ_ERR_CUDA;
  const int64_t max_tok = std::min(static_cast<int64_t>(src_MP) * src->page_size,
                                   static_cast<int64_t>(dst_MP) * dst->page_size);
  const int64_t blocks = (max_tok + kHoBlock - 1) / kHoBlock;
  const int64_t gy = B < 65535 ? B : 65535;
  const int64_t waves16 = 16LL * 2 * sms;  // 2 CTAs per SM
  const int64_t gx = std::min((blocks + kHoBlocksPerCta - 1) / kHoBlocksPerCta,
                              std::max<int64_t>(1, (waves16 + gy - 1) / gy));
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy));
  const cudaError_t e = launch_dependent(fn, grid, kHoThreads, smem,
                                         reinterpret_cast<cudaStream_t>(stream), a);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}
