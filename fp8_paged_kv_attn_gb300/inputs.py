"""Seeded synthetic workloads for the paged FP8 decode path.

This module only draws inputs: shapes, lengths, bf16 query/key/value bit
patterns, block tables, page tags and per-tensor scales.  It contains none of
the method's arithmetic (no quantisation, no attention, no tag comparison), so
both the CPU oracle's tests and the CUDA path may use it.

The shapes follow the pages' decode workloads (8192-token prompts, 1000
generated tokens, 1 to 64 concurrent requests; integrity overhead measured at
8192 in / 1000 out) -- page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全",
tables in sections "KV 缓存量化" and "共享 KV 缓存保护" -- with head counts, head
dim, page sizes and length mixes fixed by the workload definitions below.

Recipe (all draws from numpy ``default_rng`` with the seed spelled out):
  * K/V/Q source values ~ N(0, 1) in fp32, optionally 1% of entries x20
    ("outliers"), rounded to bf16 with round-to-nearest-even.  The cached
    context of request b is drawn from seed [seed, b, 1] (K) and [seed, b, 2]
    (V) so any request can be regenerated alone.
  * per-tensor scales: amax(|K source|) / 448 and amax(|V source|) / 448 in
    fp32, taken over the cached context (calibration happens before decode).
  * block tables: pages handed out from a seeded shuffled free list, after a
    seeded history of allocate/free churn for the fragmented workloads.
  * page tags: a uint32 counter per physical page, incremented each time the
    page is handed out; a request records the tag of every page it received.
  * stale injection: a victim request's page is freed and handed out again
    (its tag moves on) while the victim keeps the old expected tag.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np

E4M3_MAX = 448.0  # largest finite e4m3 magnitude; fixes the calibration scale


# --------------------------------------------------------------------------
# bf16 bit patterns
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, outlier_frac: float = 0.0,
                outlier_mult: float = 20.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if outlier_frac > 0.0:
        mask = rng.random(size=shape, dtype=np.float32) < outlier_frac
        x[mask] *= np.float32(outlier_mult)
    return f32_to_bf16_bits(x)


def amax_bf16(b: np.ndarray) -> float:
    if b.size == 0:
        return 0.0
    # |x| of a bf16 is its bit pattern with the sign cleared; the order of
    # non-negative finite floats follows their bit patterns.
    m = int((np.asarray(b, dtype=np.uint16) & np.uint16(0x7FFF)).max())
    return float(bf16_bits_to_f32(np.array([m], dtype=np.uint16))[0])


def scale_from_amax(amax: float) -> np.float32:
    s = np.float32(amax) / np.float32(E4M3_MAX)
    return s if s > 0 else np.float32(1.0)


# --------------------------------------------------------------------------
# Host page pool with tags
# --------------------------------------------------------------------------

class PagePool:
    """Physical page ids handed out from a seeded shuffled free list.

    ``tags[p]`` counts how many times page p has been handed out (uint32,
    wrapping).  This is the state the integrity check reads.
    """

    def __init__(self, num_pages: int, rng: np.random.Generator):
        self.num_pages = int(num_pages)
        self.rng = rng
        self.free: List[int] = list(rng.permutation(self.num_pages).astype(np.int64))
        self.tags = np.zeros(self.num_pages, dtype=np.uint32)

    def alloc(self) -> Tuple[int, int]:
        if not self.free:
            raise MemoryError("page pool exhausted")
        p = int(self.free.pop())
        self.tags[p] = np.uint32((int(self.tags[p]) + 1) & 0xFFFFFFFF)
        return p, int(self.tags[p])

    def release(self, p: int) -> None:
        # freed pages go back at a random spot, so reuse order is scrambled
        i = int(self.rng.integers(0, len(self.free) + 1))
        self.free.insert(i, int(p))

    def churn(self, n_events: int, live_max: int) -> None:
        """Allocate/free history that fragments the free list and bumps tags."""
        live: List[int] = []
        for _ in range(n_events):
            if live and (len(live) >= live_max or self.rng.random() < 0.5):
                j = int(self.rng.integers(0, len(live)))
                self.release(live.pop(j))
            else:
                live.append(self.alloc()[0])
        for p in live:
            self.release(p)


# --------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------

@dataclass
class Workload:
    """One synthetic decode workload.

    ctx_lens[b]: tokens already cached for request b before the first decode
    step.  Decode step s appends one token per request at position
    ctx_lens[b] + s and then attends over ctx_lens[b] + s + 1 tokens.
    """
    name: str
    seed: int
    B: int
    Hq: int
    Hkv: int
    D: int
    P: int
    num_pages: int
    MP: int
    ctx_lens: np.ndarray                  # int32 [B]
    block_table: np.ndarray               # int32 [B, MP] (-1 past the allocation)
    page_tags: np.ndarray                 # uint32 [num_pages]
    expected_tags: np.ndarray             # uint32 [B, MP]
    outlier_frac: float = 0.0
    stale: List[int] = field(default_factory=list)
    _k_scale: Optional[np.float32] = None
    _v_scale: Optional[np.float32] = None

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def sm_scale(self) -> np.float32:
        return np.float32(1.0) / np.sqrt(np.float32(self.D))

    # ---- cached context -------------------------------------------------
    def kv_source(self, b: int) -> Tuple[np.ndarray, np.ndarray]:
        """bf16 bits [ctx_lens[b], Hkv, D] for K and V of request b's context."""
        L = int(self.ctx_lens[b])
        shape = (L, self.Hkv, self.D)
        k = normal_bf16(np.random.default_rng([self.seed, b, 1]), shape, self.outlier_frac)
        v = normal_bf16(np.random.default_rng([self.seed, b, 2]), shape, self.outlier_frac)
        return k, v

    def kv_sources(self, requests=None, threads: int = 16):
        reqs = list(range(self.B)) if requests is None else list(requests)
        with ThreadPoolExecutor(max_workers=max(1, threads)) as ex:
            return list(ex.map(self.kv_source, reqs))

    def scales(self, sources=None) -> Tuple[np.float32, np.float32]:
        """Per-tensor k_scale, v_scale = amax / 448 over the cached context."""
        if self._k_scale is None:
            if sources is None:
                sources = self.kv_sources()
            ka = max((amax_bf16(k) for k, _ in sources), default=0.0)
            va = max((amax_bf16(v) for _, v in sources), default=0.0)
            self._k_scale, self._v_scale = scale_from_amax(ka), scale_from_amax(va)
        return self._k_scale, self._v_scale

    # ---- decode steps ---------------------------------------------------
    def step_inputs(self, step: int):
        """q [B,Hq,D], k_new/v_new [B,Hkv,D] (bf16 bits), req_idx, pos (int32 [B])."""
        rng = np.random.default_rng([self.seed, 1_000_000 + step])
        q = normal_bf16(rng, (self.B, self.Hq, self.D))
        k_new = normal_bf16(rng, (self.B, self.Hkv, self.D), self.outlier_frac)
        v_new = normal_bf16(rng, (self.B, self.Hkv, self.D), self.outlier_frac)
        req_idx = np.arange(self.B, dtype=np.int32)
        pos = (self.ctx_lens + step).astype(np.int32)
        return q, k_new, v_new, req_idx, pos

    def seq_lens_after(self, step: int) -> np.ndarray:
        return (self.ctx_lens + step + 1).astype(np.int32)

    # ---- sizes ------------------------------------------------------------
    def pool_shape(self):
        return (self.num_pages, self.Hkv, self.P, self.D)

    def context_tokens(self, b: int) -> Tuple[np.ndarray, np.ndarray]:
        """(req_idx, pos) for appending request b's whole cached context."""
        L = int(self.ctx_lens[b])
        return np.full(L, b, dtype=np.int32), np.arange(L, dtype=np.int32)


def _assign_pages(pool: PagePool, B: int, MP: int, caps_pages) -> Tuple[np.ndarray, np.ndarray]:
    bt = np.full((B, MP), -1, dtype=np.int32)
    exp = np.zeros((B, MP), dtype=np.uint32)
    for b in range(B):
        for i in range(int(caps_pages[b])):
            p, t = pool.alloc()
            bt[b, i] = p
            exp[b, i] = t
    return bt, exp


def _inject_stale(w: Workload, pool: PagePool, rng: np.random.Generator, victims,
                  pages_per_victim: int = 1) -> None:
    """Free and re-hand-out a checked page of each victim: the page's tag moves
    on while the victim still expects the old one."""
    lens = w.seq_lens_after(0)
    for b in victims:
        n_pages = max(1, -(-int(lens[b]) // w.P))
        idx = rng.choice(n_pages, size=min(pages_per_victim, n_pages), replace=False)
        for i in idx:
            p = int(w.block_table[b, i])
            pool.release(p)
            # hand the same page out again (as if another request took it)
            pool.free.remove(p)
            pool.free.append(p)
            pool.alloc()
        w.stale.append(int(b))
    w.page_tags = pool.tags.copy()


def tiny(seed: int = 0) -> Workload:
    """2 requests with 37 and 64 cached tokens, 4 q heads / 1 kv head, D=64,
    page 16, a 16-page pool whose pages are a random permutation split over
    the two block tables; all tags match."""
    rng = np.random.default_rng(seed)
    B, Hq, Hkv, D, P, NP = 2, 4, 1, 64, 16, 16
    MP = NP // B
    perm = rng.permutation(NP).astype(np.int32)
    bt = perm.reshape(B, MP).copy()
    tags = np.zeros(NP, dtype=np.uint32)
    return Workload("tiny", seed, B, Hq, Hkv, D, P, NP, MP,
                    np.array([37, 64], dtype=np.int32), bt, tags,
                    np.zeros((B, MP), dtype=np.uint32))


def uniform(name: str, seed: int, B: int, ctx: int, Hq: int, Hkv: int, D: int, P: int,
            decode_steps: int = 1, pool_factor: float = 2.0, outlier_frac: float = 0.01,
            num_pages: Optional[int] = None) -> Workload:
    """B requests of equal context with shuffled block tables in a pool of
    pool_factor x the pages needed for ctx + decode_steps tokens."""
    rng = np.random.default_rng(seed)
    cap_pages = -(-(ctx + decode_steps) // P)
    NP = int(num_pages) if num_pages is not None else int(math.ceil(pool_factor * B * cap_pages))
    if B * cap_pages > NP:
        raise MemoryError(f"{name}: {B} requests need {B * cap_pages} pages, pool has {NP}")
    pool = PagePool(NP, rng)
    bt, exp = _assign_pages(pool, B, cap_pages, [cap_pages] * B)
    return Workload(name, seed, B, Hq, Hkv, D, P, NP, cap_pages,
                    np.full(B, ctx, dtype=np.int32), bt, pool.tags.copy(), exp,
                    outlier_frac=outlier_frac)


def cfg8x8k(seed: int = 1) -> Workload:
    """8 requests x 8192 cached tokens, 32 q / 8 kv heads, D=128, page 16,
    pool 2x the needed pages, 1% outliers x20, one decode step."""
    return uniform("8x8192_gqa32/8_d128_p16", seed, 8, 8192, 32, 8, 128, 16)


SWEEP_PROMPT = 8192
SWEEP_DECODE_STEPS = 1000
SWEEP_POOL_REQUESTS = 64  # FP8 pool sized for 64 requests; BF16 pool of equal bytes holds half


def sweep(B: int, kv_bytes: int = 1, seed: int = 2) -> Workload:
    """Concurrency sweep point: B requests, 8192-token prompt, room for 1000
    decode steps, 32/8 heads, D=128, page 16.  The pool holds a fixed number of
    BYTES (64 requests' worth at 1 byte per element): with 2-byte (bf16)
    elements it holds half the pages, so more than 32 requests raise
    MemoryError, like running out of KV cache."""
    P, Hkv, D = 16, 8, 128
    cap_pages = -(-(SWEEP_PROMPT + SWEEP_DECODE_STEPS) // P)
    pool_pages = SWEEP_POOL_REQUESTS * cap_pages // kv_bytes
    return uniform(f"sweep_b{B}", seed, B, SWEEP_PROMPT, 32, Hkv, D, P,
                   decode_steps=SWEEP_DECODE_STEPS, num_pages=pool_pages)


def ragged(seed: int = 3, B: int = 64, total: int = 1_370_000, lo: int = 512,
           hi: int = 131072, Hq: int = 64, Hkv: int = 8, D: int = 128, P: int = 64,
           pool_factor: float = 1.25, churn_events: Optional[int] = None) -> Workload:
    """Log-uniform lengths in [lo, hi], rescaled once so they sum to about
    `total` and clamped back into [lo, hi]; pages come from a pool 1.25x the
    need whose free list went through random allocate/free churn."""
    rng = np.random.default_rng(seed)
    raw = np.exp(rng.uniform(np.log(lo), np.log(hi), size=B))
    lens = np.clip(np.round(raw * (total / raw.sum())), lo, hi).astype(np.int64)
    caps = [-(-(int(L) + 1) // P) for L in lens]
    NP = int(math.ceil(pool_factor * sum(caps)))
    pool = PagePool(NP, rng)
    pool.churn(churn_events if churn_events is not None else 2 * NP, live_max=NP // 2)
    MP = max(caps)
    bt, exp = _assign_pages(pool, B, MP, caps)
    return Workload(f"ragged_b{B}_p{P}", seed, B, Hq, Hkv, D, P, NP, MP,
                    lens.astype(np.int32), bt, pool.tags.copy(), exp, outlier_frac=0.01)


def integrity(seed: int = 4, B: int = 256, lo: int = 1024, hi: int = 16384,
              Hq: int = 32, Hkv: int = 8, D: int = 128, P: int = 16,
              stale_frac: float = 0.001, pages_per_victim: int = 1,
              pool_factor: float = 1.25) -> Workload:
    """Lengths uniform in [lo, hi]; tags bumped over an allocate/free history;
    stale tags injected into max(1, round(stale_frac * B)) requests."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi + 1, size=B).astype(np.int64)
    caps = [-(-(int(L) + 1) // P) for L in lens]
    NP = int(math.ceil(pool_factor * sum(caps)))
    pool = PagePool(NP, rng)
    pool.churn(NP, live_max=NP // 2)
    MP = max(caps)
    bt, exp = _assign_pages(pool, B, MP, caps)
    w = Workload(f"integrity_b{B}", seed, B, Hq, Hkv, D, P, NP, MP, lens.astype(np.int32),
                 bt, pool.tags.copy(), exp, outlier_frac=0.01)
    n_victims = max(1, int(round(stale_frac * B)))
    victims = sorted(int(v) for v in rng.choice(B, size=n_victims, replace=False))
    _inject_stale(w, pool, rng, victims, pages_per_victim)
    return w


@dataclass
class Handoff:
    """A prefill -> decode handoff: B prompts held in a paged BF16 prefill
    cache (page size src_P) to be moved into the paged decode cache (page
    size dst_P).  Request b's tokens [first[b], first[b] + count[b]) move;
    both block tables come from seeded shuffled free lists.  K/V values are
    drawn like the decode workloads' (kv_source)."""
    name: str
    seed: int
    B: int
    Hkv: int
    D: int
    src_P: int
    dst_P: int
    src_pages: int
    dst_pages: int
    first: np.ndarray            # int32 [B]
    count: np.ndarray            # int32 [B]
    src_block_table: np.ndarray  # int32 [B, src_MP]
    dst_block_table: np.ndarray  # int32 [B, dst_MP]
    outlier_frac: float = 0.01

    @property
    def src_MP(self) -> int:
        return self.src_block_table.shape[1]

    @property
    def dst_MP(self) -> int:
        return self.dst_block_table.shape[1]

    def kv_source(self, b: int) -> Tuple[np.ndarray, np.ndarray]:
        """bf16 bits [first[b] + count[b], Hkv, D] for K and V of request b's
        prompt (positions 0 .. first + count - 1)."""
        L = int(self.first[b] + self.count[b])
        shape = (L, self.Hkv, self.D)
        k = normal_bf16(np.random.default_rng([self.seed, b, 1]), shape, self.outlier_frac)
        v = normal_bf16(np.random.default_rng([self.seed, b, 2]), shape, self.outlier_frac)
        return k, v

    def src_shape(self):
        return (self.src_pages, self.Hkv, self.src_P, self.D)

    def dst_shape(self):
        return (self.dst_pages, self.Hkv, self.dst_P, self.D)


def handoff(seed: int = 5, B: int = 64, lens=None, first=None, Hkv: int = 8, D: int = 128,
            src_P: int = 64, dst_P: int = 16, src_pool_factor: float = 1.25,
            decode_room: int = SWEEP_DECODE_STEPS, dst_pool_factor: float = 1.0) -> Handoff:
    """Prompts of `lens` tokens (default: B x 8192, the sweep's prompts)
    moved from a prefill pool of src_P-token pages (1.25x the need) into a
    decode pool of dst_P-token pages with room for `decode_room` more tokens
    per request.  `first` (default zeros) offsets each request's range."""
    rng = np.random.default_rng(seed)
    lens = np.full(B, SWEEP_PROMPT, dtype=np.int64) if lens is None else \
        np.asarray(lens, dtype=np.int64)
    B = int(lens.shape[0])
    first = np.zeros(B, dtype=np.int64) if first is None else np.asarray(first, dtype=np.int64)
    ends = first + lens
    src_caps = [max(1, -(-int(e) // src_P)) for e in ends]
    dst_caps = [max(1, -(-(int(e) + decode_room) // dst_P)) for e in ends]
    src_np = int(math.ceil(src_pool_factor * sum(src_caps)))
    dst_np = int(math.ceil(dst_pool_factor * sum(dst_caps)))
    src_pool = PagePool(src_np, rng)
    dst_pool = PagePool(dst_np, rng)
    sbt, _ = _assign_pages(src_pool, B, max(src_caps), src_caps)
    dbt, _ = _assign_pages(dst_pool, B, max(dst_caps), dst_caps)
    return Handoff(f"handoff_b{B}_p{src_P}to{dst_P}", seed, B, Hkv, D, src_P, dst_P, src_np,
                   dst_np, first.astype(np.int32), lens.astype(np.int32), sbt, dbt)
