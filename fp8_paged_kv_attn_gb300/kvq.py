"""Python binding of the kvq C ABI (include/kvq.h): argument marshalling only.

Every function here checks tensor devices, dtypes and shapes, takes raw
device pointers and the current CUDA stream, and calls the function of the
same name in libkvq.so.  All computation happens in the library's kernels;
there is no fallback: if the library cannot be built or loaded, every call
raises.

Tensor conventions (torch is used for device memory and streams only):
  pools          uint8 (e4m3 codes) or bfloat16, [num_pages, Hkv, P, D]
  q              bfloat16 [B, Hq, D]; out float32 [B, Hq, D]
  k_new, v_new   bfloat16 [N, Hkv, D]
  block_table    int32 [B, MP]; seq_lens, req_idx, pos int32
  page_tags      int32/uint32 [num_pages]; expected_tags [B, MP]
  abort_mask     uint8 [B]; err_word int32/uint32 [1]
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

from . import _build

KV_E4M3 = 0
KV_BF16 = 1
W_INT4 = 0
W_E4M3 = 1

ERRBIT_PAGE = 1 << 0
ERRBIT_SEQLEN = 1 << 1
ERRBIT_POS = 1 << 2
ERRBIT_REQ = 1 << 3
ERRBIT_TIMEOUT = 1 << 4
ERRBIT_EXHAUSTED = 1 << 5

STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_INVALID_ARG", 2: "KVQ_ERR_WORKSPACE", 3: "KVQ_ERR_CUDA",
          4: "KVQ_ERR_UNSUPPORTED"}

# every symbol include/kvq.h declares
EXPORTS = ("kvq_append", "kvq_append_check", "kvq_handoff_pages", "kvq_check_tags",
           "kvq_pages_update", "kvq_decode_attn_workspace_size", "kvq_decode_attn",
           "kvq_decode_attn_static", "kvq_wq_gemm", "kvq_selftest_wait", "kvq_status_string")
STATIC_SCRATCH_BYTES = 64 << 20


class KvqError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


class CCache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("kv_dtype", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libkvq.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"CUDA library missing: {_build.LIB}")
    L = ctypes.CDLL(_build.LIB)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    cp = ctypes.POINTER(CCache)
    L.kvq_append.argtypes = [cp, vp, vp, vp, vp, i32, vp, i32, i32, vp, vp]
    L.kvq_append.restype = ctypes.c_int
    L.kvq_append_check.argtypes = [cp, vp, vp, vp, vp, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp]
    L.kvq_append_check.restype = ctypes.c_int
    L.kvq_handoff_pages.argtypes = [cp, vp, i32, cp, vp, i32, vp, vp, i32, vp, vp]
    L.kvq_handoff_pages.restype = ctypes.c_int
    L.kvq_check_tags.argtypes = [vp, i32, i32, vp, i32, vp, i32, vp, vp, vp]
    L.kvq_check_tags.restype = ctypes.c_int
    L.kvq_pages_update.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, vp, vp, i32, vp, vp, vp,
                                   i32, vp, vp, vp]
    L.kvq_pages_update.restype = ctypes.c_int
    L.kvq_wq_gemm.argtypes = [i32, vp, vp, vp, vp, i32, i32, i32, vp, vp]
    L.kvq_wq_gemm.restype = ctypes.c_int
    L.kvq_selftest_wait.argtypes = [i32, vp, vp, vp, vp]
    L.kvq_selftest_wait.restype = ctypes.c_int
    L.kvq_decode_attn_workspace_size.argtypes = [i32, i32, i32, i32]
    L.kvq_decode_attn_workspace_size.restype = sz
    L.kvq_decode_attn.argtypes = [cp, vp, i32, i32, vp, i32, vp, vp, f32, vp, vp, sz, vp, vp]
    L.kvq_decode_attn.restype = ctypes.c_int
    L.kvq_decode_attn_static.argtypes = [cp, vp, i32, i32, vp, i32, vp, vp, f32, vp, vp, vp]
    L.kvq_decode_attn_static.restype = ctypes.c_int
    L.kvq_status_string.argtypes = [ctypes.c_int]
    L.kvq_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dev(t: Optional[torch.Tensor], name: str, dtypes, ndim=None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, has {t.dim()}")
    return ctypes.c_void_p(t.data_ptr())


def _check(fn: str, status: int):
    if status != 0:
        raise KvqError(fn, status)


I32 = (torch.int32,)
U32 = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
U8 = (torch.uint8, torch.bool)
BF16 = (torch.bfloat16,)


@dataclass
class KVCache:
    """Caller-owned paged K/V pools ([num_pages, Hkv, P, D]) and their scales."""
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def kv_dtype(self) -> int:
        return KV_E4M3 if self.k_pool.element_size() == 1 else KV_BF16

    @property
    def shape(self):
        return tuple(self.k_pool.shape)

    def c(self) -> CCache:
        dt = (torch.uint8, torch.float8_e4m3fn, torch.bfloat16)
        _dev(self.k_pool, "k_pool", dt, 4)
        _dev(self.v_pool, "v_pool", dt, 4)
        if self.k_pool.shape != self.v_pool.shape or self.k_pool.dtype != self.v_pool.dtype:
            raise ValueError("k_pool and v_pool must match")
        NP, H, P, D = self.k_pool.shape
        return CCache(self.k_pool.data_ptr(), self.v_pool.data_ptr(), self.kv_dtype, NP, P, H, D,
                      float(self.k_scale), float(self.v_scale))

    @staticmethod
    def empty(num_pages, num_kv_heads, page_size, head_dim, kv_dtype=KV_E4M3, k_scale=1.0,
              v_scale=1.0, device="cuda"):
        dt = torch.uint8 if kv_dtype == KV_E4M3 else torch.bfloat16
        shape = (num_pages, num_kv_heads, page_size, head_dim)
        return KVCache(torch.empty(shape, dtype=dt, device=device),
                       torch.empty(shape, dtype=dt, device=device), k_scale, v_scale)


# ----------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ----------------------------------------------------------------------------

def kvq_append(cache: KVCache, k_new, v_new, req_idx, pos, block_table, err_word=None,
               stream=None) -> None:
    L = load()
    c = cache.c()
    N = int(req_idx.shape[0])
    B, MP = block_table.shape
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        if tuple(t.shape) != (N, c.num_kv_heads, c.head_dim):
            raise ValueError(f"{n} must be [{N}, {c.num_kv_heads}, {c.head_dim}]")
    st = L.kvq_append(ctypes.byref(c), _dev(k_new, "k_new", BF16, 3), _dev(v_new, "v_new", BF16, 3),
                      _dev(req_idx, "req_idx", I32, 1), _dev(pos, "pos", I32, 1), N,
                      _dev(block_table, "block_table", I32, 2), B, MP,
                      _dev(err_word, "err_word", U32), _stream(stream))
    _check("kvq_append", st)


def kvq_append_check(cache: KVCache, k_new, v_new, req_idx, pos, block_table, seq_lens,
                     page_tags, expected_tags, abort_mask, err_word=None, stream=None) -> None:
    """kvq_append and kvq_check_tags (the cache's page size and page count)
    in one launch, with the same results as the two calls."""
    L = load()
    c = cache.c()
    N = int(req_idx.shape[0])
    B, MP = block_table.shape
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        if tuple(t.shape) != (N, c.num_kv_heads, c.head_dim):
            raise ValueError(f"{n} must be [{N}, {c.num_kv_heads}, {c.head_dim}]")
    if tuple(expected_tags.shape) != (B, MP) or abort_mask.shape[0] != B or \
            seq_lens.shape[0] != B or page_tags.shape[0] != c.num_pages:
        raise ValueError("expected_tags must be [B, MP], seq_lens and abort_mask [B], "
                         "page_tags [num_pages]")
    st = L.kvq_append_check(ctypes.byref(c), _dev(k_new, "k_new", BF16, 3),
                            _dev(v_new, "v_new", BF16, 3), _dev(req_idx, "req_idx", I32, 1),
                            _dev(pos, "pos", I32, 1), N, _dev(block_table, "block_table", I32, 2),
                            B, MP, _dev(seq_lens, "seq_lens", I32, 1),
                            _dev(page_tags, "page_tags", U32, 1),
                            _dev(expected_tags, "expected_tags", U32, 2),
                            _dev(abort_mask, "abort_mask", U8, 1), _dev(err_word, "err_word", U32),
                            _stream(stream))
    _check("kvq_append_check", st)


def kvq_handoff_pages(src: KVCache, src_block_table, dst: KVCache, dst_block_table, count,
                      first=None, err_word=None, stream=None) -> None:
    """Prefill -> decode handoff: tokens [first[b], first[b] + count[b]) of
    every request b, read from the paged bf16 cache `src` through
    src_block_table [B, src_MP] and stored into `dst` through
    dst_block_table [B, dst_MP] with kvq_append's rounding."""
    L = load()
    cs, cd = src.c(), dst.c()
    B, src_MP = src_block_table.shape
    if dst_block_table.shape[0] != B or count.shape[0] != B or \
            (first is not None and first.shape[0] != B):
        raise ValueError("dst_block_table, count and first must have B rows")
    st = L.kvq_handoff_pages(ctypes.byref(cs), _dev(src_block_table, "src_block_table", I32, 2),
                             src_MP, ctypes.byref(cd),
                             _dev(dst_block_table, "dst_block_table", I32, 2),
                             int(dst_block_table.shape[1]), _dev(first, "first", I32, 1),
                             _dev(count, "count", I32, 1), B, _dev(err_word, "err_word", U32),
                             _stream(stream))
    _check("kvq_handoff_pages", st)


def kvq_check_tags(block_table, seq_lens, page_size: int, page_tags, expected_tags, abort_mask,
                   stream=None) -> None:
    L = load()
    B, MP = block_table.shape
    if tuple(expected_tags.shape) != (B, MP) or abort_mask.shape[0] != B:
        raise ValueError("expected_tags must be [B, MP] and abort_mask [B]")
    st = L.kvq_check_tags(_dev(block_table, "block_table", I32, 2), B, MP,
                          _dev(seq_lens, "seq_lens", I32, 1), int(page_size),
                          _dev(page_tags, "page_tags", U32, 1), int(page_tags.shape[0]),
                          _dev(expected_tags, "expected_tags", U32, 2),
                          _dev(abort_mask, "abort_mask", U8, 1), _stream(stream))
    _check("kvq_check_tags", st)


@dataclass
class PageState:
    """The page allocator's device state (include/kvq.h, kvq_pages_update):
    free_stack int32 [num_pages] with free_count[0] live entries (top = last),
    page_tags int32/uint32 [num_pages], block_table int32 [B, MP] and
    expected_tags int32/uint32 [B, MP] (the tables kvq_check_tags reads)."""
    free_stack: torch.Tensor
    free_count: torch.Tensor
    page_tags: torch.Tensor
    block_table: torch.Tensor
    expected_tags: torch.Tensor


def kvq_pages_update(state: PageState, rel_req=None, rel_npages=None, acq_req=None,
                     acq_first=None, acq_npages=None, acq_ok=None, err_word=None,
                     stream=None) -> None:
    """One batch of page releases then acquisitions (see include/kvq.h)."""
    L = load()
    num_pages = int(state.free_stack.shape[0])
    B, MP = state.block_table.shape
    if tuple(state.page_tags.shape) != (num_pages,) or state.free_count.numel() != 1:
        raise ValueError("page_tags must be [num_pages] and free_count [1]")
    if tuple(state.expected_tags.shape) != (B, MP):
        raise ValueError("expected_tags must match block_table")
    n_rel = 0 if rel_req is None else int(rel_req.shape[0])
    n_acq = 0 if acq_req is None else int(acq_req.shape[0])
    if n_rel and rel_npages.shape != rel_req.shape:
        raise ValueError("rel_npages must match rel_req")
    if n_acq and (acq_first.shape != acq_req.shape or acq_npages.shape != acq_req.shape or
                  acq_ok is None or acq_ok.shape != acq_req.shape):
        raise ValueError("acq_first, acq_npages and acq_ok must match acq_req")
    st = L.kvq_pages_update(_dev(state.free_stack, "free_stack", I32, 1),
                            _dev(state.free_count, "free_count", I32),
                            _dev(state.page_tags, "page_tags", U32, 1), num_pages,
                            _dev(state.block_table, "block_table", I32, 2),
                            _dev(state.expected_tags, "expected_tags", U32, 2), B, MP,
                            _dev(rel_req, "rel_req", I32, 1), _dev(rel_npages, "rel_npages", I32, 1),
                            n_rel, _dev(acq_req, "acq_req", I32, 1),
                            _dev(acq_first, "acq_first", I32, 1),
                            _dev(acq_npages, "acq_npages", I32, 1), n_acq,
                            _dev(acq_ok, "acq_ok", U8, 1), _dev(err_word, "err_word", U32),
                            _stream(stream))
    _check("kvq_pages_update", st)


def kvq_wq_gemm(w_dtype: int, w, scales, x, y, err_word=None, stream=None) -> None:
    """y [M, N] fp32 = x [M, K] bf16 times the quantised weights (include/kvq.h):
    W_INT4: w uint8 [N, K/2], scales bf16 (or int16 bits) [N, K/128];
    W_E4M3: w uint8 [N, K], scales fp32 [N].  err_word: optional int32 [1]
    device tensor that collects KVQ_ERRBIT_TIMEOUT."""
    L = load()
    M, K = x.shape
    N = int(w.shape[0])
    if tuple(y.shape) != (M, N):
        raise ValueError("y must be [M, N]")
    if w_dtype == W_INT4:
        if tuple(w.shape) != (N, K // 2) or tuple(scales.shape) != (N, K // 128):
            raise ValueError("INT4 weights must be [N, K/2] with scales [N, K/128]")
        sc = _dev(scales, "scales", (torch.bfloat16, torch.int16), 2)
    else:
        if tuple(w.shape) != (N, K) or tuple(scales.shape) != (N,):
            raise ValueError("e4m3 weights must be [N, K] with scales [N]")
        sc = _dev(scales, "scales", (torch.float32,), 1)
    st = L.kvq_wq_gemm(int(w_dtype), _dev(w, "w", U8, 2), sc, _dev(x, "x", BF16, 2),
                       _dev(y, "y", (torch.float32,), 2), M, N, K,
                       _dev(err_word, "err_word", U32), _stream(stream))
    _check("kvq_wq_gemm", st)


def kvq_selftest_wait(which: int, src, err_word, landed, stream=None) -> None:
    """Launch the bounded-wait self-test (include/kvq.h): which = 0 the split
    attention kernels' wait, 1 the weight ring's.  src: 16 int32 on the
    device; err_word, landed: int32 [1] device tensors."""
    L = load()
    st = L.kvq_selftest_wait(int(which), _dev(src, "src", U32), _dev(err_word, "err_word", U32),
                             _dev(landed, "landed", U32), _stream(stream))
    _check("kvq_selftest_wait", st)


def kvq_decode_attn_workspace_size(B: int, Hq: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load().kvq_decode_attn_workspace_size(B, Hq, num_kv_heads, head_dim))


def workspace(B: int, Hq: int, num_kv_heads: int, head_dim: int, device="cuda") -> torch.Tensor:
    """Allocate (with torch) a workspace of the size kvq_decode_attn needs."""
    n = kvq_decode_attn_workspace_size(B, Hq, num_kv_heads, head_dim)
    return torch.empty(n, dtype=torch.uint8, device=device)


def kvq_decode_attn(cache: KVCache, q, block_table, seq_lens, out, workspace, abort_mask=None,
                    sm_scale: Optional[float] = None, err_word=None, stream=None) -> None:
    L = load()
    c = cache.c()
    B, Hq, D = q.shape
    if D != c.head_dim or tuple(out.shape) != (B, Hq, D):
        raise ValueError("q / out shapes do not match the cache")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens must have B rows")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    st = L.kvq_decode_attn(ctypes.byref(c), _dev(q, "q", BF16, 3), B, Hq,
                           _dev(block_table, "block_table", I32, 2), int(block_table.shape[1]),
                           _dev(seq_lens, "seq_lens", I32, 1),
                           _dev(abort_mask, "abort_mask", U8, 1), float(sm_scale),
                           _dev(out, "out", (torch.float32,), 3),
                           _dev(workspace, "workspace", (torch.uint8,), 1),
                           workspace.numel() * workspace.element_size(),
                           _dev(err_word, "err_word", U32), _stream(stream))
    _check("kvq_decode_attn", st)


def kvq_decode_attn_static(cache: KVCache, q, block_table, seq_lens, out, abort_mask=None,
                           sm_scale: Optional[float] = None, err_word=None, stream=None) -> None:
    """kvq_decode_attn with the library's own static scratch instead of a
    caller workspace, for callers that cannot allocate device memory (see
    include/kvq.h).  Calls that can overlap on the GPU must not be issued."""
    L = load()
    c = cache.c()
    B, Hq, D = q.shape
    if D != c.head_dim or tuple(out.shape) != (B, Hq, D):
        raise ValueError("q / out shapes do not match the cache")
    if block_table.shape[0] != B or seq_lens.shape[0] != B:
        raise ValueError("block_table / seq_lens must have B rows")
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    st = L.kvq_decode_attn_static(ctypes.byref(c), _dev(q, "q", BF16, 3), B, Hq,
                                  _dev(block_table, "block_table", I32, 2),
                                  int(block_table.shape[1]), _dev(seq_lens, "seq_lens", I32, 1),
                                  _dev(abort_mask, "abort_mask", U8, 1), float(sm_scale),
                                  _dev(out, "out", (torch.float32,), 3),
                                  _dev(err_word, "err_word", U32), _stream(stream))
    _check("kvq_decode_attn_static", st)
