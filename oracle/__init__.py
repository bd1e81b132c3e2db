"""CPU oracle for the FP8 paged-KV decode path -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrappers over ``kvq_oracle.c`` (plain C, fp64 attention, scalar
e4m3 codec, linear-scan tag check, sequential page allocator).  Only the tests, the smoke check and the
benchmark's CPU-baseline / reference arm may import this package; the
product library never does.  It shares no code with the CUDA path.

Arrays are numpy arrays in the library's layouts:
  bf16 tensors as uint16 bit patterns, pools as uint8 (e4m3) or uint16 (bf16)
  arrays of shape [num_pages, Hkv, P, D], block tables int32 [B, MP].

Sources: page "大规模服务 Kimi 与 GLM：KV 缓存量化、权重压缩与缓存安全",
sections "KV 缓存量化" (e4m3 cache, convert on read) and "共享 KV 缓存保护"
(page tags and the batched check); the OCP 8-bit floating point
specification for the E4M3 bit format.
"""
import contextlib
import ctypes

import numpy as np

from . import build as _build

KV_E4M3 = 0
KV_BF16 = 1

ERR_PAGE = 1 << 0
ERR_SEQLEN = 1 << 1
ERR_POS = 1 << 2
ERR_REQ = 1 << 3
ERR_EXHAUSTED = 1 << 5

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


@contextlib.contextmanager
def use_library(path):
    """Temporarily route every wrapper through another build of the oracle
    (the mutation tests load deliberately broken copies this way)."""
    global _lib
    saved = _lib
    _lib = _load(path)
    try:
        yield
    finally:
        _lib = saved


def _load(path):
    L = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    i32, i64, f32, u32 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_uint32
    L.oracle_e4m3_encode.argtypes = [f32]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_decode.restype = ctypes.c_double
    L.oracle_e4m3_encode_array.argtypes = [vp, vp, i64]
    L.oracle_e4m3_decode_array.argtypes = [vp, vp, i64]
    L.oracle_quantise.argtypes = [ctypes.c_uint16, f32]
    L.oracle_quantise.restype = ctypes.c_uint8
    L.oracle_quantise_array.argtypes = [vp, vp, i64, f32]
    L.oracle_quant_append.argtypes = [i32, vp, vp, i32, i32, i32, i32, f32, f32,
                                      vp, vp, vp, vp, i32, vp, i32, i32]
    L.oracle_quant_append.restype = u32
    L.oracle_handoff_pages.argtypes = [vp, vp, i32, i32, vp, i32, i32, vp, vp, i32, i32, vp, i32,
                                       i32, i32, f32, f32, vp, vp, i32, vp]
    L.oracle_handoff_pages.restype = u32
    L.oracle_check_tags.argtypes = [vp, i32, i32, vp, i32, vp, i32, vp, vp]
    L.oracle_check_tags.restype = None
    L.oracle_wq_gemm.argtypes = [i32, vp, vp, vp, vp, i32, i32, i32, i32]
    L.oracle_wq_gemm.restype = None
    L.oracle_pages_update.argtypes = [vp, vp, vp, i32, vp, vp, i32, i32, vp, vp, i32,
                                      vp, vp, vp, i32, vp]
    L.oracle_pages_update.restype = u32
    L.oracle_decode_attn.argtypes = [i32, vp, vp, i32, i32, i32, i32, f32, f32,
                                     vp, i32, i32, vp, i32, vp, vp, f32, vp,
                                     vp, i32, i32, vp, i64]
    L.oracle_decode_attn.restype = u32
    L.oracle_has_openmp.argtypes = []
    L.oracle_has_openmp.restype = i32
    return L


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.dtype(dtype), (a.dtype, dtype)
    return a


def has_openmp() -> bool:
    return bool(lib().oracle_has_openmp())


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> e4m3 codes (RNE, saturating to +-448, NaN -> 0x7F)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(c) -> np.ndarray:
    """e4m3 codes -> exact float64 values (NaN for 0x7F / 0xFF)."""
    c = np.ascontiguousarray(np.asarray(c, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def quantise(bf16_bits, scale: float) -> np.ndarray:
    """Quantised e4m3 code of each bf16 element: e4m3(fp32(x) / scale)."""
    b = np.ascontiguousarray(np.asarray(bf16_bits, dtype=np.uint16))
    out = np.empty(b.shape, dtype=np.uint8)
    lib().oracle_quantise_array(_ptr(b), _ptr(out), b.size, float(np.float32(scale)))
    return out


def quant_append(kv_dtype, k_pool, v_pool, k_scale, v_scale, k_new, v_new, req_idx, pos,
                 block_table) -> int:
    """Append N tokens into the pools in place; returns the error bits."""
    NP, H, P, D = k_pool.shape
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == (np.uint8 if kv_dtype == KV_E4M3 else np.uint16)
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    req_idx = _c(req_idx, np.int32)
    pos = _c(pos, np.int32)
    block_table = _c(block_table, np.int32)
    B, MP = block_table.shape
    n = req_idx.shape[0]
    return int(lib().oracle_quant_append(kv_dtype, _ptr(k_pool), _ptr(v_pool), NP, P, H, D,
                                         float(k_scale), float(v_scale), _ptr(k_new),
                                         _ptr(v_new), _ptr(req_idx), _ptr(pos), n,
                                         _ptr(block_table), B, MP))


def handoff_pages(src_k, src_v, src_block_table, dst_dtype, dst_k, dst_v, dst_block_table,
                  k_scale, v_scale, count, first=None) -> int:
    """Prefill -> decode handoff in place: tokens [first[b], first[b] +
    count[b]) of every request, gathered from the bf16 pools src_k / src_v
    (uint16 [pages, Hkv, Ps, D]) through src_block_table [B, src_MP] and
    appended into dst_k / dst_v through dst_block_table [B, dst_MP].
    Returns the error bits."""
    SNP, H, SP, D = src_k.shape
    DNP, H2, DP, D2 = dst_k.shape
    assert (H, D) == (H2, D2) and src_v.shape == src_k.shape and dst_v.shape == dst_k.shape
    src_k, src_v = _c(src_k, np.uint16), _c(src_v, np.uint16)
    assert dst_k.flags.c_contiguous and dst_v.flags.c_contiguous
    assert dst_k.dtype == (np.uint8 if dst_dtype == KV_E4M3 else np.uint16)
    sbt = _c(src_block_table, np.int32)
    dbt = _c(dst_block_table, np.int32)
    B, SMP = sbt.shape
    assert dbt.shape[0] == B
    count = _c(count, np.int32)
    first = None if first is None else _c(first, np.int32)
    scratch = np.empty(2 * H * D, dtype=np.uint16)
    return int(lib().oracle_handoff_pages(_ptr(src_k), _ptr(src_v), SNP, SP, _ptr(sbt), SMP,
                                          dst_dtype, _ptr(dst_k), _ptr(dst_v), DNP, DP,
                                          _ptr(dbt), dbt.shape[1], H, D, float(k_scale),
                                          float(v_scale), _ptr(first), _ptr(count), B,
                                          _ptr(scratch)))


def check_tags(block_table, seq_lens, page_size, page_tags, expected_tags) -> np.ndarray:
    """abort_mask[b] = 1 if any checked page of request b mismatches."""
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    page_tags = _c(page_tags, np.uint32)
    expected_tags = _c(expected_tags, np.uint32)
    B, MP = block_table.shape
    out = np.empty(B, dtype=np.uint8)
    lib().oracle_check_tags(_ptr(block_table), B, MP, _ptr(seq_lens), page_size,
                            _ptr(page_tags), page_tags.shape[0], _ptr(expected_tags),
                            _ptr(out))
    return out


class PageState:
    """The page allocator's state (host arrays, updated in place by
    pages_update): free_stack [num_pages] int32 with free_count live entries
    (top = last), page_tags [num_pages] uint32, block_table [B, MP] int32 and
    expected_tags [B, MP] uint32."""

    def __init__(self, free_stack, free_count, page_tags, block_table, expected_tags):
        self.free_stack = np.ascontiguousarray(free_stack, dtype=np.int32)
        self.free_count = np.array([free_count], dtype=np.int32)
        self.page_tags = np.ascontiguousarray(page_tags, dtype=np.uint32)
        self.block_table = np.ascontiguousarray(block_table, dtype=np.int32)
        self.expected_tags = np.ascontiguousarray(expected_tags, dtype=np.uint32)

    @staticmethod
    def fresh(num_pages, B, MP, order=None):
        stack = np.arange(num_pages, dtype=np.int32) if order is None else order
        return PageState(stack, num_pages, np.zeros(num_pages, np.uint32),
                         np.full((B, MP), -1, np.int32), np.zeros((B, MP), np.uint32))

    def copy(self):
        return PageState(self.free_stack.copy(), int(self.free_count[0]), self.page_tags.copy(),
                         self.block_table.copy(), self.expected_tags.copy())


def pages_update(state: PageState, rel_req=(), rel_npages=(), acq_req=(), acq_first=(),
                 acq_npages=()):
    """One batch of releases then acquisitions on `state` (in place).
    Returns (acq_ok uint8 [n_acq], error bits)."""
    rel_req = _c(np.asarray(rel_req, dtype=np.int32), np.int32)
    rel_npages = _c(np.asarray(rel_npages, dtype=np.int32), np.int32)
    acq_req = _c(np.asarray(acq_req, dtype=np.int32), np.int32)
    acq_first = _c(np.asarray(acq_first, dtype=np.int32), np.int32)
    acq_npages = _c(np.asarray(acq_npages, dtype=np.int32), np.int32)
    assert rel_req.shape == rel_npages.shape
    assert acq_req.shape == acq_first.shape == acq_npages.shape
    ok = np.zeros(acq_req.shape[0], dtype=np.uint8)
    B, MP = state.block_table.shape
    err = lib().oracle_pages_update(
        _ptr(state.free_stack), _ptr(state.free_count), _ptr(state.page_tags),
        state.page_tags.shape[0], _ptr(state.block_table), _ptr(state.expected_tags), B, MP,
        _ptr(rel_req), _ptr(rel_npages), rel_req.shape[0], _ptr(acq_req), _ptr(acq_first),
        _ptr(acq_npages), acq_req.shape[0], _ptr(ok))
    return ok, int(err)


W_INT4 = 0
W_E4M3 = 1


def wq_gemm(wdtype, w, scales, x, group=128) -> np.ndarray:
    """y fp32 [M, N] = x [M, K] (bf16 bits) times the quantised weights
    w [N, K/2] (INT4, two nibbles a byte) or [N, K] (e4m3 codes), with bf16
    group scales [N, K/group] (INT4) or fp32 channel scales [N] (e4m3)."""
    w = _c(w, np.uint8)
    x = _c(x, np.uint16)
    M, K = x.shape
    N = w.shape[0]
    if wdtype == W_INT4:
        assert w.shape == (N, K // 2) and K % group == 0
        scales = _c(scales, np.uint16)
        assert scales.shape == (N, K // group)
    else:
        assert w.shape == (N, K)
        scales = _c(scales, np.float32)
        assert scales.shape == (N,)
    y = np.empty((M, N), dtype=np.float32)
    lib().oracle_wq_gemm(wdtype, _ptr(w), _ptr(scales), _ptr(x), _ptr(y), M, N, K, group)
    return y


def decode_attn(kv_dtype, k_pool, v_pool, k_scale, v_scale, q, block_table, seq_lens,
                abort_mask=None, sm_scale=None, rows=None, nthreads=1, out=None):
    """fp64 decode attention; returns (out fp32 [B, Hq, D], error bits).

    rows: optional iterable of (b, h) pairs; only those rows are computed
    (the others stay zero, or as in ``out`` if given).
    """
    NP, H, P, D = k_pool.shape
    q = _c(q, np.uint16)
    B, Hq, Dq = q.shape
    assert Dq == D and Hq % H == 0
    block_table = _c(block_table, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    MP = block_table.shape[1]
    if sm_scale is None:
        sm_scale = float(np.float32(1.0) / np.sqrt(np.float32(D)))
    if abort_mask is not None:
        abort_mask = _c(abort_mask, np.uint8)
    if out is None:
        out = np.zeros((B, Hq, D), dtype=np.float32)
    rows_arr = None
    n_rows = 0
    if rows is not None:
        rows_arr = np.array([b * Hq + h for b, h in rows], dtype=np.int32)
        n_rows = rows_arr.size
    nthreads = max(1, int(nthreads))
    max_len = int(max(0, seq_lens.max(initial=0)))
    max_len = min(max_len, MP * P)
    per_thread = max_len + D + 1
    scratch = np.empty(per_thread * nthreads, dtype=np.float64)
    err = lib().oracle_decode_attn(kv_dtype, _ptr(k_pool), _ptr(v_pool), NP, P, H, D,
                                   float(k_scale), float(v_scale), _ptr(q), B, Hq,
                                   _ptr(block_table), MP, _ptr(seq_lens), _ptr(abort_mask),
                                   float(sm_scale), _ptr(out), _ptr(rows_arr), n_rows,
                                   nthreads, _ptr(scratch), per_thread)
    return out, int(err)
