"""CPU checks of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every symbol include/kvq.h declares, and rejects bad host
arguments before launching anything."""
import ctypes
import os
import re

import pytest

from fp8_paged_kv_attn_gb300 import kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    return sorted(set(re.findall(r"KVQ_API\s+[\w\s\*]*?\b(kvq_\w+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_symbols() == sorted(kvq.EXPORTS)


def test_library_loads_and_exports_every_symbol():
    lib = kvq.load()
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.kvq_status_string(0) == b"KVQ_OK"
    assert lib.kvq_status_string(2) == b"KVQ_ERR_WORKSPACE"


def test_workspace_size_grows_with_batch_and_group():
    f = kvq.kvq_decode_attn_workspace_size
    a = f(1, 32, 8, 128)
    b = f(64, 32, 8, 128)
    c = f(64, 64, 8, 128)
    assert 0 < a < b < c
    assert b % 256 == 0
    assert f(4, 6, 4, 128) == 0  # Hq not a multiple of Hkv


def _cache(**kw):
    c = kvq.CCache(16, 16, 0, 8, 16, 2, 128, 1.0, 1.0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("kw,want", [
    ({"k_pool": None}, 1), ({"kv_dtype": 7}, 1), ({"num_pages": 0}, 1), ({"k_pool": 8}, 1),
    ({"page_size": 8}, 4), ({"head_dim": 96}, 4), ({"k_scale": -1.0}, 1),
    ({"v_scale": float("inf")}, 1)])
def test_bad_cache_rejected_before_launch(kw, want):
    lib = kvq.load()
    c = _cache(**kw)
    st = lib.kvq_append(ctypes.byref(c), 16, 16, 16, 16, 1, 16, 1, 4, None, None)
    assert st == want
    st = lib.kvq_append_check(ctypes.byref(c), 16, 16, 16, 16, 1, 16, 1, 4, 16, 16, 16, 16,
                              None, None)
    assert st == want
    st = lib.kvq_decode_attn(ctypes.byref(c), 16, 1, 4, 16, 4, 16, None, 0.1, 16, 256, 1 << 30,
                             None, None)
    assert st == want


def test_bad_call_arguments_rejected_before_launch():
    lib = kvq.load()
    c = _cache()
    # null inputs / misaligned bf16 source
    assert lib.kvq_append(ctypes.byref(c), None, 16, 16, 16, 1, 16, 1, 4, None, None) == 1
    assert lib.kvq_append(ctypes.byref(c), 18, 16, 16, 16, 1, 16, 1, 4, None, None) == 1
    # zero tokens is a no-op, no device touched
    assert lib.kvq_append(ctypes.byref(c), None, None, None, None, 0, None, 1, 4, None, None) == 0
    # Hq not a multiple of Hkv, unsupported group size, misaligned q
    assert lib.kvq_decode_attn(ctypes.byref(c), 16, 1, 3, 16, 4, 16, None, 0.1, 16, 256, 1 << 30,
                               None, None) == 1
    assert lib.kvq_decode_attn(ctypes.byref(c), 16, 1, 32, 16, 4, 16, None, 0.1, 16, 256,
                               1 << 30, None, None) == 4
    assert lib.kvq_decode_attn(ctypes.byref(c), 8, 1, 4, 16, 4, 16, None, 0.1, 16, 256, 1 << 30,
                               None, None) == 1
    # workspace too small / misaligned
    assert lib.kvq_decode_attn(ctypes.byref(c), 16, 1, 4, 16, 4, 16, None, 0.1, 16, 256, 64,
                               None, None) == 2
    assert lib.kvq_decode_attn(ctypes.byref(c), 16, 1, 4, 16, 4, 16, None, 0.1, 16, 128, 1 << 30,
                               None, None) == 2
    # non-finite softmax scale
    assert lib.kvq_decode_attn(ctypes.byref(c), 16, 1, 4, 16, 4, 16, None, float("nan"), 16, 256,
                               1 << 30, None, None) == 1
    # tag check: bad sizes, null pointers; B == 0 is a no-op
    assert lib.kvq_check_tags(16, 1, 0, 16, 16, 16, 8, 16, 16, None) == 1
    assert lib.kvq_check_tags(None, 1, 4, 16, 16, 16, 8, 16, 16, None) == 1
    assert lib.kvq_check_tags(None, 0, 4, None, 16, None, 8, None, None, None) == 0
    # append and check in one launch: either half's argument errors; nothing to
    # do at all is a no-op
    assert lib.kvq_append_check(ctypes.byref(c), None, 16, 16, 16, 1, 16, 1, 4, 16, 16, 16, 16,
                                None, None) == 1
    assert lib.kvq_append_check(ctypes.byref(c), 16, 16, 16, 16, 1, 16, 1, 4, None, 16, 16, 16,
                                None, None) == 1
    assert lib.kvq_append_check(ctypes.byref(c), 16, 16, 16, 16, 1, 16, 1, 4, 16, 16, 16, None,
                                None, None) == 1
    assert lib.kvq_append_check(ctypes.byref(c), 16, 16, 16, 16, 1, 16, 1, 0, 16, 16, 16, 16,
                                None, None) == 1
    assert lib.kvq_append_check(ctypes.byref(c), None, None, None, None, 0, None, 0, 4, None,
                                None, None, None, None, None) == 0
