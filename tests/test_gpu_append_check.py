"""GPU parity of kvq_append and kvq_check_tags against the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_attn_gb300 import inputs
from gpu_harness import Run, dev, dev_bf16, dev_u32, SENTINEL

pytestmark = pytest.mark.gpu

SCALES = [1.0, 3.0, 0.1, 1.0 / 3.0, 0.0123, 37.5, 1e-3, 2.0 ** -20,
          # amax / 448 for round amax values: a power of two (the product
          # path) and 3 * 2^k (many quotients exactly on e4m3 boundaries)
          0.25, 3.0 / 256, 0.75]
# the kernel's reciprocal fast path is exact only while 1/scale is a normal
# float: scales at and past both ends of that range, and seeded random
# scales over 2^-40 .. 2^40
EDGE_SCALES = [2.0 ** -126, 1e-38, 1e-45, 2.0 ** 126, 3.0e38, 3.4028235e38]
RANDOM_SCALES = [float(np.float32(2.0 ** e))
                 for e in np.random.default_rng(11).uniform(-40, 40, 12)]


def _v_scale(s32):
    """Twice the K scale (exact), or the K scale where twice would overflow."""
    v = 2.0 * float(s32)
    return v if v <= float(np.finfo(np.float32).max) else float(s32)


def _exhaustive_tokens():
    """All 65,536 bf16 bit patterns laid out as 512 tokens x 1 head x 128 dims."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(512, 1, 128)
    return bits


@pytest.mark.parametrize("scale", SCALES + EDGE_SCALES + RANDOM_SCALES)
def test_append_every_bf16_value(kvq, scale):
    """Every bf16 input (including inf and NaN) at several scales: the same
    e4m3 byte as the oracle; NaN inputs give a NaN code."""
    bits = _exhaustive_tokens()
    N, H, D, P = bits.shape[0], 1, 128, 16
    MP = N // P
    bt = np.random.default_rng(5).permutation(MP).astype(np.int32).reshape(1, MP)
    req = np.zeros(N, dtype=np.int32)
    pos = np.arange(N, dtype=np.int32)
    s32 = np.float32(scale)
    cache = kvq.KVCache(torch.full((MP, H, P, D), SENTINEL, dtype=torch.uint8, device="cuda"),
                        torch.full((MP, H, P, D), SENTINEL, dtype=torch.uint8, device="cuda"),
                        float(s32), _v_scale(s32))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_append(cache, dev_bf16(bits), dev_bf16(bits[::-1].copy()), dev(req), dev(pos), dev(bt),
                   err_word=err)
    hk = np.full((MP, H, P, D), SENTINEL, dtype=np.uint8)
    hv = hk.copy()
    assert oracle.quant_append(oracle.KV_E4M3, hk, hv, np.float32(cache.k_scale),
                               np.float32(cache.v_scale), bits, bits[::-1].copy(),
                               req, pos, bt) == 0
    gk = cache.k_pool.cpu().numpy()
    gv = cache.v_pool.cpu().numpy()
    assert int(err.item()) == 0
    for g, h in ((gk, hk), (gv, hv)):
        nan = (h & 0x7F) == 0x7F
        assert np.array_equal(g[~nan], h[~nan])
        assert np.all((g[nan] & 0x7F) == 0x7F)


def test_append_bf16_pool_copies(kvq):
    w = inputs.uniform("bf16copy", 41, B=3, ctx=77, Hq=8, Hkv=2, D=128, P=16)
    r = Run(w, kv_dtype=kvq.KV_BF16)
    r.fill_context()
    r.assert_pools_equal(w.ctx_lens, whole=True)
    assert r.err_word() == 0


@pytest.mark.parametrize("mk", [inputs.tiny,
                                lambda: inputs.uniform("u64", 42, B=4, ctx=300, Hq=16, Hkv=2,
                                                       D=64, P=64, outlier_frac=0.01),
                                lambda: inputs.ragged(seed=43, B=7, total=5000, lo=1, hi=2000,
                                                      Hq=8, Hkv=8, D=128, P=32)],
                         ids=["tiny", "u64", "ragged"])
def test_append_context_and_step(kvq, mk):
    """Bulk prompt append then one decode-step append: the whole pool equals
    the oracle's byte for byte (untouched bytes keep their sentinel)."""
    w = mk()
    r = Run(w)
    r.fill_context()
    r.assert_pools_equal(w.ctx_lens, whole=True)
    r.append_step(0)
    torch.cuda.synchronize()
    r.assert_pools_equal(w.seq_lens_after(0), whole=True)
    assert r.err_word() == 0


@pytest.mark.parametrize("kv_dtype", ["e4m3", "bf16"])
def test_prompt_handoff_one_call_8x8192(kvq, kv_dtype):
    """The prefill -> decode handoff at the 8-request x 8192-token size: all
    65,536 prompt tokens quantised by one call, every byte of both pools equal
    to the oracle's (pages no request uses keep their sentinel)."""
    w = inputs.cfg8x8k()
    r = Run(w, kv_dtype=kvq.KV_E4M3 if kv_dtype == "e4m3" else kvq.KV_BF16)
    assert r.fill_context_one_call() == int(w.ctx_lens.sum())
    r.assert_pools_equal(w.ctx_lens, whole=True)
    assert r.err_word() == 0


def test_prompt_handoff_one_call_64x8192(kvq):
    """The handoff at the 64-request sweep size (524,288 tokens, 1.07 GB of bf16
    K and of V, in one call): every page of 6 sampled requests equals the
    oracle's byte for byte."""
    w = inputs.sweep(64, kv_bytes=1)
    sel = [0, 13, 27, 40, 52, 63]
    r = Run(w, host_requests=sel, sources=w.kv_sources(threads=16))
    assert r.fill_context_one_call() == 64 * 8192
    r.assert_pools_equal(w.ctx_lens)
    assert r.err_word() == 0


def test_append_errors(kvq):
    w = inputs.tiny()
    r = Run(w)
    k = np.ones((4, w.Hkv, w.D), dtype=np.uint16) * 0x3F80
    req = np.array([5, 0, 0, -1], dtype=np.int32)
    pos = np.array([0, -1, w.MP * w.P, 0], dtype=np.int32)
    bt = w.block_table.copy()
    kvq.kvq_append(r.cache, dev_bf16(k), dev_bf16(k), dev(req), dev(pos), dev(bt), err_word=r.err)
    torch.cuda.synchronize()
    assert r.err_word() == (kvq.ERRBIT_REQ | kvq.ERRBIT_POS)
    r.err.zero_()
    bt[0, 0] = w.num_pages
    kvq.kvq_append(r.cache, dev_bf16(k[:1]), dev_bf16(k[:1]), dev(req[1:2]), dev(pos[3:4]),
                   dev(bt), err_word=r.err)
    torch.cuda.synchronize()
    assert r.err_word() == kvq.ERRBIT_PAGE
    gk, gv = r.pool_bytes()
    assert np.all(gk == SENTINEL) and np.all(gv == SENTINEL)


def test_append_invalid_args_return_status(kvq):
    w = inputs.tiny()
    r = Run(w)
    k = dev_bf16(np.zeros((1, w.Hkv, w.D), dtype=np.uint16))
    bad = kvq.KVCache(r.cache.k_pool, r.cache.v_pool, -1.0, 1.0)
    with pytest.raises(kvq.KvqError):
        kvq.kvq_append(bad, k, k, dev(np.zeros(1, np.int32)), dev(np.zeros(1, np.int32)), r.bt)


# ----------------------------------------------------------------------------
# tag check
# ----------------------------------------------------------------------------

def _gpu_check(kvq, w, lens, bt=None, tags=None, exp=None):
    bt = w.block_table if bt is None else bt
    tags = w.page_tags if tags is None else tags
    exp = w.expected_tags if exp is None else exp
    mask = torch.full((w.B,), 7, dtype=torch.uint8, device="cuda")
    kvq.kvq_check_tags(dev(bt), dev(lens), w.P, dev_u32(tags), dev_u32(exp), mask)
    return mask.cpu().numpy()


@pytest.mark.parametrize("B,frac,ppv", [(256, 0.001, 1), (256, 0.1, 3), (64, 0.5, 2)])
def test_check_integrity_workload(kvq, oracle_mod, B, frac, ppv):
    """The integrity workload at full size (256 requests of 1k-16k tokens,
    page 16): the GPU mask equals the oracle's and flags exactly the
    requests that received stale tags."""
    w = inputs.integrity(B=B, stale_frac=frac, pages_per_victim=ppv)
    lens = w.seq_lens_after(0)
    got = _gpu_check(kvq, w, lens)
    ref = oracle_mod.check_tags(w.block_table, lens, w.P, w.page_tags, w.expected_tags)
    assert np.array_equal(got, ref)
    assert set(np.nonzero(got)[0].tolist()) == set(w.stale)


def test_check_edges(kvq, oracle_mod):
    w = inputs.ragged(seed=44, B=9, total=3000, lo=1, hi=900, Hq=8, Hkv=8, D=64, P=16)
    lens = w.seq_lens_after(0).copy()
    lens[0] = 0
    lens[1] = w.MP * w.P + 1          # over capacity
    lens[2] = -5
    lens[4] = 5                       # one page; the rest of its row is garbage
    lens[6] = 17                      # two pages
    bt = w.block_table.copy()
    bt[3, 0] = w.num_pages            # page id out of range
    bt[4, 1:] = -1                    # past the request's length: never read
    exp = w.expected_tags.copy()
    n5 = -(-int(lens[5]) // w.P)
    exp[5, n5 - 1] ^= 1               # last checked page stale
    exp[6, 2:] += 3                   # entries past the length are ignored
    got = _gpu_check(kvq, w, lens, bt=bt, exp=exp)
    ref = oracle_mod.check_tags(bt, lens, w.P, w.page_tags, exp)
    assert np.array_equal(got, ref)
    assert got[:6].tolist() == [0, 1, 1, 1, 0, 1]


# ----------------------------------------------------------------------------
# append and check in one launch
# ----------------------------------------------------------------------------

def _two_ways(kvq, w, kv_dtype, k, v, req, pos, bt, lens, tags, exp):
    """The step's append and tag check as two calls and as one launch, each
    on its own sentinel-filled pools: (pools, mask, error word) of both."""
    res = []
    for fused in (False, True):
        fp8 = kv_dtype == kvq.KV_E4M3
        dt = torch.uint8 if fp8 else torch.int16
        fill = SENTINEL if fp8 else (SENTINEL | (SENTINEL << 8)) - 65536
        kp = torch.full(w.pool_shape(), fill, dtype=dt, device="cuda")
        vp = kp.clone()
        if not fp8:
            kp, vp = kp.view(torch.bfloat16), vp.view(torch.bfloat16)
        cache = kvq.KVCache(kp, vp, 0.037, 0.041)
        mask = torch.full((w.B,), 7, dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = (dev_bf16(k), dev_bf16(v), dev(req), dev(pos), dev(bt))
        if fused:
            kvq.kvq_append_check(cache, *args, dev(lens), dev_u32(tags), dev_u32(exp), mask,
                                 err_word=err)
        else:
            kvq.kvq_append(cache, *args, err_word=err)
            kvq.kvq_check_tags(dev(bt), dev(lens), w.P, dev_u32(tags), dev_u32(exp), mask)
        torch.cuda.synchronize()
        view = torch.uint8 if fp8 else torch.int16
        res.append((kp.view(view).cpu().numpy(), vp.view(view).cpu().numpy(),
                    mask.cpu().numpy(), int(err.item())))
    return res


@pytest.mark.parametrize("D,kv", [(128, "e4m3"), (64, "e4m3"), (128, "bf16")])
def test_append_check_matches_two_calls(kvq, oracle_mod, D, kv):
    """kvq_append_check gives what kvq_append then kvq_check_tags give: the
    same pool bytes, the same mask (the oracle's) and the same error word, on
    37 ragged requests with stale tags injected."""
    w = inputs.ragged(seed=45, B=37, total=20000, lo=1, hi=2000, Hq=8, Hkv=8, D=D, P=16)
    kv_dtype = kvq.KV_E4M3 if kv == "e4m3" else kvq.KV_BF16
    _, k, v, req, pos = w.step_inputs(0)
    lens = w.seq_lens_after(0)
    exp = w.expected_tags.copy()
    for b in (3, 17, 30):
        exp[b, int(lens[b]) // w.P // 2] ^= 5
    (k0, v0, m0, e0), (k1, v1, m1, e1) = _two_ways(kvq, w, kv_dtype, k, v, req, pos,
                                                   w.block_table, lens, w.page_tags, exp)
    ref = oracle_mod.check_tags(w.block_table, lens, w.P, w.page_tags, exp)
    assert np.array_equal(m0, ref) and np.array_equal(m1, ref)
    assert sorted(np.nonzero(ref)[0].tolist()) == [3, 17, 30]
    assert np.array_equal(k0, k1) and np.array_equal(v0, v1)
    assert e0 == e1 == 0


def test_append_check_errors_match_two_calls(kvq, oracle_mod):
    """Bad request, position and page in the append, impossible lengths and a
    page id outside the pool in the check: the same error bits, bytes and
    mask from the one launch as from the two calls."""
    w = inputs.ragged(seed=44, B=9, total=3000, lo=1, hi=900, Hq=8, Hkv=8, D=64, P=16)
    _, k, v, req, pos = w.step_inputs(0)
    req, pos = req.copy(), pos.copy()
    req[1], pos[2], pos[4] = w.B, -1, w.MP * w.P
    lens = w.seq_lens_after(0).copy()
    lens[0], lens[5] = -5, w.MP * w.P + 1
    bt = w.block_table.copy()
    bt[3, 0] = w.num_pages
    bt[6, pos[6] // w.P] = w.num_pages + 3  # the page request 6's token goes to
    (k0, v0, m0, e0), (k1, v1, m1, e1) = _two_ways(kvq, w, kvq.KV_E4M3, k, v, req, pos, bt,
                                                   lens, w.page_tags, w.expected_tags)
    ref = oracle_mod.check_tags(bt, lens, w.P, w.page_tags, w.expected_tags)
    assert np.array_equal(m0, ref) and np.array_equal(m1, ref)
    assert m1[[0, 3, 5, 6]].tolist() == [1, 1, 1, 1]
    assert np.array_equal(k0, k1) and np.array_equal(v0, v1)
    assert e0 == e1 and e1 & kvq.ERRBIT_REQ and e1 & kvq.ERRBIT_POS and e1 & kvq.ERRBIT_PAGE
