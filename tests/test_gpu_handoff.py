"""GPU parity of kvq_handoff_pages (the prefill -> decode handoff: prompts
read from a paged BF16 prefill cache and stored into the paged e4m3 decode
cache) against the oracle, bit for bit.

The prefill pool is filled on the GPU by kvq_append into a bf16 cache (a
copy) and on the host by the oracle's bf16 append; the handoff then runs on
both sides and the decode pools are compared byte for byte (sentinel bytes
included, so nothing outside the moved tokens may change).
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
from fp8_paged_kv_attn_gb300 import inputs
from gpu_harness import SENTINEL, assert_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


def _src_pools(kvq, h, requests):
    """Prefill pools holding every request's prompt (positions 0 .. first +
    count - 1) on the GPU, and the listed requests' on the host."""
    src = kvq.KVCache(torch.full(h.src_shape(), 0xBEEF - 65536, dtype=torch.int16,
                                 device="cuda").view(torch.bfloat16),
                      torch.full(h.src_shape(), 0xBEEF - 65536, dtype=torch.int16,
                                 device="cuda").view(torch.bfloat16))
    hk = np.full(h.src_shape(), 0xBEEF, dtype=np.uint16)
    hv = hk.copy()
    sbt = dev(h.src_block_table)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    amax_k = amax_v = 0.0
    for b in range(h.B):
        k, v = h.kv_source(b)
        if k.shape[0] == 0:
            continue
        amax_k = max(amax_k, inputs.amax_bf16(k))
        amax_v = max(amax_v, inputs.amax_bf16(v))
        req = np.full(k.shape[0], b, dtype=np.int32)
        pos = np.arange(k.shape[0], dtype=np.int32)
        kvq.kvq_append(src, dev_bf16(k), dev_bf16(v), dev(req), dev(pos), sbt, err_word=err)
        if b in requests:
            assert oracle.quant_append(oracle.KV_BF16, hk, hv, 1.0, 1.0, k, v, req, pos,
                                       h.src_block_table) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return src, hk, hv, float(inputs.scale_from_amax(amax_k)), \
        float(inputs.scale_from_amax(amax_v))


def _run(kvq, h, kv_dtype, src, ks, vs, count=None, first=None, sbt=None, dbt=None):
    fp8 = kv_dtype == kvq.KV_E4M3
    fill = SENTINEL if fp8 else SENTINEL | (SENTINEL << 8)
    dt = torch.uint8 if fp8 else torch.int16
    dk = torch.full(h.dst_shape(), fill if fp8 else fill - 65536, dtype=dt, device="cuda")
    dv = dk.clone()
    if not fp8:
        dk, dv = dk.view(torch.bfloat16), dv.view(torch.bfloat16)
    dst = kvq.KVCache(dk, dv, ks, vs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_handoff_pages(src, dev(h.src_block_table if sbt is None else sbt), dst,
                          dev(h.dst_block_table if dbt is None else dbt),
                          dev(h.count if count is None else count),
                          first=dev(h.first if first is None else first), err_word=err)
    torch.cuda.synchronize()
    view = torch.uint8 if fp8 else torch.int16
    npdt = np.uint8 if fp8 else np.uint16
    return (dst, dk.view(view).cpu().numpy().view(npdt), dv.view(view).cpu().numpy().view(npdt),
            int(err.item()) & 0xFFFFFFFF)


def _oracle(h, kv_dtype, hk, hv, ks, vs, count=None, first=None, sbt=None, dbt=None):
    fp8 = kv_dtype == oracle.KV_E4M3
    ok = np.full(h.dst_shape(), SENTINEL if fp8 else SENTINEL | (SENTINEL << 8),
                 dtype=np.uint8 if fp8 else np.uint16)
    ov = ok.copy()
    e = oracle.handoff_pages(hk, hv, h.src_block_table if sbt is None else sbt, kv_dtype, ok, ov,
                             h.dst_block_table if dbt is None else dbt, ks, vs,
                             h.count if count is None else count,
                             h.first if first is None else first)
    return ok, ov, e


CASES = [(64, 16, 128, "e4m3"), (16, 16, 128, "e4m3"), (16, 64, 64, "e4m3"), (32, 16, 128, "bf16"),
         (64, 32, 64, "e4m3"), (16, 32, 128, "bf16")]


@pytest.mark.parametrize("src_P,dst_P,D,dtype", CASES,
                         ids=[f"p{a}to{b}_d{d}_{t}" for a, b, d, t in CASES])
def test_handoff_whole_pool(kvq, src_P, dst_P, D, dtype):
    """Seven requests of 0 to 1,500 tokens, some starting past position 0 and
    ending mid-page: the whole decode pool equals the oracle's, byte for byte."""
    h = inputs.handoff(seed=100 + src_P + dst_P + D, lens=[0, 1, 37, 300, 1000, 1500, 65],
                       first=[0, 0, 5, 0, 17, 0, 64], Hkv=8, D=D, src_P=src_P, dst_P=dst_P,
                       decode_room=50, dst_pool_factor=1.3)
    kd = kvq.KV_E4M3 if dtype == "e4m3" else kvq.KV_BF16
    src, hk, hv, ks, vs = _src_pools(kvq, h, range(h.B))
    _, gk, gv, gerr = _run(kvq, h, kd, src, ks, vs)
    ok, ov, oerr = _oracle(h, kd, hk, hv, ks, vs)
    assert gerr == 0 and oerr == 0
    assert np.array_equal(gk, ok), "K pool differs from the oracle"
    assert np.array_equal(gv, ov), "V pool differs from the oracle"


@pytest.mark.parametrize("Hkv,D,src_P,dst_P", [(1, 64, 16, 64), (2, 128, 32, 16), (4, 64, 64, 32)])
def test_handoff_head_counts(kvq, Hkv, D, src_P, dst_P):
    """One, two and four kv heads (a stage is one head of a 64-token block):
    the whole decode pool byte for byte."""
    h = inputs.handoff(seed=61 + Hkv, lens=[700, 1, 129, 64, 1000], first=[0, 3, 63, 64, 5],
                       Hkv=Hkv, D=D, src_P=src_P, dst_P=dst_P, decode_room=20,
                       dst_pool_factor=1.3)
    src, hk, hv, ks, vs = _src_pools(kvq, h, range(h.B))
    _, gk, gv, gerr = _run(kvq, h, kvq.KV_E4M3, src, ks, vs)
    ok, ov, oerr = _oracle(h, oracle.KV_E4M3, hk, hv, ks, vs)
    assert gerr == 0 and oerr == 0
    assert np.array_equal(gk, ok), "K pool differs from the oracle"
    assert np.array_equal(gv, ov), "V pool differs from the oracle"


@pytest.mark.parametrize("scale", [1.0, 0.25, 3.0 / 256, 0.0123, 1e-39])
def test_handoff_scales(kvq, scale):
    """The quantiser's paths: power-of-two scales (a product), 3 * 2^k (many
    quotients exactly on e4m3 boundaries), an arbitrary scale (the bracket)
    and one whose reciprocal overflows (the division): byte for byte."""
    h = inputs.handoff(seed=41, lens=[300, 1000, 65], first=[0, 17, 64], Hkv=8, D=128,
                       src_P=64, dst_P=16, decode_room=16, dst_pool_factor=1.2)
    src, hk, hv, _, _ = _src_pools(kvq, h, range(h.B))
    ks, vs = float(np.float32(scale)), float(np.float32(2 * scale))
    _, gk, gv, gerr = _run(kvq, h, kvq.KV_E4M3, src, ks, vs)
    ok, ov, oerr = _oracle(h, oracle.KV_E4M3, hk, hv, ks, vs)
    assert gerr == 0 and oerr == 0
    assert np.array_equal(gk, ok), "K pool differs from the oracle"
    assert np.array_equal(gv, ov), "V pool differs from the oracle"


def test_handoff_errors(kvq):
    """Ranges past either table, a negative count, a prefill page outside the
    pool (negative and one past the end), a decode page outside the pool:
    the same error bits as the oracle and the same untouched bytes."""
    h = inputs.handoff(seed=7, lens=[300, 200, 100, 50, 400, 64], first=[0, 0, 5, 0, 40, 0],
                       Hkv=8, D=128, src_P=32, dst_P=16, decode_room=16, dst_pool_factor=1.2)
    src, hk, hv, ks, vs = _src_pools(kvq, h, range(h.B))
    cnt, fst = h.count.copy(), h.first.copy()
    sbt, dbt = h.src_block_table.copy(), h.dst_block_table.copy()
    cnt[0] = h.dst_MP * h.dst_P + 1
    cnt[1] = -1
    sbt[2, 1] = -1
    sbt[3, 0] = h.src_pages
    dbt[4, (40 + 3) // h.dst_P] = h.dst_pages
    _, gk, gv, gerr = _run(kvq, h, kvq.KV_E4M3, src, ks, vs, cnt, fst, sbt, dbt)
    ok, ov, oerr = _oracle(h, oracle.KV_E4M3, hk, hv, ks, vs, cnt, fst, sbt, dbt)
    assert oerr == oracle.ERR_POS | oracle.ERR_PAGE
    assert gerr == oerr
    assert np.array_equal(gk, ok) and np.array_equal(gv, ov)


def test_handoff_matches_append(kvq):
    """A prompt handed off is stored exactly as the same tokens appended by
    kvq_append (the decode path's own quantisation)."""
    h = inputs.handoff(seed=9, lens=[700, 1300, 5], first=[0, 30, 2], Hkv=8, D=128, src_P=64,
                       dst_P=16, decode_room=16)
    src, _, _, ks, vs = _src_pools(kvq, h, [])
    dst, gk, gv, _ = _run(kvq, h, kvq.KV_E4M3, src, ks, vs)
    ref = kvq.KVCache(torch.full(h.dst_shape(), SENTINEL, dtype=torch.uint8, device="cuda"),
                      torch.full(h.dst_shape(), SENTINEL, dtype=torch.uint8, device="cuda"), ks, vs)
    dbt = dev(h.dst_block_table)
    for b in range(h.B):
        k, v = h.kv_source(b)
        f = int(h.first[b])
        pos = np.arange(f, k.shape[0], dtype=np.int32)
        kvq.kvq_append(ref, dev_bf16(k[f:]), dev_bf16(v[f:]), dev(np.full(pos.shape, b, np.int32)),
                       dev(pos), dbt)
    torch.cuda.synchronize()
    assert np.array_equal(ref.k_pool.cpu().numpy(), gk)
    assert np.array_equal(ref.v_pool.cpu().numpy(), gv)


def test_handoff_full_64x8192_then_decode(kvq):
    """The sweep's 64 requests x 8192-token prompts, prefill pages of 64
    tokens into the decode pool of 64 requests x 575 pages of 16, in one
    call: every page of four sampled requests bit for bit against the oracle,
    then decode attention over the handed-off cache (sampled rows) against
    the oracle's attention over the oracle's pool."""
    h = inputs.handoff()
    picks = [0, 21, 42, 63]
    src, hk, hv, ks, vs = _src_pools(kvq, h, picks)
    dst, gk, gv, gerr = _run(kvq, h, kvq.KV_E4M3, src, ks, vs)
    assert gerr == 0
    only = np.zeros(h.B, dtype=np.int32)
    only[picks] = h.count[picks]
    ok, ov, oerr = _oracle(h, oracle.KV_E4M3, hk, hv, ks, vs, count=only)
    assert oerr == 0
    pages = np.sort(np.concatenate([h.dst_block_table[b][:-(-int(h.count[b]) // h.dst_P)]
                                    for b in picks]))
    assert np.array_equal(gk[pages], ok[pages]), "K pages differ from the oracle"
    assert np.array_equal(gv[pages], ov[pages]), "V pages differ from the oracle"
    # decode attention over the handed-off prompts (no new token)
    Hq = 32
    rng = np.random.default_rng(11)
    q = inputs.normal_bf16(rng, (h.B, Hq, h.D))
    lens = h.count.astype(np.int32)
    out = torch.full((h.B, Hq, h.D), float("nan"), device="cuda")
    ws = kvq.workspace(h.B, Hq, h.Hkv, h.D)
    sm = float(np.float32(1.0) / np.sqrt(np.float32(h.D)))
    kvq.kvq_decode_attn(dst, dev_bf16(q), dev(h.dst_block_table), dev(lens), out, ws, sm_scale=sm)
    rows = [(b, hh) for b in picks for hh in (0, 11, 31)]
    ref, e = oracle.decode_attn(oracle.KV_E4M3, ok, ov, ks, vs, q, h.dst_block_table, lens,
                                sm_scale=sm, rows=rows, nthreads=16)
    assert e == 0
    got = out.cpu().numpy()
    for b, hh in rows:
        assert_close(got[b, hh], ref[b, hh], f"row ({b},{hh}) over the handed-off cache")
