"""GPU parity of kvq_pages_update (the page allocator that sets the tags)
against the oracle: bit-exact stack, free count, tags, block table, expected
tags, served flags and error bits after every batch; then the whole loop on
the GPU (allocate -> append -> check -> attention) with a stale request."""
import json

import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
from fp8_paged_kv_attn_gb300 import inputs, kvq
from gpu_harness import assert_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(np.asarray(a).astype(np.int64).astype(np.int32)))


def to_gpu(st: oracle.PageState) -> kvq.PageState:
    return kvq.PageState(_i32(st.free_stack).cuda(), _i32(st.free_count).cuda(),
                         torch.from_numpy(st.page_tags.view(np.int32).copy()).cuda(),
                         _i32(st.block_table).cuda(),
                         torch.from_numpy(st.expected_tags.view(np.int32).copy()).cuda())


def from_gpu(g: kvq.PageState) -> oracle.PageState:
    return oracle.PageState(g.free_stack.cpu().numpy(), int(g.free_count.item()),
                            g.page_tags.cpu().numpy().view(np.uint32),
                            g.block_table.cpu().numpy(),
                            g.expected_tags.cpu().numpy().view(np.uint32))


def gpu_update(g, rel_req, rel_n, acq_req, acq_first, acq_n):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    n_acq = len(acq_req)
    ok = torch.full((n_acq,), 0xAB, dtype=torch.uint8, device="cuda")
    t = lambda x: dev(np.asarray(x, dtype=np.int32)) if len(x) else None  # noqa: E731
    kvq.kvq_pages_update(g, rel_req=t(rel_req), rel_npages=t(rel_n), acq_req=t(acq_req),
                         acq_first=t(acq_first), acq_npages=t(acq_n),
                         acq_ok=ok if n_acq else None, err_word=err)
    torch.cuda.synchronize()
    return ok.cpu().numpy(), int(err.item()) & 0xFFFFFFFF


def assert_same(g: oracle.PageState, h: oracle.PageState, what=""):
    c = int(h.free_count[0])
    assert int(g.free_count[0]) == c, (what, "count", int(g.free_count[0]), c)
    assert np.array_equal(g.free_stack[:c], h.free_stack[:c]), (what, "stack")
    assert np.array_equal(g.page_tags, h.page_tags), (what, "tags")
    assert np.array_equal(g.block_table, h.block_table), (what, "block table")
    assert np.array_equal(g.expected_tags, h.expected_tags), (what, "expected tags")


def run_both(g, h, op, what):
    ok_g, err_g = gpu_update(g, *op)
    ok_h, err_h = oracle.pages_update(h, *op)
    assert np.array_equal(ok_g, ok_h), (what, "served", ok_g, ok_h)
    assert err_g == err_h, (what, "error bits", err_g, err_h)
    assert_same(from_gpu(g), h, what)
    return ok_g, err_g


def test_pages_golden_example_on_gpu(kvq):
    with open(pins.GOLDEN_PAGES) as f:
        gold = json.load(f)
    B, MP = gold["B"], gold["MP"]
    st = pins._state_from(oracle, gold["initial"], B, MP)
    g = to_gpu(st)
    for n, op in enumerate(gold["ops"]):
        rel, acq = op["release"], op["acquire"]
        ok, err = gpu_update(g, [r[0] for r in rel], [r[1] for r in rel], [a[0] for a in acq],
                             [a[1] for a in acq], [a[2] for a in acq])
        pins._assert_expect(from_gpu(g), ok, err, op["expect"], f"gpu op {n + 1}")
    w = gold["wrap"]
    g = to_gpu(pins._state_from(oracle, w["initial"], w["B"], w["MP"]))
    ok, err = gpu_update(g, [], [], *[[a[i] for a in w["acquire"]] for i in range(3)])
    pins._assert_expect(from_gpu(g), ok, err, w["expect"], "gpu wrap")


@pytest.mark.parametrize("seed,num_pages,B,MP,fail_often", [
    (1, 64, 12, 10, False), (2, 64, 12, 10, True), (3, 17, 5, 6, True),
    (4, 3000, 300, 24, False), (5, 700, 300, 24, True)])
def test_pages_random_sequences(kvq, seed, num_pages, B, MP, fail_often):
    rng = np.random.default_rng(seed)
    h = oracle.PageState.fresh(num_pages, B, MP, order=rng.permutation(num_pages).astype(np.int32))
    g = to_gpu(h)
    for step in range(40):
        op = pins.next_page_ops(rng, h.block_table, fail_often,
                                bad_release=fail_often and step % 7 == 3)
        run_both(g, h, op, f"step {step}")


def test_pages_long_lists_and_whole_prompts(kvq):
    """Lists of more than 1024 entries (several rounds of the kernel) and
    entries of hundreds of pages: admit 64 requests x 575 pages into a pool
    of exactly 36,800 pages (the last fits exactly), then 1,500 one-page
    acquisitions against an empty stack, then release 40 requests (23,000
    pages) and serve 2,100 requests of 8-15 pages, of which only part fit."""
    num_pages, B, MP = 36800, 2200, 600
    rng = np.random.default_rng(7)
    h = oracle.PageState.fresh(num_pages, B, MP, order=rng.permutation(num_pages).astype(np.int32))
    g = to_gpu(h)
    run_both(g, h, ([], [], list(range(64)), [0] * 64, [575] * 64), "admit")
    assert int(h.free_count[0]) == 0
    reqs = list(range(64, 64 + 1500))
    ok, err = run_both(g, h, ([], [], reqs, [0] * 1500, [1] * 1500), "exhausted")
    assert err == oracle.ERR_EXHAUSTED and not ok.any()
    rel = [int(b) for b in rng.choice(64, 40, replace=False)]
    reqs = list(range(64, 64 + 2100))
    ok, err = run_both(g, h, (rel, [575] * 40, reqs, [0] * 2100,
                               [int(x) for x in rng.integers(8, 16, 2100)]), "release and refill")
    assert err == oracle.ERR_EXHAUSTED and ok.any() and not ok.all()
    assert int(h.free_count[0]) < 16


def test_pages_bad_state_and_arguments(kvq):
    h = oracle.PageState.fresh(8, 2, 4)
    h.free_count[0] = 9
    g = to_gpu(h)
    run_both(g, h, ([], [], [0], [0], [1]), "bad count")
    g = to_gpu(oracle.PageState.fresh(8, 2, 4))
    one = dev(np.array([0], np.int32))
    with pytest.raises(ValueError):  # the binding refuses a missing acq_ok
        kvq.kvq_pages_update(g, acq_req=one, acq_first=one, acq_npages=one, acq_ok=None)
    # and so does the C ABI, before any launch
    L = kvq.load()
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = L.kvq_pages_update(p(g.free_stack), p(g.free_count), p(g.page_tags), 8,
                            p(g.block_table), p(g.expected_tags), 2, 4, None, None, 0,
                            p(one), p(one), p(one), 1, None, None, None)
    assert st == 1


def test_allocate_append_check_attend_loop(kvq):
    """The integrity loop on the GPU: requests get their pages from
    kvq_pages_update, their prompts are appended, one request finishes and
    its pages are handed to a newcomer (tags bumped); a stale copy of the
    finished request's rows fails kvq_check_tags and its attention rows are
    zero, while every live request passes and matches the oracle."""
    Hq, Hkv, D, P = 8, 2, 128, 16
    num_pages, B, MP = 40, 5, 8
    rng = np.random.default_rng(12)
    h = oracle.PageState.fresh(num_pages, B, MP, order=rng.permutation(num_pages).astype(np.int32))
    g = to_gpu(h)
    lens0 = np.array([70, 33, 100, 16, 0], np.int32)
    need = (lens0 + P - 1) // P
    run_both(g, h, ([], [], [0, 1, 2, 3], [0] * 4, [int(x) for x in need[:4]]), "admit")
    scale = np.float32(0.02)
    cache = kvq.KVCache(torch.zeros((num_pages, Hkv, P, D), dtype=torch.uint8, device="cuda"),
                        torch.zeros((num_pages, Hkv, P, D), dtype=torch.uint8, device="cuda"),
                        float(scale), float(scale))
    hk = np.zeros((num_pages, Hkv, P, D), np.uint8)
    hv = hk.copy()

    def append(b, L):
        k = inputs.normal_bf16(rng, (L, Hkv, D))
        v = inputs.normal_bf16(rng, (L, Hkv, D))
        req = np.full(L, b, np.int32)
        pos = np.arange(L, dtype=np.int32)
        kvq.kvq_append(cache, dev_bf16(k), dev_bf16(v), dev(req), dev(pos), g.block_table)
        assert oracle.quant_append(oracle.KV_E4M3, hk, hv, scale, scale, k, v, req, pos,
                                   h.block_table) == 0

    for b in range(4):
        append(b, int(lens0[b]))
    stale_bt, stale_exp = h.block_table[0].copy(), h.expected_tags[0].copy()
    # request 0 finishes; request 4 arrives and takes its pages (LIFO)
    run_both(g, h, ([0], [int(need[0])], [4], [0], [5]), "turnover")
    append(4, 80)
    lens = np.array([0, 33, 100, 16, 80], np.int32)
    # a server that kept request 0's old rows would present them here
    bt = h.block_table.copy()
    exp = h.expected_tags.copy()
    bt[0], exp[0] = stale_bt, stale_exp
    lens[0] = lens0[0]
    mask = torch.zeros(B, dtype=torch.uint8, device="cuda")
    kvq.kvq_check_tags(dev(bt), dev(lens), P, g.page_tags, dev(exp.view(np.int32)), mask)
    ab = mask.cpu().numpy()
    ref = oracle.check_tags(bt, lens, P, h.page_tags, exp)
    assert np.array_equal(ab, ref) and list(ab) == [1, 0, 0, 0, 0]
    q = inputs.normal_bf16(rng, (B, Hq, D))
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvq.workspace(B, Hq, Hkv, D)
    kvq.kvq_decode_attn(cache, dev_bf16(q), dev(bt), dev(lens), out, ws, abort_mask=mask,
                        sm_scale=1.0 / np.sqrt(D))
    got = out.cpu().numpy()
    want, err = oracle.decode_attn(oracle.KV_E4M3, hk, hv, scale, scale, q, bt, lens,
                                   abort_mask=ref, sm_scale=1.0 / np.sqrt(D))
    assert err == 0
    assert np.all(got[0] == 0)
    assert_close(got, want, "loop attention")
