"""GPU parity of kvq_decode_attn (FP8 and BF16 caches) against the fp64
oracle: |gpu - ref| <= 1e-3 + 1e-3 |ref| elementwise, plus exact cases."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
from fp8_paged_kv_attn_gb300 import inputs
from gpu_harness import Run, assert_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


def step_and_compare(kvq, w, kv_dtype=None, rows=None, host_requests=None, abort=None,
                     check_pools=True):
    kv_dtype = kvq.KV_E4M3 if kv_dtype is None else kv_dtype
    r = Run(w, kv_dtype=kv_dtype, host_requests=host_requests)
    r.fill_context()
    q = r.append_step(0)
    lens = w.seq_lens_after(0)
    got = r.attend(q, lens, abort=abort)
    if check_pools:
        r.assert_pools_equal(lens)
    if rows is None:
        rows = [(b, h) for b in r.host_requests for h in range(w.Hq)]
    ref, err = r.oracle_rows(q, lens, rows, abort=abort)
    assert err == 0 and r.err_word() == 0
    for b, h in rows:
        assert_close(got[b, h], ref[b, h], f"{w.name} row ({b},{h})")
    return r, got, ref, q, lens


def test_tiny_fp8(kvq):
    step_and_compare(kvq, inputs.tiny())


def test_tiny_bf16(kvq):
    step_and_compare(kvq, inputs.tiny(), kv_dtype=kvq.KV_BF16)


SHAPES = [(G, D, P) for G in (1, 2, 4, 8) for D in (64, 128) for P in (16, 32, 64)]


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
@pytest.mark.parametrize("G,D,P", SHAPES, ids=[f"g{g}_d{d}_p{p}" for g, d, p in SHAPES])
def test_shapes(kvq, G, D, P, dtype):
    """Every compiled (group size, head dim, page size) with ragged lengths
    that span several work items and end mid-page."""
    Hkv = 2
    w = inputs.ragged(seed=100 + G + D + P, B=4, total=2600, lo=1, hi=1500, Hq=G * Hkv, Hkv=Hkv,
                      D=D, P=P)
    step_and_compare(kvq, w, kv_dtype=kvq.KV_E4M3 if dtype == "e4m3" else kvq.KV_BF16)


def test_ragged_many_items(kvq):
    """Lengths from 1 to ~6000 in one batch: each request splits into a
    different number of items, tails end mid-stage."""
    w = inputs.ragged(seed=7, B=12, total=30000, lo=1, hi=6000, Hq=32, Hkv=8, D=128, P=16)
    step_and_compare(kvq, w)


def test_one_token_is_exact(kvq):
    """A 1-token context gives exactly v_scale * e4m3(v) (softmax weight 1)."""
    w = inputs.uniform("one", 9, B=3, ctx=0, Hq=16, Hkv=4, D=128, P=16, outlier_frac=0.01)
    r = Run(w)
    q = r.append_step(0)
    lens = w.seq_lens_after(0)
    got = r.attend(q, lens)
    for b in range(w.B):
        page = w.block_table[b, 0]
        for h in range(w.Hq):
            v = (pins.torch_decode(r.hv[page, h // w.G, 0, :]) * float(r.v_scale)).astype(np.float32)
            assert np.array_equal(got[b, h], v), (b, h)


def test_equal_keys_mean_of_v(kvq):
    w = inputs.uniform("eqk", 10, B=2, ctx=333, Hq=8, Hkv=2, D=64, P=16)
    r = Run(w)
    r.fill_context()
    r.cache.k_pool.fill_(0x3C)
    r.hk[...] = 0x3C
    q, *_ = w.step_inputs(0)
    got = r.attend(q, w.ctx_lens)
    for b in range(w.B):
        L = int(w.ctx_lens[b])
        j = np.arange(L)
        v = pins.torch_decode(r.hv[w.block_table[b, j // w.P], :, j % w.P, :]) * float(r.v_scale)
        for h in range(w.Hq):
            assert_close(got[b, h], v[:, h // w.G].mean(axis=0), "mean of V")


def test_page_permutation_bitwise_and_deterministic(kvq):
    """Moving every page to another physical slot leaves the GPU output bit
    for bit unchanged; repeated calls give identical bits."""
    w = inputs.ragged(seed=11, B=6, total=9000, lo=1, hi=4000, Hq=32, Hkv=8, D=128, P=16)
    r = Run(w)
    r.fill_context()
    q, *_ = w.step_inputs(0)
    a = r.attend(q, w.ctx_lens)
    b = r.attend(q, w.ctx_lens)
    assert np.array_equal(a, b)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(w.num_pages)).cuda()
    kp = torch.empty_like(r.cache.k_pool)
    vp = torch.empty_like(r.cache.v_pool)
    kp[perm] = r.cache.k_pool
    vp[perm] = r.cache.v_pool
    r.cache.k_pool, r.cache.v_pool = kp, vp
    bt = w.block_table
    r.bt = dev(np.where(bt >= 0, perm.cpu().numpy()[np.maximum(bt, 0)], -1).astype(np.int32))
    c = r.attend(q, w.ctx_lens)
    assert np.array_equal(a, c)


def test_abort_reads_nothing(kvq):
    """An aborted request's pages are filled with NaN codes: its output rows
    are exactly zero and every other row is unaffected."""
    w = inputs.uniform("abort", 12, B=5, ctx=700, Hq=16, Hkv=4, D=128, P=16)
    r = Run(w)
    r.fill_context()
    q, *_ = w.step_inputs(0)
    base = r.attend(q, w.ctx_lens)
    victims = [1, 3]
    for b in victims:
        n = -(-int(w.ctx_lens[b]) // w.P)
        pages = torch.from_numpy(w.block_table[b, :n].astype(np.int64)).cuda()
        r.cache.k_pool[pages] = 0x7F
        r.cache.v_pool[pages] = 0xFF
    mask = np.zeros(w.B, dtype=np.uint8)
    mask[victims] = 1
    got = r.attend(q, w.ctx_lens, abort=mask)
    assert not np.isnan(got).any()
    for b in range(w.B):
        if b in victims:
            assert not got[b].any()
        else:
            assert np.array_equal(got[b], base[b])
    assert r.err_word() == 0


def test_errors_zero_rows(kvq):
    w = inputs.uniform("errs", 13, B=4, ctx=100, Hq=8, Hkv=2, D=64, P=16)
    r = Run(w)
    r.fill_context()
    q, *_ = w.step_inputs(0)
    lens = w.ctx_lens.copy()
    base = r.attend(q, lens)
    lens[0] = 0
    lens[1] = w.MP * w.P + 1
    bt = w.block_table.copy()
    bt[2, 3] = w.num_pages + 1
    r.bt = dev(bt)
    r.err.zero_()
    got = r.attend(q, lens)
    assert not got[0].any() and not got[1].any() and not got[2].any()
    assert np.array_equal(got[3], base[3])
    assert r.err_word() == (kvq.ERRBIT_SEQLEN | kvq.ERRBIT_PAGE)


def test_all_aborted_and_empty_batch(kvq):
    w = inputs.uniform("none", 14, B=3, ctx=40, Hq=8, Hkv=2, D=64, P=16)
    r = Run(w)
    r.fill_context()
    q, *_ = w.step_inputs(0)
    got = r.attend(q, w.ctx_lens, abort=np.ones(w.B, dtype=np.uint8))
    assert not got.any()
    got = r.attend(q, np.zeros(w.B, dtype=np.int32))
    assert not got.any()


def test_invalid_args(kvq):
    w = inputs.tiny()
    r = Run(w)
    q = dev_bf16(np.zeros((w.B, w.Hq, w.D), dtype=np.uint16))
    out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attn(r.cache, q, r.bt, dev(w.ctx_lens), out, small)
    assert e.value.status == 2
    ws = kvq.workspace(w.B, w.Hq, w.Hkv, w.D)
    r3 = kvq.KVCache(r.cache.k_pool, r.cache.v_pool, float("nan"), 1.0)
    with pytest.raises(kvq.KvqError):
        kvq.kvq_decode_attn(r3, q, r.bt, dev(w.ctx_lens), out, ws)


# ----------------------------------------------------------------------------
# full-size workloads (sampled rows)
# ----------------------------------------------------------------------------

def test_full_8x8192(kvq):
    """8 requests x 8192 cached tokens (+1 appended), 32/8 heads, D=128,
    page 16, pool 2x: every row of requests 0, 3 and 7."""
    w = inputs.cfg8x8k()
    step_and_compare(kvq, w, host_requests=[0, 3, 7])


def test_full_sweep_b64(kvq):
    """The concurrency-sweep point the benchmark times (64 requests, 8192-token
    prompts, page 16, FP8 pool of 64 requests' bytes), after the step that
    appends token 8193: sampled requests, all heads."""
    w = inputs.sweep(64)
    step_and_compare(kvq, w, host_requests=[0, 21, 63],
                     rows=[(b, h) for b in (0, 21, 63) for h in (0, 5, 13, 31)])


def test_full_sweep_bf16_b32(kvq):
    w = inputs.sweep(32, kv_bytes=2)
    step_and_compare(kvq, w, kv_dtype=kvq.KV_BF16, host_requests=[2, 31],
                     rows=[(b, h) for b in (2, 31) for h in (1, 30)])


def test_full_ragged(kvq):
    """64 requests, log-uniform 512..131072 tokens (~1.37M total), 64/8 heads,
    page 64, fragmented pool: shortest, median and longest requests."""
    w = inputs.ragged()
    order = np.argsort(w.ctx_lens)
    picks = [int(order[0]), int(order[len(order) // 2]), int(order[-1])]
    rows = [(b, h) for b in picks for h in (0, 9, 63)]
    step_and_compare(kvq, w, host_requests=picks, rows=rows)


def test_full_integrity(kvq, oracle_mod):
    """256 requests of 1k-16k tokens with one stale tag: the GPU check's mask
    feeds the GPU attention; the stale request's rows are zero, sampled
    survivors match the oracle."""
    w = inputs.integrity()
    lens = w.seq_lens_after(0)
    mask_ref = oracle_mod.check_tags(w.block_table, lens, w.P, w.page_tags, w.expected_tags)
    victim = w.stale[0]
    picks = [0, victim, 128, 255]
    r = Run(w, host_requests=picks)
    r.fill_context()
    q = r.append_step(0)
    mask = torch.empty(w.B, dtype=torch.uint8, device="cuda")
    from gpu_harness import dev_u32
    kvq.kvq_check_tags(r.bt, dev(lens), w.P, dev_u32(w.page_tags), dev_u32(w.expected_tags), mask)
    assert np.array_equal(mask.cpu().numpy(), mask_ref)
    got = r.attend(q, lens, abort=mask.cpu().numpy())
    rows = [(b, h) for b in picks for h in (0, 17, 31)]
    ref, err = r.oracle_rows(q, lens, rows, abort=mask_ref)
    assert err == 0
    assert not got[victim].any()
    for b, h in rows:
        assert_close(got[b, h], ref[b, h], f"integrity row ({b},{h})")


@pytest.mark.parametrize("dtype", ["e4m3", "bf16"])
@pytest.mark.parametrize("lens", [[8000], [5000, 20, 3000], [1, 12000],
                                  [4100, 3900, 4000, 4200, 3800, 4050]],
                         ids=["one", "mix", "two", "six"])
def test_few_long_requests(kvq, dtype, lens):
    """Few requests with long contexts: every row is split over many CTAs (25
    to ~270 parts) and merged by the combine kernel's CTA-per-row path (rows
    of at most 8 parts take its warp-per-row path; that one is covered by
    the other tests)."""
    B = len(lens)
    w = inputs.uniform("few", 50 + B, B=B, ctx=max(lens), Hq=32, Hkv=8, D=128, P=16,
                       outlier_frac=0.01)
    w.ctx_lens = np.array(lens, dtype=np.int32)
    step_and_compare(kvq, w, kv_dtype=kvq.KV_E4M3 if dtype == "e4m3" else kvq.KV_BF16,
                     rows=[(b, h) for b in range(B) for h in (0, 3, 17, 31)])


def test_workspace_reused_across_calls(kvq):
    """One workspace serves a mixed sequence of calls of different shapes
    (every call's plan rewrites the per-call state: bad-page flags, the two
    lists of rows the combine kernel merges): rows of many parts, merged by a
    combine CTA per output row (A), rows of a few parts, merged by a combine
    warp per output row, with two aborted requests and an out-of-pool page
    (B), and the head_dim-64 CUDA-core kernel (C), each checked against the
    oracle, repeats bit-identical."""
    wa = inputs.uniform("reuseA", 71, B=2, ctx=9000, Hq=32, Hkv=8, D=128, P=16, outlier_frac=0.01)
    wa.ctx_lens = np.array([9000, 4100], dtype=np.int32)
    wb = inputs.uniform("reuseB", 72, B=64, ctx=1200, Hq=32, Hkv=8, D=128, P=16)
    wc = inputs.uniform("reuseC", 73, B=16, ctx=2000, Hq=16, Hkv=4, D=64, P=16)
    runs = {}
    for name, w in (("A", wa), ("B", wb), ("C", wc)):
        r = Run(w, host_requests={"A": [0, 1], "B": [0, 3, 5, 11, 40], "C": [0, 3, 9, 15]}[name])
        r.fill_context()
        q = r.append_step(0)
        runs[name] = (r, q, w.seq_lens_after(0))
    size = max(kvq.kvq_decode_attn_workspace_size(w.B, w.Hq, w.Hkv, w.D) for w in (wa, wb, wc))
    ws = torch.zeros(size, dtype=torch.uint8, device="cuda")
    # B: requests 3 and 11 aborted; request 5 has an out-of-pool page (a row
    # split over several CTAs sets its bad-page flag)
    abort_b = np.zeros(wb.B, dtype=np.uint8)
    abort_b[[3, 11]] = 1
    bt_b = wb.block_table.copy()
    bt_b[5, 40] = wb.num_pages + 7
    ref = {}
    for name in ("A", "B", "C"):
        r, q, lens = runs[name]
        rows = [(b, h) for b in r.host_requests for h in range(0, r.w.Hq, 5)]
        if name == "B":
            want, err = oracle.decode_attn(oracle.KV_E4M3, r.hk, r.hv, r.k_scale, r.v_scale, q,
                                           bt_b, lens, abort_mask=abort_b, sm_scale=r.w.sm_scale,
                                           rows=rows, nthreads=16)
            assert err == kvq.ERRBIT_PAGE
        else:
            want, err = r.oracle_rows(q, lens, rows)
            assert err == 0
        ref[name] = (want, rows)
    first = {}
    for name in ("A", "B", "C", "A", "B", "C", "A"):
        r, q, lens = runs[name]
        r.err.zero_()
        if name == "B":
            got = r.attend(q, lens, abort=abort_b, ws=ws, bt=dev(bt_b))
            assert r.err_word() == kvq.ERRBIT_PAGE
            assert not got[3].any() and not got[11].any() and not got[5].any()
        else:
            got = r.attend(q, lens, ws=ws)
            assert r.err_word() == 0
        want, rows = ref[name]
        for b, h in rows:
            assert_close(got[b, h], want[b, h], f"{name} row ({b},{h})")
        if name in first:
            assert np.array_equal(got, first[name]), f"{name}: repeated call differs"
        else:
            first[name] = got


@pytest.mark.parametrize("G,page", [(4, 100), (8, 100), (8, 101)],
                         ids=["g4_p100", "g8_p100", "g8_p101"])
def test_combine_path_bad_page(kvq, G, page):
    """Rows split over many CTAs, merged by the combine kernel, with an
    out-of-pool page in request 2 (for G = 8, whose consumers take two stages
    per step, at two neighbouring pages, so that it falls in either stage of
    a pair): that request's rows are zero, the page error is raised, the
    other requests match the oracle."""
    w = inputs.uniform("warpbad", 81 + G, B=6, ctx=4000, Hq=8 * G, Hkv=8, D=128, P=16)
    r = Run(w, host_requests=[0, 2, 5])
    r.fill_context()
    q = r.append_step(0)
    lens = w.seq_lens_after(0)
    bt = w.block_table.copy()
    bt[2, page] = -3
    got = r.attend(q, lens, bt=dev(bt))
    assert r.err_word() == kvq.ERRBIT_PAGE
    assert not got[2].any()
    rows = [(b, h) for b in (0, 5) for h in range(0, w.Hq, 3)]
    want, err = oracle.decode_attn(oracle.KV_E4M3, r.hk, r.hv, r.k_scale, r.v_scale, q, bt, lens,
                                   sm_scale=w.sm_scale, rows=rows, nthreads=16)
    for b, h in rows:
        assert_close(got[b, h], want[b, h], f"row ({b},{h})")


# The tensor-core split kernel schedules itself (before the plan kernel has
# finished) for batches of up to 32 x (kv heads per group + 1) x 16 requests,
# and takes the plan's schedule for larger ones: 1,024 requests when a group
# is one kv head, 4,608 when it is eight.
@pytest.mark.parametrize("Hkv,B", [(1, 1024), (1, 1100), (8, 4608), (8, 4700)],
                         ids=["hg1_own_1024", "hg1_plan_1100", "hg8_own_4608", "hg8_plan_4700"])
def test_schedule_at_and_past_the_own_scan_limit(kvq, Hkv, B):
    """Short ragged requests (1-60 tokens) in numbers at and just past the
    limit: sampled rows from the start, the end and around the boundary
    requests match the oracle, and every other row is finite."""
    w = inputs.ragged(seed=900 + B + Hkv, B=B, total=B * 25, lo=1, hi=60, Hq=4 * Hkv, Hkv=Hkv,
                      D=128, P=16)
    host = sorted({0, 1, 2, B // 2, 1023, 1024, B - 2, B - 1} & set(range(B)))
    r = Run(w, host_requests=host)
    r.fill_context()
    q = r.append_step(0)
    lens = w.seq_lens_after(0)
    got = r.attend(q, lens)
    assert r.err_word() == 0
    assert np.isfinite(got).all()
    rows = [(b, h) for b in host for h in range(w.Hq)]
    ref, err = r.oracle_rows(q, lens, rows)
    assert err == 0
    for b, h in rows:
        assert_close(got[b, h], ref[b, h], f"row ({b},{h})")


def test_schedule_skips_runs_of_empty_and_aborted_requests(kvq):
    """The split CTAs walk requests by their own lengths and abort flags:
    runs of empty (L = 0) and aborted requests longer than 32, at the start,
    in the middle and at the end of the batch, own no units; the rows between
    them match the oracle and the skipped rows are zero."""
    B = 200
    w = inputs.uniform("skips", 91, B=B, ctx=600, Hq=32, Hkv=8, D=128, P=16)
    real = list(range(50, 61)) + list(range(151, 160)) + [185]
    r = Run(w, host_requests=real)
    r.fill_context()
    q = r.append_step(0)
    lens = w.seq_lens_after(0).copy()
    abort = np.zeros(B, dtype=np.uint8)
    others = np.setdiff1d(np.arange(B), real)
    lens[others[::2]] = 0          # empty
    abort[others[1::2]] = 1        # aborted
    lens[185] = 1                  # one token: its row is that token's V
    got = r.attend(q, lens, abort=abort)
    assert r.err_word() == 0
    assert not got[others].any()
    rows = [(b, h) for b in real for h in range(0, 32, 3)]
    ref, err = r.oracle_rows(q, lens, rows, abort=abort)
    assert err == 0
    for b, h in rows:
        assert_close(got[b, h], ref[b, h], f"row ({b},{h})")


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_softmax_weights_kept_to_fp32_accuracy(kvq, G):
    """Two cached tokens whose scores differ by a fraction (weights that f16
    cannot hold) and V rows of +100 and -100 r_d with r_d spanning 0.05..20
    over the dims, so that in every head some output dims nearly cancel.
    Rounding the weights to f16 alone would break the tolerance in every
    head (checked here on the CPU from the oracle's dequantised cache); the
    kernel, which carries each weight as f16 hi + lo (for G <= 4 through the
    MMA's free head slots), matches the oracle everywhere."""
    D, Hkv, L = 128, 2, 2
    w = inputs.uniform("cancel", 95 + G, B=2, ctx=L, Hq=G * Hkv, Hkv=Hkv, D=D, P=16,
                       outlier_frac=0.0)
    r_d = np.exp(np.linspace(np.log(0.05), np.log(20.0), D))
    k = np.zeros((L, Hkv, D), np.float32)
    k[0], k[1] = 1.0, 1.5
    v = np.zeros((L, Hkv, D), np.float32)
    v[0], v[1] = 100.0, -100.0 * r_d
    sources = [(_bf16_bits(k), _bf16_bits(v)) for _ in range(w.B)]
    r = Run(w, sources=sources)
    r.fill_context()
    c = 0.05 + 0.0137 * np.arange(w.Hq)  # a score gap of 0.3 to 1.6 between the two tokens
    q = _bf16_bits(np.broadcast_to(c[None, :, None], (w.B, w.Hq, D)))
    lens = w.ctx_lens.astype(np.int32)
    got = r.attend(q, lens)
    assert r.err_word() == 0
    rows = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    ref, err = r.oracle_rows(q, lens, rows)
    assert err == 0
    for b, h in rows:
        assert_close(got[b, h], ref[b, h], f"G={G} row ({b},{h})")
    # the case is sensitive: f16 weights alone fail in every head
    for b, h in rows:
        g = h // G
        pages = w.block_table[b, np.arange(L) // w.P]
        slots = np.arange(L) % w.P
        K = pins.torch_decode(r.hk[pages, g, slots, :]) * float(r.k_scale)
        V = pins.torch_decode(r.hv[pages, g, slots, :]) * float(r.v_scale)
        qf = (q[b, h].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        s = (K @ qf) * float(w.sm_scale)
        p = 128.0 * np.exp(s - s.max())
        o16 = (p.astype(np.float16).astype(np.float64) @ V) / p.sum()
        assert (np.abs(o16 - ref[b, h]) > 1e-3 + 1e-3 * np.abs(ref[b, h])).any(), \
            f"row ({b},{h}) does not distinguish f16 weights"


@pytest.mark.parametrize("G", [1, 8])
def test_softmax_weights_bf16_cache(kvq, G):
    """The cancellation case of test_softmax_weights_kept_to_fp32_accuracy on
    the bf16-cache kernel (weights as bf16 hi + lo, about 16 significant
    bits): every row matches the oracle."""
    D, Hkv, L = 128, 2, 2
    w = inputs.uniform("cancel_bf16", 97 + G, B=2, ctx=L, Hq=G * Hkv, Hkv=Hkv, D=D, P=16,
                       outlier_frac=0.0)
    r_d = np.exp(np.linspace(np.log(0.05), np.log(20.0), D))
    k = np.zeros((L, Hkv, D), np.float32)
    k[0], k[1] = 1.0, 1.5
    v = np.zeros((L, Hkv, D), np.float32)
    v[0], v[1] = 100.0, -100.0 * r_d
    sources = [(_bf16_bits(k), _bf16_bits(v)) for _ in range(w.B)]
    r = Run(w, kv_dtype=kvq.KV_BF16, sources=sources)
    r.fill_context()
    q = _bf16_bits(np.broadcast_to((0.05 + 0.0137 * np.arange(w.Hq))[None, :, None],
                                   (w.B, w.Hq, D)))
    lens = w.ctx_lens.astype(np.int32)
    got = r.attend(q, lens)
    assert r.err_word() == 0
    rows = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    ref, err = r.oracle_rows(q, lens, rows)
    assert err == 0
    for b, h in rows:
        assert_close(got[b, h], ref[b, h], f"bf16 G={G} row ({b},{h})")


def test_bad_page_rows_are_zero_even_with_nan_codes(kvq):
    """A request with a page outside the pool is written as zeros, including
    when its other pages hold NaN codes (0x7F), for a row held by one CTA
    (short request) and for a row split across CTAs (long request); the
    other requests match the oracle."""
    B = 120
    w = inputs.uniform("badnan", 93, B=B, ctx=3000, Hq=32, Hkv=8, D=128, P=16)
    lens = np.full(B, 40, dtype=np.int32)  # short rows: most are held by one CTA
    lens[7] = 3000                          # a long row, split across CTAs
    w.ctx_lens = lens.copy()
    good = [0, 6, 8, 119]
    r = Run(w, host_requests=good)
    r.fill_context()
    bt = w.block_table.copy()
    for b_bad, page_bad, page_nan in ((3, 1, 0), (7, 100, 5)):
        bt[b_bad, page_bad] = w.num_pages + 5
        p = int(w.block_table[b_bad, page_nan])
        r.cache.k_pool.view(torch.uint8)[p, :, 3, :] = 0x7F
        r.cache.v_pool.view(torch.uint8)[p, :, 3, :] = 0x7F
    q, *_ = w.step_inputs(0)
    got = r.attend(q, lens, bt=dev(bt))
    assert r.err_word() == kvq.ERRBIT_PAGE
    for b_bad in (3, 7):
        assert np.array_equal(got[b_bad], np.zeros_like(got[b_bad])), f"request {b_bad}"
    rows = [(b, h) for b in good for h in range(0, 32, 3)]
    want, err = oracle.decode_attn(oracle.KV_E4M3, r.hk, r.hv, r.k_scale, r.v_scale, q, bt, lens,
                                   sm_scale=w.sm_scale, rows=rows, nthreads=16)
    for b, h in rows:
        assert_close(got[b, h], want[b, h], f"row ({b},{h})")


def test_concurrent_calls_from_host_threads(kvq):
    """Four host threads call kvq_decode_attn at once (ctypes releases the
    GIL), each on its own stream with its own workspace and output, for a
    shape whose kernels this process has not launched yet (the first call
    sets up the kernel and caches its occupancy); every result equals a
    single-threaded call's, bit for bit."""
    import threading
    w = inputs.uniform("threads", 99, B=5, ctx=2500, Hq=16, Hkv=8, D=128, P=16)
    r = Run(w, kv_dtype=kvq.KV_BF16, host_requests=[0])
    r.fill_context()
    q, *_ = w.step_inputs(0)
    lens = w.ctx_lens.astype(np.int32)
    qd, ld = dev_bf16(q), dev(lens)
    outs, errs = [None] * 4, []

    def run(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                ws = kvq.workspace(w.B, w.Hq, w.Hkv, w.D)
                out = torch.empty((w.B, w.Hq, w.D), dtype=torch.float32, device="cuda")
                for _ in range(3):
                    kvq.kvq_decode_attn(r.cache, qd, r.bt, ld, out, ws, sm_scale=float(w.sm_scale))
            s.synchronize()
            outs[i] = out.cpu().numpy()
        except Exception as e:  # reported below
            errs.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errs, errs
    ref = r.attend(q, lens)
    for i in range(4):
        assert np.array_equal(outs[i], ref), f"thread {i}"
