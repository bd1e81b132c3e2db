"""Pins for the CPU oracle: facts fixed by the pages, the e4m3 format and
mathematics, checked WITHOUT the oracle's own arithmetic.

Each ``pin_*`` function raises AssertionError when the oracle disagrees.  The
test modules call them against the real oracle; ``test_oracle_mutants``
calls them against deliberately broken copies of the oracle to show that a
plausible mistake is caught.

Independent references used here:
  * PyTorch's ``float8_e4m3fn`` dtype (a separate implementation of the OCP
    E4M3 format; it rounds to nearest-even and turns |x| >= 465 into NaN
    instead of saturating, so it is compared only where both agree);
  * brute-force nearest-value search over the 253 finite e4m3 values;
  * ``torch.nn.functional.scaled_dot_product_attention`` in float64 on K/V
    gathered with torch indexing;
  * closed forms: one-token context, identical keys, page permutation,
    a pool of 1-byte elements taking half the bytes of 2-byte elements.
"""
import numpy as np
import torch

from fp8_paged_kv_attn_gb300 import inputs

E4M3 = torch.float8_e4m3fn


# ----------------------------------------------------------------------------
# reference helpers (independent of the oracle)
# ----------------------------------------------------------------------------

def torch_decode(codes) -> np.ndarray:
    c = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return c.view(E4M3).to(torch.float64).numpy()


def torch_encode(x) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(E4M3).view(torch.uint8).numpy()


def finite_grid():
    """(values, codes) of all non-negative finite e4m3 numbers, via torch."""
    codes = np.arange(0x7F, dtype=np.uint8)  # 0x00 .. 0x7E
    return torch_decode(codes), codes


def brute_force_encode(x: np.ndarray) -> np.ndarray:
    """Nearest finite e4m3 value; on an exact tie the code with an even
    mantissa; beyond 448 saturate to 448 (the satfinite reading)."""
    vals, codes = finite_grid()
    a = np.abs(x.astype(np.float64))
    d = np.abs(a[:, None] - vals[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    even = (codes[None, :] & 1) == 0
    pick_even = cand & even
    has_even = pick_even.any(axis=1)
    idx = np.where(has_even, pick_even.argmax(axis=1), cand.argmax(axis=1))
    out = codes[idx].astype(np.uint8)
    out[a > 448.0] = 0x7E
    out |= np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    out[np.isnan(x)] = 0x7F
    return out


def all_fp32_sample() -> np.ndarray:
    """All bf16 bit patterns widened with several low halves: 393,216 fp32
    values that include every binade, both signs and rounding boundaries."""
    hi = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF], dtype=np.uint32)
    return (hi[:, None] | lows[None, :]).reshape(-1).view(np.float32)


def near_midpoints() -> np.ndarray:
    """Every midpoint between adjacent non-negative e4m3 values, +-3 fp32 ulps,
    with both signs."""
    vals, _ = finite_grid()
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)  # exact in fp32
    pts = [mids]
    for k in (1, 2, 3):
        up = mids.copy()
        dn = mids.copy()
        for _ in range(k):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
        pts += [up, dn]
    x = np.concatenate(pts).astype(np.float32)
    return np.concatenate([x, -x])


# ----------------------------------------------------------------------------
# codec pins
# ----------------------------------------------------------------------------

def pin_decode_all_codes(oracle):
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    ref = torch_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "NaN codes differ"
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(got[~nan], ref[~nan]), "decoded values differ from torch e4m3fn"
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def pin_decode_structure(oracle):
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0), "positive codes must increase strictly"
    assert pos[0x7E] == 448.0 and pos[0x01] == 2.0 ** -9 and pos[0x08] == 2.0 ** -6
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)


def pin_encode_roundtrip(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = torch_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def pin_encode_vs_torch(oracle):
    x = all_fp32_sample()
    x = x[np.isfinite(x) & (np.abs(x) < 464.0)]
    assert np.array_equal(oracle.e4m3_encode(x), torch_encode(x)), "encode differs from torch RNE"


def pin_encode_brute_force(oracle):
    x = near_midpoints()
    rng = np.random.default_rng(123)
    extra = np.concatenate([
        rng.uniform(-500, 500, 20000).astype(np.float32),
        (rng.standard_normal(20000) * 2.0 ** rng.integers(-14, 9, 20000)).astype(np.float32),
    ])
    x = np.concatenate([x, extra])
    assert np.array_equal(oracle.e4m3_encode(x), brute_force_encode(x))


def pin_encode_special(oracle):
    f = np.float32
    cases = [  # (value, code); a list because 0.0 == -0.0 as dict keys
        (448.0, 0x7E), (-448.0, 0xFE), (464.0, 0x7E), (465.0, 0x7E), (1e30, 0x7E),
        (float("inf"), 0x7E), (float("-inf"), 0xFE), (2.0 ** -9, 0x01),
        (2.0 ** -10, 0x00),                                   # tie -> even (0)
        (float(np.nextafter(f(2.0 ** -10), f(1))), 0x01),
        (3 * 2.0 ** -10, 0x02),                               # tie 1 vs 2 -> 2
        (5 * 2.0 ** -10, 0x02),                               # tie 2 vs 3 -> 2
        (0.0, 0x00), (-0.0, 0x80), (2.0 ** -6, 0x08), (1.0, 0x38), (1.0625, 0x38),
        (1.1875, 0x3A), (240.0, 0x77), (256.0, 0x78), (1e-30, 0x00), (-1e-30, 0x80),
    ]
    x = np.array([c[0] for c in cases], dtype=np.float32)
    want = np.array([c[1] for c in cases], dtype=np.uint8)
    got = oracle.e4m3_encode(x)
    assert np.array_equal(got, want), list(zip(x, got, want))
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


QUANT_SCALES = [1.0, 3.0, 0.1, 7.0, 1.0 / 3.0, 0.0123, 37.5, 1e-3]


def pin_quantise_exhaustive(oracle):
    """Every bf16 input, several scales: one IEEE fp32 division (torch on the
    CPU divides in IEEE fp32) then RNE into e4m3; beyond 448 saturate."""
    bits = np.arange(65536, dtype=np.uint16)
    x = torch.from_numpy(inputs.bf16_bits_to_f32(bits))
    for s in QUANT_SCALES:
        s32 = np.float32(s)
        got = oracle.quantise(bits, s32)
        y = (x / torch.tensor(s32)).numpy()
        ok = np.isfinite(y) & (np.abs(y) < 464.0)
        assert np.array_equal(got[ok], torch_encode(y[ok])), f"scale {s}"
        big = np.isfinite(x.numpy()) & ~ok & ~np.isnan(y)
        assert np.all(got[big] & 0x7F == 0x7E), f"saturation at scale {s}"
        assert np.all(got[np.isnan(y)] & 0x7F == 0x7F)


# ----------------------------------------------------------------------------
# append pins
# ----------------------------------------------------------------------------

SENTINEL = 0xA5


def _fill_context(oracle, w, dtype=None, sources=None):
    dtype = oracle.KV_E4M3 if dtype is None else dtype
    np_dtype = np.uint8 if dtype == oracle.KV_E4M3 else np.uint16
    kp = np.full(w.pool_shape(), SENTINEL, dtype=np_dtype)
    vp = np.full(w.pool_shape(), SENTINEL, dtype=np_dtype)
    sources = w.kv_sources() if sources is None else sources
    ks, vs = w.scales(sources)
    err = 0
    for b, (k, v) in enumerate(sources):
        req, pos = w.context_tokens(b)
        err |= oracle.quant_append(dtype, kp, vp, ks, vs, k, v, req, pos, w.block_table)
    return kp, vp, ks, vs, sources, err


def pin_append_slots(oracle, w):
    """Every appended token is found, quantised as torch would, at the slot the
    block table names; every other byte keeps its sentinel."""
    kp, vp, ks, vs, sources, err = _fill_context(oracle, w)
    assert err == 0
    touched = np.zeros((w.num_pages, w.P), dtype=bool)  # [page, slot]
    bt = torch.from_numpy(w.block_table.astype(np.int64))
    for b, (k, v) in enumerate(sources):
        L = k.shape[0]
        j = torch.arange(L)
        pages = bt[b, j // w.P].numpy()
        slots = (j % w.P).numpy()
        got_k = kp[pages, :, slots, :]
        got_v = vp[pages, :, slots, :]
        kf = torch.from_numpy(inputs.bf16_bits_to_f32(k))
        vf = torch.from_numpy(inputs.bf16_bits_to_f32(v))
        want_k = (kf / torch.tensor(ks)).to(E4M3).view(torch.uint8).numpy()
        want_v = (vf / torch.tensor(vs)).to(E4M3).view(torch.uint8).numpy()
        assert np.array_equal(got_k, want_k), f"K of request {b}"
        assert np.array_equal(got_v, want_v), f"V of request {b}"
        touched[pages, slots] = True
    by_slot_k = kp.transpose(0, 2, 1, 3)  # [page, slot, head, dim]
    by_slot_v = vp.transpose(0, 2, 1, 3)
    assert np.all(by_slot_k[~touched] == SENTINEL) and np.all(by_slot_v[~touched] == SENTINEL)


def pin_append_bf16_copy(oracle, w):
    kp, vp, _, _, sources, err = _fill_context(oracle, w, dtype=oracle.KV_BF16)
    assert err == 0
    for b, (k, v) in enumerate(sources):
        L = k.shape[0]
        j = np.arange(L)
        pages = w.block_table[b, j // w.P]
        assert np.array_equal(kp[pages, :, j % w.P, :], k)
        assert np.array_equal(vp[pages, :, j % w.P, :], v)


def handoff_case(rng=None):
    """A small handoff: 5 requests (an empty one, ranges that start past 0
    and end mid-page), prefill pages of 32 tokens, decode pages of 16, GQA
    head count 2, D 64; the prefill pools hold random bf16 values where the
    requests' tokens live and a sentinel elsewhere."""
    h = inputs.handoff(seed=61, lens=[37, 0, 100, 16, 61], first=[0, 3, 5, 0, 40], Hkv=2, D=64,
                       src_P=32, dst_P=16, decode_room=20, dst_pool_factor=1.5)
    rng = np.random.default_rng(62) if rng is None else rng
    # one spare page past the pool, so that a page id one past the end stays
    # inside the allocation even for code that does not check it
    spare = (h.src_pages + 1,) + h.src_shape()[1:]
    sk = np.full(spare, 0xBEEF, dtype=np.uint16)[:h.src_pages]
    sv = np.full(spare, 0xBEEF, dtype=np.uint16)[:h.src_pages]
    for b in range(h.B):
        k, v = h.kv_source(b)
        j = np.arange(k.shape[0])
        pages = h.src_block_table[b, j // h.src_P]
        sk[pages, :, j % h.src_P, :] = k
        sv[pages, :, j % h.src_P, :] = v
    ks = inputs.scale_from_amax(inputs.amax_bf16(sk[sk != 0xBEEF]))
    vs = inputs.scale_from_amax(inputs.amax_bf16(sv[sv != 0xBEEF]))
    return h, sk, sv, ks, vs


def pin_handoff_vs_torch(oracle):
    """The handoff: every moved token is found at its decode slot, quantised
    as torch would quantise the bf16 value torch indexing reads from its
    prefill slot (fp32 division by the scale, then float8_e4m3fn); a bf16
    decode pool receives the bits unchanged; every other decode byte keeps
    its sentinel; bad ranges and pages raise their bits and write nothing."""
    h, sk, sv, ks, vs = handoff_case()
    for dt in (oracle.KV_E4M3, oracle.KV_BF16):
        npdt = np.uint8 if dt == oracle.KV_E4M3 else np.uint16
        sent = SENTINEL if dt == oracle.KV_E4M3 else 0xA5A5
        dk = np.full(h.dst_shape(), sent, dtype=npdt)
        dv = np.full(h.dst_shape(), sent, dtype=npdt)
        err = oracle.handoff_pages(sk, sv, h.src_block_table, dt, dk, dv, h.dst_block_table, ks, vs,
                                   h.count, h.first)
        assert err == 0
        touched = np.zeros((h.dst_pages, h.dst_P), dtype=bool)
        tsk, tsv = torch.from_numpy(sk.view(np.int16)), torch.from_numpy(sv.view(np.int16))
        for b in range(h.B):
            p = torch.arange(int(h.first[b]), int(h.first[b] + h.count[b]))
            if p.numel() == 0:
                continue
            spg = torch.from_numpy(h.src_block_table[b].astype(np.int64))[p // h.src_P]
            src_k = tsk[spg, :, p % h.src_P, :].view(torch.bfloat16)
            src_v = tsv[spg, :, p % h.src_P, :].view(torch.bfloat16)
            dpg = h.dst_block_table[b][(p // h.dst_P).numpy()]
            dsl = (p % h.dst_P).numpy()
            if dt == oracle.KV_E4M3:
                want_k = (src_k.float() / torch.tensor(ks)).to(E4M3).view(torch.uint8).numpy()
                want_v = (src_v.float() / torch.tensor(vs)).to(E4M3).view(torch.uint8).numpy()
            else:
                want_k = src_k.view(torch.int16).numpy().view(np.uint16)
                want_v = src_v.view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(dk[dpg, :, dsl, :], want_k), f"K of request {b}"
            assert np.array_equal(dv[dpg, :, dsl, :], want_v), f"V of request {b}"
            touched[dpg, dsl] = True
        assert np.all(dk.transpose(0, 2, 1, 3)[~touched] == sent)
        assert np.all(dv.transpose(0, 2, 1, 3)[~touched] == sent)
    # errors: a range past the decode table, a negative count, a prefill
    # page outside the pool, a decode page outside the pool
    cnt = h.count.copy()
    fst = h.first.copy()
    sbt = h.src_block_table.copy()
    dbt = h.dst_block_table.copy()
    cnt[0] = h.dst_MP * h.dst_P + 1        # request 0: past the capacity
    cnt[1] = -1                            # request 1: negative
    sbt[2, (5 + 10) // h.src_P] = -1       # request 2: token 10 of its range (and its page-mates)
    sbt[3, 0] = h.src_pages                # request 3: one past the prefill pool
    dbt[4, (40 + 3) // h.dst_P] = h.dst_pages  # request 4: the decode page of its token 3
    dk = np.full(h.dst_shape(), SENTINEL, dtype=np.uint8)
    dv = np.full(h.dst_shape(), SENTINEL, dtype=np.uint8)
    err = oracle.handoff_pages(sk, sv, sbt, oracle.KV_E4M3, dk, dv, dbt, ks, vs, cnt, fst)
    assert err == oracle.ERR_POS | oracle.ERR_PAGE
    for b in (0, 1, 3):  # nothing of these requests is written
        pages = h.dst_block_table[b][h.dst_block_table[b] >= 0]
        assert np.all(dk[pages] == SENTINEL) and np.all(dv[pages] == SENTINEL)
    # request 2: the tokens on the bad prefill page are not written, the rest are
    p = np.arange(5, 105)
    on_bad = (p // h.src_P) == (5 + 10) // h.src_P
    dpg, dsl = h.dst_block_table[2][p // h.dst_P], p % h.dst_P
    assert np.all(dk[dpg[on_bad], :, dsl[on_bad], :] == SENTINEL)
    assert not np.any(np.all(dk[dpg[~on_bad], :, dsl[~on_bad], :] == SENTINEL, axis=(1, 2)))


def pin_half_bytes(w):
    """An e4m3 pool holds the same tokens as a bf16 pool in half the bytes; at
    equal pool bytes the bf16 pool admits half the requests (the pages' BF16
    cache runs out past 32 concurrent requests while FP8 serves 64)."""
    fp8 = np.zeros(w.pool_shape(), dtype=np.uint8)
    bf16 = np.zeros(w.pool_shape(), dtype=np.uint16)
    assert 2 * fp8.nbytes == bf16.nbytes
    s8 = inputs.sweep(64, kv_bytes=1)
    s16 = inputs.sweep(32, kv_bytes=2)
    per_page = s8.Hkv * s8.P * s8.D
    assert s8.num_pages * per_page * 1 == s16.num_pages * per_page * 2
    assert s8.num_pages == 2 * s16.num_pages
    try:
        inputs.sweep(33, kv_bytes=2)
    except MemoryError:
        pass
    else:
        raise AssertionError("33 bf16 requests must not fit the equal-bytes pool")


def pin_append_errors(oracle):
    w = inputs.tiny()
    kp = np.full(w.pool_shape(), SENTINEL, dtype=np.uint8)
    vp = kp.copy()
    k = np.zeros((4, w.Hkv, w.D), dtype=np.uint16)
    req = np.array([5, 0, 0, 0], dtype=np.int32)
    pos = np.array([0, -1, w.MP * w.P, 0], dtype=np.int32)
    bt = w.block_table.copy()
    bt[0, 0] = w.num_pages  # out of the pool
    err = oracle.quant_append(oracle.KV_E4M3, kp, vp, 1.0, 1.0, k, k, req, pos, bt)
    assert err == (oracle.ERR_REQ | oracle.ERR_POS | oracle.ERR_PAGE)
    assert np.all(kp == SENTINEL) and np.all(vp == SENTINEL)


# ----------------------------------------------------------------------------
# tag-check pins
# ----------------------------------------------------------------------------

def brute_force_check(w, seq_lens, page_tags, expected, bt):
    """Python set comparison: requests whose recorded (page, tag) pairs are not
    all current."""
    current = {(p, int(t)) for p, t in enumerate(page_tags)}
    out = np.zeros(w.B, dtype=np.uint8)
    for b in range(w.B):
        L = int(seq_lens[b])
        if L < 0 or L > w.MP * w.P:
            out[b] = 1
            continue
        n = -(-L // w.P)
        want = {(int(bt[b, i]), int(expected[b, i])) for i in range(n)}
        if not want <= current:
            out[b] = 1
    return out


def pin_check_injected(oracle, w):
    lens = w.seq_lens_after(0)
    got = oracle.check_tags(w.block_table, lens, w.P, w.page_tags, w.expected_tags)
    assert np.array_equal(got, brute_force_check(w, lens, w.page_tags, w.expected_tags,
                                                 w.block_table))
    assert set(np.nonzero(got)[0].tolist()) == set(w.stale)


def pin_check_edges(oracle):
    w = inputs.tiny()
    lens = w.seq_lens_after(0)
    assert not oracle.check_tags(w.block_table, lens, w.P, w.page_tags, w.expected_tags).any()
    # a stale tag on a page past the checked range is ignored; on the last
    # checked page it aborts
    for b in range(w.B):
        n = -(-int(lens[b]) // w.P)
        exp = w.expected_tags.copy()
        exp[b, n] += 1
        assert not oracle.check_tags(w.block_table, lens, w.P, w.page_tags, exp).any()
        exp = w.expected_tags.copy()
        exp[b, n - 1] += 1
        m = oracle.check_tags(w.block_table, lens, w.P, w.page_tags, exp)
        assert m.tolist() == [int(i == b) for i in range(w.B)]
    bt = w.block_table.copy()
    bt[1, 0] = -3
    assert oracle.check_tags(bt, lens, w.P, w.page_tags, w.expected_tags).tolist() == [0, 1]
    bad_len = lens.copy()
    bad_len[0] = w.MP * w.P + 1
    assert oracle.check_tags(w.block_table, bad_len, w.P, w.page_tags,
                             w.expected_tags).tolist() == [1, 0]
    zero = np.zeros_like(lens)
    assert not oracle.check_tags(w.block_table, zero, w.P, w.page_tags, w.expected_tags).any()


# ----------------------------------------------------------------------------
# attention pins
# ----------------------------------------------------------------------------

def sdpa_reference(kv_dtype_is_fp8, kp, vp, ks, vs, q_bits, bt, lens, Hkv, sm_scale):
    """float64 SDPA on K/V gathered by torch indexing; fp8 decoded by torch."""
    B, Hq, D = q_bits.shape
    g = Hq // Hkv
    P = kp.shape[2]
    q = torch.from_numpy(inputs.bf16_bits_to_f32(q_bits)).to(torch.float64)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        L = int(lens[b])
        if L == 0:
            continue
        j = np.arange(L)
        pages = bt[b, j // P]
        kb = kp[pages, :, j % P, :]  # [L, Hkv, D]
        vb = vp[pages, :, j % P, :]
        if kv_dtype_is_fp8:
            k = torch_decode(kb) * float(ks)
            v = torch_decode(vb) * float(vs)
        else:
            k = inputs.bf16_bits_to_f32(kb).astype(np.float64)
            v = inputs.bf16_bits_to_f32(vb).astype(np.float64)
        k = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, dim=0)  # [Hq, L, D]
        v = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b][:, None, :], k, v, scale=float(sm_scale))
        out[b] = o[:, 0, :].numpy()
    return out


def _attend(oracle, w, kv_dtype, kp, vp, ks, vs, q, lens, **kw):
    return oracle.decode_attn(kv_dtype, kp, vp, ks, vs, q, w.block_table, lens,
                              sm_scale=w.sm_scale, **kw)


def pin_attn_vs_sdpa(oracle, w, kv_dtype=None):
    kv_dtype = oracle.KV_E4M3 if kv_dtype is None else kv_dtype
    kp, vp, ks, vs, _, _ = _fill_context(oracle, w, dtype=kv_dtype)
    q, *_ = w.step_inputs(0)
    lens = w.ctx_lens
    got, err = _attend(oracle, w, kv_dtype, kp, vp, ks, vs, q, lens)
    assert err == 0
    ref = sdpa_reference(kv_dtype == oracle.KV_E4M3, kp, vp, ks, vs, q, w.block_table,
                         lens, w.Hkv, w.sm_scale)
    np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-7)


def pin_attn_one_token(oracle):
    """One cached token: softmax weight 1, the output is that token's V."""
    w = inputs.uniform("one", 7, B=3, ctx=1, Hq=8, Hkv=2, D=64, P=16, outlier_frac=0.01)
    kp, vp, ks, vs, _, _ = _fill_context(oracle, w)
    q, *_ = w.step_inputs(0)
    got, err = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, w.ctx_lens)
    assert err == 0
    for b in range(w.B):
        page = w.block_table[b, 0]
        for h in range(w.Hq):
            v = torch_decode(vp[page, h // w.G, 0, :]) * float(vs)
            assert np.array_equal(got[b, h], v.astype(np.float32))


def pin_attn_equal_keys(oracle):
    """All keys identical: uniform weights, the output is the mean of V."""
    w = inputs.uniform("eqk", 8, B=2, ctx=45, Hq=4, Hkv=2, D=64, P=16)
    kp, vp, ks, vs, _, _ = _fill_context(oracle, w)
    kp[...] = 0x3C  # every key element 1.5
    q, *_ = w.step_inputs(0)
    got, err = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, w.ctx_lens)
    assert err == 0
    for b in range(w.B):
        L = int(w.ctx_lens[b])
        j = np.arange(L)
        pages = w.block_table[b, j // w.P]
        v = torch_decode(vp[pages, :, j % w.P, :]) * float(vs)  # [L, Hkv, D]
        mean = v.mean(axis=0)
        for h in range(w.Hq):
            np.testing.assert_allclose(got[b, h], mean[h // w.G], rtol=1e-6, atol=1e-7)


def pin_attn_page_permutation(oracle, w):
    """Moving pages to other physical slots (and fixing the block table) leaves
    the output bit-for-bit unchanged."""
    kp, vp, ks, vs, _, _ = _fill_context(oracle, w)
    q, *_ = w.step_inputs(0)
    base, err = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, w.ctx_lens)
    assert err == 0
    perm = np.random.default_rng(99).permutation(w.num_pages)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    bt2 = np.where(w.block_table >= 0, perm[np.maximum(w.block_table, 0)], -1).astype(np.int32)
    got, err = oracle.decode_attn(oracle.KV_E4M3, kp2, vp2, ks, vs, q, bt2, w.ctx_lens,
                                  sm_scale=w.sm_scale)
    assert err == 0 and np.array_equal(got, base)


def pin_attn_abort_and_errors(oracle):
    w = inputs.tiny()
    kp, vp, ks, vs, _, _ = _fill_context(oracle, w)
    q, *_ = w.step_inputs(0)
    lens = w.ctx_lens
    full, err = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, lens)
    assert err == 0 and np.all(np.abs(full).sum(axis=2) > 0)
    mask = np.array([1, 0], dtype=np.uint8)
    got, err = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, lens, abort_mask=mask)
    assert err == 0 and not got[0].any() and np.array_equal(got[1], full[1])
    bt = w.block_table.copy()
    bt[1, 2] = w.num_pages + 4
    got, err = oracle.decode_attn(oracle.KV_E4M3, kp, vp, ks, vs, q, bt, lens,
                                  sm_scale=w.sm_scale)
    assert err == oracle.ERR_PAGE and not got[1].any() and np.array_equal(got[0], full[0])
    bad = lens.copy()
    bad[0] = w.MP * w.P + 1
    got, err = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, bad)
    assert err == oracle.ERR_SEQLEN and not got[0].any()
    zero = np.array([0, lens[1]], dtype=np.int32)
    got, err = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, zero)
    assert err == 0 and not got[0].any() and np.array_equal(got[1], full[1])
    rows = [(1, 3), (0, 0)]
    part, _ = _attend(oracle, w, oracle.KV_E4M3, kp, vp, ks, vs, q, lens, rows=rows)
    for b, h in rows:
        assert np.array_equal(part[b, h], full[b, h])


# ----------------------------------------------------------------------------
# page allocator
# ----------------------------------------------------------------------------

GOLDEN_PAGES = __import__("os").path.join(__import__("os").path.dirname(__file__), "golden",
                                          "page_allocator_example.json")


def _golden_pages():
    import json
    with open(GOLDEN_PAGES) as f:
        return json.load(f)


def _state_from(oracle, g, B, MP):
    n = len(g["tags"])
    stack = np.full(n, -7, dtype=np.int32)  # entries above the count are never read
    stack[:len(g["stack"])] = g["stack"]
    return oracle.PageState(stack, g["count"], np.array(g["tags"], dtype=np.uint32),
                            np.full((B, MP), -1, np.int32), np.zeros((B, MP), np.uint32))


def _assert_expect(st, ok, err, e, what):
    assert err == e["err"], (what, "err", err, e["err"])
    assert list(ok) == e["ok"], (what, "ok", list(ok), e["ok"])
    c = int(st.free_count[0])
    assert c == e["count"], (what, "count", c, e["count"])
    if "stack" in e:
        assert list(st.free_stack[:c]) == e["stack"], (what, "stack", list(st.free_stack[:c]))
    assert list(st.page_tags) == e["tags"], (what, "tags", list(st.page_tags), e["tags"])
    for b, row in e["bt"].items():
        assert list(st.block_table[int(b)]) == row, (what, "bt", b, list(st.block_table[int(b)]))
    for b, row in e["exp"].items():
        assert list(st.expected_tags[int(b)]) == row, (what, "exp", b,
                                                       list(st.expected_tags[int(b)]))


def _run_golden_op(oracle, st, op):
    rel = op.get("release", [])
    acq = op.get("acquire", [])
    return oracle.pages_update(st, [r[0] for r in rel], [r[1] for r in rel],
                               [a[0] for a in acq], [a[1] for a in acq], [a[2] for a in acq])


def pin_pages_golden(oracle):
    """The hand-worked allocator example (tests/golden/page_allocator_example.json):
    every op's error bits, served flags, stack, tags, block-table and
    expected-tag rows; the tag check after op 2 (live requests pass, a stale
    copy of a released request fails); uint32 tag wrap-around."""
    g = _golden_pages()
    B, MP, P = g["B"], g["MP"], g["page_size"]
    st = _state_from(oracle, g["initial"], B, MP)
    snapshot = None
    for n, op in enumerate(g["ops"]):
        if n == 1:
            snapshot = st.copy()
        ok, err = _run_golden_op(oracle, st, op)
        _assert_expect(st, ok, err, op["expect"], f"op {n + 1}")
        if "check" in op:
            live = op["check"]["live"]
            rq = live["requests"]
            ab = oracle.check_tags(st.block_table[rq], np.array(live["seq_lens"], np.int32), P,
                                   st.page_tags, st.expected_tags[rq])
            assert list(ab) == live["abort"], ("live check", list(ab))
            stale = op["check"]["stale"]
            assert list(snapshot.block_table[0]) == stale["bt"]
            assert list(snapshot.expected_tags[0]) == stale["exp"]
            ab = oracle.check_tags(np.array([stale["bt"]], np.int32),
                                   np.array([stale["seq_len"]], np.int32), P, st.page_tags,
                                   np.array([stale["exp"]], np.uint32))
            assert list(ab) == [stale["abort"]], ("stale check", list(ab))
    w = g["wrap"]
    st = _state_from(oracle, w["initial"], w["B"], w["MP"])
    ok, err = _run_golden_op(oracle, st, w)
    _assert_expect(st, ok, err, w["expect"], "wrap")


def mapped_prefix(block_table):
    """Per request slot, how many leading block-table entries are mapped."""
    unm = block_table < 0
    return np.where(unm.any(axis=1), unm.argmax(axis=1), block_table.shape[1])


def next_page_ops(rng, block_table, fail_often=False, bad_release=False):
    """One seeded (release, acquire) batch for the current mapping, keeping
    the allocator's preconditions (a request returns exactly its mapped
    prefix, acquires only unmapped entries, appears at most once per list):
    some live requests finish, some grow by a page or two, some free slots
    admit a new request.  `fail_often` asks for three times as many pages;
    `bad_release` makes one release reach past its mapped prefix (which the
    allocator must refuse as a batch)."""
    B, MP = block_table.shape
    held = mapped_prefix(block_table)
    rel_req, rel_n = [], []
    for b in np.nonzero(held > 0)[0]:
        if rng.random() < 0.15:
            rel_req.append(int(b))
            rel_n.append(int(held[b]))
    if bad_release and rel_req and held[rel_req[0]] < MP:
        rel_n[0] += 1
    acq = []
    for b in rng.permutation(B):
        b = int(b)
        if b in rel_req:
            continue
        if held[b] > 0 and held[b] < MP and rng.random() < 0.4:
            n = int(rng.integers(1, 3))
        elif held[b] == 0 and rng.random() < 0.3:
            n = int(rng.integers(1, max(2, MP // 2)))
        else:
            continue
        if fail_often:
            n *= 3
        acq.append((b, int(held[b]), int(min(MP - held[b], n))))
    return (rel_req, rel_n, [a[0] for a in acq], [a[1] for a in acq], [a[2] for a in acq])


def pin_pages_invariants(oracle, seed=3, num_pages=64, B=12, MP=10, n_ops=60):
    """Properties every op must keep, whatever the implementation:
    conservation (the free stack and the live block-table entries hold every
    page exactly once), LIFO order (the pages an op hands out are the top of
    the stack after its releases, in pop order), one tag increment per page
    handed out and none otherwise, served requests = the valid requests in
    order up to the first that does not fit, expected tag = current tag on
    every live entry (so the check passes every live request and fails a
    stale copy of a request whose pages were handed out again)."""
    for fail_often in (False, True):
        rng = np.random.default_rng(seed)
        order = rng.permutation(num_pages).astype(np.int32)
        st = oracle.PageState.fresh(num_pages, B, MP, order=order)
        stale = []
        for step in range(n_ops):
            rel_req, rel_n, acq_req, acq_first, acq_n = next_page_ops(
                rng, st.block_table, fail_often, bad_release=fail_often and step % 7 == 3)
            before = st.copy()
            # releases of entries that were never mapped are refused as a batch
            rel_ok = all(np.all(before.block_table[b, :n] >= 0) for b, n in zip(rel_req, rel_n))
            if rel_ok:
                for b in rel_req:
                    stale.append((before.block_table[b].copy(), before.expected_tags[b].copy()))
            ok, err = oracle.pages_update(st, rel_req, rel_n, acq_req, acq_first, acq_n)
            # after the releases (if accepted): the stack as the acquisitions see it
            stack = list(before.free_stack[:before.free_count[0]])
            if rel_ok:
                for b, n in zip(rel_req, rel_n):
                    stack.extend(int(p) for p in before.block_table[b, :n])
            else:
                assert err & oracle.ERR_PAGE
            # served = valid requests in order until the first that does not fit
            avail = len(stack)
            expect_ok, stopped, handed = [], False, []
            for b, f, n in zip(acq_req, acq_first, acq_n):
                if stopped or n > avail:
                    stopped = True
                    expect_ok.append(0)
                    continue
                expect_ok.append(1)
                for k in range(n):
                    handed.append((b, f + k, stack[len(stack) - 1 - (len(handed))]))
                avail -= n
            assert list(ok) == expect_ok, (list(ok), expect_ok)
            assert bool(err & oracle.ERR_EXHAUSTED) == stopped
            assert int(st.free_count[0]) == len(stack) - len(handed)
            assert list(st.free_stack[:st.free_count[0]]) == stack[:len(stack) - len(handed)]
            # tags: +1 for each page handed out, unchanged otherwise
            bump = np.zeros(num_pages, dtype=np.uint32)
            for _, _, p in handed:
                bump[p] += 1
            assert np.array_equal(st.page_tags, before.page_tags + bump)
            for b, k, p in handed:
                assert st.block_table[b, k] == p
                assert st.expected_tags[b, k] == st.page_tags[p]
            if rel_ok:
                for b, n in zip(rel_req, rel_n):
                    assert np.all(st.block_table[b, :n] < 0)
            else:
                for b in rel_req:
                    assert np.array_equal(st.block_table[b], before.block_table[b])
            # conservation
            live = st.block_table[st.block_table >= 0]
            allp = np.sort(np.concatenate([st.free_stack[:st.free_count[0]], live]))
            assert np.array_equal(allp, np.arange(num_pages)), "a page was lost or duplicated"
            # expected tag = current tag on every live entry: the check passes
            # every request over its mapped prefix
            for b in range(B):
                row = st.block_table[b]
                n = int(np.argmax(row < 0)) if np.any(row < 0) else MP
                if n == 0:
                    continue
                ab = oracle.check_tags(row[None, :], np.array([n * 4], np.int32), 4,
                                       st.page_tags, st.expected_tags[b][None, :])
                assert ab[0] == 0
        # a stale copy of a released request fails the check once one of its
        # pages has been handed out again
        flagged = 0
        for bt_row, exp_row in stale:
            n = int(np.argmax(bt_row < 0)) if np.any(bt_row < 0) else MP
            if n == 0:
                continue
            reused = any(st.page_tags[p] != exp_row[i] for i, p in enumerate(bt_row[:n]))
            ab = oracle.check_tags(bt_row[None, :], np.array([n * 4], np.int32), 4,
                                   st.page_tags, exp_row[None, :])
            assert ab[0] == int(reused)
            flagged += int(reused)
        assert flagged > 0


def pin_pages_overflow_and_state(oracle):
    """A release that would push more pages than the pool holds is refused as
    a whole (page error); so is a call on a free count outside [0, pages]."""
    st = oracle.PageState.fresh(4, 2, 4)
    st.block_table[0, :2] = [1, 2]  # a mapping to pages that are also free
    before = st.copy()
    ok, err = oracle.pages_update(st, [0], [2], [1], [0], [1])
    assert err & oracle.ERR_PAGE
    # the release is refused but the acquisition still runs on the full stack
    assert list(ok) == [1] and st.block_table[0, 0] == 1
    assert int(st.free_count[0]) == 3 and st.block_table[1, 0] == before.free_stack[3]
    bad = oracle.PageState.fresh(4, 2, 4)
    bad.free_count[0] = 5
    snap = bad.copy()
    ok, err = oracle.pages_update(bad, [], [], [0], [0], [1])
    assert err == oracle.ERR_PAGE and list(ok) == [0]
    assert np.array_equal(bad.free_stack, snap.free_stack)
    assert np.array_equal(bad.page_tags, snap.page_tags)
    assert int(bad.free_count[0]) == 5


# ----------------------------------------------------------------------------
# weight-only quantised matrix product
# ----------------------------------------------------------------------------

def _bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def numpy_int4_weights(w, scales, group):
    """Dequantised INT4 weights [N, K] in float64, unpacked with numpy bit
    operations (independent of the oracle): even k = low nibble, odd k = high
    nibble, two's complement."""
    w = np.asarray(w, dtype=np.uint8)
    lo = (w & 0x0F).astype(np.int64)
    hi = (w >> 4).astype(np.int64)
    q = np.empty((w.shape[0], w.shape[1] * 2), dtype=np.int64)
    q[:, 0::2], q[:, 1::2] = lo, hi
    q = np.where(q >= 8, q - 16, q)
    s = np.repeat(_bf16_to_f64(scales), group, axis=1)
    return q.astype(np.float64) * s


def random_wq_case(rng, wdtype, M, N, K, group=128):
    x = inputs.normal_bf16(rng, (M, K))
    if wdtype == 0:
        w = rng.integers(0, 256, (N, K // 2), dtype=np.uint8)
        amax = np.abs(rng.standard_normal((N, K // group))).astype(np.float32) * 0.02 + 1e-3
        s = (amax.view(np.uint32) >> 16).astype(np.uint16)  # bf16 scales
    else:
        w = rng.integers(0, 256, (N, K), dtype=np.uint8)
        w[(w & 0x7F) == 0x7F] ^= 0x01  # no NaN codes in weights
        s = (np.abs(rng.standard_normal(N)) * 0.01 + 1e-3).astype(np.float32)
    return w, s, x


def wide_range_x(rng, M, K):
    """bf16 activations [M, K] (bit patterns) over bf16's whole range, one
    regime per row (cycled): N(0,1) with entries of +-1e5 and +-3e4 (beyond
    f16's 65504); magnitudes log-uniform over 13 decades in one row; all
    near 1e-6; bf16 subnormals only; subnormals mixed with 1e-30; near 1e30;
    zeros but one 1e5; all zeros."""
    x = np.zeros((M, K), dtype=np.float32)
    for m in range(M):
        kind = m % 8
        z = rng.standard_normal(K).astype(np.float32)
        if kind == 0:
            z[rng.choice(K, 6, replace=False)] = np.float32([1e5, -1e5, 3e4, -3e4, 99999.0, -65520.0])
            x[m] = z
        elif kind == 1:
            x[m] = z * np.float32(10.0) ** rng.uniform(-8, 5, K).astype(np.float32)
        elif kind == 2:
            x[m] = z * np.float32(1e-6)
        elif kind == 4:
            x[m] = z * np.float32(1e-30)
        elif kind == 5:
            x[m] = z * np.float32(1e30)
        elif kind == 6:
            x[m, rng.integers(K)] = np.float32(1e5)
    bits = inputs.f32_to_bf16_bits(x)
    for m in range(M):
        kind = m % 8
        if kind in (3, 4):  # bf16 subnormals: exponent field 0, mantissa 1..127
            sub = rng.integers(1, 128, K).astype(np.uint16) | \
                (rng.integers(0, 2, K).astype(np.uint16) << np.uint16(15))
            if kind == 3:
                bits[m] = sub
            else:
                pick = rng.random(K) < 0.5
                bits[m] = np.where(pick, sub, bits[m])
    return bits


def pin_wq_wide_range_x(oracle):
    """Activations over bf16's whole range (wide_range_x): the oracle still
    equals a float64 matmul of independently dequantised weights to within
    the last fp32 bit, for both weight types."""
    rng = np.random.default_rng(33)
    for wdtype in (0, 1):
        w, s, _ = random_wq_case(rng, wdtype, 8, 40, 640)
        x = wide_range_x(rng, 8, 640)
        if wdtype == 0:
            wd = numpy_int4_weights(w, s, 128)
        else:
            wd = torch.from_numpy(w).view(E4M3).to(torch.float64).numpy() * \
                s.astype(np.float64)[:, None]
        ref = _bf16_to_f64(x) @ wd.T
        got = oracle.wq_gemm(oracle.W_INT4 if wdtype == 0 else oracle.W_E4M3, w, s, x)
        assert np.all(np.isfinite(got))
        np.testing.assert_allclose(got, ref, rtol=2e-7, atol=1e-44)
        assert np.any(np.abs(got[0]) > 1e4) and np.all(got[7] == 0.0)


def pin_int4_nibbles(oracle):
    """Every byte value: with a one-hot x picking k = 0 or k = 1 and scale 1,
    y is the low or high nibble read as a signed 4-bit number."""
    b = np.arange(256, dtype=np.uint8)
    w = np.zeros((256, 64), dtype=np.uint8)
    w[:, 0] = b
    one = np.uint16(0x3F80)
    s = np.full((256, 1), one, dtype=np.uint16)
    for k, nib in ((0, b & 0x0F), (1, b >> 4)):
        x = np.zeros((1, 128), dtype=np.uint16)
        x[0, k] = one
        y = oracle.wq_gemm(oracle.W_INT4, w, s, x)[0]
        want = np.where(nib >= 8, nib.astype(np.int64) - 16, nib.astype(np.int64))
        assert np.array_equal(y, want.astype(np.float32)), k


def pin_wq_vs_numpy(oracle):
    """Random INT4 and e4m3 weights: the oracle equals a float64 matmul of
    weights dequantised independently (numpy nibbles; torch's float8_e4m3fn),
    to within the last fp32 bit (the two sum in different orders)."""
    rng = np.random.default_rng(31)
    for M, N, K in ((1, 16, 128), (5, 33, 384), (16, 64, 1024)):
        w, s, x = random_wq_case(rng, 0, M, N, K)
        ref = _bf16_to_f64(x) @ numpy_int4_weights(w, s, 128).T
        got = oracle.wq_gemm(oracle.W_INT4, w, s, x)
        np.testing.assert_allclose(got, ref, rtol=2e-7, atol=1e-30)
        w, s, x = random_wq_case(rng, 1, M, N, K)
        wd = torch.from_numpy(w).view(E4M3).to(torch.float64).numpy() * s.astype(np.float64)[:, None]
        ref = _bf16_to_f64(x) @ wd.T
        got = oracle.wq_gemm(oracle.W_E4M3, w, s, x)
        np.testing.assert_allclose(got, ref, rtol=2e-7, atol=1e-30)


def pin_wq_single_weight(oracle):
    """One nonzero weight: y is exactly x times that weight times its scale,
    in the row and the group the weight sits in; other outputs are 0."""
    K, N = 256, 3
    x = inputs.normal_bf16(np.random.default_rng(32), (2, K))
    w = np.zeros((N, K // 2), dtype=np.uint8)
    w[1, 150 // 2] = 0x30  # k = 151 (high nibble) holds 3; k = 150 holds 0
    s = np.full((N, K // 128), 0x3F80, dtype=np.uint16)
    s[1, 1] = 0x4040  # 3.0 for group 1 (k 128..255)
    y = oracle.wq_gemm(oracle.W_INT4, w, s, x)
    want = _bf16_to_f64(x[:, 151]) * 3 * 3.0
    assert np.array_equal(y[:, 1], want.astype(np.float32))
    assert not y[:, 0].any() and not y[:, 2].any()
