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
