"""The argument behind kvq_append's division-free quantisation, checked on the
CPU with the oracle's encoder (no GPU, no kernel code).

The kernel takes y = RN(1/s), r_lo = RN(y (1 - 2^-21)), r_hi = RN(y (1 + 2^-21))
(host fp32 arithmetic) and the e4m3 codes of RN(x r_lo) and RN(x r_hi); when
the two codes agree it stores that code, else it divides.  The claim:
whenever the two codes agree they equal the code of the correctly rounded
quotient RN(x / s), provided y, r_lo and r_hi are normal floats.  Here
numpy's float32 arithmetic (IEEE, round to nearest even) plays the kernel's
and the claim is checked for every bf16 input at many scales.  The test
also counts how often the kernel would fall back to the division.
"""
import numpy as np

import oracle

SHRINK = np.float32(1.0 - 2.0 ** -21)
GROW = np.float32(1.0 + 2.0 ** -21)


def _all_bf16_as_f32():
    bits = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    return bits.view(np.float32)


def _scales():
    rng = np.random.default_rng(17)
    fixed = [1.0, 3.0, 0.1, 1.0 / 3.0, 0.0123, 37.5, 1e-3, 2.0 ** -20, 2.0 ** -126, 1e-38,
             2.0 ** 126, 1.7e38, 448.0, 1.0 / 448.0, 0.999999, 1.000001]
    rand = [2.0 ** e for e in rng.uniform(-60, 60, 24)]
    return [np.float32(s) for s in fixed + rand]


def test_fast_path_agrees_with_division():
    x = _all_bf16_as_f32()
    finite = np.isfinite(x)
    fallbacks = 0
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        for s in _scales():
            rcp = np.float32(1.0) / s
            r_lo, r_hi = rcp * SHRINK, rcp * GROW
            if not (np.isfinite(rcp) and np.isfinite(r_hi) and r_lo >= np.finfo(np.float32).tiny):
                continue  # the kernel divides every element for such a scale
            exact = oracle.e4m3_encode(x / s)  # float32 division: RN(x / s)
            lo = oracle.e4m3_encode(x * r_lo)
            hi = oracle.e4m3_encode(x * r_hi)
            agree = lo == hi
            # NaN inputs give a NaN code on both paths; compare the rest
            ok = agree & finite
            bad = np.nonzero(lo[ok] != exact[ok])[0]
            assert bad.size == 0, (float(s), x[ok][bad[:5]], lo[ok][bad[:5]], exact[ok][bad[:5]])
            assert np.all((lo[agree & ~finite] & 0x7F) == (exact[agree & ~finite] & 0x7F))
            fallbacks += int((~agree).sum())
    # the fall-back is rare for scales that are not powers of two
    assert fallbacks < 0.02 * 65536 * len(_scales())


def test_margin_is_needed():
    """Without the margin (lo = hi = q) the reciprocal product alone is wrong
    for some inputs: the interval check is doing work."""
    x = _all_bf16_as_f32()
    wrong = 0
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        for s in _scales():
            fin = np.isfinite(x)
            exact = oracle.e4m3_encode(x[fin] / s)
            naive = oracle.e4m3_encode(x[fin] * (np.float32(1.0) / s))
            wrong += int((naive != exact).sum())
    assert wrong > 0


EXACT_AMAX = (1.75, 3.5, 5.25, 7.0, 10.5, 224.0)  # amax / 448 exact in fp32
OTHER_AMAX = (2.0, 0.75, 96.0, 83.0, 81.5, 121.0, 0.0123, 1e5)


def _wide_scales():
    """Seeded scales with full significands (amax / 448 for arbitrary amax)."""
    rng = np.random.default_rng(23)
    return [np.float32(a / 448.0) for a in rng.uniform(0.5, 500.0, 24)]


def _amax_scales():
    """amax / 448 (fp32, as the host rounds it) for amax values that make it
    exact (a power of two times 1 or 3: many quotients then fall exactly on
    e4m3 boundaries) and for others."""
    return [np.float32(a / 448.0) for a in EXACT_AMAX + OTHER_AMAX]


def test_exact_remainder_step():
    """The second step: where the two codes differ, q = RN(x y) and
    t = RN(x - q s) (one fma); t = 0 must mean RN(x / s) = q, so the code is
    e4m3(q).  Checked for every bf16 input and scale (scale >= 2^-92, the
    host's condition for the step); what is left goes to the division.  On
    round amax / 448 scales nothing is left: every differing element is an
    exact quotient.  On scales whose significand (trailing zeros dropped)
    has 8 or more bits no differing element is exact, which is why the
    kernel skips the step for them."""
    x = _all_bf16_as_f32()
    fin = np.isfinite(x)
    left_round = 0
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        for s in _scales() + _amax_scales() + _wide_scales():
            rcp = np.float32(1.0) / s
            r_lo, r_hi = rcp * SHRINK, rcp * GROW
            if not (np.isfinite(rcp) and np.isfinite(r_hi) and r_lo >= np.finfo(np.float32).tiny):
                continue
            if s < np.float32(2.0 ** -92):
                continue
            differ = (oracle.e4m3_encode(x * r_lo) != oracle.e4m3_encode(x * r_hi)) & fin
            xd = x[differ]
            q = xd * rcp  # float32 product: RN(x y)
            # x - q s exactly (a float64 product of two floats is exact, and the
            # difference of two values this close is exact too), rounded once
            t = (xd.astype(np.float64) - q.astype(np.float64) * np.float64(s)).astype(np.float32)
            exact = t == 0
            want = oracle.e4m3_encode(xd / s)
            got = oracle.e4m3_encode(q)
            bad = np.nonzero(exact & (got != want))[0]
            assert bad.size == 0, (float(s), xd[bad[:5]], got[bad[:5]], want[bad[:5]])
            if any(s == r for r in _amax_scales()[:len(EXACT_AMAX)]):
                left_round += int((~exact).sum())
            else:  # quotients near a boundary but not on it: rare
                assert (~exact).sum() <= 256, float(s)  # 0.4% of the inputs
            if _odd_significand(s) >= 256:  # the kernel skips the step: it never fires
                assert not exact.any(), float(s)
    assert left_round == 0


def _odd_significand(s):
    """The significand of a float32 with its trailing zero bits dropped (the
    kernel's host test: the remainder step runs only when this is < 256)."""
    m, _ = np.frexp(np.float64(s))
    sig = int(m * 2 ** 24)
    while sig and sig % 2 == 0:
        sig //= 2
    return sig


def test_exact_remainder_step_is_needed():
    """On an exact amax / 448 scale the bracket alone leaves about one in 16
    values of e4m3's normal range undecided (so most 16-value groups would
    go to the division): the exact step is what keeps them off it."""
    x = _all_bf16_as_f32()
    for a in EXACT_AMAX:
        s = np.float32(a / 448.0)
        rcp = np.float32(1.0) / s
        with np.errstate(all="ignore"):
            sel = np.isfinite(x) & (np.abs(x / s) >= 2.0 ** -6) & (np.abs(x / s) <= 448)
        xs = x[sel]
        differ = oracle.e4m3_encode(xs * (rcp * SHRINK)) != oracle.e4m3_encode(xs * (rcp * GROW))
        assert differ.mean() > 0.05, a


def test_power_of_two_scale_is_a_product():
    """For a power-of-two scale (1 / scale normal) the kernel stores the code
    of RN(x * (1 / scale)) with no bracket: the same real number as x / scale,
    so the same code for every bf16 input."""
    x = _all_bf16_as_f32()
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        for k in (-120, -60, -9, -2, 0, 1, 3, 8, 60, 120, 126):
            s = np.float32(2.0 ** k)
            got = oracle.e4m3_encode(x * (np.float32(1.0) / s))
            want = oracle.e4m3_encode(x / s)
            assert np.array_equal(got, want), k

