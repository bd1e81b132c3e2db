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
