"""The index split the weight-only product uses when it stages a CTA's INT4
group scales, checked on the CPU (no GPU, no kernel code).

Item e of a CTA's (row pair, group) list is split as p = e / ng, g = e - p ng
without an integer division: p = trunc((float(e) + 1/2) * RN(1/ng)) in fp32.
The claim: for every group count ng up to 2048 and every item e below
64 ng (64 row pairs is the most a CTA stages), this equals floor(e / ng).
numpy's float32 arithmetic (IEEE, round to nearest even) plays the kernel's.
"""
import numpy as np


def test_reciprocal_split_is_exact():
    for ng in range(1, 2049):
        inv = np.float32(1.0) / np.float32(ng)
        e = np.arange(64 * ng, dtype=np.int64)
        p = ((e.astype(np.float32) + np.float32(0.5)) * inv).astype(np.int64)
        assert np.array_equal(p, e // ng), ng


def test_plain_product_without_the_half_is_not_exact():
    """The +1/2 matters: trunc(e * RN(1/ng)) alone is one short at some e."""
    bad = 0
    for ng in (3, 5, 7, 11, 13, 40, 41, 97):
        inv = np.float32(1.0) / np.float32(ng)
        e = np.arange(64 * ng, dtype=np.int64)
        p = (e.astype(np.float32) * inv).astype(np.int64)
        bad += int(np.sum(p != e // ng))
    assert bad > 0
