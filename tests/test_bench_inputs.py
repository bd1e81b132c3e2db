"""The benchmark's packed step inputs on the CPU: every field lands where its
view reads it, byte for byte, and every field starts on a 256-byte boundary
(the library wants 16-byte aligned q, k_new and v_new)."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _step(rng, B, Hq, Hkv, D):
    return {"q": rng.integers(0, 1 << 16, (B, Hq, D), dtype=np.uint16),
            "k": rng.integers(0, 1 << 16, (B, Hkv, D), dtype=np.uint16),
            "v": rng.integers(0, 1 << 16, (B, Hkv, D), dtype=np.uint16),
            "pos": rng.integers(0, 1 << 20, B, dtype=np.int32),
            "lens": rng.integers(1, 1 << 20, B, dtype=np.int32)}


def test_pack_round_trip_and_alignment():
    rng = np.random.default_rng(5)
    for B, Hq, Hkv, D in ((1, 4, 1, 64), (3, 32, 8, 128), (64, 64, 8, 128)):
        p = bench.StepInputs(torch, B, Hq, Hkv, D)
        steps = [_step(rng, B, Hq, Hkv, D) for _ in range(3)]
        rows = p.pack(steps)
        assert rows.shape == (3, p.nbytes) and p.nbytes % 256 == 0
        for _, off, n, _, _ in p.fields:
            assert off % 256 == 0
        for i, st in enumerate(steps):
            v = p.views(rows[i])
            for name in ("q", "k", "v"):
                got = v[name].view(torch.int16).numpy().view(np.uint16)
                assert v[name].dtype == torch.bfloat16
                np.testing.assert_array_equal(got, st[name])
            for name in ("pos", "lens"):
                assert v[name].dtype == torch.int32
                np.testing.assert_array_equal(v[name].numpy(), st[name])


def test_pack_rejects_wrong_sizes():
    rng = np.random.default_rng(6)
    p = bench.StepInputs(torch, 2, 4, 1, 64)
    st = _step(rng, 2, 4, 1, 64)
    st["pos"] = st["pos"][:1]
    try:
        p.pack([st])
    except AssertionError:
        return
    raise AssertionError("a short field was packed")
