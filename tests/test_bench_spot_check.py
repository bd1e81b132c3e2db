"""The benchmark's oracle check of the last timed step, on the CPU.

bench.oracle_spot_check rebuilds the sampled requests' pools from their
prompts and the packed step rows, in the order the run appended them, and
compares the last step's output rows and abort mask with the oracle.  Here
the "device" result is made by replaying the same appends through the oracle
for every request, so the check must pass; a single perturbed element, a
wrong mask bit or a skipped append must make it fail.
"""
import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_attn_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(w, args, gen, skip_append_of=None):
    """The pools and last-step result a device run would leave, via the oracle."""
    sources = w.kv_sources()
    ks, vs = w.scales(sources)
    hk = np.zeros(w.pool_shape(), dtype=np.uint8)
    hv = np.zeros_like(hk)
    for b, (k, v) in enumerate(sources):
        req, pos = w.context_tokens(b)
        assert oracle.quant_append(oracle.KV_E4M3, hk, hv, ks, vs, k, v, req, pos,
                                   w.block_table) == 0
    packer = bench.StepInputs(torch, w.B, w.Hq, w.Hkv, w.D)
    rows = []
    for i, gi in enumerate(gen):
        q, k_new, v_new, req, pos = w.step_inputs(gi)
        rows.append({"q": q, "k": k_new, "v": v_new, "pos": pos, "lens": w.seq_lens_after(gi)})
        if i != skip_append_of:
            assert oracle.quant_append(oracle.KV_E4M3, hk, hv, ks, vs, k_new, v_new, req, pos,
                                       w.block_table) == 0
    h_rows = packer.pack(rows)
    lens = rows[-1]["lens"]
    mask = oracle.check_tags(w.block_table, lens, w.P, w.page_tags, w.expected_tags)
    out, e = oracle.decode_attn(oracle.KV_E4M3, hk, hv, ks, vs, rows[-1]["q"], w.block_table,
                                lens, abort_mask=mask, sm_scale=w.sm_scale)
    assert e == 0
    kept = {b: sources[b] for b in bench.spot_check_requests(w.B)}
    return ks, vs, kept, packer, h_rows, out, mask


@pytest.fixture(scope="module")
def case():
    w = inputs.uniform("spot", 3, B=5, ctx=40, Hq=8, Hkv=2, D=64, P=16, decode_steps=12)
    args = SimpleNamespace(warmup=2, steps=4, check="on")
    gen = [3 + i for i in range(args.warmup + args.steps)]
    return w, args, gen


def test_spot_check_passes_on_the_same_appends(case):
    w, args, gen = case
    ks, vs, kept, packer, h_rows, out, mask = _run(w, args, gen)
    res = bench.oracle_spot_check(args, w, ks, vs, 1, kept, packer, h_rows, gen, None, out, mask)
    assert res["ok"] and res["requests"] == [0, 2, 4] and res["rows"] == 3 * w.Hq
    assert res["max_abs_err"] == 0.0 and res["abort_mask_bit_exact"]


def test_spot_check_fails_on_a_wrong_value_or_mask(case):
    w, args, gen = case
    ks, vs, kept, packer, h_rows, out, mask = _run(w, args, gen)
    bad = out.copy()
    bad[2, 3, 5] += 0.01 + 0.01 * abs(bad[2, 3, 5])
    with pytest.raises(RuntimeError):
        bench.oracle_spot_check(args, w, ks, vs, 1, kept, packer, h_rows, gen, None, bad, mask)
    m = mask.copy()
    m[1] ^= 1
    with pytest.raises(RuntimeError):
        bench.oracle_spot_check(args, w, ks, vs, 1, kept, packer, h_rows, gen, None, out, m)


def test_spot_check_fails_when_a_step_was_not_appended(case):
    w, args, gen = case
    # the run "skipped" the append of the last step: the rows differ
    ks, vs, kept, packer, h_rows, out, mask = _run(w, args, gen, skip_append_of=len(gen) - 1)
    with pytest.raises(RuntimeError):
        bench.oracle_spot_check(args, w, ks, vs, 1, kept, packer, h_rows, gen, None, out, mask)
