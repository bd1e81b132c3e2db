"""The decode step as the benchmark times it -- kvq_append -> kvq_check_tags ->
kvq_decode_attn captured once into a CUDA graph and replayed over staged
inputs -- against the oracle.

Captured, the step's programmatic dependent launches (append, check, split,
combine; plus the plan kernel for very large batches) become programmatic
edges of the graph.  The split kernel reads the sequence lengths and the
abort mask right after its grid-dependency wait, which is correct only if the
graph orders it after the tag check exactly as the stream does; eager calls
(every other test) do not show that.  Here the
benchmark's own DecodeStep captures the step once, then replays it for four
consecutive decode steps, each staged with one device copy into the graph's
static buffers.  Before one replay a page of one request is re-tagged on the
device (the page was handed to another owner), so that replay's check must
abort that request and its attention rows must be zero; the tag is put back
for the next replay.  After every replay:
  * the abort mask equals the oracle's linear scan bit for bit;
  * the K/V pools equal the oracle's on every page of the sampled requests
    (the step's appended token included), bit for bit;
  * sampled output rows are within 1e-3 + 1e-3*|ref| of the fp64 oracle;
  * the graph's output equals an eager kvq_decode_attn call on the same
    inputs bit for bit (same kernels, same schedule);
  * no device error bit is set.
Shapes: the benchmark's 64-request concurrency-sweep point (G = 4, page 16)
and a ragged batch with G = 8 and page 64 (the paired-stage path).
"""
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from fp8_paged_kv_attn_gb300 import inputs
from gpu_harness import Run, assert_close, dev_u32

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.gpu

STEPS = 4
STALE_STEP = 2


def _replay_and_compare(kvq, w, host_requests, heads, victim):
    assert victim in host_requests
    r = Run(w, host_requests=host_requests)
    r.fill_context()
    B, Hq, Hkv, D = w.B, w.Hq, w.Hkv, w.D
    packer = bench.StepInputs(torch, B, Hq, Hkv, D)
    step_rows = []
    for s in range(STEPS):
        q, k_new, v_new, req, pos = w.step_inputs(s)
        assert np.array_equal(req, np.arange(B, dtype=np.int32))
        step_rows.append({"q": q, "k": k_new, "v": v_new, "pos": pos,
                          "lens": w.seq_lens_after(s)})
    d_rows = packer.pack(step_rows).cuda()
    host_tags = w.page_tags.copy()
    tags = dev_u32(host_tags)
    exp_tags = dev_u32(w.expected_tags)
    mask = torch.full((B,), 0xEE, dtype=torch.uint8, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    ws = kvq.workspace(B, Hq, Hkv, D)
    step = bench.DecodeStep(torch, kvq, r.cache, r.bt, w.P, float(w.sm_scale), packer, out, ws,
                            err=r.err, check=True, tags=tags, exp_tags=exp_tags, mask=mask,
                            graph=True)
    # one eager run of step 0 (library set-up), then the capture; every step
    # below, step 0 included, runs as a replay of the captured graph
    step.capture(d_rows[0])
    torch.cuda.synchronize()

    stale_page = int(w.block_table[victim, 0])
    eager_out = torch.empty_like(out)
    eager_ws = kvq.workspace(B, Hq, Hkv, D)
    rows = [(b, h) for b in host_requests for h in heads]
    for s in range(STEPS):
        if s == STALE_STEP:  # the page was handed to another owner: its tag moves on
            host_tags[stale_page] = np.uint32((int(host_tags[stale_page]) + 1) & 0xFFFFFFFF)
        elif s == STALE_STEP + 1:
            host_tags[stale_page] = w.page_tags[stale_page]
        tags.copy_(dev_u32(host_tags))
        out.fill_(float("nan"))
        step.run(d_rows[s])
        torch.cuda.synchronize()
        lens = w.seq_lens_after(s)
        q_bits = r.oracle_append_step(s)

        assert r.err_word() == 0, f"step {s}: device error bits {r.err_word():#x}"
        ref_mask = oracle.check_tags(w.block_table, lens, w.P, host_tags, w.expected_tags)
        got_mask = mask.cpu().numpy()
        assert np.array_equal(got_mask, ref_mask), f"step {s}: abort mask differs"
        assert bool(ref_mask[victim]) == (s == STALE_STEP)
        r.assert_pools_equal(lens)
        got = out.cpu().numpy()
        ref, oerr = r.oracle_rows(q_bits, lens, rows, abort=ref_mask)
        assert oerr == 0
        for b, h in rows:
            assert_close(got[b, h], ref[b, h], f"graph step {s} row ({b},{h})")
        if s == STALE_STEP:
            assert not got[victim].any(), "the aborted request's rows are not zero"
        # the same attention call made eagerly on the staged inputs
        v = step.static
        kvq.kvq_decode_attn(r.cache, v["q"], r.bt, v["lens"], eager_out, eager_ws,
                            abort_mask=mask, sm_scale=float(w.sm_scale), err_word=r.err)
        torch.cuda.synchronize()
        assert np.array_equal(eager_out.cpu().numpy().view(np.uint32), got.view(np.uint32)), \
            f"step {s}: graph output differs from the eager call"


def test_graph_step_sweep_b64(kvq):
    """The benchmark's headline workload: 64 requests x 8192-token prompts,
    GQA 32/8, page 16, e4m3 pool of 64 requests' bytes."""
    w = inputs.sweep(64)
    _replay_and_compare(kvq, w, host_requests=[0, 17, 40, 63], heads=(0, 5, 13, 31), victim=17)


def test_graph_step_ragged_g8_p64(kvq):
    """Ragged lengths, 64 query / 8 kv heads (G = 8), page 64, fragmented pool."""
    w = inputs.ragged(seed=31, B=16, total=100_000, lo=512, hi=40_000)
    w.ctx_lens = (w.ctx_lens - STEPS).astype(np.int32)  # room for the steps' tokens
    order = [int(b) for b in np.argsort(w.ctx_lens)]
    picks = sorted({order[0], order[len(order) // 2], order[-1]})
    _replay_and_compare(kvq, w, host_requests=picks, heads=(0, 9, 63), victim=picks[-1])
