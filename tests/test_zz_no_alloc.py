"""kvq_decode_attn_static: decode attention for callers that cannot allocate.

Serving runtimes that reserve all device memory up front, plugin hosts that
forbid allocation in their execute callback and latency-bound loops that
cannot afford cudaMalloc have no workspace to pass to kvq_decode_attn.  The
static entry point takes its scratch from a device array owned by the
library.  This test calls it through the C ABI twice in a row (different
lengths, so the second call runs on the first call's leftover scratch) and
checks each output against kvq_decode_attn's on the same inputs, within the
attention tolerance.  It lives in its own file, collected last, and passes
both alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

from fp8_paged_kv_attn_gb300 import inputs
from gpu_harness import Run, assert_close, dev, dev_bf16

pytestmark = pytest.mark.gpu


def test_static_scratch_matches_workspace_entry_point(kvq):
    w = inputs.ragged(seed=77, B=6, total=20000, lo=1, hi=9000, Hq=32, Hkv=8, D=128, P=16)
    r = Run(w)
    r.fill_context()
    q_bits, *_ = w.step_inputs(0)
    q = dev_bf16(q_bits)
    for call, lens in enumerate([w.ctx_lens, np.maximum(w.ctx_lens // 3, 1).astype(np.int32)]):
        d_lens = dev(lens)
        ref = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
        ws = kvq.workspace(w.B, w.Hq, w.Hkv, w.D)
        kvq.kvq_decode_attn(r.cache, q, r.bt, d_lens, ref, ws, sm_scale=float(w.sm_scale))
        got = torch.full_like(ref, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.kvq_decode_attn_static(r.cache, q, r.bt, d_lens, got, sm_scale=float(w.sm_scale),
                                   err_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error bits"
        assert_close(got.cpu().numpy(), ref.cpu().numpy(), f"static call {call}")


def test_static_scratch_rejects_oversized_batches(kvq):
    w = inputs.tiny()
    r = Run(w)
    too_many = 1 << 16  # the workspace for 65,536 requests exceeds the static array
    q = torch.zeros((too_many, w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((too_many, w.Hq, w.D), dtype=torch.float32, device="cuda")
    bt = torch.zeros((too_many, w.MP), dtype=torch.int32, device="cuda")
    lens = torch.zeros(too_many, dtype=torch.int32, device="cuda")
    assert kvq.kvq_decode_attn_workspace_size(too_many, w.Hq, w.Hkv, w.D) > kvq.STATIC_SCRATCH_BYTES
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attn_static(r.cache, q, bt, lens, out)
    assert e.value.status == 2
