"""kvq_decode_attn_static: decode attention for callers that cannot allocate.

Serving runtimes that reserve all device memory up front, plugin hosts that
forbid allocation in their execute callback and latency-bound loops that
cannot afford cudaMalloc have no workspace to pass to kvq_decode_attn.  The
static entry point takes its scratch from a device array owned by the
library.  This test calls it through the C ABI twice in a row (different
lengths, so the second call runs on the first call's leftover scratch).  The
same kernels run on the same inputs as kvq_decode_attn, only with another
workspace address, so each output must equal kvq_decode_attn's bit for bit;
the first call is also checked against the oracle within the attention
tolerance.  It covers the tensor-core kernel with an e4m3 and a bf16 cache
and the head_dim-64 CUDA-core kernel, whose partials are laid out
differently in the scratch.  It lives in its own file, collected last, and
passes both alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

from fp8_paged_kv_attn_gb300 import inputs
from gpu_harness import Run, assert_close, dev, dev_bf16

pytestmark = pytest.mark.gpu

CASES = [("e4m3", 128), ("bf16", 128), ("e4m3", 64)]


@pytest.mark.parametrize("dtype,D", CASES, ids=[f"{d}_d{D}" for d, D in CASES])
def test_static_scratch_matches_workspace_entry_point(kvq, dtype, D):
    w = inputs.ragged(seed=77, B=6, total=20000, lo=1, hi=9000, Hq=32, Hkv=8, D=D, P=16)
    r = Run(w, kv_dtype=kvq.KV_E4M3 if dtype == "e4m3" else kvq.KV_BF16)
    r.fill_context()
    q_bits, *_ = w.step_inputs(0)
    q = dev_bf16(q_bits)
    calls = [w.ctx_lens, np.maximum(w.ctx_lens // 3, 1).astype(np.int32)]
    for call, lens in enumerate(calls):
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
        g = got.cpu().numpy()
        assert np.array_equal(g.view(np.uint32), ref.cpu().numpy().view(np.uint32)), \
            f"call {call}: static entry point differs from kvq_decode_attn"
        if call == 0:
            rows = [(b, h) for b in range(w.B) for h in (0, 7, 31)]
            oref, oerr = r.oracle_rows(q_bits, lens, rows)
            assert oerr == 0
            for b, h in rows:
                assert_close(g[b, h], oref[b, h], f"static call 0 row ({b},{h}) vs oracle")


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
