"""Run a synthetic workload through the CUDA library and through the oracle
on the same seeded inputs.  Used by the GPU parity tests and the smoke check.

Nothing here computes the method: the CUDA side goes through the C ABI
binding, the expected side through ``oracle``.
"""
import numpy as np
import torch

import oracle
from fp8_paged_kv_attn_gb300 import inputs
from fp8_paged_kv_attn_gb300 import kvq

SENTINEL = 0xA5
TOL_ABS = 1e-3
TOL_REL = 1e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def dev_u32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).cuda()


def assert_close(got: np.ndarray, ref: np.ndarray, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = TOL_ABS + TOL_REL * np.abs(ref)
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements off, worst at {i}: "
                             f"got {got[i]}, ref {ref[i]}, |err| {err[i]:.3g}")


class Run:
    """A workload's cache on the GPU and (optionally) on the host for the oracle."""

    def __init__(self, w: inputs.Workload, kv_dtype=kvq.KV_E4M3, host_requests=None,
                 sources=None):
        self.w = w
        self.kv_dtype = kv_dtype
        fp8 = kv_dtype == kvq.KV_E4M3
        self.np_dtype = np.uint8 if fp8 else np.uint16
        self.sources = w.kv_sources() if sources is None else sources
        self.k_scale, self.v_scale = w.scales(self.sources)
        shape = w.pool_shape()
        tdt = torch.uint8 if fp8 else torch.int16
        # the same sentinel byte in every byte of the pool
        fill = SENTINEL if fp8 else int(np.array([SENTINEL | (SENTINEL << 8)],
                                                 dtype=np.uint16).view(np.int16)[0])
        kp = torch.full(shape, fill, dtype=tdt, device="cuda")
        vp = torch.full(shape, fill, dtype=tdt, device="cuda")
        if not fp8:
            kp, vp = kp.view(torch.bfloat16), vp.view(torch.bfloat16)
        self.cache = kvq.KVCache(kp, vp, float(self.k_scale), float(self.v_scale))
        self.bt = dev(w.block_table)
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        # the host pools hold only the requests the oracle will look at
        self.host_requests = list(range(w.B)) if host_requests is None else list(host_requests)
        self.hk = np.full(shape, SENTINEL, dtype=np.uint8) if fp8 else \
            np.full(shape, SENTINEL | (SENTINEL << 8), dtype=np.uint16)
        self.hv = self.hk.copy()
        self.oracle_dtype = oracle.KV_E4M3 if fp8 else oracle.KV_BF16

    # ---- context fill (bulk append) ----------------------------------------
    def fill_context(self):
        for b, (k, v) in enumerate(self.sources):
            if k.shape[0] == 0:
                continue
            req, pos = self.w.context_tokens(b)
            kvq.kvq_append(self.cache, dev_bf16(k), dev_bf16(v), dev(req), dev(pos), self.bt,
                           err_word=self.err)
            if b in self.host_requests:
                e = oracle.quant_append(self.oracle_dtype, self.hk, self.hv, self.k_scale,
                                        self.v_scale, k, v, req, pos, self.w.block_table)
                assert e == 0
        torch.cuda.synchronize()

    def fill_context_one_call(self):
        """The prompt handoff: every request's whole prompt quantised into the
        pages by ONE kvq_append call (N = sum of the prompt lengths)."""
        ks, vs, reqs, poss = [], [], [], []
        for b, (k, v) in enumerate(self.sources):
            if k.shape[0] == 0:
                continue
            req, pos = self.w.context_tokens(b)
            ks.append(k)
            vs.append(v)
            reqs.append(req)
            poss.append(pos)
        k, v = np.concatenate(ks), np.concatenate(vs)
        req, pos = np.concatenate(reqs), np.concatenate(poss)
        kvq.kvq_append(self.cache, dev_bf16(k), dev_bf16(v), dev(req), dev(pos), self.bt,
                       err_word=self.err)
        sel = np.isin(req, np.array(self.host_requests, dtype=np.int32))
        e = oracle.quant_append(self.oracle_dtype, self.hk, self.hv, self.k_scale, self.v_scale,
                                np.ascontiguousarray(k[sel]), np.ascontiguousarray(v[sel]),
                                np.ascontiguousarray(req[sel]), np.ascontiguousarray(pos[sel]),
                                self.w.block_table)
        assert e == 0
        torch.cuda.synchronize()
        return int(req.shape[0])

    def append_step(self, step: int):
        q, k_new, v_new, req, pos = self.w.step_inputs(step)
        kvq.kvq_append(self.cache, dev_bf16(k_new), dev_bf16(v_new), dev(req), dev(pos), self.bt,
                       err_word=self.err)
        self.oracle_append_step(step)
        return q

    def oracle_append_step(self, step: int):
        """The oracle's side of decode step `step`'s append (host requests
        only); the GPU side is whatever ran the step (an eager call or a
        replayed graph)."""
        q, k_new, v_new, req, pos = self.w.step_inputs(step)
        sel = np.array(self.host_requests, dtype=np.int64)
        e = oracle.quant_append(self.oracle_dtype, self.hk, self.hv, self.k_scale, self.v_scale,
                                k_new[sel], v_new[sel], req[sel], pos[sel], self.w.block_table)
        assert e == 0
        return q

    # ---- comparisons ---------------------------------------------------------
    def pages_of(self, requests, upto_lens):
        pages = []
        for b in requests:
            n = -(-int(upto_lens[b]) // self.w.P)
            pages.extend(int(p) for p in self.w.block_table[b, :n])
        return np.array(sorted(set(pages)), dtype=np.int64)

    def pool_bytes(self, pages=None):
        kp = self.cache.k_pool.view(torch.uint8 if self.np_dtype == np.uint8 else torch.int16)
        vp = self.cache.v_pool.view(torch.uint8 if self.np_dtype == np.uint8 else torch.int16)
        if pages is not None:
            idx = torch.from_numpy(pages).cuda()
            kp, vp = kp[idx], vp[idx]
        k = kp.cpu().numpy().view(self.np_dtype)
        v = vp.cpu().numpy().view(self.np_dtype)
        return k, v

    def assert_pools_equal(self, upto_lens, whole=False):
        """Bit-exact append parity: the GPU pools equal the oracle's, on every
        page of the host requests (or the whole pool)."""
        pages = None if whole else self.pages_of(self.host_requests, upto_lens)
        gk, gv = self.pool_bytes(pages)
        hk = self.hk if pages is None else self.hk[pages]
        hv = self.hv if pages is None else self.hv[pages]
        assert np.array_equal(gk, hk), "K pool bytes differ from the oracle"
        assert np.array_equal(gv, hv), "V pool bytes differ from the oracle"

    def attend(self, q_bits, lens, abort=None, sm_scale=None, ws=None, bt=None):
        """kvq_decode_attn on this cache; `ws` is a workspace to reuse (a fresh
        zeroed one by default), `bt` a block table to use instead of the
        workload's (device tensor)."""
        w = self.w
        qd = dev_bf16(q_bits)
        out = torch.full((w.B, w.Hq, w.D), float("nan"), dtype=torch.float32, device="cuda")
        if ws is None:
            ws = kvq.workspace(w.B, w.Hq, w.Hkv, w.D)
        ab = None if abort is None else dev(abort.astype(np.uint8))
        kvq.kvq_decode_attn(self.cache, qd, self.bt if bt is None else bt, dev(lens), out, ws,
                            abort_mask=ab,
                            sm_scale=float(w.sm_scale if sm_scale is None else sm_scale),
                            err_word=self.err)
        return out.cpu().numpy()

    def oracle_rows(self, q_bits, lens, rows, abort=None, nthreads=16):
        w = self.w
        ref, err = oracle.decode_attn(self.oracle_dtype, self.hk, self.hv, self.k_scale,
                                      self.v_scale, q_bits, w.block_table, lens,
                                      abort_mask=abort, sm_scale=w.sm_scale, rows=rows,
                                      nthreads=nthreads)
        return ref, err

    def err_word(self) -> int:
        return int(self.err.item()) & 0xFFFFFFFF
