"""GPU parity of kvq_wq_gemm (weight-only INT4 / e4m3 decode matrix product)
against the oracle.

Tolerance, derived from the arithmetic: the kernel's products are exact
(INT4 and e4m3 values are exact in bf16 / f16, and so is x in the range
used), and a sum of K terms in fp32 -- tensor-core accumulation, split-K
partial sums added with atomics -- is within K * u * sum|w x| of the exact
sum (u = 2^-24, the standard worst-case bound for recursive summation);
the test allows twice that, K * 2^-23 * sum_k |w[n][k] x[m][k]|, elementwise.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins as pins
from fp8_paged_kv_attn_gb300 import inputs, kvq
from gpu_harness import dev

pytestmark = pytest.mark.gpu

E4M3 = torch.float8_e4m3fn


def _dequant(wdtype, w, s):
    if wdtype == oracle.W_INT4:
        return pins.numpy_int4_weights(w, s, 128)
    return torch.from_numpy(w).view(E4M3).to(torch.float64).numpy() * s.astype(np.float64)[:, None]


def run_gpu(wdtype, w, s, x):
    M, N = x.shape[0], w.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    sd = dev(s.view(np.int16)) if wdtype == oracle.W_INT4 else dev(s)
    xd = dev(x.view(np.int16)).view(torch.bfloat16)
    kvq.kvq_wq_gemm(wdtype, dev(w), sd, xd, y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def check(wdtype, w, s, x, rows=None, what=""):
    got = run_gpu(wdtype, w, s, x)
    if rows is not None:
        w, s, got = w[rows], s[rows], got[:, rows]
    ref = oracle.wq_gemm(wdtype, w, s, x)
    K = x.shape[1]
    absum = np.abs(pins._bf16_to_f64(x)) @ np.abs(_dequant(wdtype, w, s)).T
    bound = K * 2.0 ** -23 * absum + 1e-30
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= bound), (what, float((err / bound).max()))
    return float((err / np.maximum(absum, 1e-30)).max())


SHAPES = [(1, 16, 128), (3, 100, 384), (8, 64, 1024), (13, 200, 640), (33, 64, 256),
          (64, 130, 1280), (17, 1, 128), (64, 257, 5120), (32, 200, 1024), (26, 300, 5120),
          (48, 129, 768)]


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_wq_gemm_shapes(kvq, wdtype, M, N, K):
    rng = np.random.default_rng(M * 1000 + N + K + wdtype)
    w, s, x = pins.random_wq_case(rng, wdtype, M, N, K)
    check(wdtype, w, s, x, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
def test_wq_gemm_every_code(kvq, wdtype):
    """Every INT4 byte value / every finite e4m3 code (subnormals, +-448, -0)
    in every lane position of a 128-wide group, against dense random x."""
    rng = np.random.default_rng(40 + wdtype)
    M, N, K = 9, 64, 512
    x = inputs.normal_bf16(rng, (M, K))
    if wdtype == 0:
        base = np.arange(256, dtype=np.uint8)
        w = np.resize(base, (N, K // 2)).astype(np.uint8)
        s = np.full((N, K // 128), 0x3C00, dtype=np.uint16)  # 2^-7
    else:
        codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
        w = np.resize(codes, (N, K)).astype(np.uint8)
        s = np.full(N, 0.01, dtype=np.float32)
    w = np.ascontiguousarray(w)
    check(wdtype, w, s, x, what="codes")


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(1, 1792, 5120), (64, 5120, 1536), (8, 3072, 5120),
                                   (64, 28672, 5120)])
def test_wq_gemm_full_size_sampled(kvq, wdtype, M, N, K):
    """GLM-like shapes at 8-way tensor parallelism (and one large projection):
    the whole product on the GPU, 96 sampled output channels against the
    oracle."""
    rng = np.random.default_rng(N + K + M + wdtype)
    w, s, x = pins.random_wq_case(rng, wdtype, M, N, K)
    rows = np.sort(rng.choice(N, min(N, 96), replace=False))
    check(wdtype, w, s, x, rows=rows, what=f"{M}x{N}x{K}")


def test_wq_gemm_arguments(kvq):
    L = kvq.load()
    y = torch.zeros(4, dtype=torch.float32, device="cuda")
    w = torch.zeros(64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(8, dtype=torch.float32, device="cuda")
    x = torch.zeros(128 * 65, dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 65, 1, 128, None) == 4   # M > 64
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 1, 1, 200, None) == 4   # K % 128
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 1, 1, 100, None) == 1   # K < 128
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 0, 1, 128, None) == 1   # M < 1
    assert L.kvq_wq_gemm(2, p(w), p(s), p(x), p(y), 1, 1, 128, None) == 1   # dtype
    assert L.kvq_wq_gemm(0, p(w) + 8, p(s), p(x), p(y), 1, 1, 128, None) == 1  # alignment
    assert L.kvq_wq_gemm(0, None, p(s), p(x), p(y), 1, 1, 128, None) == 1
