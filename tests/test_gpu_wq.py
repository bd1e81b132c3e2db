"""GPU parity of kvq_wq_gemm (weight-only INT4 / e4m3 decode matrix product)
against the oracle.

Tolerance, derived from the kernel's arithmetic.  The oracle is exact up to
one final fp32 rounding.  The kernel:
  * scales each token's x, per 128-wide k group, by a power of two 2^e (the
    group's largest finite |x| into [2^14, 2^15)) and rounds it to f16:
    exact for values down to 2^-32 of that largest, otherwise off by at most
    2^-25 * 2^-e (the test computes e per token and group as the kernel does);
  * multiplies exactly (INT4, e4m3 and scaled x are exact in f16) and sums a
    group with fp32 tensor-core accumulation, 8 mma.sync steps, each a
    rounding of at most 2^-22 of the running sum's magnitude (allowing for an
    accumulator that truncates instead of rounding to nearest); then one
    fused multiply-add per group into the output (2^-e is exact, and so is
    the INT4 group scale's product with it), the split-K atomics and the e4m3
    channel scale, each an fp32 rounding (2^-24).  Groups per CTA and split-K
    parts are each at most G = K / 128.
So elementwise, with A = sum_k |W[n][k] x[m][k]|,
  |err| <= (8 2^-22 + (2 G + 3) 2^-24) A + sum_g 2^-25 2^-e(m,g) sum_{k in g} |W[n][k]|
plus (2 G + 1) 2^-126: the split-K partial sums are added with fp32 atomic
adds, which flush subnormal operands and results, so each of the (at most
G) adds can lose a partial and a running sum below fp32's normal range,
2^-126 (seen on rows made only of bf16 subnormals).
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


def wq_bound(wdtype, w, s, x):
    wd = _dequant(wdtype, w, s)
    xf = pins._bf16_to_f64(x)
    M, K = xf.shape
    G = K // 128
    absum = np.abs(xf) @ np.abs(wd).T
    rel = 8 * 2.0 ** -22 + (2 * G + 3) * 2.0 ** -24
    # per token and group: 2^-25 2^-e, e from the group's largest finite |x|
    ax = np.where(np.isfinite(xf), np.abs(xf), 0.0).reshape(M, G, 128).max(axis=2)
    e = np.where(ax > 0, 14 - np.floor(np.log2(np.where(ax > 0, ax, 1.0))), 0.0)
    wg = np.abs(wd).reshape(wd.shape[0], G, 128).sum(axis=2)  # [N, G]
    xround = (2.0 ** (-25 - e)) @ wg.T
    return rel * absum + xround + (2 * G + 1) * 2.0 ** -126, absum


def check(wdtype, w, s, x, rows=None, what=""):
    got = run_gpu(wdtype, w, s, x)
    if rows is not None:
        w, s, got = w[rows], s[rows], got[:, rows]
    ref = oracle.wq_gemm(wdtype, w, s, x)
    bound, absum = wq_bound(wdtype, w, s, x)
    err = np.abs(got.astype(np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= bound), (what, float((err / bound).max()))
    return float((err / np.maximum(absum, 1e-300)).max())


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
@pytest.mark.parametrize("M", [1, 2, 9], ids=["ring1", "ring", "registers"])
def test_wq_gemm_every_code(kvq, wdtype, M):
    """Every INT4 byte value / every finite e4m3 code (subnormals, +-448, -0)
    in every lane position of a 128-wide group, against dense random x (1
    and 2 tokens: the TMA-ring kernel; 9: the register-ring kernel)."""
    rng = np.random.default_rng(40 + wdtype)
    N, K = 64, 512
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


# Up to eight tokens run the TMA-ring kernel where the shape suits it (one
# token its own specialisation): k split over clusters of 1 to 8 CTAs (3, 4,
# 5, 6 and 7 included), rows past N zero-filled by the copy, odd group counts
# per CTA, one group in all; 3 to 8 tokens on the projections of a layer.
RING_SHAPES = [(1, 200, 1536), (2, 1000, 640), (1, 130, 3584), (2, 5000, 1536), (1, 64, 128),
               (2, 65, 256), (1, 8000, 768), (2, 777, 2560), (3, 300, 2560), (4, 1792, 5120),
               (5, 1000, 1536), (7, 130, 640), (8, 5120, 1536), (8, 777, 5120)]


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
@pytest.mark.parametrize("M,N,K", RING_SHAPES)
def test_wq_ring_shapes(kvq, wdtype, M, N, K):
    rng = np.random.default_rng(7 * M + N + K + wdtype)
    w, s, x = pins.random_wq_case(rng, wdtype, M, N, K)
    rows = None if N <= 1000 else np.sort(rng.choice(N, 128, replace=False))
    check(wdtype, w, s, x, rows=rows, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
@pytest.mark.parametrize("M", [2, 8])
def test_wq_ring_deterministic(kvq, wdtype, M):
    """The split-K sums of the ring kernel are added in cluster-rank order, not
    by atomics: two calls give the same bits, and no wait gives up."""
    rng = np.random.default_rng(90 + wdtype + M)
    N, K = (1792, 5120) if M == 2 else (5120, 1536)
    w, s, x = pins.random_wq_case(rng, wdtype, M, N, K)
    sd = dev(s.view(np.int16)) if wdtype == oracle.W_INT4 else dev(s)
    xd = dev(x.view(np.int16)).view(torch.bfloat16)
    wd = dev(w)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = []
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        kvq.kvq_wq_gemm(wdtype, wd, sd, xd, y, err_word=err)
        ys.append(y)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(ys[0].view(torch.int32), ys[1].view(torch.int32))


def test_wq_gemm_arguments(kvq):
    L = kvq.load()
    y = torch.zeros(4, dtype=torch.float32, device="cuda")
    w = torch.zeros(64, dtype=torch.uint8, device="cuda")
    s = torch.zeros(8, dtype=torch.float32, device="cuda")
    x = torch.zeros(128 * 65, dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()  # noqa: E731
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 65, 1, 128, None, None) == 4   # M > 64
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 1, 1, 200, None, None) == 4   # K % 128
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 1, 1, 100, None, None) == 1   # K < 128
    assert L.kvq_wq_gemm(0, p(w), p(s), p(x), p(y), 0, 1, 128, None, None) == 1   # M < 1
    assert L.kvq_wq_gemm(2, p(w), p(s), p(x), p(y), 1, 1, 128, None, None) == 1   # dtype
    assert L.kvq_wq_gemm(0, p(w) + 8, p(s), p(x), p(y), 1, 1, 128, None, None) == 1  # alignment
    assert L.kvq_wq_gemm(0, None, p(s), p(x), p(y), 1, 1, 128, None, None) == 1


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
@pytest.mark.parametrize("M,N,K", [(8, 200, 1280), (13, 130, 5120), (1, 64, 384), (64, 129, 768),
                                   (24, 300, 2560)])
def test_wq_gemm_wide_range_x(kvq, wdtype, M, N, K):
    """Activations over bf16's whole range: +-1e5 and +-3e4 (beyond f16's
    65504), 13 decades within a row, ~1e-6, bf16 subnormals, ~1e-30 and
    ~1e30, zero rows (oracle_pins.wide_range_x)."""
    rng = np.random.default_rng(7 * M + N + K + wdtype)
    w, s, _ = pins.random_wq_case(rng, wdtype, M, N, K)
    x = pins.wide_range_x(rng, M, K)
    check(wdtype, w, s, x, what=f"wide x {M}x{N}x{K}")


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
@pytest.mark.parametrize("N,K", [(200, 1536), (70, 640)])
def test_wq_ring_wide_range_x(kvq, wdtype, N, K):
    """Each of the eight wide-range activation regimes through the ring
    kernel: as one token (its own instantiation) and in pairs of tokens."""
    rng = np.random.default_rng(N + K + 10 * wdtype)
    w, s, _ = pins.random_wq_case(rng, wdtype, 1, N, K)
    x8 = pins.wide_range_x(rng, 8, K)
    for m in range(8):
        check(wdtype, w, s, x8[m:m + 1], what=f"regime {m}, one token, {N}x{K}")
    for m in range(0, 8, 2):
        check(wdtype, w, s, x8[m:m + 2], what=f"regimes {m},{m + 1}, two tokens, {N}x{K}")


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
@pytest.mark.parametrize("M", [1, 2, 9], ids=["ring1", "ring", "registers"])
def test_wq_gemm_nan_inf_propagate(kvq, wdtype, M):
    """NaN and infinities in x propagate as IEEE arithmetic has them: a NaN in
    a token's k range makes every output of that token NaN; +-inf gives +-inf
    or NaN (inf * 0, inf - inf) exactly where the fp64 oracle does; the other
    tokens stay within the bound."""
    rng = np.random.default_rng(50 + 3 * M + wdtype)
    N, K = 150, 768
    w, s, x = pins.random_wq_case(rng, wdtype, M, N, K)
    x = x.copy()
    nan_b, inf_b, ninf_b = np.uint16(0x7FC0), np.uint16(0x7F80), np.uint16(0xFF80)
    x[0, 300] = nan_b
    if M > 1:
        x[1, 5] = inf_b
        x[1, 700] = ninf_b
    got = run_gpu(wdtype, w, s, x).astype(np.float64)
    ref = oracle.wq_gemm(wdtype, w, s, x)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "NaN positions differ"
    assert np.array_equal(np.isposinf(got), np.isposinf(ref)), "+inf positions differ"
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "-inf positions differ"
    assert np.all(np.isnan(got[0])), "a NaN input must make its token's outputs NaN"
    if M > 2:
        bound, _ = wq_bound(wdtype, w, s, x[2:])
        assert np.all(np.abs(got[2:] - ref[2:]) <= bound)


@pytest.mark.parametrize("wdtype", [0, 1], ids=["int4", "e4m3"])
def test_wq_gemm_wide_range_x_full_size(kvq, wdtype):
    """The large projection (28672 x 5120) at 64 tokens with wide-range
    activations: 96 sampled output channels."""
    rng = np.random.default_rng(90 + wdtype)
    M, N, K = 64, 28672, 5120
    w, s, _ = pins.random_wq_case(rng, wdtype, M, N, K)
    x = pins.wide_range_x(rng, M, K)
    rows = np.sort(rng.choice(N, 96, replace=False))
    check(wdtype, w, s, x, rows=rows, what="wide x full size")
