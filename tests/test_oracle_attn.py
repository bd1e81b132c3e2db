"""Pins of the oracle's fp64 paged decode attention."""
import pytest

import oracle_pins as pins  # noqa: E402
from fp8_paged_kv_attn_gb300 import inputs


def attn_workloads():
    return [inputs.tiny(),
            inputs.uniform("mha_g1", 31, B=2, ctx=50, Hq=2, Hkv=2, D=64, P=16),
            inputs.uniform("gqa_g8", 32, B=2, ctx=100, Hq=16, Hkv=2, D=128, P=16,
                           outlier_frac=0.01),
            inputs.ragged(seed=33, B=3, total=500, lo=30, hi=300, Hq=8, Hkv=2, D=64, P=64)]


@pytest.mark.parametrize("w", attn_workloads(), ids=lambda w: w.name)
def test_attn_vs_sdpa_fp8(oracle_mod, w):
    pins.pin_attn_vs_sdpa(oracle_mod, w)


@pytest.mark.parametrize("w", attn_workloads()[:2], ids=lambda w: w.name)
def test_attn_vs_sdpa_bf16(oracle_mod, w):
    pins.pin_attn_vs_sdpa(oracle_mod, w, kv_dtype=oracle_mod.KV_BF16)


def test_attn_one_token(oracle_mod):
    pins.pin_attn_one_token(oracle_mod)


def test_attn_equal_keys(oracle_mod):
    pins.pin_attn_equal_keys(oracle_mod)


def test_attn_page_permutation(oracle_mod):
    pins.pin_attn_page_permutation(oracle_mod, attn_workloads()[2])


def test_attn_abort_and_errors(oracle_mod):
    pins.pin_attn_abort_and_errors(oracle_mod)
