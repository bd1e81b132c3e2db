"""Pins of the oracle's quantise-and-append and tag check."""
import pytest

import oracle_pins as pins  # noqa: E402
from fp8_paged_kv_attn_gb300 import inputs


def small_workloads():
    return [inputs.tiny(),
            inputs.uniform("u1", 11, B=3, ctx=70, Hq=8, Hkv=2, D=128, P=16, outlier_frac=0.01),
            inputs.ragged(seed=12, B=5, total=900, lo=40, hi=400, Hq=8, Hkv=4, D=64, P=64)]


@pytest.mark.parametrize("w", small_workloads(), ids=lambda w: w.name)
def test_append_slots(oracle_mod, w):
    pins.pin_append_slots(oracle_mod, w)


@pytest.mark.parametrize("w", small_workloads(), ids=lambda w: w.name)
def test_append_bf16(oracle_mod, w):
    pins.pin_append_bf16_copy(oracle_mod, w)


def test_append_errors(oracle_mod):
    pins.pin_append_errors(oracle_mod)


def test_half_bytes():
    pins.pin_half_bytes(inputs.tiny())


@pytest.mark.parametrize("B,pages_per_victim,frac", [(256, 1, 0.001), (64, 3, 0.1)])
def test_check_injected(oracle_mod, B, pages_per_victim, frac):
    w = inputs.integrity(seed=21, B=B, lo=16, hi=600, stale_frac=frac,
                         pages_per_victim=pages_per_victim)
    pins.pin_check_injected(oracle_mod, w)


def test_check_edges(oracle_mod):
    pins.pin_check_edges(oracle_mod)
