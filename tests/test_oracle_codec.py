"""Pins of the oracle's e4m3 codec (OCP E4M3; the pages name the format only)."""
import pytest

import oracle_pins as pins  # noqa: E402


@pytest.mark.parametrize("pin", [pins.pin_decode_all_codes, pins.pin_decode_structure,
                                 pins.pin_encode_roundtrip, pins.pin_encode_vs_torch,
                                 pins.pin_encode_brute_force, pins.pin_encode_special,
                                 pins.pin_quantise_exhaustive])
def test_codec_pin(oracle_mod, pin):
    pin(oracle_mod)
