"""The oracle's prefill -> decode handoff against its pin: torch indexing of
the prefill slots, torch's fp32 division and float8_e4m3fn conversion, and
the error cases (bad ranges and pages write nothing)."""
import oracle
import oracle_pins as pins


def test_handoff_vs_torch():
    pins.pin_handoff_vs_torch(oracle)
