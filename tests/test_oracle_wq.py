"""The oracle's weight-only quantised matrix product against its pins: every
INT4 byte value through one-hot activations, float64 matmuls of weights
dequantised independently (numpy bit operations; torch's float8_e4m3fn), and
single-weight closed forms."""
import oracle
import oracle_pins as pins


def test_int4_nibbles():
    pins.pin_int4_nibbles(oracle)


def test_wq_vs_numpy_and_torch():
    pins.pin_wq_vs_numpy(oracle)


def test_wq_single_weight():
    pins.pin_wq_single_weight(oracle)


def test_wq_wide_range_x():
    pins.pin_wq_wide_range_x(oracle)
