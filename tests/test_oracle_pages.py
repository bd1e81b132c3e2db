"""The oracle's page allocator against its pins: the hand-worked example
(tests/golden/page_allocator_example.json) and the invariants any correct
allocator keeps (conservation, LIFO order, one tag increment per hand-out,
served-in-order-until-the-first-misfit, check consistency)."""
import oracle
import oracle_pins as pins


def test_pages_golden_example():
    pins.pin_pages_golden(oracle)


def test_pages_invariants():
    pins.pin_pages_invariants(oracle)


def test_pages_invariants_other_shapes():
    pins.pin_pages_invariants(oracle, seed=9, num_pages=17, B=5, MP=6, n_ops=80)
    pins.pin_pages_invariants(oracle, seed=10, num_pages=300, B=40, MP=16, n_ops=40)


def test_pages_overflow_and_bad_state():
    pins.pin_pages_overflow_and_state(oracle)
