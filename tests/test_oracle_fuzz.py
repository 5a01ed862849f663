"""The oracle's batch build against its independent pins on many random
small steps (hypothesis draws the shapes: block sizes 1 to 16, one to three
KV-cache groups, sliding windows, decode/prefill mixes, recycled rows), not
only on the fixed seeded cases of ``oracle_pins.small_workloads``: the
flattening by concatenation, slots by brute-force enumeration, the
invariants of the definitions, and the gathered block-table rows."""
from unittest import mock

import pytest

import oracle
import pkv_workloads as workloads
from tests import oracle_pins

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies

PINS = [oracle_pins.pin_flatten_by_concatenation, oracle_pins.pin_slots_brute_force,
        oracle_pins.pin_invariants, oracle_pins.pin_block_tables]


@hypothesis.settings(max_examples=80, deadline=None, derandomize=True)
@hypothesis.given(
    seed=st.integers(0, 10_000),
    n=st.integers(1, 24),
    block_sizes=st.lists(st.sampled_from([1, 2, 3, 4, 5, 7, 8, 16]), min_size=1, max_size=3),
    max_ctx=st.integers(1, 120),
    max_chunk=st.integers(1, 30),
    decode_frac=st.floats(0.0, 1.0),
    window=st.sampled_from([0, 0, 4, 9, 32]),
)
def test_prepare_pins_on_random_steps(seed, n, block_sizes, max_ctx, max_chunk, decode_frac,
                                      window):
    wl = workloads.random_small(seed=seed, num_requests=n, block_sizes=tuple(block_sizes),
                                max_ctx=max_ctx, max_chunk=max_chunk,
                                decode_frac=decode_frac, window=window)
    lib = oracle.load()
    with mock.patch.object(oracle_pins, "small_workloads", lambda: [wl]):
        for pin in PINS:
            pin(lib)
