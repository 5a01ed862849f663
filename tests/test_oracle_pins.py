"""The CPU oracle against its pins (no GPU needed)."""
import pytest

import oracle
from tests import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_generators_are_seeded():
    a = oracle_pins.small_workloads()
    b = oracle_pins.small_workloads()
    for x, y in zip(a, b):
        assert x.schedule == y.schedule
        for (ka, ra), (kb, rb) in zip(x.ops, y.ops):
            assert ka == kb
            if ka == "add":
                assert (ra.token_ids == rb.token_ids).all()
                assert all((p == q).all() for p, q in zip(ra.blocks, rb.blocks))
