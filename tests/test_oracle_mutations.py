"""Each planted mistake in the oracle must make at least one pin fail.

This shows the pins are sharp enough to catch a dropped term, a wrong sign or
index, or a transposed operand anywhere in the oracle."""

import pytest

import oracle
import pins


@pytest.mark.parametrize("name", sorted(oracle.MUTATIONS))
def test_mutation_is_caught(name):
    failed = []
    with oracle.mutation(name):
        for pin_name, pin in pins.ALL_PINS.items():
            try:
                ok, _ = pin()
            except Exception:
                ok = False
            if not ok:
                failed.append(pin_name)
                break
    assert failed, f"planted mistake {name!r} passed every pin"
    assert oracle._load().oracle_get_mutation() == 0
