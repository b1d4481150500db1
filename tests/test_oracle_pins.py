"""The oracle against its pins (closed forms, stated invariants, golden cases, brute force)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_every_oracle_function_is_pinned():
    names = {p.__name__ for p in oracle_pins.ALL_PINS}
    for prefix in ("pin_logits", "pin_topk", "pin_walk", "pin_pair", "pin_conv", "pin_ce"):
        assert any(n.startswith(prefix) for n in names), prefix
