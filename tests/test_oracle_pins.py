"""The CPU oracle against what the source pages and plain mathematics fix (no GPU)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(oracle_mod, pin):
    if pin in (oracle_pins.pin_cos_sin_mpmath, oracle_pins.pin_position_scale, oracle_pins.pin_glu_activation,
               oracle_pins.pin_double_to_bf16, oracle_pins.pin_glu_gradient):
        pytest.importorskip("mpmath")
    pin(oracle_mod)
