"""Closed-form pins of the oracle's RoPE frequency, attention scale, layer composition and LM
head (CPU). The checks live in _layer_pins.py so that test_oracle_mutations.py can run them on
oracle copies with one planted mistake each."""
import pytest

import oracle as orc

from _layer_pins import PINS


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_layer_pin(name):
    PINS[name](orc)
