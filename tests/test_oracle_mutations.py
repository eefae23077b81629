"""The pins have teeth: each oracle build with one planted mistake (a swapped
combine, the decay without A, the sign of A lost, delta dropped from b, the D
residual dropped, the gate applied to x, chunk states off by one, the delta
bias ignored, exp in place of softplus, three mistakes of the backward and two
of the SSD form)
fails at
least one pin.  The mistakes are compiled into separate copies of the oracle
on the CPU; the real oracle is untouched."""
import pytest

import pins

PLANTS = {1: "combine operands swapped", 2: "decay exp(-delta) without A",
          3: "sign of A lost", 4: "delta dropped from b", 5: "D residual dropped",
          6: "gate applied to x", 7: "chunk state one step early",
          8: "dt_bias ignored", 9: "exp in place of softplus",
          10: "backward adjoint carried with the next step's decay",
          11: "backward dA without its delta factor", 12: "backward dz without silu'",
          13: "SSD input read without the head offset", 14: "SSD input decayed with the state"}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda k: PLANTS[k].replace(" ", "_"))
def test_planted_mistake_is_caught(oracle, plant):
    assert oracle.plant_id(plant) == plant
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(plant=plant)
        except (AssertionError, FloatingPointError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches planted mistake {plant} ({PLANTS[plant]})"
