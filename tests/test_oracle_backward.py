"""The gradient oracle (fp64 autograd of the sequential recurrence) checked
against what does not depend on it (CPU only): central finite differences of
the C forward oracle along random directions, and two closed forms --
causal linear attention (b = 0, w = 1, no decay) and pure decay (b = w = 0).
The pins live in tests/pins_backward.py; tests/test_oracle_backward_mutants.py
shows that each catches planted mistakes."""
import pytest

import oracle
import pins_backward


@pytest.mark.parametrize("name", sorted(pins_backward.PINS))
def test_backward_oracle_meets_pin(name):
    score = pins_backward.PINS[name](oracle.backward)
    assert score <= pins_backward.TOL[name], f"{name}: {score:.3e}"
