"""A planted mistake in the oracle must fail at least one pin (CPU only).

The page's own tests include a planted error that must fail ("Add opt-in
FP32 KDA chunk computation", section Validation); here every plausible
mistake in the oracle's arithmetic -- a dropped term, a wrong order, a wrong
index, a transposed operand -- is planted in turn."""
import pytest

import oracle
import pinlib

# The NumPy restatement of the same formula is not counted as a pin.
_RESTATEMENTS = {"numpy_matrix_form"}


@pytest.mark.parametrize("name", [n for n, m in oracle.MUTATIONS.items() if m])
def test_planted_mistake_is_caught(name):
    failing = [p for p in pinlib.failing_pins(oracle.MUTATIONS[name]) if p not in _RESTATEMENTS]
    assert failing, f"planted mistake {name!r} passes every pin"
