"""The CPU oracle against what the pages, the mathematics and independent
library routines fix (hand-worked golden relayouts, textbook cos/sin values,
all-gather formulation of the all-to-all, torch rms_norm, complex rotation)."""
import pytest

import oracle_pins


@pytest.mark.parametrize("check", oracle_pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check, olib):
    check(olib)
