"""The fp64 oracle against facts other than itself (CPU only)."""
import numpy as np
import pytest

import oracle_pins


@pytest.mark.parametrize("name", list(oracle_pins.ALL_PINS))
def test_pin(name):
    err, tol = oracle_pins.ALL_PINS[name]()
    assert err <= tol, f"{name}: error {err} above {tol}"


def test_golden_fixture_cites_its_source():
    text = open(oracle_pins.os.path.join(oracle_pins.GOLDEN, "worked_example_locations.txt")).read()
    assert "section 2.2" in text and "un.csdn.net/8fh7s5u7wxgo" in text
    rows = oracle_pins.read_worked_example()
    assert rows.shape == (4, 6)
    np.testing.assert_allclose(rows[:, 4:6], rows[:, 0:2] + rows[:, 2:4], atol=1e-15)
