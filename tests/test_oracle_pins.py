"""The fp64 oracle against what the pages and mathematics fix (CPU only)."""
import pytest

from oracle_pins import PINS


@pytest.mark.parametrize("name", sorted(PINS))
def test_oracle_pin(oracle_lib, name):
    fn, tol = PINS[name]
    err = fn(oracle_lib)
    assert err <= tol, f"pin {name}: error {err:.3e} > {tol:.0e}"
