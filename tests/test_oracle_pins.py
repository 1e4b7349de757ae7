"""The CPU oracle against its pins (no GPU).

Each test ties the oracle to something other than itself: hand-worked rows,
library decoders, brute-force nearest-value rounding, numpy binary32 sums,
exact rational arithmetic, and invariants of the method on seeded inputs.
"""
import pytest

import oracle
import pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def test_worked_rows(orc):
    pins.check_worked_rows(orc)


def test_inv_rms_statistic(orc):
    pins.check_inv_rms_r2(orc)


def test_one_rounding_from_exact(orc):
    pins.check_one_rounding(orc)


def test_exact_tiny_bruteforce(orc):
    pins.check_exact_tiny(orc)


def test_strided_rows(orc):
    pins.check_strided(orc)


def test_f32_partials_bruteforce(orc):
    pins.check_f32_partials(orc)


def test_widen_exhaustive(orc):
    pins.check_widen(orc)


def test_roundtrip_exhaustive(orc):
    pins.check_roundtrip(orc)


def test_narrow_f32_bruteforce_and_library(orc):
    pins.check_narrow_f32(orc)


def test_narrow_f64_one_rounding(orc):
    pins.check_narrow_f64(orc)


@pytest.mark.parametrize("name", list(pins.SMALL_M))
def test_invariants_seeded(orc, name):
    pins.check_invariants(orc, names=(name,))


def test_rejects_bad_arguments(orc):
    import numpy as np
    p = np.zeros((2, 8), np.uint16)
    with pytest.raises(ValueError):
        orc.run(pins.RMSNORM, [p], None, None, 1e-6)  # RMS needs residual and gamma
    assert orc.lib.arf_oracle_run(5, 1, None, None, None, 0.0, None, None, 1, 8, 0) == 1


def test_empty_rows(orc):
    import numpy as np
    p = np.zeros((0, 8), np.uint16)
    out, ro = orc.run(pins.RMSNORM, [p, p], p, np.ones(8, np.uint16), 1e-6)
    assert out.shape == (0, 8) and ro.shape == (0, 8)
