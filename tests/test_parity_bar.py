"""The float bar of the parity tests: bf16 ulps and the rounding slack (CPU)."""
import numpy as np
import pytest

from helpers import bf16_ulp, float_parity


def test_bf16_ulp():
    assert bf16_ulp(np.array([1.0, 1.99, 2.0, 12.0, -12.0, 0.75]))[:].tolist() == [2 ** -7, 2 ** -7, 2 ** -6,
                                                                                   2 ** -4, 2 ** -4, 2 ** -8]
    assert bf16_ulp(np.array([0.0]))[0] == 2.0 ** -133


def test_one_ulp_flip_passes_only_with_the_bf16_bar():
    ref = np.array([12.0] + [0.5] * 99)          # rms about 1.3: 2e-2 * rms = 0.026 < one ulp at 12 (0.0625)
    got = ref.copy()
    got[0] = 12.0625
    with pytest.raises(AssertionError):
        float_parity(got, ref)
    float_parity(got, ref, bf16=True)
    got[0] = 12.125                               # two ulps: over the bar either way
    with pytest.raises(AssertionError):
        float_parity(got, ref, bf16=True)


def test_sum_of_rounded_parts():
    parts = [np.array([3.0, 0.25]), np.array([3.0, 0.25]), np.array([3.0, 0.25])]
    ref = np.array([9.0, 0.75])
    got = sum(parts) + np.array([0.05, 0.0])      # within 2e-2 rms + (3 ulp(3) + ulp(9)) / 2 = 0.13 + 0.055
    float_parity(got, ref, bf16_terms=parts)
    with pytest.raises(AssertionError):
        float_parity(got + np.array([0.2, 0.0]), ref, bf16_terms=parts)
