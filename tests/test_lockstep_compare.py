"""The lockstep harness's output comparison, on the CPU.

The tolerances the parity tests apply: fp32 rows within 1e-5 of the row's
largest magnitude; bf16 elements within one bf16 ulp of the larger value
(at least 2^-15) and never beyond 2e-2; HiKV Stage II rows whose selection
float32 rounding could change must equal one of the oracle's admissible
outputs at those same tolerances.  Checked here on constructed arrays, so a
loosened or inverted bound fails without a GPU.
"""
import numpy as np
import pytest

import workloads as W
from tests.lockstep import Lockstep, Report, bf16_ulp


def _harness(dtype):
    ls = Lockstep.__new__(Lockstep)
    ls.w = W.WORKLOADS[0].with_(dtype=dtype, d=8, hq=4)
    ls.rep = Report()
    return ls


def test_fp32_rows_at_the_relative_bound():
    ls = _harness("f32")
    want = np.ones((2, 4, 8), np.float32)
    got = want.copy()
    got[1, 2, 3] += 0.9e-5
    ls.compare_out(got, want, 0)
    got[1, 2, 3] += 0.2e-5          # 1.1e-5 of a row whose largest value is 1
    with pytest.raises(AssertionError):
        ls.compare_out(got, want, 0)


def test_bf16_ulp_spacing():
    assert bf16_ulp(1.0) == 2.0 ** -7
    assert bf16_ulp(1.99) == 2.0 ** -7
    assert bf16_ulp(2.0) == 2.0 ** -6
    assert bf16_ulp(-0.3) == 2.0 ** -9          # 0.3 in [2^-2, 2^-1)


def test_bf16_elements_within_one_ulp():
    ls = _harness("bf16")
    want = np.full((2, 4, 8), 0.3, np.float32)
    got = want.copy()
    got[0, 0, 0] = 0.3 + 2.0 ** -9              # one ulp at 0.3: a rounding boundary between the sums
    ls.compare_out(got, want, 0)
    assert ls.rep.bf16_over_1ulp == 0
    got[0, 0, 0] = 0.3 + 2 * 2.0 ** -9          # two ulps: a real difference, far below 2e-2
    with pytest.raises(AssertionError):
        ls.compare_out(got, want, 0)


def test_bf16_small_values_use_the_floor():
    ls = _harness("bf16")
    want = np.full((2, 4, 8), 1e-6, np.float32)
    got = want.copy()
    got[1, 3, 7] = 1e-6 + 2.0 ** -16            # many ulps of 1e-6, within the 2^-15 floor
    ls.compare_out(got, want, 0)
    assert ls.rep.bf16_over_1ulp == 1
    got[1, 3, 7] = 1e-6 + 2.0 ** -14
    with pytest.raises(AssertionError):
        ls.compare_out(got, want, 0)


def test_stage2_rows_match_an_admissible_selection():
    ls = _harness("f32")
    want = np.ones((2, 4, 8), np.float32)
    got = want.copy()
    other = want[0, 1].copy()
    other[0] += 0.01                     # the output of the other admissible selection
    got[0, 1] = other
    alts = {(0, 1): np.stack([want[0, 1], other])}
    ls.compare_out(got, want, 0, alternatives=alts)
    assert ls.rep.stage2_near_tie_rows == 1 and ls.rep.stage2_alt_matches == 1
    with pytest.raises(AssertionError):  # the same row without alternatives fails
        ls.compare_out(got, want, 0)
    got[0, 1, 0] = 1.005                 # matches neither selection
    with pytest.raises(AssertionError):
        ls.compare_out(got, want, 0, alternatives=alts)
    got[0, 1] = want[0, 1]               # the exact selection is one of them
    ls.compare_out(got, want, 0, alternatives=alts)
    assert ls.rep.stage2_alt_matches == 1
