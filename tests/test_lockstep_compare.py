"""The lockstep harness's output comparison, on the CPU.

The tolerances the parity tests apply: fp32 rows within 1e-5 of the row's
largest magnitude, bf16 elements within 2e-2, and HiKV Stage II rows the
oracle flags as near-ties within 2e-2 whatever the dtype.  Checked here on
constructed arrays, so a loosened or inverted bound fails without a GPU.
"""
import numpy as np
import pytest

import workloads as W
from tests.lockstep import Lockstep, Report


def _harness(dtype):
    ls = Lockstep.__new__(Lockstep)
    ls.w = W.WORKLOADS[0].with_(dtype=dtype, d=8)
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


def test_bf16_elements_at_the_absolute_bound():
    ls = _harness("bf16")
    want = np.zeros((2, 4, 8), np.float32)
    got = want.copy()
    got[0, 0, 0] = 0.019
    ls.compare_out(got, want, 0)
    got[0, 0, 0] = 0.021
    with pytest.raises(AssertionError):
        ls.compare_out(got, want, 0)


def test_near_tie_rows_are_held_to_the_loose_bound_only():
    ls = _harness("f32")
    want = np.ones((2, 4, 8), np.float32)
    got = want.copy()
    got[0, 1, :] += 0.01                 # a swapped chunk entry in a flagged row
    skip = np.zeros((2, 4), bool)
    skip[0, 1] = True
    ls.compare_out(got, want, 0, skip=skip)
    assert ls.rep.stage2_near_tie_rows == 1
    with pytest.raises(AssertionError):  # the same error in an unflagged row fails
        ls.compare_out(got, want, 0)
    got[0, 1, 0] = 1.03                  # beyond the loose bound even when flagged
    with pytest.raises(AssertionError):
        ls.compare_out(got, want, 0, skip=skip)
