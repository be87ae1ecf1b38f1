"""The comparison helpers the GPU parity tests use are not vacuous: they
pass results within the stated bounds and fail the plausible wrong answers,
including the one the element-wise bound alone would let through (an
all-zero latent when the reference is far smaller than 2e-2, as at long
contexts).  CPU only."""

import numpy as np
import pytest
import torch

from tests.parity import assert_bf16_close, assert_lse_close

rng = np.random.default_rng(0)
REF = rng.normal(0, 0.5, (64, 512))
SMALL = REF * 8e-3                      # |ref| ~ 4e-3: long-context latent magnitude


def test_bf16_within_bounds_passes():
    got = torch.from_numpy(REF).to(torch.bfloat16)          # bf16 rounding: ~2^-9 relative
    assert_bf16_close(got, REF)
    assert_bf16_close(REF + 1e-3, REF)


@pytest.mark.parametrize("bad", [
    lambda r: r * 1.05,                                      # 5 % scale error on O(1) values
    lambda r: r + 0.03,                                      # offset past abs 2e-2
    lambda r: np.where(np.arange(r.size).reshape(r.shape) == 7, np.nan, r),   # one NaN
    lambda r: r[::-1],                                       # rows permuted
])
def test_bf16_wrong_answers_fail(bad):
    with pytest.raises(AssertionError):
        assert_bf16_close(bad(REF), REF)


def test_all_zero_answer_fails_on_small_references():
    """abs 2e-2 alone accepts zeros against |ref| ~ 4e-3; the scale-aware
    bound max|err| / max|ref| <= 2e-2 does not."""
    zeros = np.zeros_like(SMALL)
    assert np.all(np.abs(zeros - SMALL) <= 2e-2 + 2e-2 * np.abs(SMALL))   # the element-wise bound passes
    with pytest.raises(AssertionError, match="max\\|err\\|/max\\|ref\\|"):
        assert_bf16_close(zeros, SMALL)
    with pytest.raises(AssertionError):
        assert_bf16_close(SMALL * 1.1, SMALL)                # 10 % off, still far below 2e-2 absolute
    assert_bf16_close(SMALL * 1.005, SMALL)


def test_mask_excludes_unspecified_entries():
    got = REF.copy()
    got[3] = np.nan                                          # an unused split's o
    mask = np.ones(REF.shape[0], bool)
    mask[3] = False
    assert_bf16_close(got, REF, mask=mask)
    with pytest.raises(AssertionError):
        assert_bf16_close(got, REF)


def test_lse_bounds_and_neg_inf_pattern():
    ref = rng.normal(5, 2, (8, 12))
    ref[2] = -np.inf
    assert_lse_close(ref + 9e-4, ref)
    with pytest.raises(AssertionError):
        assert_lse_close(ref + 2e-3, ref)
    flipped = ref.copy()
    flipped[2] = 0.0                                         # an empty row given a finite LSE
    with pytest.raises(AssertionError, match="-inf pattern"):
        assert_lse_close(flipped, ref)
    nan = ref.copy()
    nan[0, 0] = np.nan
    with pytest.raises(AssertionError):
        assert_lse_close(nan, ref)
