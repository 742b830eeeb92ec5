"""The comparison rules of tests/parity.py, pinned on the CPU: the bf16
rounding against torch's conversion, half an ulp against the binade
definition, and cases just inside and just outside each bound."""
import numpy as np
import pytest
import torch

from tests.parity import OUT_TOL, bf16_half_ulp, bf16_round, check_out


def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-30, 30, 200000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    assert np.array_equal(bf16_round(x.astype(np.float64)), ref)


def test_bf16_round_ties_go_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even significand (1) wins;
    # 1 + 3 * 2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: 1 + 2^-6 wins
    assert bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert bf16_round(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert bf16_round(np.array([-(1 + 2.0 ** -8)]))[0] == -1.0


def test_half_ulp_by_binade():
    vals = np.array([0.3, 0.5, 0.75, 0.999, 1.0, 1.5, 2.0, 3.9, -2.5, 0.0])
    expect = np.array([2.0 ** -10, 2.0 ** -9, 2.0 ** -9, 2.0 ** -8, 2.0 ** -8, 2.0 ** -8, 2.0 ** -7, 2.0 ** -7,
                       2.0 ** -7, 0.0])
    assert np.array_equal(bf16_half_ulp(vals), expect)
    # just below 2: bf16 rounds up to 2.0 once past the midpoint 2 - 2^-8
    assert bf16_half_ulp(np.array([2 - 2.0 ** -8]))[0] == 2.0 ** -7
    assert bf16_half_ulp(np.array([2 - 2.0 ** -7]))[0] == 2.0 ** -8


def test_bf16_rule_accepts_a_correct_rounding_and_rejects_a_kernel_error_above_2e3():
    rng = np.random.default_rng(6)
    ref = rng.standard_normal(4096) * 2
    # a kernel that was within 1.9e-3 before rounding passes
    good = bf16_round(ref + rng.uniform(-1.9e-3, 1.9e-3, ref.shape))
    check_out(good, ref, bf16=True)
    # one value 2.5e-3 off before rounding fails on some element, although
    # the rounded result can sit within 2e-3 + half an ulp of the oracle
    bad = bf16_round(ref + 2.5e-3)
    with pytest.raises(AssertionError):
        check_out(bad, ref, bf16=True)
    assert np.all(np.abs(bad - ref) <= OUT_TOL + bf16_half_ulp(ref) + 2.5e-3)


def test_fp32_rule_is_the_literal_bound():
    ref = np.linspace(-3, 3, 1001)
    check_out(ref + 1.99e-3, ref, bf16=False)
    with pytest.raises(AssertionError):
        check_out(ref + 2.01e-3, ref, bf16=False)
