"""The parity tests' own comparison logic, on CPU: the routing check accepts
a different choice only where the ranking sits inside the logits' error band,
and only when that choice is still a valid top-K within the band."""
import numpy as np
import pytest

from _helpers import LOGIT_TOL, check_routing, decided_tokens


def _case():
    # 3 tokens, 5 experts, K = 2; scale 1 everywhere -> band 2e-5 per logit
    L64 = np.array([[3.0, 2.0, 1.0, 0.0, -1.0],          # clear margins
                    [1.0, 0.5, 0.5 - 1e-6, 0.0, -1.0],   # slots 2 and 3 nearly tied
                    [2.0, 2.0 - 3e-5, 1.0, 0.0, -1.0]])  # slots 1 and 2 within the band
    scale = np.ones_like(L64)
    ref = np.array([[0, 1], [0, 1], [0, 1]])
    return L64, scale, ref


def test_decided_tokens():
    L64, scale, _ = _case()
    assert decided_tokens(L64, scale, 2).tolist() == [True, False, False]
    # K = E: every consecutive gap counts
    assert decided_tokens(L64[:1], scale[:1], 5).tolist() == [True]


def test_identical_routing_passes():
    L64, scale, ref = _case()
    assert check_routing(ref.copy(), ref, L64, scale, 2).all()


def test_decided_token_routed_differently_fails():
    L64, scale, ref = _case()
    got = ref.copy()
    got[0] = [0, 2]
    with pytest.raises(AssertionError, match="decided"):
        check_routing(got, ref, L64, scale, 2)


def test_near_tie_swap_is_accepted():
    L64, scale, ref = _case()
    got = ref.copy()
    got[1] = [0, 2]              # expert 2 instead of its near twin 1
    got[2] = [1, 0]              # the two near-equal leaders in the other order
    same = check_routing(got, ref, L64, scale, 2)
    assert same.tolist() == [True, False, False]


def test_invalid_choice_inside_the_band_still_fails():
    L64, scale, ref = _case()
    got = ref.copy()
    got[1] = [0, 4]              # expert 4 is far below experts 1 and 2
    with pytest.raises(AssertionError):
        check_routing(got, ref, L64, scale, 2)
    got[1] = [1, 0]              # slot order reversed beyond the band
    with pytest.raises(AssertionError):
        check_routing(got, ref, L64, scale, 2)


def test_band_is_twice_the_tolerance():
    assert LOGIT_TOL == 1e-5
    L64 = np.array([[1.0, 1.0 - 4.1e-5, 0.0]])
    assert decided_tokens(L64, np.ones_like(L64), 1).tolist() == [True]
    L64 = np.array([[1.0, 1.0 - 3.9e-5, 0.0]])
    assert decided_tokens(L64, np.ones_like(L64), 1).tolist() == [False]
