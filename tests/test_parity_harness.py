"""Host logic of the GPU-vs-oracle parity harness (runs on the CPU).

The harness decides which kept-set and budget differences count as the
near-tie divergences the method's parity contract allows (the oracle's
scores within 1e-6 relative) and fails every other difference; the tests
then require zero divergences.  These checks pin those decisions.
"""
import numpy as np
import pytest

from . import parity


def _keys(keys, pos, prot=None):
    pos = np.asarray(pos, np.int32)
    return {"key": np.asarray(keys, np.float32), "pos": pos,
            "prot": np.zeros(len(pos), bool) if prot is None else np.asarray(prot, bool)}


def test_kept_near_tie_is_accepted():
    # oracle keeps 10 and 11; 12's key is 1e-7 relative below the cut: a swap
    # of 11 and 12 is a near-tie
    k = _keys([0.5, 0.3, 0.2, 0.2 * (1 - 1e-7), 0.1], [9, 10, 11, 12, 13])
    kept_o = {9, 10, 11}
    kept_g = {9, 10, 12}
    assert parity._legit_kept_divergence(k, kept_o, kept_g)


def test_kept_real_difference_is_rejected():
    # 13's key is far below the cut (0.2): not a near-tie
    k = _keys([0.5, 0.3, 0.2, 0.2 * (1 - 1e-7), 0.1], [9, 10, 11, 12, 13])
    assert not parity._legit_kept_divergence(k, {9, 10, 11}, {9, 10, 13})
    # a position the oracle never ranked
    assert not parity._legit_kept_divergence(k, {9, 10, 11}, {9, 10, 99})
    # just outside the 1e-6 relative band
    k2 = _keys([0.5, 0.2, 0.2 * (1 - 3e-6)], [1, 2, 3])
    assert not parity._legit_kept_divergence(k2, {1, 2}, {1, 3})


def test_protected_tokens_do_not_set_the_cut():
    # the protected token 20 has the lowest key but is kept by rule; the cut
    # is the lowest key among the kept candidates (0.4)
    k = _keys([0.01, 0.4, 0.4 * (1 + 5e-7), 0.3], [20, 5, 6, 7], [1, 0, 0, 0])
    assert parity._legit_kept_divergence(k, {20, 5}, {20, 6})
    assert not parity._legit_kept_divergence(k, {20, 5}, {20, 7})


def test_budget_near_tie_rule():
    assert parity.budget_near_tie(0.5 * (1 + 4e-7), 0.5)
    assert parity.budget_near_tie(0.5 * (1 - 4e-7), 0.5)
    assert not parity.budget_near_tie(0.5 + 1e-5, 0.5)      # the old 1e-5 rule accepted this
    assert not parity.budget_near_tie(0.49, 0.5)


def test_check_requires_every_lane_step_and_no_divergence():
    r = parity.Report()
    r.rc = 0
    r.total = r.compared = 10
    assert parity.check(r) is r
    r.kept_div, r.uncompared, r.compared = 1, 3, 7
    with pytest.raises(AssertionError):
        parity.check(r)
    assert parity.check(r, allowed_divergences=1) is r
    r.compared = 6                        # a lane-step neither compared nor counted
    with pytest.raises(AssertionError):
        parity.check(r, allowed_divergences=1)
    r2 = parity.Report()
    r2.rc, r2.total, r2.compared = 0, 10, 9
    with pytest.raises(AssertionError):
        parity.check(r2)
    r2.compared, r2.rc = 10, -5
    with pytest.raises(AssertionError):
        parity.check(r2)
