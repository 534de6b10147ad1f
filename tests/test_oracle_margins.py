"""Pins of the oracle's boundary outputs, which decide what the GPU parity rule allows.

- the top-p cut ("The decoding loop and MTP", "Why a hand-written decoding loop": top-p
  keeps the smallest top set whose mass reaches p): on rows with hand-set masses, the
  group count the rule keeps, its margin, and the range of counts a computation off by
  less than delta can reach (S_g < p + delta and S_{g+1} >= p - delta);
- a forced cut keeps exactly that many groups and renormalises over them;
- the inverse-CDF draw ("MPT (MTP, Multi-Token Prediction) 原理详解", 三 stage 3): for U
  placed a hand-chosen distance from a cell edge, the drawn id, the two distances to the
  cell's edges and the neighbouring ids with positive weight.
Masses are given as logits log(m) in float64 rounded to float32, so the sums are only
within ~1e-7 of the hand-set values; every expected boundary distance here is either
far larger or set up to be within 1e-6.
"""
import numpy as np
import pytest

import oracle


def _logits(masses):
    return np.log(np.asarray(masses, np.float64)).astype(np.float32)


# ---------------------------------------------------------------- top-p cuts

def test_cut_range_when_a_group_straddles_p():
    # masses 0.5, 0.3, 0.2: S_1 = 0, S_2 = 0.5, S_3 = 0.8, S_4 = 1
    t = _logits([0.5, 0.3, 0.2])
    cases = [
        # p, delta, (rule, lowest, highest)
        (0.7, 1e-5, (2, 2, 2)),          # S_2 < 0.7 <= S_3, far from both
        (0.8 - 1e-6, 1e-5, (2, 2, 3)),   # S_3 only 1e-6 above p: the third group may stay
        (0.8 + 1e-6, 1e-5, (3, 2, 3)),   # S_3 only 1e-6 below p: it stays, may drop
        (0.5 + 1e-6, 1e-5, (2, 1, 2)),   # S_2 1e-6 below p: the second group may drop
        (0.8 - 1e-6, 1e-7, (2, 2, 2)),   # a window narrower than the distance
        (0.3, 0.25, (1, 1, 2)),          # a wide window reaches the next group
    ]
    for p, delta, want in cases:
        r = oracle.verify_unit(t, None, 0, 1.0, 0, p, 0.5, 0.5, draw=False, delta=delta)
        assert r["cut_t"] == want, (p, delta, r["cut_t"])


def test_top_p_margin_is_the_distance_of_the_deciding_masses():
    t = _logits([0.5, 0.3, 0.2])
    # kept groups 1-2; the margin is min(p - S_2, |S_3 - p|)
    r = oracle.verify_unit(t, None, 0, 1.0, 0, 0.78, 0.5, 0.5, draw=False)
    assert abs(r["margin_t"] - 0.02) < 1e-6
    r = oracle.verify_unit(t, None, 0, 1.0, 0, 0.55, 0.5, 0.5, draw=False)
    assert abs(r["margin_t"] - 0.05) < 1e-6
    r = oracle.verify_unit(t, None, 0, 1.0, 0, 0.8 - 1e-6, 0.5, 0.5, draw=False)
    assert 5e-7 < r["margin_t"] < 1.5e-6
    # top-p off: no margin
    r = oracle.verify_unit(t, None, 0, 1.0, 0, 1.0, 0.5, 0.5, draw=False)
    assert r["margin_t"] == np.inf and r["cut_t"] == (3, 3, 3)


def test_ties_form_one_group():
    # two equal logits of mass 0.25 each after the top: one group, kept or dropped together
    t = _logits([0.4, 0.25, 0.25, 0.1])
    r = oracle.verify_unit(t, None, 1, 1.0, 0, 0.5, 0.5, 0.5, draw=False, delta=1e-5)
    assert r["cut_t"] == (2, 2, 2)
    assert abs(r["pt"] - 0.25 / 0.9) < 1e-6


def test_forced_cut_keeps_that_many_groups():
    t = _logits([0.5, 0.3, 0.15, 0.05])
    q = _logits([0.25, 0.25, 0.25, 0.25])
    # p = 0.7: the rule keeps 2 groups (p(0) = 0.5/0.8); forced 3 keeps 0.95 of the mass
    r = oracle.verify_unit(t, q, 0, 1.0, 0, 0.7, 0.5, 0.5, draw=False)
    assert abs(r["pt"] - 0.5 / 0.8) < 1e-6
    r3 = oracle.verify_unit(t, q, 0, 1.0, 0, 0.7, 0.5, 0.5, draw=False, gt=3)
    assert abs(r3["pt"] - 0.5 / 0.95) < 1e-6
    r1 = oracle.verify_unit(t, q, 2, 1.0, 0, 0.7, 0.5, 0.5, draw=False, gt=1)
    assert r1["pt"] == 0.0
    # the draft row's cut: all four ids tie, one group, kept whatever p is
    assert r["cut_q"] == (1, 1, 1)
    rq = oracle.verify_unit(t, q, 3, 1.0, 0, 0.7, 0.5, 0.5, draw=False, gq=1)
    assert abs(rq["pd"] - 0.25) < 1e-6


def test_cut_counts_follow_top_k():
    # top-k 2 leaves two groups (0.4, 0.3; Z = 0.7); top-p acts inside them
    t = _logits([0.4, 0.3, 0.2, 0.1])
    r = oracle.verify_unit(t, None, 0, 1.0, 2, 1.0, 0.5, 0.5, draw=False)
    assert r["cut_t"] == (2, 2, 2)
    # p = 0.5: S_2 = 0.4 / 0.7 = 0.571 >= p, so only the top id stays
    r = oracle.verify_unit(t, None, 0, 1.0, 2, 0.5, 0.5, 0.5, draw=False, delta=1e-5)
    assert r["cut_t"] == (1, 1, 1) and abs(r["pt"] - 1.0) < 1e-12
    # p just above 4/7: the second group stays, and may drop
    r = oracle.verify_unit(t, None, 0, 1.0, 2, 0.4 / 0.7 + 1e-6, 0.5, 0.5, draw=False,
                           delta=1e-5)
    assert r["cut_t"] == (2, 1, 2) and abs(r["pt"] - 0.4 / 0.7) < 1e-6


# ---------------------------------------------------------------- inverse-CDF draws

@pytest.mark.parametrize("u,tok,lo,hi,prev,nxt", [
    (0.30, 1, 0.05, 0.20, 0, 3),          # inside cell 1 = [0.25, 0.5)
    (0.5 - 1e-6, 1, 0.25 - 1e-6, 1e-6, 0, 3),   # 1e-6 below the edge with cell 3
    (0.5 + 1e-6, 3, 1e-6, 0.5 - 1e-6, 1, -1),   # 1e-6 above it (id 2 has no weight)
    (0.1, 0, 0.1, 0.15, -1, 1),           # the first cell
])
def test_inverse_cdf_cell_and_neighbours(u, tok, lo, hi, prev, nxt):
    # bonus draw from weights 0.25, 0.25, 0, 0.5 (id 2 is outside the support: top-k 3)
    t = _logits([0.25, 0.25, 1e-9, 0.5])
    r = oracle.verify_unit(t, None, -1, 1.0, 3, 1.0, 0.5, u, bonus=True)
    assert r["token"] == tok
    assert abs(r["cdf_lo"] - lo) < 1e-7 and abs(r["cdf_hi"] - hi) < 1e-7
    assert r["tok_prev"] == prev and r["tok_next"] == nxt
    assert abs(r["cdf_margin"] - min(lo, hi)) < 1e-7


def test_residual_draw_neighbours_skip_zero_weights():
    # residual max(0, p - q): p = (0.4, 0.3, 0.2, 0.1), q = (0.1, 0.5, 0.25, 0.15) gives
    # (0.3, 0, 0, 0), normalised (1, 0, 0, 0): a point mass, no neighbours
    t = _logits([0.4, 0.3, 0.2, 0.1])
    q = _logits([0.1, 0.5, 0.25, 0.15])
    r = oracle.verify_unit(t, q, 1, 1.0, 0, 1.0, 0.999, 0.7)
    assert not r["accept"] and r["token"] == 0
    assert r["tok_prev"] == -1 and r["tok_next"] == -1
    assert abs(r["cdf_lo"] - 0.7) < 1e-6 and abs(r["cdf_hi"] - 0.3) < 1e-6
