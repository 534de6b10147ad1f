"""Pins of the oracle's sampling distribution: temperature, then top-k, then top-p
(page "The decoding loop and MTP", "Why a hand-written decoding loop").

Each check states the filter another way than the oracle's sorted walk:
- no filter is scipy's softmax of x / tau;
- top-k by rank: a token is kept iff fewer than k logits are strictly larger;
- top-p by definition: a token is kept iff the filtered mass of strictly larger logits
  is < p, summed directly over all pairs (O(V^2));
- special cases: k = 1 is the argmax, a tiny p keeps only the largest logits, all -inf
  is the argmax's point mass.
"""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from verify_spec_greedy_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits


def _brute(x, tau, k, p):
    x = np.asarray(x, np.float64)
    V = x.size
    keep = np.ones(V, bool)
    if 1 <= k < V:
        keep = np.array([(x > x[i]).sum() < k for i in range(V)])
    pi = np.zeros(V)
    pi[keep] = softmax(x[keep] / tau)
    if p < 1:
        keep2 = np.array([keep[i] and pi[(x > x[i]) & keep].sum() < p for i in range(V)])
        keep = keep2
    out = np.zeros(V)
    out[keep] = softmax(x[keep] / tau)
    return out


def test_no_filter_is_softmax():
    rng = np.random.default_rng(0)
    for V in (1, 2, 7, 100, 1000):
        x = (rng.standard_normal(V) * 3).astype(np.float32)
        for tau in (0.3, 1.0, 2.5):
            got = oracle.filter_probs(x, tau)
            np.testing.assert_allclose(got, softmax(x.astype(np.float64) / tau), rtol=1e-12,
                                       atol=1e-300)


@pytest.mark.parametrize("V", [5, 16, 33, 200])
def test_filters_match_brute_force(V):
    rng = np.random.default_rng(V)
    for trial in range(30):
        if trial % 3 == 0:
            x = rng.integers(-4, 5, V).astype(np.float32)  # heavy ties
        else:
            x = (rng.standard_normal(V) * 2).astype(np.float32)
        tau = float(rng.choice([0.5, 1.0, 1.7]))
        k = int(rng.choice([0, 1, 2, V // 3 + 1, V - 1, V, V + 5]))
        p = float(rng.choice([1.0, 0.9, 0.5, 0.05, 0.999]))
        got = oracle.filter_probs(x, tau, k, p)
        want = _brute(x, tau, k, p)
        np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-15)
        assert abs(got.sum() - 1) < 1e-12
        # the support is a set of largest logits: every kept value >= every dropped one
        kept = got > 0
        if (~kept).any():
            assert x[kept].min() >= x[~kept].max() - 0.0


def test_top_k_keeps_boundary_ties():
    x = np.array([5, 4, 4, 4, 3, 2], np.float32)
    got = oracle.filter_probs(x, 1.0, k=2)
    assert (got[:4] > 0).all() and (got[4:] == 0).all()
    np.testing.assert_allclose(got[:4], softmax(x[:4].astype(np.float64)), rtol=1e-13)


def test_top_k_one_is_argmax_and_tiny_p_keeps_the_top():
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = (rng.standard_normal(300) * 3).astype(np.float32)
        g = int(np.argmax(x))
        onehot = np.zeros(300)
        onehot[g] = 1
        np.testing.assert_array_equal(oracle.filter_probs(x, 0.8, k=1), onehot)
        np.testing.assert_array_equal(oracle.filter_probs(x, 0.8, p=1e-6), onehot)


def test_top_p_boundary_is_strict():
    # probabilities 0.5, 0.25, 0.25 (tau = 1): with p = 0.5 the second token sees exactly
    # 0.5 above it, which is not < 0.5, so it is dropped; with p = 0.5 + 1e-9 it stays.
    x = np.log(np.array([0.5, 0.25, 0.25]))
    x = x.astype(np.float64)
    p1 = oracle.filter_probs(np.array([2.0, 1.0, 1.0], np.float32), 1 / np.log(2), p=0.5)
    assert p1.tolist() == [1.0, 0.0, 0.0]
    p2 = oracle.filter_probs(np.array([2.0, 1.0, 1.0], np.float32), 1 / np.log(2), p=0.500001)
    np.testing.assert_allclose(p2, [0.5, 0.25, 0.25], rtol=1e-12)


def test_negative_infinity():
    x = np.array([-np.inf, 1.0, -np.inf, 0.0], np.float32)
    got = oracle.filter_probs(x, 1.0)
    np.testing.assert_allclose(got, [0, 1 / (1 + np.exp(-1)), 0, np.exp(-1) / (1 + np.exp(-1))])
    allninf = np.full(5, -np.inf, np.float32)
    assert oracle.filter_probs(allninf, 0.7, k=2, p=0.5).tolist() == [1, 0, 0, 0, 0]


def test_bf16_is_storage_only():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(500) * 2.5).astype(np.float32)
    b = f32_to_bf16_bits(x)
    np.testing.assert_array_equal(oracle.filter_probs(b, 1.0, 64, 0.95),
                                  oracle.filter_probs(bf16_bits_to_f32(b), 1.0, 64, 0.95))


def test_margin_reports_distance_to_p():
    p_in = np.array([0.5, 0.3, 0.2])
    x = np.log(p_in).astype(np.float32)
    probs, margin = oracle.filter_probs(x, 1.0, p=0.79, with_margin=True)
    # kept: 0.5 (0 above) and 0.3 (0.5 above); dropped: 0.2 (0.8 above)
    assert (probs > 0).tolist() == [True, True, False]
    assert abs(margin - 0.01) < 1e-6
