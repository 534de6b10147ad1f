"""Exact pin of the oracle's speculative sampling: the output distribution integrated over
the uniforms, with no sampling noise.

Page "MPT (MTP, Multi-Token Prediction) 原理详解", section 三 stage 3 (accept a draft x
drawn from q with probability min(1, p(x)/q(x)), otherwise draw the replacement from the
residual) and page "The decoding loop and MTP", "MTP speculative decoding" item 3 (the
extra token from the target when every guess holds).  For one position over a vocabulary
of at most 6 ids:

- the accept test is a threshold on U_acc: the oracle accepts just below min(1, p/q) and
  rejects just above it, so P(accept | x) = min(1, p(x)/q(x));
- the draw is a step function of U_smp: the oracle's token at the middle of each cell of
  the cumulative weights is that cell's id, so P(token = y | reject x) = r_x(y) / R_x;
- summing over x with weight q(x) gives P(accept) = sum_y min(p_y, q_y) and
  P(first token = y) = min(p_y, q_y) + (1 - sum min) r(y)/R = p_y, both to 1e-12;
- the bonus draw at position D: P(token = y) = p_D(y).

The filters (temperature, top-k, top-p) are on in most cases, so p and q are the
filtered distributions, as the oracle's own filter gives them.
"""
import numpy as np
import pytest

import oracle

CASES = [
    # V, tau, k, p, seed
    (2, 1.0, 0, 1.0, 1),
    (3, 0.7, 0, 1.0, 2),
    (4, 1.3, 3, 1.0, 3),
    (5, 1.0, 0, 0.8, 4),
    (6, 0.6, 4, 0.9, 5),
    (6, 2.0, 0, 0.5, 6),
    (6, 1.0, 5, 0.95, 7),
]


def _rows(V, seed):
    rng = np.random.default_rng(seed)
    t = (rng.standard_normal(V) * 1.5).astype(np.float32)
    q = (t + rng.standard_normal(V) * 1.2).astype(np.float32)
    return t, q


def _accept_prob(t, q, x, tau, k, p):
    """P(accept | draft x): the oracle's accept region in U_acc, located and measured."""
    r = oracle.verify_unit(t, q, x, tau, k, p, 0.5, 0.5, draw=False)
    pt, pd = r["pt"], r["pd"]
    if pt == 0.0:
        assert not oracle.verify_unit(t, q, x, tau, k, p, 1e-12, 0.5, draw=False)["accept"]
        return 0.0
    ratio = r["ratio"]
    assert np.isclose(ratio, pt / pd, rtol=1e-12), (ratio, pt, pd)
    if ratio >= 1.0:
        assert oracle.verify_unit(t, q, x, tau, k, p, 1.0 - 2.0 ** -24, 0.5, draw=False)["accept"]
        return 1.0
    below = oracle.verify_unit(t, q, x, tau, k, p, ratio * (1 - 1e-12), 0.5, draw=False)
    above = oracle.verify_unit(t, q, x, tau, k, p, ratio * (1 + 1e-12), 0.5, draw=False)
    assert below["accept"] and not above["accept"]
    return ratio


def _draw_dist(t, q, x, tau, k, p, bonus=False):
    """P(token = y) of the draw at a rejection of x (or at the bonus position): cells of
    the oracle's cumulative draw weights in id order, each checked at its middle."""
    V = t.size
    args = (t, None if bonus else q, -1 if bonus else x, tau, k, p, np.inf)
    w = oracle.verify_unit(*args, 0.5, bonus=bonus, with_weights=True)["w_draw"]
    S = w.sum()
    assert S > 0
    c = np.concatenate([[0.0], np.cumsum(w)]) / S
    dist = np.zeros(V)
    for y in range(V):
        if w[y] <= 0:
            continue
        mid = 0.5 * (c[y] + c[y + 1])
        tok = oracle.verify_unit(*args, mid, bonus=bonus)["token"]
        assert tok == y, (y, tok)
        dist[y] = c[y + 1] - c[y]
    return dist


@pytest.mark.parametrize("V,tau,k,p,seed", CASES)
def test_first_token_distribution_is_exact(V, tau, k, p, seed):
    t, q = _rows(V, seed)
    P = oracle.filter_probs(t, tau, k, p)
    Qd = oracle.filter_probs(q, tau, k, p)
    acc_total = 0.0
    out = np.zeros(V)
    for x in range(V):
        if Qd[x] == 0.0:
            continue
        a = _accept_prob(t, q, x, tau, k, p)
        acc_total += Qd[x] * a
        out[x] += Qd[x] * a
        if a < 1.0:
            out += Qd[x] * (1.0 - a) * _draw_dist(t, q, x, tau, k, p)
    assert abs(acc_total - np.minimum(P, Qd).sum()) <= 1e-12
    np.testing.assert_allclose(out, P, rtol=0, atol=1e-12)


@pytest.mark.parametrize("V,tau,k,p,seed", CASES)
def test_one_hot_draft_distribution_is_exact(V, tau, k, p, seed):
    # a one-hot draft x (drawn by a greedy drafter, here with probability g(x) from an
    # arbitrary guess distribution): kept with probability p(x), else a draw from p
    # without x; the first token follows p whatever g is
    t, _ = _rows(V, seed)
    P = oracle.filter_probs(t, tau, k, p)
    g = np.linspace(1.0, 2.0, V)
    g /= g.sum()
    out = np.zeros(V)
    for x in range(V):
        r = oracle.verify_unit(t, None, x, tau, k, p, 0.5, 0.5, draw=False)
        assert r["pd"] == 1.0 and np.isclose(r["pt"], P[x], rtol=1e-12, atol=0)
        a = _accept_prob(t, None, x, tau, k, p) if P[x] > 0 else 0.0
        out[x] += g[x] * a
        if a < 1.0:
            d = _draw_dist(t, None, x, tau, k, p)
            assert d[x] == 0.0
            out += g[x] * (1.0 - a) * d
    np.testing.assert_allclose(out, P, rtol=0, atol=1e-12)


@pytest.mark.parametrize("V,tau,k,p,seed", CASES)
def test_bonus_draw_distribution_is_exact(V, tau, k, p, seed):
    t, _ = _rows(V, seed + 100)
    P = oracle.filter_probs(t, tau, k, p)
    np.testing.assert_allclose(_draw_dist(t, None, -1, tau, k, p, bonus=True), P, rtol=0,
                               atol=1e-12)


def test_verify_unit_matches_the_row_oracle():
    # the unit entry point with Philox's uniforms gives the row oracle's decisions
    V, B = 40, 30
    rng = np.random.default_rng(9)
    T = (rng.standard_normal((B, 2, V)) * 2).astype(np.float32)
    Q = (T[:, :1] + rng.standard_normal((B, 1, V))).astype(np.float32)
    d = rng.integers(0, V, (B, 1)).astype(np.int32)
    tau = np.full(B, 0.9, np.float32)
    k = np.full(B, 12, np.int32)
    p = np.full(B, 0.85, np.float32)
    r = oracle.verify_sample(T, Q, d, tau, k, p, seed=77)
    for b in range(B):
        ua, us = oracle.uniforms(77, b, 0)
        u = oracle.verify_unit(T[b, 0], Q[b, 0], int(d[b, 0]), float(tau[b]), 12, float(p[b]), ua,
                                us)
        assert u["pt"] == r["p_target"][b, 0] and u["pd"] == r["p_draft"][b, 0]
        assert u["accept"] == (r["num_accepted"][b] == 1)
        if not u["accept"]:
            assert u["token"] == r["out"][b, 0]
        else:
            ua, us = oracle.uniforms(77, b, 1)
            bo = oracle.verify_unit(T[b, 1], None, -1, float(tau[b]), 12, float(p[b]), ua, us,
                                    bonus=True)
            assert bo["token"] == r["out"][b, 1]
