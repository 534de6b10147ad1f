"""Pins of the oracle's speculative-sampling verification (page "MPT (MTP, Multi-Token
Prediction) 原理详解", section 三 stage 3; page "The decoding loop and MTP", "MTP
speculative decoding" item 3).

- lossless: with the draft drawn from q, the first emitted token follows the filtered
  target distribution p (chi-square over 20,000 trials, the trial count the second page
  names for its own check);
- per-draft acceptance rate min(1, p(x)/q(x)), overall sum_x min(p(x), q(x));
- a rejected draft is replaced by a draw from max(0, p - q) / R;
- special cases: a one-hot draft distribution is kept with probability p(x) and otherwise
  replaced by a draw from p without x; k = 1 and a vanishing temperature reduce to the
  greedy rule;
- every verification emits 1 to D+1 tokens;
- a decoding loop of repeated verifications (D = 3, drafts drawn from q) against a
  stationary target emits independent draws from p: non-overlapping pairs follow p x p.
"""
import numpy as np
import pytest
from scipy import stats

import oracle
from verify_spec_greedy_gb300.inputs import Workload, make_verify_inputs


def _rows(T1, Q1, B):
    T = np.ascontiguousarray(np.broadcast_to(T1, (B,) + T1.shape))
    Q = np.ascontiguousarray(np.broadcast_to(Q1, (B,) + Q1.shape))
    return T, Q


def _chi2_ok(counts, probs, alpha=1e-3):
    n = counts.sum()
    nz = probs > 0
    assert counts[~nz].sum() == 0
    exp = probs[nz] * n
    return stats.chisquare(counts[nz], exp).pvalue > alpha


def test_lossless_first_token_chi_square():
    V, N = 16, 20000
    rng = np.random.default_rng(11)
    t = (rng.standard_normal(V) * 1.5).astype(np.float32)
    q = (t + rng.standard_normal(V).astype(np.float32) * 1.2).astype(np.float32)
    tau, k, p = 0.8, 12, 0.9
    P = oracle.filter_probs(t, tau, k, p)
    Qd = oracle.filter_probs(q, tau, k, p)
    T1 = np.stack([t, t])          # D = 1: positions 0 and 1
    Q1 = q[None]
    T, Q = _rows(T1, Q1, N)
    d = rng.choice(V, size=(N, 1), p=Qd).astype(np.int32)
    r = oracle.verify_sample(T, Q, d, np.full(N, tau, np.float32), np.full(N, k, np.int32),
                             np.full(N, p, np.float32), seed=123)
    first = r["out"][:, 0]
    counts = np.bincount(first, minlength=V)
    assert _chi2_ok(counts, P)
    # when the draft held, the bonus token follows p at position 1
    held = r["num_accepted"] == 1
    assert held.sum() > 1000
    assert _chi2_ok(np.bincount(r["out"][held, 1], minlength=V), P)
    assert (r["out"][~held, 1] == -1).all()


def test_acceptance_rates_and_residual():
    V, N = 5, 6000
    t = np.log(np.array([0.4, 0.3, 0.15, 0.1, 0.05])).astype(np.float32)
    q = np.log(np.array([0.1, 0.5, 0.2, 0.05, 0.15])).astype(np.float32)
    P = oracle.filter_probs(t, 1.0)
    Qd = oracle.filter_probs(q, 1.0)
    T, Q = _rows(np.stack([t, t]), q[None], N)
    resid = np.maximum(P - Qd, 0)
    resid /= resid.sum()
    for x in range(V):
        d = np.full((N, 1), x, np.int32)
        r = oracle.verify_sample(T, Q, d, np.ones(N, np.float32), seed=1000 + x)
        acc = r["num_accepted"] == 1
        want = min(1.0, P[x] / Qd[x])
        sd = np.sqrt(want * (1 - want) / N) + 1e-9
        assert abs(acc.mean() - want) <= 4.5 * sd + 1e-12, (x, acc.mean(), want)
        np.testing.assert_allclose(r["p_target"][:, 0], P[x], rtol=1e-12)
        np.testing.assert_allclose(r["p_draft"][:, 0], Qd[x], rtol=1e-12)
        if (~acc).sum() > 200:
            counts = np.bincount(r["out"][~acc, 0], minlength=V)
            assert _chi2_ok(counts, resid)
    # overall acceptance with the draft drawn from q is sum(min(p, q))
    rng = np.random.default_rng(5)
    d = rng.choice(V, size=(N, 1), p=Qd).astype(np.int32)
    r = oracle.verify_sample(T, Q, d, np.ones(N, np.float32), seed=77)
    want = np.minimum(P, Qd).sum()
    assert abs((r["num_accepted"] == 1).mean() - want) <= 4.5 * np.sqrt(want * (1 - want) / N)


def test_one_hot_draft_distribution():
    # q is a point mass on x: the guess is kept with probability p(x) and otherwise the
    # token comes from the other candidates in proportion to p
    V, N, x = 8, 20000, 2
    rng = np.random.default_rng(9)
    t = (rng.standard_normal(V) * 1.0).astype(np.float32)
    q = np.full(V, -np.inf, np.float32)
    q[x] = 0.0
    P = oracle.filter_probs(t, 1.0)
    T, Q = _rows(np.stack([t, t]), q[None], N)
    r = oracle.verify_sample(T, Q, np.full((N, 1), x, np.int32), np.ones(N, np.float32), seed=4)
    acc = r["num_accepted"] == 1
    assert abs(acc.mean() - P[x]) <= 4.5 * np.sqrt(P[x] * (1 - P[x]) / N)
    others = P.copy()
    others[x] = 0
    others /= others.sum()
    assert _chi2_ok(np.bincount(r["out"][~acc, 0], minlength=V), others)


def test_top_k_one_and_zero_temperature_reduce_to_greedy():
    rng = np.random.default_rng(21)
    B, D, V = 200, 3, 64
    T = (rng.standard_normal((B, D + 1, V)) * 2).astype(np.float32)
    Q = (T[:, :D] + rng.standard_normal((B, D, V)).astype(np.float32)).astype(np.float32)
    # drafts: the draft model's argmax, or the target's argmax, or random ids
    choice = rng.integers(0, 3, (B, D))
    d = np.where(choice == 0, Q.argmax(-1), np.where(choice == 1, T[:, :D].argmax(-1),
                                                      rng.integers(0, V, (B, D)))).astype(np.int32)
    g_out, g_acc, _ = oracle.verify_greedy(T, d)
    r = oracle.verify_sample(T, Q, d, np.full(B, 0.9, np.float32), np.ones(B, np.int32), seed=3)
    np.testing.assert_array_equal(r["out"], g_out)
    np.testing.assert_array_equal(r["num_accepted"], g_acc)
    z = oracle.verify_sample(T, Q, d, np.zeros(B, np.float32), seed=3)
    np.testing.assert_array_equal(z["out"], g_out)
    # a vanishing temperature with drafts taken from the draft model's argmax
    d2 = np.where(choice == 0, Q.argmax(-1), T[:, :D].argmax(-1)).astype(np.int32)
    g2, a2, _ = oracle.verify_greedy(T, d2)
    s2 = oracle.verify_sample(T, Q, d2, np.full(B, 1e-4, np.float32), seed=8)
    np.testing.assert_array_equal(s2["out"], g2)
    np.testing.assert_array_equal(s2["num_accepted"], a2)


def test_emitted_bounds_and_format_on_workload():
    w = Workload(name="t", B=40, D=4, V=300, H=8, tau_range=(0.5, 1.2), greedy_frac=0.25,
                 top_k=20, top_p=0.9, seed=2, philox_seed=2)
    x = make_verify_inputs(w)
    r = oracle.verify_sample(x["T"], x["Q"], x["d"], x["tau"], x["top_k"], x["top_p"], x["seed"])
    for b in range(w.B):
        a = r["num_accepted"][b]
        assert 0 <= a <= w.D
        assert r["out"][b, :a].tolist() == x["d"][b, :a].tolist()
        assert 0 <= r["out"][b, a] < w.V
        assert (r["out"][b, a + 1:] == -1).all()
    # rows are independent: a subset with the right row offset reproduces the batch
    sub = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], x["top_k"], x["top_p"],
                                    x["seed"], rows=[3, 17, 39])
    np.testing.assert_array_equal(sub["out"], r["out"][[3, 17, 39]])


def test_invalid_draft_rejected_and_flagged():
    rng = np.random.default_rng(0)
    T = rng.standard_normal((2, 3, 10)).astype(np.float32)
    Q = rng.standard_normal((2, 2, 10)).astype(np.float32)
    d = np.array([[10, 1], [1, -5]], np.int32)
    r = oracle.verify_sample(T, Q, d, np.ones(2, np.float32), seed=0)
    assert r["status"] == oracle.STATUS_BAD_DRAFT_ID
    assert r["num_accepted"][0] == 0
    assert r["p_target"][0, 0] == 0 and r["p_draft"][0, 0] == 0


def test_draft_outside_draft_support_is_always_accepted():
    # d is in the target's top-k but outside the draft's top-k: q(d) = 0 and p(d) > 0,
    # so min(1, p/q) = 1 and the draft is kept in every trial
    # q's top-3 is {0, 3, 2}; id 1 misses it by a hair, so the ratio it would have had
    # inside the support is about 0.39, far from 1
    V, N = 6, 3000
    t = np.array([3.0, 1.0, -5.0, -5.0, -6.0, -6.0], np.float32)
    q = np.array([3.0, 2.9, 2.95, 2.99, -6.0, -6.0], np.float32)
    T, Q = _rows(np.stack([t, t]), q[None], N)
    r = oracle.verify_sample(T, Q, np.full((N, 1), 1, np.int32), np.ones(N, np.float32),
                             np.full(N, 3, np.int32), seed=5)
    assert (r["p_draft"][:, 0] == 0).all() and (r["p_target"][:, 0] > 0).all()
    assert (r["num_accepted"] == 1).all()
    # and a draft outside the target's support is rejected in every trial
    r = oracle.verify_sample(T, Q, np.full((N, 1), 4, np.int32), np.ones(N, np.float32),
                             np.full(N, 3, np.int32), seed=6)
    assert (r["num_accepted"] == 0).all()


def test_draws_take_the_inverse_cdf_in_ascending_id_order():
    # equal logits make p uniform over the n kept ids, so the ascending-order inverse
    # CDF picks kept id number floor(U_smp * n); U_smp is pinned by the Philox vectors
    N, V = 500, 10
    t = np.zeros(V, np.float32)
    t[[1, 4, 6, 7]] = 1.0          # kept ids under top-k = 4, in ascending order
    T, Q = _rows(np.stack([t, t]), t[None], N)
    d = np.full((N, 1), 4, np.int32)
    r = oracle.verify_sample(T, Q, d, np.ones(N, np.float32), np.full(N, 4, np.int32), seed=99)
    assert (r["num_accepted"] == 1).all()  # p = q: every draft holds
    kept = [1, 4, 6, 7]
    for b in range(N):
        us = oracle.uniforms(99, b, 1)[1]
        assert r["out"][b, 1] == kept[int(us * 4)]


def test_all_negative_infinity_rows_are_point_masses_on_id_0():
    V, N = 6, 2000
    t = np.full(V, -np.inf, np.float32)
    q = np.array([0.0, 1.0, -1.0, 0.5, -np.inf, 2.0], np.float32)
    T, Q = _rows(np.stack([t, t]), q[None], N)
    Qd = oracle.filter_probs(q, 1.0)
    # draft 0: p(0) = 1 >= q(0), always kept; any other draft: outside p's support
    r = oracle.verify_sample(T, Q, np.zeros((N, 1), np.int32), np.ones(N, np.float32), seed=1)
    assert (r["num_accepted"] == 1).all() and (r["out"][:, 1] == 0).all()
    np.testing.assert_allclose(r["p_draft"][:, 0], Qd[0])
    r = oracle.verify_sample(T, Q, np.full((N, 1), 3, np.int32), np.ones(N, np.float32), seed=2)
    assert (r["num_accepted"] == 0).all() and (r["out"][:, 0] == 0).all()
    # the draft side degenerate: q = point mass on 0, accepted with probability p(0)
    T2, Q2 = _rows(np.stack([q, q]), t[None], N)
    r = oracle.verify_sample(T2, Q2, np.zeros((N, 1), np.int32), np.ones(N, np.float32), seed=3)
    want = oracle.filter_probs(q, 1.0)[0]
    assert abs((r["num_accepted"] == 1).mean() - want) < 4.5 * np.sqrt(want * (1 - want) / N)


def test_one_hot_mode_equals_point_mass_draft_rows():
    # without draft logits the drafter's distribution is the point mass on its token: the
    # same verification as draft rows of -inf but 0 at the token (same uniforms, same
    # expressions), and q(d) = 1
    rng = np.random.default_rng(21)
    B, D, V = 40, 3, 300
    T = (rng.standard_normal((B, D + 1, V)) * 2.0).astype(np.float32)
    d = rng.integers(0, V, (B, D)).astype(np.int32)
    # half the drafts are the target's argmax, so that some are held
    am = T[:, :D, :].argmax(-1).astype(np.int32)
    d = np.where(rng.random((B, D)) < 0.5, am, d).astype(np.int32)
    Q = np.full((B, D, V), -np.inf, np.float32)
    np.put_along_axis(Q, d[:, :, None], 0.0, axis=2)
    tau = rng.uniform(0.5, 1.5, B).astype(np.float32)
    tk = rng.choice([0, 5, 40], B).astype(np.int32)
    tp = rng.choice([1.0, 0.9, 0.6], B).astype(np.float32)
    a = oracle.verify_sample(T, Q, d, tau, tk, tp, seed=3)
    b = oracle.verify_sample(T, None, d, tau, tk, tp, seed=3)
    np.testing.assert_array_equal(a["out"], b["out"])
    np.testing.assert_array_equal(a["num_accepted"], b["num_accepted"])
    np.testing.assert_array_equal(a["p_target"], b["p_target"])
    np.testing.assert_array_equal(b["p_draft"], np.ones((B, D)))
    assert 0 < (b["num_accepted"] > 0).sum() < B


def test_one_hot_mode_lossless_and_acceptance():
    # a fixed drafted token x: kept with probability p(x); the first emitted token follows
    # p whatever x is (chi-square over 20,000 trials)
    V, N = 16, 20000
    rng = np.random.default_rng(31)
    t = (rng.standard_normal(V) * 1.5).astype(np.float32)
    tau, k, p = float(np.float32(0.9)), 10, float(np.float32(0.9))  # as the verify sees them
    P = oracle.filter_probs(t, tau, k, p)
    x = int(np.argsort(-P)[1])    # a likely but not the likeliest token
    T = np.ascontiguousarray(np.broadcast_to(np.stack([t, t]), (N, 2, V)))
    r = oracle.verify_sample(T, None, np.full((N, 1), x, np.int32), np.full(N, tau, np.float32),
                             np.full(N, k, np.int32), np.full(N, p, np.float32), seed=17)
    acc = r["num_accepted"] == 1
    assert abs(acc.mean() - P[x]) <= 4.5 * np.sqrt(P[x] * (1 - P[x]) / N)
    assert _chi2_ok(np.bincount(r["out"][:, 0], minlength=V), P)
    np.testing.assert_allclose(r["p_target"][:, 0], P[x], rtol=1e-12)
    # an id outside the vocabulary is rejected and flagged; the token then follows p
    r = oracle.verify_sample(T[:4000], None, np.full((4000, 1), V, np.int32),
                             np.full(4000, tau, np.float32), np.full(4000, k, np.int32),
                             np.full(4000, p, np.float32), seed=18)
    assert r["status"] & oracle.STATUS_BAD_DRAFT_ID
    assert (r["num_accepted"] == 0).all() and (r["p_draft"] == 0).all()
    assert _chi2_ok(np.bincount(r["out"][:, 0], minlength=V), P)


def test_emitted_stream_is_iid_from_the_target():
    # a stationary target (every position has the same filtered distribution p) and a
    # drafter that draws each guess from q: a decoding loop that verifies again and again
    # must emit a stream of independent draws from p.  Non-overlapping pairs of the stream
    # are checked against p x p, which a wrong residual or bonus at any position, or a
    # uniform shared between positions, would fail.  top-k 4 leaves p > 0 on an id that q
    # never proposes, so the residual must supply it.
    V, D, B, calls = 5, 3, 400, 40
    rng = np.random.default_rng(21)
    t = np.array([1.0, 0.3, -0.4, 0.6, -1.0], np.float32)
    q = np.array([0.2, 0.9, -0.1, -0.3, 0.5], np.float32)
    tau, k, p = 1.0, 4, 1.0
    P = oracle.filter_probs(t, tau, k, p)
    Qd = oracle.filter_probs(q, tau, k, p)
    assert P[3] > 0 and Qd[3] == 0
    T, Q = _rows(np.stack([t] * (D + 1)), np.stack([q] * D), B)
    streams = [[] for _ in range(B)]
    for c in range(calls):
        d = rng.choice(V, size=(B, D), p=Qd).astype(np.int32)
        r = oracle.verify_sample(T, Q, d, np.full(B, tau, np.float32), np.full(B, k, np.int32),
                                 np.full(B, p, np.float32), seed=1000 + c)
        for b in range(B):
            streams[b].extend(int(x) for x in r["out"][b] if x >= 0)
    marg = np.zeros(V, np.int64)
    pairs = np.zeros((V, V), np.int64)
    for s in streams:
        a = np.array(s[: len(s) // 2 * 2])
        marg += np.bincount(a, minlength=V)
        np.add.at(pairs, (a[0::2], a[1::2]), 1)
    assert pairs.sum() > 12000
    assert _chi2_ok(marg, P)
    assert _chi2_ok(pairs.ravel(), np.outer(P, P).ravel())
