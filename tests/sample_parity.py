"""The parity rule for sampling verification: the GPU's rows against the oracle's.

Token ids and accepted counts must be bit-exact, except where a floating-point decision
sits so close to its boundary that the GPU's fp32 arithmetic may land on either side.
There the GPU's row must equal the oracle's result for one of the other sides, which the
oracle computes itself (``oracle.verify_unit``); nothing is excused outright:

- **top-p boundary** ("The decoding loop and MTP", "Why a hand-written decoding loop": the
  nucleus is the smallest top set whose mass reaches p): group g of equal logits stays
  when the mass S_g strictly above it is < p.  A cut after g groups is allowed when
  S_g < p + DELTA and S_{g+1} >= p - DELTA.  The GPU's p(d) and q(d) of the unit must
  match (1e-5 relative) the oracle's under the cut it is taken to have used, and its
  accept decision and draw are then checked under that cut.
- **inverse-CDF draw** ("MPT (MTP, Multi-Token Prediction) 原理详解", section 三 stage 3:
  the replacement drawn from the residual): the drawn id must be the oracle's, or the
  neighbouring id with positive weight when U*R lies within DELTA*R of the shared edge.
- **accept test** (same section: accept when U <= p/q): a decision opposite to the
  oracle's is allowed only where |U - p/q| < ACC_MARGIN, the tolerance stated for this
  path.  Rows holding such a unit are counted, and must stay below 1e-4 of the rows of
  each test (at least one row is allowed in a test).

DELTA is a bound on the GPU's rounding, not a budget.  The GPU forms every weight as
2^(x*c - m*c) in fp32: the exponent carries an absolute error of a few ulp of numbers up
to ~30 (about 4e-6) and ex2.approx adds ~2^-22 relative, so every weight and every sum of
weights is within ~3e-6 relative of its exact value, and a normalised mass S <= 1 within
~6e-6.  DELTA = 1e-5 covers that with room to spare; a kernel that kept one group too
many, dropped one, or drew the neighbouring token anywhere else fails.
"""
from __future__ import annotations

import math

import numpy as np

import oracle

DELTA = 1e-5
ACC_MARGIN = 1e-5
P_RTOL = 1e-5
P_ATOL = 1e-30


def _close(a, b):
    return abs(float(a) - float(b)) <= P_RTOL * abs(float(b)) + P_ATOL


def _row_params(x, b):
    tau = float(x["tau"][b])
    k = int(x["top_k"][b]) if x.get("top_k") is not None else 0
    p = float(x["top_p"][b]) if x.get("top_p") is not None else 1.0
    return tau, k, p


def _match_cut(fn, lo, hi, want):
    """Cut counts g in [lo, hi] whose probability fn(g) matches want: fn is 0 below the group
    of the draft token and decreasing from it, so a bisection finds the group's first cut
    and another the matching value; returns up to three candidates around the match."""
    if hi - lo <= 4:
        return [g for g in range(lo, hi + 1) if _close(want, fn(g))]
    if want == 0.0:
        return [lo] if _close(0.0, fn(lo)) else []
    a, b = lo, hi   # first cut keeping the draft token
    if fn(b) == 0.0:
        return []
    while a < b:
        m = (a + b) // 2
        if fn(m) > 0.0:
            b = m
        else:
            a = m + 1
    a, b = a, hi    # decreasing from here: the last cut whose value is >= want
    while a < b:
        m = (a + b + 1) // 2
        if fn(m) >= want * (1 - P_RTOL):
            a = m
        else:
            b = m - 1
    return [g for g in (a - 1, a, a + 1) if lo <= g <= hi and _close(want, fn(g))]


def _alternatives(t_row, q_row, d, tau, k, p, ua, us, gpt=None, gpd=None):
    """(gt, gq, result) for the top-p cuts within DELTA, the rule's first; when the window
    holds many cuts (p near 1), only those whose probabilities match the GPU's."""
    base = oracle.verify_unit(t_row, q_row, d, tau, k, p, ua, us, draw=False, delta=DELTA)
    rule_t = base["cut_t"][0]
    rule_q = base["cut_q"][0] if q_row is not None else -1
    out = [(rule_t, rule_q, base)]
    gts = list(range(base["cut_t"][1], base["cut_t"][2] + 1))
    gqs = list(range(base["cut_q"][1], base["cut_q"][2] + 1)) if q_row is not None else [-1]
    if gpt is not None and (len(gts) > 5 or len(gqs) > 5):
        cache = {}

        def unit(gt, gq):
            if (gt, gq) not in cache:
                cache[(gt, gq)] = oracle.verify_unit(t_row, q_row, d, tau, k, p, ua, us,
                                                     draw=False, gt=gt, gq=gq)
            return cache[(gt, gq)]
        if len(gts) > 5:
            gts = _match_cut(lambda g: unit(g, rule_q)["pt"], gts[0], gts[-1], float(gpt))
        if len(gqs) > 5 and q_row is not None:
            gqs = _match_cut(lambda g: unit(rule_t, g)["pd"], gqs[0], gqs[-1], float(gpd))
    for gt in gts:
        for gq in gqs:
            if gt == out[0][0] and gq == out[0][1]:
                continue
            r = oracle.verify_unit(t_row, q_row, d, tau, k, p, ua, us, draw=False, gt=gt, gq=gq)
            out.append((gt, gq, r))
    return out


def _allowed_tokens(r):
    toks = {r["token"]}
    if r["cdf_lo"] < DELTA and r["tok_prev"] >= 0:
        toks.add(r["tok_prev"])
    if r["cdf_hi"] < DELTA and r["tok_next"] >= 0:
        toks.add(r["tok_next"])
    return toks


def _check_row(gout, gna, gpt, gpd, x, b, one_hot):
    """Explain one GPU row that differs from the oracle's exact result.  Returns the
    categories it used, or a string saying why it cannot be explained."""
    T = x["T"][b]
    Q = None if one_hot else x["Q"][b]
    d = x["d"][b]
    D = len(d)
    tau, k, p = _row_params(x, b)
    seed = x["seed"]
    used = set()
    matched = []
    for j in range(D):
        ua, us = oracle.uniforms(seed, b, j)
        alts = _alternatives(T[j], None if Q is None else Q[j], int(d[j]), tau, k, p, ua, us,
                             gpt[j], gpd[j])
        m = [a for a in alts if _close(gpt[j], a[2]["pt"]) and _close(gpd[j], a[2]["pd"])]
        if not m:
            return (f"position {j}: p_target {gpt[j]:.9g} / p_draft {gpd[j]:.9g} match no top-p "
                    f"cut within the window (the rule gives {alts[0][2]['pt']:.9g} / "
                    f"{alts[0][2]['pd']:.9g}, cuts {alts[0][2]['cut_t']} {alts[0][2]['cut_q']})")
        if m[0] is not alts[0]:
            used.add("topp")
        matched.append((m, ua, us))
    a = int(gna)
    if not 0 <= a <= D:
        return f"accepted count {a} outside [0, {D}]"
    for j in range(a):
        m = matched[j][0]
        if not any(r["accept"] for _, _, r in m):
            if not any(r["acc_margin"] < ACC_MARGIN for _, _, r in m):
                return f"position {j} accepted on the GPU, rejected by the oracle outside the margin"
            used.add("accept")
    if a < D:
        m, ua, us = matched[a]
        if not any(not r["accept"] for _, _, r in m):
            if not any(r["acc_margin"] < ACC_MARGIN for _, _, r in m):
                return f"position {a} rejected on the GPU, accepted by the oracle outside the margin"
            used.add("accept")
        toks, exact_tok = set(), None
        for gt, gq, r in m:
            if r["accept"] and not r["acc_margin"] < ACC_MARGIN:
                continue
            # the draw under this cut, with the accept test forced to reject
            rr = oracle.verify_unit(T[a], None if Q is None else Q[a], int(d[a]), tau, k, p,
                                    math.inf, us, draw=True, gt=gt, gq=gq)
            if exact_tok is None:
                exact_tok = rr["token"]
            toks |= _allowed_tokens(rr)
    else:
        ua, us = oracle.uniforms(seed, b, D)
        base = oracle.verify_unit(T[D], None, -1, tau, k, p, ua, us, bonus=True, delta=DELTA)
        exact_tok = base["token"]
        toks = _allowed_tokens(base)
        lo_, hi_ = base["cut_t"][1], base["cut_t"][2]
        # the bonus has no probability to match: every cut of a narrow window, else the
        # window's ends and the rule's neighbours
        cuts = range(lo_, hi_ + 1) if hi_ - lo_ <= 8 else sorted(
            {lo_, lo_ + 1, hi_ - 1, hi_, base["cut_t"][0] - 1, base["cut_t"][0] + 1})
        for gt in cuts:
            if gt != base["cut_t"][0] and lo_ <= gt <= hi_:
                toks |= _allowed_tokens(oracle.verify_unit(T[D], None, -1, tau, k, p, ua, us,
                                                           bonus=True, gt=gt))
    tok = int(gout[a])
    if tok not in toks:
        return f"token {tok} at position {a} is not among the allowed draws {sorted(toks)}"
    if tok != exact_tok:
        used.add("cdf")
    want = np.full(D + 1, -1, np.int32)
    want[:a] = d[:a]
    want[a] = tok
    if not np.array_equal(np.asarray(gout), want):
        return f"output {list(gout)} is not the accepted drafts then the token: {list(want)}"
    return used


def check(g, o, x, rows=None, one_hot=False, label=""):
    """Assert the parity rule on GPU outputs g against the oracle's exact outputs o (both
    restricted to ``rows`` of the inputs x, in that order).  Returns the counts per
    category and prints them."""
    B = len(o["out"])
    rows = list(range(B)) if rows is None else [int(r) for r in rows]
    if len(g["out"]) != B:
        g = {kk: (v[rows] if isinstance(v, np.ndarray) else v) for kk, v in g.items()}
    D = g["p_target"].shape[1]
    counts = dict(rows=B, exact=0, topp_alt_rows=0, cdf_alt_rows=0, accept_flip_rows=0,
                  accept_margin_rows=0)
    acc_lit = (o["margins"][:, :D, 0] < ACC_MARGIN).any(1)
    counts["accept_margin_rows"] = int(acc_lit.sum())
    errors = []
    for i, b in enumerate(rows):
        same = (np.array_equal(g["out"][i], o["out"][i])
                and int(g["num_accepted"][i]) == int(o["num_accepted"][i])
                and all(_close(g["p_target"][i, j], o["p_target"][i, j])
                        and _close(g["p_draft"][i, j], o["p_draft"][i, j]) for j in range(D)))
        if same:
            counts["exact"] += 1
            continue
        tau = float(x["tau"][b])
        if not tau > 0:
            errors.append(f"row {b} (greedy) differs: gpu {g['out'][i]} oracle {o['out'][i]}")
            continue
        r = _check_row(g["out"][i], g["num_accepted"][i], g["p_target"][i], g["p_draft"][i], x,
                       b, one_hot)
        if isinstance(r, str):
            errors.append(f"row {b}: {r}; gpu {list(g['out'][i])} oracle {list(o['out'][i])}")
            continue
        counts["topp_alt_rows"] += "topp" in r
        counts["cdf_alt_rows"] += "cdf" in r
        counts["accept_flip_rows"] += "accept" in r
    print(f"[{label}] parity: {counts}")
    assert not errors, f"{label}: {len(errors)} rows unexplained, e.g. " + "; ".join(errors[:3])
    assert counts["accept_margin_rows"] <= max(1, 1e-4 * B), (
        f"{label}: {counts['accept_margin_rows']} of {B} rows hold an accept margin < "
        f"{ACC_MARGIN}")
    assert counts["accept_flip_rows"] <= counts["accept_margin_rows"]
    return counts
