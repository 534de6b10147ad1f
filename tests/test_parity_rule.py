"""The sampling parity rule (tests/sample_parity.py) on the CPU: it accepts the oracle's own
results and the other side of a decision that sits within the window, and rejects a row
that a wrong kernel would produce.  Rows stand in for GPU outputs; they are built from the
oracle's unit entry point with chosen top-p cuts and uniforms."""
import numpy as np
import pytest

import oracle
import sample_parity
from sample_parity import DELTA, check
from verify_spec_greedy_gb300.inputs import Workload, make_verify_inputs


def _as_gpu(o):
    return dict(out=o["out"].copy(), num_accepted=o["num_accepted"].copy(),
                p_target=o["p_target"].astype(np.float32),
                p_draft=o["p_draft"].astype(np.float32), status=o["status"])


def _inputs(B=40, V=64, D=1, p=0.9, k=0, seed=3):
    w = Workload(name="pr", B=B, D=D, V=V, H=8, tau_range=(0.6, 1.2), top_k=k, top_p=p,
                 t_std=2.0, q_noise=1.0, seed=seed, philox_seed=seed)
    return make_verify_inputs(w)


def _row(x, b, gts=None, uniforms=None, flip=None):
    """Row b as a kernel that keeps gts[j] top-p groups of T at position j (None: the
    rule) would emit, with the given uniforms per position (default: Philox's)."""
    T, Q, d = x["T"][b], x["Q"][b], x["d"][b]
    D = len(d)
    tau, k, p = sample_parity._row_params(x, b)
    uni = uniforms or [oracle.uniforms(x["seed"], b, j) for j in range(D + 1)]
    gts = gts or [-1] * (D + 1)
    out = np.full(D + 1, -1, np.int32)
    pt, pd = np.zeros(D, np.float32), np.zeros(D, np.float32)
    a = D
    for j in range(D):
        r = oracle.verify_unit(T[j], Q[j], int(d[j]), tau, k, p, *uni[j], gt=gts[j])
        pt[j], pd[j] = r["pt"], r["pd"]
        acc = r["accept"] if flip != j else not r["accept"]
        if not acc and a == D:
            a = j
            if flip == j:
                r = oracle.verify_unit(T[j], Q[j], int(d[j]), tau, k, p, np.inf, uni[j][1],
                                       gt=gts[j])
            out[j] = r["token"]
    if a == D:
        out[D] = oracle.verify_unit(T[D], None, -1, tau, k, p, *uni[D], bonus=True,
                                    gt=gts[D])["token"]
    out[:a] = d[:a]
    return out, a, pt, pd


def _replace(g, b, row):
    out, a, pt, pd = row
    g["out"][b], g["num_accepted"][b], g["p_target"][b], g["p_draft"][b] = out, a, pt, pd


def test_the_oracles_own_rows_pass():
    x = _inputs(D=3, k=20)
    o = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], x["top_k"], x["top_p"],
                                  x["seed"])
    c = check(_as_gpu(o), o, x, label="self")
    assert c["exact"] == c["rows"] == 40


def test_a_changed_token_fails():
    x = _inputs()
    o = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], None, x["top_p"], x["seed"])
    g = _as_gpu(o)
    b = 5
    a = g["num_accepted"][b]
    g["out"][b, a] = (g["out"][b, a] + 17) % 64
    with pytest.raises(AssertionError, match="unexplained"):
        check(g, o, x, label="changed token")


def _marginal_p(t_row, tau, K, gap):
    """A top-p value whose boundary after K groups sits `gap` below S_{K+1}."""
    P = oracle.filter_probs(t_row, tau, 0, 1.0)
    s = np.sort(P[P > 0])[::-1]
    return float(np.cumsum(s)[K - 1] - gap)


def test_a_cut_one_group_past_a_marginal_boundary_passes():
    x = _inputs()
    b = 7
    tau = float(x["tau"][b])
    x["top_p"][b] = _marginal_p(x["T"][b, 0], tau, 4, 3e-6)
    o = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], None, x["top_p"], x["seed"])
    rule = oracle.verify_unit(x["T"][b, 0], None, -1, tau, 0, float(x["top_p"][b]), 0.5, 0.5,
                              bonus=True, delta=DELTA)["cut_t"]
    assert rule[0] == 4 and rule[2] == 5
    g = _as_gpu(o)
    _replace(g, b, _row(x, b, gts=[5, -1]))
    assert not np.isclose(g["p_target"][b, 0], o["p_target"][b, 0], rtol=1e-5)
    c = check(g, o, x, label="alt cut")
    assert c["topp_alt_rows"] == 1 and c["exact"] == 39


def test_an_extra_group_on_a_clear_boundary_fails():
    x = _inputs()
    o = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], None, x["top_p"], x["seed"])
    g = _as_gpu(o)
    b = 11
    tau = float(x["tau"][b])
    cut = oracle.verify_unit(x["T"][b, 0], None, -1, tau, 0, float(x["top_p"][b]), 0.5, 0.5,
                             bonus=True, delta=DELTA)["cut_t"]
    assert cut[1] == cut[0] == cut[2]
    _replace(g, b, _row(x, b, gts=[cut[0] + 1, -1]))
    with pytest.raises(AssertionError, match="match no top-p cut"):
        check(g, o, x, label="extra group")


def test_an_accept_flip_outside_the_margin_fails():
    x = _inputs()
    o = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], None, x["top_p"], x["seed"])
    b = int(np.nonzero(o["margins"][:, 0, 0] > 1e-3)[0][0])
    g = _as_gpu(o)
    _replace(g, b, _row(x, b, flip=0))
    with pytest.raises(AssertionError, match="outside the margin"):
        check(g, o, x, label="flip")


def test_the_neighbouring_draw_at_a_cell_edge(monkeypatch):
    # uniforms chosen so that position 0 rejects and U_smp lands 2e-6 from a cell edge;
    # the neighbouring token passes, a token two cells away fails
    x = _inputs(B=16)
    for b in range(16):  # a row whose first draft can be rejected, with a wide residual
        T, Q, d = x["T"][b], x["Q"][b], x["d"][b]
        tau, k, p = sample_parity._row_params(x, b)
        r = oracle.verify_unit(T[0], Q[0], int(d[0]), tau, k, p, np.inf, 0.5, with_weights=True)
        w = r["w_draw"]
        if (w > 0).sum() >= 4 and r["ratio"] < 0.99:
            break
    c = np.cumsum(w) / w.sum()
    pos = [i for i in np.nonzero(w > 0)[0][:-1]]
    edge_id = pos[len(pos) // 2]
    u_smp = float(c[edge_id] - 2e-6)
    uni = [(0.9999999, u_smp), oracle.uniforms(x["seed"], b, 1)]
    real = oracle.uniforms
    monkeypatch.setattr(oracle, "uniforms",
                        lambda seed, row, pos: uni[pos] if row == b else real(seed, row, pos))
    exact = _row(x, b, uniforms=uni)
    assert exact[1] == 0 and exact[0][0] == edge_id
    o = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], None, x["top_p"], x["seed"])
    _replace(o, b, exact)
    o["margins"][b, 0, 0] = 1.0
    g = _as_gpu(o)
    nxt = int(np.nonzero(w[edge_id + 1:] > 0)[0][0]) + edge_id + 1
    g["out"][b, 0] = nxt
    cnt = check(g, o, x, label="cdf neighbour")
    assert cnt["cdf_alt_rows"] == 1
    far = int(np.nonzero(w[nxt + 1:] > 0)[0][0]) + nxt + 1
    g["out"][b, 0] = far
    with pytest.raises(AssertionError, match="allowed draws"):
        check(g, o, x, label="cdf far")
