"""GPU parity of spec_verify_sample against the CPU oracle.

The rule (tests/sample_parity.py): token ids and accepted counts are bit-exact, and
p_target / p_draft agree to 1e-5 relative on every unit, except where a floating-point
decision sits within the GPU's rounding of its boundary.  There the GPU's row must equal
the oracle's result on one of the sides (a top-p cut one group up or down, the
neighbouring inverse-CDF cell), and an accept decision may differ only where
|U - p/q| < 1e-5, in fewer than 1e-4 of each test's rows.  Every category is counted and
printed per test.
"""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import (WORKLOADS, Workload, f32_to_bf16_bits,
                                             make_verify_inputs)

from sample_parity import check

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def gpu_verify(x, T_dev=None, Q_dev=None, one_hot=False):
    B, D = x["d"].shape
    T = _dev(x["T"]) if T_dev is None else T_dev
    Q = None if one_hot else (_dev(x["Q"]) if Q_dev is None else Q_dev)
    out = torch.full((B, D + 1), -9, dtype=torch.int32, device=DEV)
    na = torch.full((B,), -9, dtype=torch.int32, device=DEV)
    pt = torch.full((B, D), -1.0, dtype=torch.float32, device=DEV)
    pd = torch.full((B, D), -1.0, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, T.shape[-1]), dtype=torch.uint8,
                     device=DEV)
    lib.spec_verify_sample(T, Q, _dev(x["d"]), _dev(x["tau"]), _dev(x.get("top_k")),
                           _dev(x.get("top_p")), x["seed"], out, na, pt, pd, ws, st)
    torch.cuda.synchronize()
    return dict(out=out.cpu().numpy(), num_accepted=na.cpu().numpy(), p_target=pt.cpu().numpy(),
                p_draft=pd.cpu().numpy(), status=int(st.item()))


def oracle_verify(x, rows=None, one_hot=False):
    return oracle.verify_sample_rows(x["T"], None if one_hot else x["Q"], x["d"], x["tau"],
                                     x.get("top_k"), x.get("top_p"), x["seed"], rows=rows)


def compare(g, o, x, rows=None, label="", one_hot=False):
    """Assert the parity rule (tests/sample_parity.py); returns the per-category counts."""
    return check(g, o, x, rows=rows, one_hot=one_hot, label=label)


# ---------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_full_size(name):
    w = WORKLOADS[name]
    if w.mode == "greedy":
        w = w.scaled(mode="sample", tau=0.9, top_k=40, top_p=0.95, greedy_frac=0.0)
    x = make_verify_inputs(w)
    g = gpu_verify(x)
    o = oracle_verify(x)
    assert g["status"] == o["status"] == 0
    compare(g, o, x, label=name)
    assert ((g["num_accepted"] >= 0) & (g["num_accepted"] <= w.D)).all()


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_serving_mix_more_seeds(seed):
    w = WORKLOADS["serve_b256_d3_v152k"].scaled(B=96, seed=seed, philox_seed=seed * 7)
    x = make_verify_inputs(w)
    compare(gpu_verify(x), oracle_verify(x), x, label=f"serve seed {seed}")


# ---------------------------------------------------------------- ragged sizes, filters

CASES = [
    # V, D, dtype, tau, k, p
    (16, 1, "f32", 1.0, 0, 1.0),
    (17, 2, "f32", 0.7, 5, 0.9),
    (33, 3, "bf16", 1.0, 8, 0.95),
    (1000, 2, "f32", 0.5, 1, 1.0),
    (4097, 5, "f32", 1.3, 0, 0.8),
    (4099, 3, "bf16", 0.9, 100, 0.6),
    (40001, 4, "f32", 0.8, 2000, 0.9),
    (65537, 2, "bf16", 1.0, 0, 0.97),
    (151936, 1, "f32", 2.0, 0, 0.5),
    (262147, 2, "bf16", 1.0, 64, 0.95),
]


@pytest.mark.parametrize("V,D,dtype,tau,k,p", CASES)
def test_ragged_and_filters(V, D, dtype, tau, k, p):
    w = Workload(name="c", B=6 if V > 60000 else 24, D=D, V=V, H=8, dtype=dtype, tau=tau,
                 top_k=k, top_p=p, t_std=3.0, q_noise=1.0, seed=V + D, philox_seed=V)
    x = make_verify_inputs(w)
    compare(gpu_verify(x), oracle_verify(x), x, label=f"V={V} D={D} {dtype} k={k} p={p}")


def test_mixed_rows_in_one_batch():
    # per-row temperature (0 = greedy), top-k and top-p all differ across the batch
    rng = np.random.default_rng(3)
    w = Workload(name="mix", B=48, D=3, V=20011, H=8, tau=1.0, t_std=3.0, q_noise=1.5, seed=9,
                 philox_seed=99)
    x = make_verify_inputs(w)
    x["tau"] = rng.choice([0.0, 0.3, 0.8, 1.5, 4.0], size=w.B).astype(np.float32)
    x["top_k"] = rng.choice([0, 1, 3, 50, 20011, 30000], size=w.B).astype(np.int32)
    x["top_p"] = rng.choice([1.0, 0.99, 0.9, 0.5, 1e-4], size=w.B).astype(np.float32)
    compare(gpu_verify(x), oracle_verify(x), x, label="mixed rows")


@pytest.mark.parametrize("p", [0.9999, 0.99999])
def test_top_p_near_one_uses_exact_search(p):
    # the boundary falls where the weights are below the binned range
    w = Workload(name="p1", B=8, D=2, V=30000, H=8, tau=0.25, top_p=p, t_std=3.0, q_noise=0.5,
                 seed=4, philox_seed=4)
    x = make_verify_inputs(w)
    compare(gpu_verify(x), oracle_verify(x), x, label=f"p={p}")


def test_large_k_and_flat_rows_use_exact_search():
    # k far beyond the binned range at a small temperature; and rows of one repeated value
    w = Workload(name="k", B=8, D=2, V=50000, H=8, tau=0.05, top_k=40000, top_p=0.9, t_std=3.0,
                 q_noise=0.5, seed=5, philox_seed=5)
    x = make_verify_inputs(w)
    compare(gpu_verify(x), oracle_verify(x), x, label="large k")
    w2 = Workload(name="flat", B=6, D=2, V=9000, H=8, dtype="bf16", tau=1.0, top_k=100,
                  top_p=0.5, seed=6, philox_seed=6)
    x2 = make_verify_inputs(w2)
    x2["T"][:] = f32_to_bf16_bits(np.float32(1.5))
    x2["T"][:, :, ::7] = f32_to_bf16_bits(np.float32(1.25))
    compare(gpu_verify(x2), oracle_verify(x2), x2, label="flat bf16")


@pytest.mark.parametrize("C", [2, 6, 16])
def test_top_k_bound_edge_cases(C, monkeypatch):
    # top-k rows with a small k gather every element at or above a lower bound on the k-th
    # largest logit: k on both sides of the largest k that takes the bound, the top logits
    # packed into the first CTA's slice (the bound then admits too many candidates, and the
    # exact search takes over), and logits on a coarse grid (many ties at the bound)
    monkeypatch.setenv("MTPSPEC_VERIFY_CLUSTER", str(C))
    w = Workload(name="kb", B=8, D=2, V=30011, H=8, tau=0.8, top_k=50, top_p=0.95, t_std=3.0,
                 q_noise=1.0, seed=30 + C, philox_seed=30 + C)
    x = make_verify_inputs(w)
    x["top_k"] = np.array([1, 2, 7, 64, 127, 128, 129, 50], np.int32)
    x["top_p"][5] = 1.0
    x["T"][1, :, :500] += 12.0
    x["Q"][1, :, :500] += 12.0
    x["T"][2] = np.round(x["T"][2] * 2.0) / 2.0
    x["Q"][2] = np.round(x["Q"][2] * 2.0) / 2.0
    compare(gpu_verify(x), oracle_verify(x), x, label=f"top-k bound C={C}")


def test_negative_infinity_and_degenerate_rows():
    w = Workload(name="ninf", B=12, D=2, V=5000, H=8, tau=1.0, top_k=30, top_p=0.9, seed=7,
                 philox_seed=7)
    x = make_verify_inputs(w)
    x["T"][:, :, 100:4000] = -np.inf
    x["Q"][:, :, 200:4500] = -np.inf
    x["T"][0] = -np.inf          # row 0: every target position is a point mass on id 0
    x["Q"][1] = -np.inf          # row 1: every draft position is a point mass on id 0
    x["d"][0] = 0
    x["d"][1, 0] = 0
    compare(gpu_verify(x), oracle_verify(x), x, label="-inf")


def test_invalid_draft_ids_and_bad_params_set_status():
    w = Workload(name="bad", B=6, D=3, V=3001, H=8, tau=1.0, top_p=0.9, seed=8, philox_seed=8)
    x = make_verify_inputs(w)
    x["d"][2, 1] = w.V
    x["d"][3, 0] = -5
    g = gpu_verify(x)
    o = oracle_verify(x)
    assert g["status"] & lib.STATUS_BAD_DRAFT_ID
    assert o["status"] & oracle.STATUS_BAD_DRAFT_ID
    compare(g, o, x, label="bad ids")
    assert g["num_accepted"][3] == 0 and g["p_target"][3, 0] == 0
    # a negative temperature is reported and the row is verified greedily
    x["tau"][4] = -1.0
    g = gpu_verify(x)
    assert g["status"] & lib.STATUS_BAD_PARAM
    go, gn, _ = oracle.verify_greedy(x["T"][4:5], x["d"][4:5])
    np.testing.assert_array_equal(g["out"][4], go[0])


def test_unaligned_rows():
    # V odd: rows start at arbitrary 4- or 2-byte offsets
    for dtype in ("f32", "bf16"):
        w = Workload(name="odd", B=10, D=3, V=12343, H=8, dtype=dtype, tau=0.9, top_k=64,
                     top_p=0.92, seed=10, philox_seed=10)
        x = make_verify_inputs(w)
        compare(gpu_verify(x), oracle_verify(x), x, label=f"odd {dtype}")


def test_deterministic_and_seed_sensitive():
    w = WORKLOADS["sample_b8_d3_v152k"]
    x = make_verify_inputs(w)
    a, b = gpu_verify(x), gpu_verify(x)
    for k in ("out", "num_accepted", "p_target", "p_draft"):
        np.testing.assert_array_equal(a[k], b[k])
    x2 = dict(x, seed=x["seed"] + 1)
    c = gpu_verify(x2)
    compare(c, oracle_verify(x2), x2, label="seed+1")


def test_margin_rows_are_rare():
    # many rows at a moderate vocabulary: rows whose accept margin is below 1e-5 stay under
    # 1e-4 of the rows (asserted by the rule on this test's rows alone)
    w = Workload(name="many", B=4000, D=3, V=2048, H=8, tau_range=(0.5, 1.2), top_k=200,
                 top_p=0.9, t_std=3.0, q_noise_range=(0.3, 2.0), seed=12, philox_seed=12)
    x = make_verify_inputs(w)
    c = compare(gpu_verify(x), oracle_verify(x), x, label="many rows")
    assert c["accept_margin_rows"] <= 1


@pytest.mark.parametrize("C", [2, 3, 5, 6, 7, 9, 10, 11, 16])
def test_cluster_sizes(C, monkeypatch):
    # every cluster size the launch can choose (odd ones split the candidate slots unevenly
    # and leave slices ragged) gives the oracle's results
    monkeypatch.setenv("MTPSPEC_VERIFY_CLUSTER", str(C))
    for dtype, k in (("f32", 0), ("bf16", 50)):
        w = Workload(name="cl", B=12, D=3, V=20011, H=8, dtype=dtype, tau_range=(0.5, 1.2),
                     top_k=k, top_p=0.9, t_std=3.0, q_noise_range=(0.3, 2.0), seed=20 + C,
                     philox_seed=20 + C)
        x = make_verify_inputs(w)
        compare(gpu_verify(x), oracle_verify(x), x, label=f"C={C} {dtype}")


@pytest.mark.parametrize("order", ["row", "position"])
@pytest.mark.parametrize("one_hot", [False, True])
def test_unit_orders(order, one_hot, monkeypatch):
    # both unit orders (row-major; position-major with the draws behind a rejected position
    # skipped) give the oracle's results, and the same outputs as each other
    monkeypatch.setenv("MTPSPEC_VERIFY_ORDER", order)
    w = Workload(name="ord", B=40, D=4, V=20011, H=8, tau_range=(0.5, 1.2), top_p=0.9,
                 t_std=3.0, q_noise_range=(0.3, 2.0), seed=31, philox_seed=31, greedy_frac=0.2)
    x = make_verify_inputs(w)
    got = gpu_verify(x, one_hot=one_hot)
    compare(got, oracle_verify(x, one_hot=one_hot), x, label=f"{order} one_hot={one_hot}",
            one_hot=one_hot)
    monkeypatch.setenv("MTPSPEC_VERIFY_ORDER", "row" if order == "position" else "position")
    other = gpu_verify(x, one_hot=one_hot)
    for key in got:
        np.testing.assert_array_equal(np.asarray(got[key]), np.asarray(other[key]), err_msg=key)


# ---------------------------------------------------------------- one-hot drafts

def _argmax_drafts(x):
    """The target's argmax at every draft position."""
    am = x["T"][:, :-1, :]
    if am.dtype == np.uint16:
        am = (am.astype(np.uint32) << 16).view(np.float32)
    return am.argmax(-1).astype(np.int32)


def _greedy_half(x, rng):
    """Half the drafts become the target's argmax, so that some of them are held."""
    am = _argmax_drafts(x)
    x["d"] = np.where(rng.random(x["d"].shape) < 0.5, am, x["d"]).astype(np.int32)
    return x


@pytest.mark.parametrize("V,D,dtype,tau,k,p", [
    (17, 2, "f32", 0.7, 5, 0.9),
    (4099, 3, "bf16", 0.9, 100, 0.6),
    (40001, 4, "f32", 0.8, 2000, 0.9),
    (151936, 3, "f32", 1.0, 0, 0.9),
    (262147, 2, "bf16", 1.0, 64, 0.95),
])
def test_one_hot_draft_mode(V, D, dtype, tau, k, p):
    # no draft logits: each draft is the point mass on its token
    w = Workload(name="oh", B=8 if V > 60000 else 24, D=D, V=V, H=8, dtype=dtype, tau=tau,
                 top_k=k, top_p=p, t_std=3.0, q_noise=1.0, seed=V + 7, philox_seed=V + 1)
    x = _greedy_half(make_verify_inputs(w), np.random.default_rng(V))
    g, o = gpu_verify(x, one_hot=True), oracle_verify(x, one_hot=True)
    assert g["status"] == o["status"] == 0
    compare(g, o, x, label=f"one-hot V={V} {dtype} k={k} p={p}", one_hot=True)
    if V < 60000:  # (over the large vocabularies even the argmax holds only a few percent)
        assert (g["num_accepted"] > 0).any()


def test_one_hot_draft_serving_mix():
    w = WORKLOADS["serve_b256_d3_v152k"].scaled(B=64, seed=41, philox_seed=43)
    x = _greedy_half(make_verify_inputs(w), np.random.default_rng(41))
    compare(gpu_verify(x, one_hot=True), oracle_verify(x, one_hot=True), x, label="one-hot serve",
            one_hot=True)


# ---------------------------------------------------------------- limits

@pytest.mark.parametrize("dtype,one_hot,V,k", [
    ("f32", False, 407552, 0),      # the largest vocabularies a cluster stages
    ("bf16", False, 815104, 50),
    ("f32", True, 651776, 50),
    ("bf16", True, 1303552, 0),
])
def test_maximum_vocabulary(dtype, one_hot, V, k):
    w = Workload(name="vmax", B=2, D=2, V=V, H=8, dtype=dtype, tau=1.0, top_k=k, top_p=0.9,
                 t_std=3.0, q_noise=1.0, seed=V % 1000, philox_seed=V)
    x = _greedy_half(make_verify_inputs(w), np.random.default_rng(V))
    g, o = gpu_verify(x, one_hot=one_hot), oracle_verify(x, one_hot=one_hot)
    assert g["status"] == o["status"] == 0
    compare(g, o, x, label=f"V={V} {dtype} one-hot={one_hot} k={k}", one_hot=one_hot)


@pytest.mark.parametrize("V,D,dtype", [(1000, 64, "f32"), (4099, 16, "bf16"),
                                       (151936, 16, "f32")])
def test_long_drafts(V, D, dtype):
    # peaked targets, and every draft of rows 0-1 (half of those of rows 2-3) the target's
    # argmax, so that long accepted prefixes occur (40 of 64 in one row at V = 1000)
    w = Workload(name="long", B=4, D=D, V=V, H=8, dtype=dtype, tau=0.5, top_k=0, top_p=0.95,
                 t_std=8.0, q_noise=1.0, seed=D + V, philox_seed=D)
    x = _greedy_half(make_verify_inputs(w), np.random.default_rng(D))
    x["d"][:2] = _argmax_drafts(x)[:2]
    g, o = gpu_verify(x), oracle_verify(x)
    assert o["num_accepted"].max() >= min(D, 9)
    assert g["status"] == o["status"] == 0
    compare(g, o, x, label=f"V={V} D={D} {dtype}")


WITHOUT_P = {
    # the serving mix (its sampled rows are top-p only)
    "serve": lambda: WORKLOADS["serve_b256_d3_v152k"].scaled(B=96, seed=61, philox_seed=67),
    # bf16 top-p rows, four drafts
    "topp_bf16": lambda: Workload(name="tpb", B=64, D=4, V=65537, H=8, dtype="bf16",
                                  tau_range=(0.5, 1.5), top_p=0.95, t_std=3.0,
                                  q_noise_range=(0.2, 1.5), seed=71, philox_seed=73),
    # drafts close to their targets: most drafts accepted
    "topp_close": lambda: Workload(name="tpc", B=128, D=3, V=30011, H=8, tau_range=(0.6, 1.2),
                                   top_p=0.8, t_std=3.0, q_noise=0.1, seed=81, philox_seed=83),
}


@pytest.mark.parametrize("case,one_hot", [("serve", False), ("serve", True),
                                          ("topp_bf16", False), ("topp_close", False)])
def test_outputs_without_probabilities_equal_those_with(case, one_hot):
    # without p_target and p_draft only the positions up to each row's first rejection are
    # read, so a unit behind a rejection the cluster already knows of is skipped, and a
    # draft whose acceptance is certain before the thresholds skips them; the tokens and
    # accepted counts must be the same, bit for bit, as when every position's
    # probabilities are requested (units position-major at these batch sizes)
    x = make_verify_inputs(WITHOUT_P[case]())
    if one_hot:
        x = _greedy_half(x, np.random.default_rng(61))
    B, D = x["d"].shape
    T, Q = _dev(x["T"]), (None if one_hot else _dev(x["Q"]))
    args = (T, Q, _dev(x["d"]), _dev(x["tau"]), None, _dev(x["top_p"]), x["seed"])
    ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, T.shape[-1]), dtype=torch.uint8,
                     device=DEV)

    def run(with_p):
        out = torch.full((B, D + 1), -9, dtype=torch.int32, device=DEV)
        na = torch.full((B,), -9, dtype=torch.int32, device=DEV)
        pt = torch.full((B, D), -1.0, device=DEV) if with_p else None
        pd = torch.full((B, D), -1.0, device=DEV) if with_p else None
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        lib.spec_verify_sample(*args, out, na, pt, pd, ws, st)
        torch.cuda.synchronize()
        return out.cpu().numpy(), na.cpu().numpy(), pt, pd, int(st.item())

    o1, n1, pt, pd, s1 = run(True)
    for _ in range(2):
        o0, n0, _, _, s0 = run(False)
        np.testing.assert_array_equal(o0, o1)
        np.testing.assert_array_equal(n0, n1)
        assert s0 == s1 == 0
    g = dict(out=o1, num_accepted=n1, p_target=pt.cpu().numpy(), p_draft=pd.cpu().numpy(), status=s1)
    rows = list(range(0, B, 3))
    compare(g, oracle_verify(x, rows=rows, one_hot=one_hot), x, rows=rows,
            label=f"{case} with probabilities, one_hot={one_hot}", one_hot=one_hot)
