"""GPU parity of mtp_lm_head_greedy (the draft output layer with the greedy pick) against
the CPU oracle.  The GPU sums the bf16 products in fp32, the oracle in double, so the pick
is compared where it is unique: with E_v = H * 2^-23 * sum_k |W[v, k] x_k| (a bound on an
fp32 sum of H exact products in any order, rounding or truncating), the GPU id must lie
in {v : exact_v >= exact_max - E_max - E_v}, and must equal the oracle's id when that set
has one member; its reported logit must lie within E of the exact one."""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import make_lm_head_input

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def gpu_lm_head(x, norm=True, hidden_dev=None, W_dev=None):
    M, H, V = x["M"], x["H"], x["V"]
    ids = torch.full((M,), -7, dtype=torch.int32, device=DEV)
    lg = torch.full((M,), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(lib.mtp_lm_head_greedy_workspace_bytes(M, H, V), dtype=torch.uint8, device=DEV)
    lib.mtp_lm_head_greedy(_bf(x["hidden"]) if hidden_dev is None else hidden_dev,
                           _bf(x["W"]) if W_dev is None else W_dev, ids,
                           norm_w=_bf(x["norm_w"]) if norm else None, eps=x["eps"],
                           out_logit=lg, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return ids.cpu().numpy(), lg.cpu().numpy()


def check(x, ids, lg, toks, norm=True):
    H = x["H"]
    exact, ad = oracle.lm_head_logits(x["hidden"], x["W"], toks,
                                      norm_w=x["norm_w"] if norm else None, eps=x["eps"],
                                      with_absdot=True)
    E = H * 2.0 ** -23 * ad
    unique = 0
    for i, t in enumerate(toks):
        e, b = exact[i], E[i]
        a = int(np.argmax(e))
        amb = np.flatnonzero(e >= e[a] - b[a] - b)
        g = int(ids[t])
        assert g in amb, (t, g, a, e[g] - e[a])
        if amb.size == 1:
            assert g == a
            unique += 1
        assert abs(float(lg[t]) - e[g]) <= b[g] + 1e-30, (t, lg[t], e[g])
    return unique


@pytest.mark.parametrize("M,H,V,norm", [
    (1, 64, 1000, False), (2, 8, 300, True), (5, 128, 4099, True), (16, 256, 32768, False),
    (17, 136, 3000, True), (33, 512, 20000, True), (64, 1024, 12345, False),
    (100, 384, 9000, True), (129, 256, 5000, False), (200, 1024, 50000, False),
    (256, 512, 7000, True), (300, 256, 10000, True), (700, 128, 2000, False),
    (3, 64, 1000003, True), (2, 64, 8388480, True)])
def test_parity_small(M, H, V, norm):
    x = make_lm_head_input(M, H, V, seed=M * 131 + H + V)
    ids, lg = gpu_lm_head(x, norm)
    toks = np.arange(M) if M * V * H <= 6e9 else np.linspace(0, M - 1, 24).astype(np.int64)
    unique = check(x, ids, lg, toks, norm)
    assert unique >= 0.8 * len(toks)


def test_ties_take_the_lowest_id():
    # a row copied to a lower and to a higher id in other vocabulary tiles: the copies give
    # the same fp32 sums, so the pick must be the lowest of the three ids
    M, H, V = 8, 256, 3000
    x = make_lm_head_input(M, H, V, seed=5)
    ids0, _ = gpu_lm_head(x, norm=False)
    W = x["W"].copy()
    t = 3
    a = int(ids0[t])
    W[(a + 1000) % V] = W[a]
    W[(a + 2000) % V] = W[a]
    x2 = dict(x, W=W)
    ids, _ = gpu_lm_head(x2, norm=False)
    assert ids[t] == min(a, (a + 1000) % V, (a + 2000) % V)


def test_vocabulary_and_token_tails():
    # V just past a 128-row tile, M just past a token tile, H not a multiple of 64
    for M, H, V in [(257, 72, 129), (1, 8, 1), (3, 8, 2), (65, 520, 257)]:
        x = make_lm_head_input(M, H, V, seed=M + V)
        ids, lg = gpu_lm_head(x)
        assert ((ids >= 0) & (ids < V)).all()
        check(x, ids, lg, np.arange(M))


def test_zero_tokens_enqueue_nothing():
    w = torch.empty((10, 64), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    ids = torch.empty(0, dtype=torch.int32, device=DEV)
    n0 = lib.mtpspec_launch_count()
    lib.mtp_lm_head_greedy(h, w, ids)
    assert lib.mtpspec_launch_count() == n0


@pytest.mark.parametrize("M,H,V", [(256, 4096, 151936), (64, 7168, 129280)])
def test_parity_full_size_sampled_tokens(M, H, V):
    # the serving workload's draft step (one token per row) and the large-hidden head, at
    # full size; the oracle checks a spread of tokens
    x = make_lm_head_input(M, H, V, seed=H + V, w_std=0.02)
    ids, lg = gpu_lm_head(x)
    assert ((ids >= 0) & (ids < V)).all()
    toks = np.unique(np.linspace(0, M - 1, 5).astype(np.int64))
    check(x, ids, lg, toks)


def gpu_topk(x, k, norm=True):
    M, H, V = x["M"], x["H"], x["V"]
    ids = torch.full((M, k), -7, dtype=torch.int32, device=DEV)
    lg = torch.full((M, k), float("nan"), dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(lib.mtp_lm_head_topk_workspace_bytes(M, H, V), dtype=torch.uint8, device=DEV)
    lib.mtp_lm_head_topk(_bf(x["hidden"]), _bf(x["W"]), ids, norm_w=_bf(x["norm_w"]) if norm else None,
                         eps=x["eps"], out_logits=lg, workspace=ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return ids.cpu().numpy(), lg.cpu().numpy()


def check_topk(x, ids, lg, toks, k, norm=True):
    """The GPU's k ids of each token against the exact logits: distinct and valid, each
    logit within its bound E, the order decreasing up to the bounds, every id that must be
    in the top k present and none that cannot be; exact equality where the oracle's k
    largest are separated by more than the bounds."""
    H = x["H"]
    exact, ad = oracle.lm_head_logits(x["hidden"], x["W"], toks,
                                      norm_w=x["norm_w"] if norm else None, eps=x["eps"],
                                      with_absdot=True)
    E = H * 2.0 ** -23 * ad
    strict = 0
    for i, t in enumerate(toks):
        e, b, g = exact[i], E[i], ids[t]
        assert len(set(g.tolist())) == k and ((g >= 0) & (g < x["V"])).all(), (t, g)
        assert (np.abs(lg[t].astype(np.float64) - e[g]) <= b[g] + 1e-30).all(), t
        for r in range(k - 1):
            assert e[g[r]] >= e[g[r + 1]] - b[g[r]] - b[g[r + 1]], (t, r)
        order = np.argsort(-e, kind="stable")          # the oracle's order: value, then id
        o = order[:k]
        kth = e[o[-1]]
        bmax = b.max()
        if k < e.size:
            nxt = order[k]
            must = o[e[o] > e[nxt] + b[o] + b[nxt]]
            assert set(must.tolist()) <= set(g.tolist()), (t, must, g)
        assert (e[g] >= kth - b[g] - bmax).all(), t
        vals = e[order[:min(k + 1, e.size)]]
        if np.all(np.diff(vals) < -2 * bmax):
            assert (g == o).all(), (t, g, o)
            strict += 1
    return strict


@pytest.mark.parametrize("M,H,V,k,norm", [
    (1, 64, 1000, 1, False), (2, 8, 300, 8, True), (5, 128, 4099, 8, True),
    (17, 136, 3000, 3, True), (33, 256, 20000, 5, False), (64, 512, 9000, 8, True),
    (130, 256, 5000, 8, False), (300, 256, 10000, 2, True), (3, 64, 8, 8, True),
    (2, 64, 1000003, 8, True)])
def test_topk_parity(M, H, V, k, norm):
    x = make_lm_head_input(M, H, V, seed=M * 7 + k + V)
    ids, lg = gpu_topk(x, k, norm)
    strict = check_topk(x, ids, lg, np.arange(M), k, norm)
    assert strict >= 0.3 * M
    # the oracle's own top k agrees with the order used above
    oi, _ = oracle.lm_head_topk(x["hidden"][:2], x["W"], k, norm_w=x["norm_w"] if norm else None,
                                eps=x["eps"])
    assert oi.shape == (min(2, M), k)


def test_topk_one_is_the_greedy_pick():
    x = make_lm_head_input(40, 256, 6000, seed=77)
    ids1, lg1 = gpu_topk(x, 1)
    g, lg = gpu_lm_head(x)
    np.testing.assert_array_equal(ids1[:, 0], g)
    np.testing.assert_array_equal(lg1[:, 0], lg)


def test_topk_ties_by_id():
    # copies of the top row at higher and lower ids in other tiles: equal logits, listed by id
    M, H, V, k = 4, 256, 3000, 4
    x = make_lm_head_input(M, H, V, seed=5)
    g, _ = gpu_lm_head(x, norm=False)
    a = int(g[1])
    W = x["W"].copy()
    c1, c2 = (a + 700) % V, (a + 1900) % V
    W[c1] = W[a]
    W[c2] = W[a]
    ids, _ = gpu_topk(dict(x, W=W), k, norm=False)
    assert ids[1, :3].tolist() == sorted([a, c1, c2])


def test_topk_serving_size_sampled_tokens():
    M, H, V, k = 256, 4096, 151936, 8
    x = make_lm_head_input(M, H, V, seed=H + V, w_std=0.02)
    ids, lg = gpu_topk(x, k)
    check_topk(x, ids, lg, np.array([0, 100, 255]), k)
