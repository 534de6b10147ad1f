"""Pins of the oracle's draft output layer with the greedy pick (the draft head's final
norm, the shared output layer and the argmax: "14. MTP: speculative decoding with the
built-in draft head", "The draft head"; "The decoding loop and MTP", "Why a hand-written
decoding loop": the lower id wins a tie).  Each pin fixes a part by something other than
the oracle itself: a closed form (a one-hot hidden state picks a column of the weight),
the tie rule on duplicated rows, a float64 matrix product, the norm's scale invariance
and its formula restated with an independent bf16 rounding."""
import numpy as np
import pytest

import oracle
from verify_spec_greedy_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_lm_head_input


def _f(b):
    return bf16_bits_to_f32(np.asarray(b, np.uint16)).astype(np.float64)


def test_one_hot_hidden_picks_a_weight_column():
    x = make_lm_head_input(4, 64, 700, seed=1)
    W = x["W"]
    h = np.zeros((4, 64), np.uint16)
    ks = [0, 5, 63, 17]
    scales = [1.0, 2.0, 0.5, -4.0]
    for t, (k, s) in enumerate(zip(ks, scales)):
        h[t, k] = f32_to_bf16_bits(np.array([s], np.float32))[0]
    ids, mx = oracle.lm_head_greedy(h, W)
    for t, (k, s) in enumerate(zip(ks, scales)):
        col = s * _f(W[:, k])
        assert ids[t] == int(np.argmax(col))        # first maximum: the lowest id
        assert mx[t] == col.max()


def test_ties_take_the_lowest_id():
    x = make_lm_head_input(3, 96, 500, seed=2)
    W = x["W"]
    V = W.shape[0]
    ids0, _ = oracle.lm_head_greedy(x["hidden"], W)
    for t in range(3):
        a = int(ids0[t])
        assert 0 < a < V - 1
        W2 = W.copy()
        W2[a // 2] = W2[a]                           # an equal logit at a lower id
        ids, _ = oracle.lm_head_greedy(x["hidden"][t:t + 1], W2)
        assert ids[0] == a // 2
        W3 = W.copy()
        W3[V - 1] = W3[a]                            # an equal logit at a higher id
        ids, _ = oracle.lm_head_greedy(x["hidden"][t:t + 1], W3)
        assert ids[0] == a


@pytest.mark.parametrize("M,H,V", [(1, 8, 10), (5, 64, 333), (7, 200, 1000)])
def test_logits_match_a_float64_product(M, H, V):
    x = make_lm_head_input(M, H, V, seed=M + H)
    ref = _f(x["hidden"]) @ _f(x["W"]).T               # bf16 products are exact in float64
    lg, ad = oracle.lm_head_logits(x["hidden"], x["W"], np.arange(M), with_absdot=True)
    np.testing.assert_allclose(lg, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    np.testing.assert_allclose(ad, np.abs(_f(x["hidden"]))[:, None, :].__mul__(
        np.abs(_f(x["W"]))[None, :, :]).sum(-1), rtol=1e-12)
    ids, mx = oracle.lm_head_greedy(x["hidden"], x["W"])
    np.testing.assert_array_equal(ids, np.argmax(ref, axis=1))
    np.testing.assert_array_equal(mx, ref.max(axis=1))


def _bf16_rne_f64(v):
    """Round float64 to bf16 (nearest, ties to even) directly, without a float32 step."""
    m, e = np.frexp(v)                       # v = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)   # 8 significant bits; np.round is RNE


def test_norm_formula():
    M, H, V, eps = 6, 128, 400, 1e-6
    x = make_lm_head_input(M, H, V, seed=9)
    h, w = _f(x["hidden"]), _f(x["norm_w"])
    r = 1.0 / np.sqrt((h * h).mean(axis=1, keepdims=True) + eps)
    xn = _bf16_rne_f64(h * r * w)
    ref = xn @ _f(x["W"]).T
    lg = oracle.lm_head_logits(x["hidden"], x["W"], np.arange(M), norm_w=x["norm_w"], eps=eps)
    np.testing.assert_allclose(lg, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    ids, _ = oracle.lm_head_greedy(x["hidden"], x["W"], norm_w=x["norm_w"], eps=eps)
    np.testing.assert_array_equal(ids, np.argmax(ref, axis=1))


def test_norm_is_scale_invariant():
    # with eps = 0, RMSNorm(2^k h) = RMSNorm(h) exactly (bf16 scaling by 2^k is exact)
    x = make_lm_head_input(5, 256, 900, seed=11)
    h2 = f32_to_bf16_bits(bf16_bits_to_f32(x["hidden"]) * np.float32(8.0))
    a = oracle.lm_head_logits(x["hidden"], x["W"], np.arange(5), norm_w=x["norm_w"], eps=0.0)
    b = oracle.lm_head_logits(h2, x["W"], np.arange(5), norm_w=x["norm_w"], eps=0.0)
    np.testing.assert_array_equal(a, b)
    # and without the norm the logits scale by the same factor
    c = oracle.lm_head_logits(x["hidden"], x["W"], np.arange(5))
    d = oracle.lm_head_logits(h2, x["W"], np.arange(5))
    np.testing.assert_array_equal(8.0 * c, d)


def test_shapes_are_checked():
    x = make_lm_head_input(2, 16, 20, seed=3)
    with pytest.raises(ValueError):
        oracle.lm_head_greedy(x["hidden"], x["W"][:, :8])


def test_topk_is_a_stable_sort_of_the_logits():
    # the k largest of a float64 product, ordered by value then id (numpy's stable sort of
    # the negated logits), with planted ties
    M, H, V, k = 4, 64, 300, 8
    x = make_lm_head_input(M, H, V, seed=12)
    W = x["W"].copy()
    W[17] = W[250]                                   # equal logits at 17 and 250
    W[5] = W[250]
    ids, vals = oracle.lm_head_topk(x["hidden"], W, k)
    ref = _f(x["hidden"]) @ _f(W).T
    for t in range(M):
        want = np.argsort(-ref[t], kind="stable")[:k]
        np.testing.assert_array_equal(ids[t], want)
        np.testing.assert_array_equal(vals[t], ref[t, want])
    # k = 1 is the greedy pick
    ids1, _ = oracle.lm_head_topk(x["hidden"], W, 1)
    g, _ = oracle.lm_head_greedy(x["hidden"], W)
    np.testing.assert_array_equal(ids1[:, 0], g)


def test_topk_of_a_one_hot_hidden_is_a_sorted_column():
    x = make_lm_head_input(1, 32, 100, seed=13)
    h = np.zeros((1, 32), np.uint16)
    h[0, 9] = f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    ids, vals = oracle.lm_head_topk(h, x["W"], 5)
    col = _f(x["W"][:, 9])
    np.testing.assert_array_equal(ids[0], np.argsort(-col, kind="stable")[:5])


def test_topk_lists_equal_logits_by_id():
    # each token's largest row copied to a lower and a higher id: the three equal logits
    # head the list in increasing id order, the next one follows
    M, H, V, k = 3, 96, 500, 5
    x = make_lm_head_input(M, H, V, seed=14)
    ids0, _ = oracle.lm_head_topk(x["hidden"], x["W"], k)
    for t in range(M):
        a = int(ids0[t, 0])
        lo, hi = (a + 7) % 3, V - 1 - (a % 2)          # two other ids, below and above a
        assert lo < a < hi
        W = x["W"].copy()
        W[lo] = W[a]
        W[hi] = W[a]
        ids, vals = oracle.lm_head_topk(x["hidden"][t:t + 1], W, k)
        np.testing.assert_array_equal(ids[0, :3], sorted([lo, a, hi]))
        assert vals[0, 0] == vals[0, 1] == vals[0, 2] > vals[0, 3]
