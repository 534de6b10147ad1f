"""Pins of the oracle's serial draft steps ("MPT (MTP, Multi-Token Prediction) 原理详解"
三 stages 1-2: each step embeds the previous token, runs the head, greedy-samples the next
draft and passes the token and the head's hidden state on; 二.2 step 1: the embedding at
position 0 is zeroed).  Closed forms: a head wired to copy its input token drafts that
token at every step; a masked position drafts as a zero embedding does; D steps equal D
single steps chained by hand; an id outside the vocabulary embeds as zeros and is
flagged."""
import numpy as np
import pytest

import oracle
from verify_spec_greedy_gb300.inputs import f32_to_bf16_bits, make_draft_input, make_lm_head_input, Workload

ONE = f32_to_bf16_bits(np.array([1.0], np.float32))[0]


def _copy_head(V, H, c=0.5):
    """Embedding rows c * e_v, eh_proj = [I | 0] (the embedding half only), unit norm
    weights, lm_head = the embedding: the head's logits peak at its input token."""
    E = np.zeros((V, H), np.uint16)
    E[np.arange(V), np.arange(V)] = f32_to_bf16_bits(np.array([c], np.float32))[0]
    W = np.zeros((H, 2 * H), np.uint16)
    W[np.arange(H), np.arange(H)] = ONE
    ones = np.full(H, ONE, np.uint16)
    return E, W, ones


@pytest.mark.parametrize("D", [1, 3, 6])
def test_copy_head_repeats_its_token(D):
    V, H, M = 48, 64, 5
    E, W, ones = _copy_head(V, H)
    rng = np.random.default_rng(D)
    ids0 = rng.integers(0, V, M).astype(np.int32)
    h0 = f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    out, hout, st = oracle.draft_steps(E, ids0, h0, ones, ones, W, E, D, eps=1e-6, norm_w=ones)
    assert st == 0
    np.testing.assert_array_equal(out, np.repeat(ids0[:, None], D, axis=1))
    # the hidden state is the normalised one-hot: sqrt(H) at the token
    hv = hout.astype(np.uint32) << 16
    assert (hv.view(np.float32)[:, np.arange(M), ids0] == 8.0).all()


def test_position_zero_drafts_as_a_zero_embedding():
    V, H, M, D = 40, 64, 4, 3
    E, W, ones = _copy_head(V, H)
    ids0 = np.array([5, 6, 7, 8], np.int32)
    h0 = np.zeros((M, H), np.uint16)
    pos = np.array([0, 3, 0, 1], np.int32)
    out, _, _ = oracle.draft_steps(E, ids0, h0, ones, ones, W, E, D, eps=1e-6, norm_w=ones,
                                   positions=pos)
    # masked rows: all logits 0 at step 0, so the lowest id (0), which then repeats
    np.testing.assert_array_equal(out[[0, 2]], 0)
    np.testing.assert_array_equal(out[[1, 3]], np.array([[6] * D, [8] * D]))
    # on a general head the mask equals a zero row in the embedding table
    x = make_lm_head_input(M, 64, V, seed=4)
    di = make_draft_input(Workload(name="x", B=1, D=1, V=16, H=64, M=M, seed=4, w_std=0.05))
    Ez = x["W"].copy()
    Ez[ids0[0]] = 0
    Ez[ids0[2]] = 0
    a = oracle.draft_steps(x["W"], ids0, x["hidden"], di["we"], di["wh"], di["W"], x["W"], 1,
                           eps=1e-6, norm_w=x["norm_w"], positions=pos)
    b = oracle.draft_steps(Ez, ids0, x["hidden"], di["we"], di["wh"], di["W"], x["W"], 1,
                           eps=1e-6, norm_w=x["norm_w"])
    np.testing.assert_array_equal(a[0][[0, 2]], b[0][[0, 2]])
    np.testing.assert_array_equal(a[1][:, [0, 2]], b[1][:, [0, 2]])


def test_steps_chain_the_token_and_the_hidden_state():
    M, H, V, D = 6, 64, 300, 4
    x = make_lm_head_input(M, H, V, seed=8, w_std=0.1)
    di = make_draft_input(Workload(name="x", B=1, D=1, V=16, H=H, M=M, seed=8, w_std=0.05))
    ids0 = np.arange(M, dtype=np.int32) * 7
    pos = np.array([0, 1, 2, 0, 5, 9], np.int32)
    out, hout, _ = oracle.draft_steps(x["W"], ids0, x["hidden"], di["we"], di["wh"], di["W"],
                                      x["W"], D, eps=1e-6, norm_w=x["norm_w"], positions=pos)
    ids, h = ids0, x["hidden"]
    for k in range(D):
        o1, h1, _ = oracle.draft_steps(x["W"], ids, h, di["we"], di["wh"], di["W"], x["W"], 1,
                                       eps=1e-6, norm_w=x["norm_w"], positions=pos + k)
        np.testing.assert_array_equal(o1[:, 0], out[:, k])
        np.testing.assert_array_equal(h1[0], hout[k])
        ids, h = o1[:, 0], h1[0]


def test_bad_ids_embed_as_zeros():
    V, H, M = 30, 64, 3
    E, W, ones = _copy_head(V, H)
    out, _, st = oracle.draft_steps(E, np.array([2, -1, 30], np.int32), np.zeros((M, H), np.uint16),
                                    ones, ones, W, E, 2, eps=1e-6, norm_w=ones)
    assert st == 1
    np.testing.assert_array_equal(out, [[2, 2], [0, 0], [0, 0]])
