"""Pins of the oracle's draft-head input stage: RMSNorm of the next token's embedding and
of the main model's hidden state, concatenated embedding first, then eh_proj [H, 2H]
(page "14. MTP: speculative decoding with the built-in draft head", "The draft head";
page "MPT (MTP, Multi-Token Prediction) 原理详解", section 二.2)."""
import os

import numpy as np
import pytest
import torch

import oracle
from verify_spec_greedy_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits


def _bits(vals):
    return f32_to_bf16_bits(np.array(vals, np.float32))


def _hand_cases(golden_dir):
    for line in open(os.path.join(golden_dir, "draft_input_hand.txt"), encoding="utf-8"):
        if line.startswith("#") or not line.strip():
            continue
        name, eps, e, h, we, wh, W, y = [t.strip() for t in line.split("|")]
        f = lambda s: [float(v) for v in s.split()]
        yield name, float(eps), f(e), f(h), f(we), f(wh), [f(r) for r in W.split(";")], f(y)


def test_hand_computed_cases(golden_dir):
    n = 0
    for name, eps, e, h, we, wh, W, y in _hand_cases(golden_dir):
        got = oracle.draft_input(_bits([e]), _bits([h]), _bits(we), _bits(wh), _bits(W), eps)
        np.testing.assert_array_equal(got[0], np.array(y), err_msg=name)
        n += 1
    assert n == 3


def test_bf16_rounding_against_torch():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(20000) * 10, rng.standard_normal(2000) * 1e-38,
                           [1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8), 3.0e38, 1e-45]]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.double_to_bf16(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, want)
    assert oracle.double_to_bf16(1 + 2**-8) == 0x3F80       # tie to even (down)
    assert oracle.double_to_bf16(1 + 3 * 2**-8) == 0x3F82   # tie to even (up)


def _rand(rng, M, H, wstd=0.05):
    e = f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    h = f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    we = f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    wh = f32_to_bf16_bits((1 + 0.1 * rng.standard_normal(H)).astype(np.float32))
    W = f32_to_bf16_bits((wstd * rng.standard_normal((H, 2 * H))).astype(np.float32))
    return e, h, we, wh, W


def test_scale_invariance_of_rmsnorm():
    rng = np.random.default_rng(1)
    e, h, we, wh, W = _rand(rng, 3, 64)
    y1 = oracle.draft_input(e, h, we, wh, W, 0.0)
    e2 = f32_to_bf16_bits(bf16_bits_to_f32(e) * 4.0)     # exact scaling by a power of two
    h2 = f32_to_bf16_bits(bf16_bits_to_f32(h) * 0.125)
    y2 = oracle.draft_input(e2, h2, we, wh, W, 0.0)
    np.testing.assert_array_equal(y1, y2)


def test_embedding_half_comes_first():
    rng = np.random.default_rng(2)
    M, H = 4, 32
    e, h, we, wh, W = _rand(rng, M, H)
    Wf = bf16_bits_to_f32(W).copy()
    Wf[:, H:] = 0
    W_e = f32_to_bf16_bits(Wf)
    h_other = f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    np.testing.assert_array_equal(oracle.draft_input(e, h, we, wh, W_e, 1e-6),
                                  oracle.draft_input(e, h_other, we, wh, W_e, 1e-6))
    e_other = f32_to_bf16_bits(rng.standard_normal((M, H)).astype(np.float32))
    assert not np.array_equal(oracle.draft_input(e, h, we, wh, W_e, 1e-6),
                              oracle.draft_input(e_other, h, we, wh, W_e, 1e-6))


def test_linear_in_weight_and_normalised_activations():
    rng = np.random.default_rng(3)
    M, H = 2, 16
    e, h, we, wh, W = _rand(rng, M, H)
    y, xn = oracle.draft_input(e, h, we, wh, W, 1e-6, return_xnorm=True)
    x = bf16_bits_to_f32(xn).astype(np.float64)
    # unit weight rows pick out single normalised activations
    for k in (0, 5, H, 2 * H - 1):
        Wk = np.zeros((H, 2 * H), np.float32)
        Wk[0, k] = 1.0
        yk = oracle.draft_input(e, h, we, wh, f32_to_bf16_bits(Wk), 1e-6)
        np.testing.assert_array_equal(yk[:, 0], x[:, k])
    # normalised activations have unit mean square before the norm weight
    ef = bf16_bits_to_f32(e).astype(np.float64)
    r = 1 / np.sqrt((ef ** 2).mean(1) + 1e-6)
    want = ef * r[:, None] * bf16_bits_to_f32(we)[None]
    np.testing.assert_allclose(x[:, :H], want, rtol=2 ** -8)


def test_selected_outputs_match_full():
    rng = np.random.default_rng(4)
    M, H = 5, 48
    e, h, we, wh, W = _rand(rng, M, H)
    y = oracle.draft_input(e, h, we, wh, W, 1e-6)
    tok = rng.integers(0, M, 50)
    col = rng.integers(0, H, 50)
    np.testing.assert_array_equal(oracle.draft_input_at(e, h, we, wh, W, 1e-6, tok, col),
                                  y[tok, col])
