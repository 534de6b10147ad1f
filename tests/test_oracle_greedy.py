"""Pins of the oracle's argmax and greedy verification.

- argmax takes the lowest id among equal maxima (page "The decoding loop and MTP",
  "Why a hand-written decoding loop"); numpy's argmax has the same rule.
- the worked example and counter-example of page "MPT (MTP, Multi-Token Prediction)
  原理详解", section 四.
- greedy speculative decoding emits exactly the tokens of plain greedy decoding (page
  "14. MTP: speculative decoding with the built-in draft head", "Acceptance rate and
  speed-up": identical token by token), on a seeded toy language model.
- every verification emits between 1 and D+1 tokens (section 三, stage 4).
"""
import os

import numpy as np
import pytest

import oracle
from verify_spec_greedy_gb300.inputs import f32_to_bf16_bits


def test_argmax_matches_first_occurrence_rule():
    rng = np.random.default_rng(0)
    for V in (1, 2, 3, 17, 100, 4097):
        for _ in range(20):
            x = rng.integers(-3, 4, size=V).astype(np.float32)  # many ties
            assert oracle.argmax(x) == int(np.argmax(x))
            b = f32_to_bf16_bits(x)
            assert oracle.argmax(b) == int(np.argmax(x))


def test_argmax_infinities_and_nan():
    x = np.full(10, -np.inf, np.float32)
    assert oracle.argmax(x) == 0
    x[7] = -1e30
    assert oracle.argmax(x) == 7
    x[3] = np.nan
    with pytest.raises(ValueError):
        oracle.argmax(x)


def test_bf16_argmax_compares_stored_values():
    # two fp32 values that differ, but round to the same bf16: the lower id wins
    x = np.array([1.0, 1.001, 0.5], np.float32)
    b = f32_to_bf16_bits(x)
    assert b[0] == b[1]
    assert oracle.argmax(b) == 0
    assert oracle.argmax(x) == 1


def _worked_example(golden_dir):
    vocab, cases = None, []
    for line in open(os.path.join(golden_dir, "worked_example_zh.txt"), encoding="utf-8"):
        line = line.strip()
        if line.startswith("vocab:"):
            vocab = line.split(":", 1)[1].split()
        elif line.startswith("case:"):
            name, drafts, am, emitted, na = [t.strip() for t in line.split(":", 1)[1].split("|")]
            cases.append((name, drafts.split(), am.split(), emitted.split(), int(na)))
    return vocab, cases


def test_worked_example(golden_dir):
    vocab, cases = _worked_example(golden_dir)
    ids = {t: i for i, t in enumerate(vocab)}
    V = len(vocab)
    for name, drafts, am, emitted, na in cases:
        D = len(drafts)
        T = np.zeros((1, D + 1, V), np.float32)
        for j, tok in enumerate(am):
            T[0, j, ids[tok]] = 5.0
        d = np.array([[ids[t] for t in drafts]], np.int32)
        out, acc, st = oracle.verify_greedy(T, d)
        assert st == 0
        assert acc[0] == na, name
        want = [ids[t] for t in emitted] + [-1] * (D + 1 - len(emitted))
        assert out[0].tolist() == want, name
        # the page's count includes the bonus token carried in from the previous round
        if name == "step_c_d":
            assert 1 + (acc[0] + 1) == 4


class ToyLM:
    """A seeded deterministic 'language model': the logits after a prefix are N(0, 2)
    drawn from a generator seeded by the prefix."""

    def __init__(self, V, salt):
        self.V, self.salt = V, salt

    def logits(self, prefix):
        h = hash((self.salt,) + tuple(prefix)) & 0xFFFFFFFFFFFF
        return (np.random.default_rng(h).standard_normal(self.V) * 2.0).astype(np.float32)


@pytest.mark.parametrize("V,D", [(64, 1), (512, 3), (4096, 6)])
def test_greedy_speculative_equals_plain_greedy(V, D):
    lm = ToyLM(V, salt=V * 10 + D)
    rng = np.random.default_rng(V + D)
    prompt = [1, 2, 3]
    n_new = 1000
    plain = list(prompt)
    while len(plain) < len(prompt) + n_new:
        plain.append(int(np.argmax(lm.logits(plain))))

    seq = list(prompt)
    steps = 0
    while len(seq) < len(prompt) + n_new:
        # a noisy drafter: the model's own pick with probability 0.7, else a random id
        drafts, ctx = [], list(seq)
        for _ in range(D):
            g = int(np.argmax(lm.logits(ctx)))
            t = g if rng.random() < 0.7 else int(rng.integers(0, V))
            drafts.append(t)
            ctx.append(t)
        T = np.stack([lm.logits(seq + drafts[:j]) for j in range(D + 1)])[None]
        out, acc, _ = oracle.verify_greedy(T, np.array([drafts], np.int32))
        emitted = [t for t in out[0].tolist() if t >= 0]
        assert 1 <= len(emitted) <= D + 1
        assert len(emitted) == acc[0] + 1
        seq += emitted
        steps += 1
    n = len(prompt) + n_new
    assert seq[:n] == plain[:n]
    assert steps < n_new  # some drafts were accepted


def test_emitted_count_bounds_random():
    rng = np.random.default_rng(3)
    for D in (1, 2, 5, 8):
        B, V = 64, 50
        T = rng.standard_normal((B, D + 1, V)).astype(np.float32)
        am = T.argmax(-1)
        d = np.where(rng.random((B, D)) < 0.8, am[:, :D], rng.integers(0, V, (B, D))).astype(np.int32)
        out, acc, st = oracle.verify_greedy(T, d)
        assert st == 0
        for b in range(B):
            a = acc[b]
            assert 0 <= a <= D
            assert out[b, :a].tolist() == d[b, :a].tolist()
            assert out[b, a] == am[b, a]
            assert (out[b, a + 1:] == -1).all()
            assert all(d[b, j] == am[b, j] for j in range(a))
            if a < D:
                assert d[b, a] != am[b, a]


def test_invalid_draft_ids_are_rejected_and_flagged():
    T = np.zeros((2, 3, 8), np.float32)
    T[:, :, 2] = 1.0
    d = np.array([[2, 99], [-1, 2]], np.int32)
    out, acc, st = oracle.verify_greedy(T, d)
    assert st == oracle.STATUS_BAD_DRAFT_ID
    assert acc.tolist() == [1, 0]
    assert out.tolist() == [[2, 2, -1], [2, -1, -1]]
