"""Pins of the oracle's post-verify state fix-up ("14. MTP: speculative decoding with the
built-in draft head", the snapshot / rollback of the decoding loop and "Rolling back":
a KV cache is truncated, the linear attention's memory tables and convolution windows are
copied before verification and restored on a miss).  The strongest pin is the definition
of correctness itself: after the fix-up (and the recomputation it asks for) a toy hybrid
model's KV length and recurrent state equal those of plain one-token-at-a-time decoding of
the kept tokens, for every accepted count."""
import numpy as np
import pytest

import oracle


def _f(S, tok):
    """A toy recurrent update: the next state from the state and one token (uint8 bytes)."""
    return ((S.astype(np.int64) * 5 + tok * 3 + np.arange(S.size) * 7 + (S[::-1] >> 1)) % 256).astype(np.uint8)


def _run(S, toks):
    for t in toks:
        S = _f(S, t)
    return S


@pytest.mark.parametrize("D", [1, 3, 6])
def test_fixup_reproduces_plain_decoding(D):
    rng = np.random.default_rng(D)
    B, nbytes = 12, 40
    S0 = rng.integers(0, 256, (B, nbytes), dtype=np.uint8)           # state before the verify
    kv0 = rng.integers(0, 1000, B).astype(np.int32)                   # KV length before
    carried = rng.integers(0, 50000, B)
    drafts = rng.integers(0, 50000, (B, D))
    a = np.array([b % (D + 1) for b in range(B)], np.int32)           # every accepted count
    backup = oracle.state_snapshot(S0)
    # the verify forward: all D + 1 positions pass the model
    Sv = np.stack([_run(S0[b], [carried[b], *drafts[b]]) for b in range(B)])
    kv, rc, S, _, st = oracle.state_fixup(a, D, kv0, Sv, backup)
    assert st == 0
    for b in range(B):
        kept = [carried[b], *drafts[b, :a[b]]]                        # the step's processed tokens
        # the recomputation the fix-up asks for: the first rc[b] kept tokens from the state
        S_b = _run(S[b], kept[:rc[b]])
        kv_b = kv[b] + rc[b]
        np.testing.assert_array_equal(S_b, _run(S0[b], kept))       # = plain decoding
        assert kv_b == kv0[b] + len(kept)
        assert rc[b] == (0 if a[b] == D else 1 + a[b])
    # an attention-only model keeps 1 + a positions and recomputes nothing
    kv, rc, _, _, _ = oracle.state_fixup(a, D, kv0)
    np.testing.assert_array_equal(kv, kv0 + 1 + a)
    assert (rc == 0).all()


def test_the_pages_one_draft_loop():
    # one draft: a hit keeps both new positions; a miss rolls back to the snapshot and
    # recomputes only the carried-in token
    S = np.arange(16, dtype=np.uint8)[None, :]
    backup = oracle.state_snapshot(S)
    after = (S + 9).astype(np.uint8)
    kv, rc, st_, _, _ = oracle.state_fixup([1], 1, [100], after, backup)
    assert kv[0] == 102 and rc[0] == 0
    np.testing.assert_array_equal(st_, after)
    kv, rc, st_, _, _ = oracle.state_fixup([0], 1, [100], after, backup)
    assert kv[0] == 100 and rc[0] == 1
    np.testing.assert_array_equal(st_, S)


def test_worked_example_keep_counts():
    # four verified positions [bonus, d1, d2, d3], two drafts accepted: an attention cache
    # keeps the bonus and the two accepted drafts
    kv, rc, _, _, _ = oracle.state_fixup([2], 3, [50])
    assert kv[0] == 53 and rc[0] == 0
    # the counter-example: the first draft rejected keeps the bonus alone
    kv, _, _, _, _ = oracle.state_fixup([0], 3, [50])
    assert kv[0] == 51


def test_snapshot_round_trip_and_untouched_hits():
    rng = np.random.default_rng(7)
    S0 = rng.integers(0, 256, (6, 64), dtype=np.uint8)
    backup = oracle.state_snapshot(S0)
    np.testing.assert_array_equal(backup, S0)
    S1 = rng.integers(0, 256, (6, 64), dtype=np.uint8)
    a = np.array([3, 0, 3, 1, 2, 3], np.int32)
    _, _, S, _, _ = oracle.state_fixup(a, 3, np.zeros(6, np.int32), S1, backup)
    for b in range(6):
        np.testing.assert_array_equal(S[b], S1[b] if a[b] == 3 else S0[b])


def test_draft_kv_is_cut_on_a_miss():
    kv0 = np.array([10, 10, 10], np.int32)
    S = np.zeros((3, 16), np.uint8)
    dk = np.array([13, 12, 9], np.int32)
    kv, _, _, dk2, _ = oracle.state_fixup([3, 1, 0], 3, kv0, S, S, draft_kv_len=dk)
    np.testing.assert_array_equal(kv, [14, 10, 10])
    np.testing.assert_array_equal(dk2, [13, 10, 9])


def test_bad_counts_leave_the_row_alone():
    S = np.full((2, 16), 5, np.uint8)
    backup = np.zeros((2, 16), np.uint8)
    kv, rc, S2, _, st = oracle.state_fixup([-1, 4], 3, [7, 7], S, backup)
    assert st == 2
    np.testing.assert_array_equal(S2, S)
    np.testing.assert_array_equal(kv, [0, 0])
