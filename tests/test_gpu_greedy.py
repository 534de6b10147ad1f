"""GPU parity of the greedy path (mtp_greedy_draft, spec_verify_greedy) against the CPU
oracle: token ids and accepted counts must be bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import (WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits,
                                             make_greedy_draft_logits, make_verify_inputs)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _rows(rng, M, V, kind, dtype):
    if kind == "normal":
        x = (rng.standard_normal((M, V)) * 2).astype(np.float32)
    elif kind == "ties":
        x = rng.integers(-3, 3, (M, V)).astype(np.float32)
    elif kind == "ninf":
        x = np.full((M, V), -np.inf, np.float32)
        x[::2, rng.integers(0, V)] = -1e30
    else:
        raise ValueError(kind)
    return x if dtype == "f32" else f32_to_bf16_bits(x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 7, 16, 17, 1000, 4097, 32768, 151936, 262147])
def test_greedy_draft_parity(dtype, V):
    rng = np.random.default_rng(V)
    for kind in ("normal", "ties", "ninf"):
        M = 5 if V > 100000 else 33
        x = _rows(rng, M, V, kind, dtype)
        ids = torch.full((M,), -7, dtype=torch.int32, device=DEV)
        lib.mtp_greedy_draft(_dev(x), ids)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(ids.cpu().numpy(), oracle.greedy_draft(x), err_msg=kind)


def test_greedy_draft_unaligned_rows_and_offsets():
    # a view that starts 1 element into a buffer: rows are not 16-byte aligned
    rng = np.random.default_rng(0)
    for dtype in ("f32", "bf16"):
        base = _rows(rng, 9, 3001, "ties", dtype)
        buf = _dev(base).reshape(-1)
        x = buf[1:1 + 8 * 3000].view(8, 3000)
        ids = torch.empty(8, dtype=torch.int32, device=DEV)
        lib.mtp_greedy_draft(x, ids)
        torch.cuda.synchronize()
        host = base.reshape(-1)[1:1 + 8 * 3000].reshape(8, 3000)
        np.testing.assert_array_equal(ids.cpu().numpy(), oracle.greedy_draft(host))


def test_greedy_draft_full_size_workload():
    w = WORKLOADS["greedy_b1_d1_v32k"]
    x = make_greedy_draft_logits(w, rows=4)
    ids = torch.empty(4, dtype=torch.int32, device=DEV)
    lib.mtp_greedy_draft(_dev(x), ids)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), oracle.greedy_draft(x))


def _verify(T, d):
    B, D1, V = T.shape
    out = torch.full((B, D1), -9, dtype=torch.int32, device=DEV)
    na = torch.full((B,), -9, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.spec_verify_greedy(_dev(T), _dev(d), out, na, st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), na.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("name", ["greedy_b1_d1_v32k", "serve_b256_d3_v152k"])
def test_verify_greedy_workloads(name):
    w = WORKLOADS[name].scaled(mode="greedy", B=min(WORKLOADS[name].B, 64))
    x = make_verify_inputs(w)
    out, na, st = _verify(x["T"], x["d"])
    o_out, o_na, o_st = oracle.verify_greedy(x["T"], x["d"])
    np.testing.assert_array_equal(out, o_out)
    np.testing.assert_array_equal(na, o_na)
    assert st == o_st == 0


@pytest.mark.parametrize("D", [1, 2, 3, 6, 8, 64])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_verify_greedy_draft_lengths(D, dtype):
    w = WORKLOADS["greedy_b1_d1_v32k"].scaled(B=12, D=D, V=4999 if D < 64 else 301, dtype=dtype,
                                               draft_hit=0.9, seed=D)
    x = make_verify_inputs(w)
    out, na, st = _verify(x["T"], x["d"])
    o_out, o_na, _ = oracle.verify_greedy(x["T"], x["d"])
    np.testing.assert_array_equal(out, o_out)
    np.testing.assert_array_equal(na, o_na)
    assert (na >= 0).all() and (na <= D).all()


def test_verify_greedy_ties_invalid_ids_and_tiny_vocab():
    rng = np.random.default_rng(5)
    B, D, V = 40, 3, 5
    T = rng.integers(0, 2, (B, D + 1, V)).astype(np.float32)  # heavy ties
    d = rng.integers(0, V, (B, D)).astype(np.int32)
    d[3, 1] = V
    d[7, 0] = -1
    out, na, st = _verify(T, d)
    o_out, o_na, o_st = oracle.verify_greedy(T, d)
    np.testing.assert_array_equal(out, o_out)
    np.testing.assert_array_equal(na, o_na)
    assert st == o_st == lib.STATUS_BAD_DRAFT_ID
    # V = 1: every argmax is 0
    T1 = np.zeros((3, 2, 1), np.float32)
    d1 = np.array([[0], [0], [1]], np.int32)
    out, na, st = _verify(T1, d1)
    np.testing.assert_array_equal(out, [[0, 0], [0, 0], [0, -1]])
    np.testing.assert_array_equal(na, [1, 1, 0])


def test_empty_batch_is_a_no_op():
    T = torch.zeros((0, 2, 10), device=DEV)
    d = torch.zeros((0, 1), dtype=torch.int32, device=DEV)
    out = torch.zeros((0, 2), dtype=torch.int32, device=DEV)
    na = torch.zeros((0,), dtype=torch.int32, device=DEV)
    lib.spec_verify_greedy(T, d, out, na)


def test_greedy_speculative_decoding_on_gpu_equals_plain_greedy():
    # a seeded toy LM; plain greedy decoding vs drafting + GPU greedy verification
    V, D = 2048, 3
    rng = np.random.default_rng(1)

    def logits(prefix):
        h = hash(("gpu",) + tuple(prefix)) & 0xFFFFFFFFFFFF
        return (np.random.default_rng(h).standard_normal(V) * 2).astype(np.float32)

    prompt = [5, 6]
    plain = list(prompt)
    while len(plain) < 300:
        plain.append(int(np.argmax(logits(plain))))
    seq = list(prompt)
    while len(seq) < 300:
        drafts, ctx = [], list(seq)
        for _ in range(D):
            g = int(np.argmax(logits(ctx)))
            t = g if rng.random() < 0.7 else int(rng.integers(0, V))
            drafts.append(t)
            ctx.append(t)
        T = np.stack([logits(seq + drafts[:j]) for j in range(D + 1)])[None]
        out, na, _ = _verify(T, np.array([drafts], np.int32))
        emitted = [t for t in out[0].tolist() if t >= 0]
        assert len(emitted) == na[0] + 1
        seq += emitted
    assert seq[:300] == plain[:300]
