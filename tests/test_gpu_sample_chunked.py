"""GPU parity of the chunked sampling verifier against the CPU oracle.

spec_verify_sample runs the cluster kernel wherever a cluster's shared memory stages a
unit's rows, and the chunked verifier beyond that (and wherever MTPSPEC_VERIFY_IMPL=chunks
asks for it).  This module reruns the cluster kernel's parity cases through the chunked
verifier, then covers what is its own: vocabularies past the cluster limits up to its
largest (256 chunks of 32 KB of logits per row), calls too small to give every resident
CTA a full chunk (the chunk shrinks), units recycling the coordination slots, and a
switch between the two verifiers on one stream.  The parity rule is the one of
tests/sample_parity.py.
"""
import numpy as np
import pytest
import torch

import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import Workload, make_verify_inputs

# the cluster kernel's cases, collected here again and run with the chunked verifier
from test_gpu_sample import (  # noqa: F401
    _greedy_half, compare, gpu_verify, oracle_verify, test_deterministic_and_seed_sensitive,
    test_invalid_draft_ids_and_bad_params_set_status, test_large_k_and_flat_rows_use_exact_search,
    test_long_drafts, test_margin_rows_are_rare, test_maximum_vocabulary,
    test_mixed_rows_in_one_batch, test_negative_infinity_and_degenerate_rows,
    test_one_hot_draft_mode, test_one_hot_draft_serving_mix, test_ragged_and_filters,
    test_serving_mix_more_seeds, test_top_p_near_one_uses_exact_search, test_unaligned_rows,
    test_workload_full_size)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def chunked(monkeypatch):
    monkeypatch.setenv("MTPSPEC_VERIFY_IMPL", "chunks")


# the largest vocabularies: 256 chunks of 8192 fp32 or 16384 bf16 logits, and a ragged tail
@pytest.mark.parametrize("dtype,one_hot,V,k", [
    ("f32", False, 2097152, 0),
    ("f32", True, 2097151, 50),
    ("bf16", False, 4194304, 50),
    ("bf16", True, 4194303, 0),
])
def test_chunked_maximum_vocabulary(dtype, one_hot, V, k):
    w = Workload(name="vmax", B=2, D=2, V=V, H=8, dtype=dtype, tau=1.0, top_k=k, top_p=0.9,
                 t_std=3.0, q_noise=1.0, seed=V % 1000, philox_seed=V)
    x = _greedy_half(make_verify_inputs(w), np.random.default_rng(V))
    g, o = gpu_verify(x, one_hot=one_hot), oracle_verify(x, one_hot=one_hot)
    assert g["status"] == o["status"] == 0
    compare(g, o, x, label=f"chunked V={V} {dtype} one-hot={one_hot} k={k}", one_hot=one_hot)


def test_past_the_cluster_limit_without_asking(monkeypatch):
    # one id past what a cluster stages (fp32 with draft logits): the call takes it anyway,
    # through the chunked verifier
    monkeypatch.delenv("MTPSPEC_VERIFY_IMPL")
    w = Workload(name="past", B=3, D=2, V=407553, H=8, tau_range=(0.6, 1.2), top_k=0,
                 top_p=0.95, t_std=3.0, q_noise=1.0, seed=8, philox_seed=8)
    x = make_verify_inputs(w)
    g, o = gpu_verify(x), oracle_verify(x)
    assert g["status"] == o["status"] == 0
    compare(g, o, x, label="V=407553 by default")


@pytest.mark.parametrize("B,D,V", [(1, 1, 1), (1, 1, 1000), (1, 1, 400000), (1, 2, 65537),
                                   (2, 1, 1048577)])
def test_small_calls_shrink_the_chunk(B, D, V):
    # few units: the chunk shrinks (to a multiple of 64 ids, at least 1024) so that every
    # resident CTA has one; V = 1 is a single chunk of one id
    w = Workload(name="few", B=B, D=D, V=V, H=8, tau=0.8, top_k=0 if V > 1000 else 7,
                 top_p=0.9, t_std=3.0, q_noise=1.0, seed=V + B, philox_seed=V + D)
    x = make_verify_inputs(w)
    g, o = gpu_verify(x), oracle_verify(x)
    assert g["status"] == o["status"] == 0
    compare(g, o, x, label=f"B={B} D={D} V={V}")


def test_many_units_recycle_the_slots():
    # 600 units through 128 coordination slots, each reused several times within a call,
    # with rows of every kind (greedy, top-k, top-p, unfiltered) interleaved
    rng = np.random.default_rng(17)
    w = Workload(name="recycle", B=150, D=3, V=12289, H=8, tau=1.0, t_std=3.0, q_noise=1.5,
                 seed=17, philox_seed=71)
    x = make_verify_inputs(w)
    x["tau"] = rng.choice([0.0, 0.5, 1.0, 2.0], size=w.B).astype(np.float32)
    x["top_k"] = rng.choice([0, 1, 20, 12289], size=w.B).astype(np.int32)
    x["top_p"] = rng.choice([1.0, 0.9, 0.3], size=w.B).astype(np.float32)
    compare(gpu_verify(x), oracle_verify(x), x, label="slot recycling")


def test_switching_verifiers_on_one_stream(monkeypatch):
    # the two verifiers, back to back on the same inputs and stream, agree with the oracle,
    # and the chunked verifier's two runs (one before, one after the other) are identical
    w = Workload(name="sw", B=32, D=3, V=30011, H=8, tau_range=(0.5, 1.2), top_k=50,
                 top_p=0.9, t_std=3.0, q_noise=1.0, seed=23, philox_seed=23)
    x = make_verify_inputs(w)
    o = oracle_verify(x)
    res = {}
    for impl in ("chunks", "clusters", "chunks"):
        monkeypatch.setenv("MTPSPEC_VERIFY_IMPL", impl)
        res.setdefault(impl, []).append(gpu_verify(x))
    for impl, runs in res.items():
        for g in runs:
            compare(g, o, x, label=impl)
    a, b = res["chunks"]
    for key in a:
        np.testing.assert_array_equal(np.asarray(a[key]), np.asarray(b[key]), err_msg=key)


def test_workspace_query_covers_the_chunked_verifier(monkeypatch):
    # asked for, the chunked verifier's workspace is part of the query's answer; a call
    # with one byte less is refused before anything runs
    B, D, V = 4, 2, 5000
    need = lib.spec_verify_workspace_bytes(B, D, V)
    monkeypatch.setenv("MTPSPEC_VERIFY_IMPL", "clusters")
    assert lib.spec_verify_workspace_bytes(B, D, V) < need
    monkeypatch.setenv("MTPSPEC_VERIFY_IMPL", "chunks")
    T = torch.zeros((B, D + 1, V), device="cuda")
    d = torch.zeros((B, D), dtype=torch.int32, device="cuda")
    tau = torch.ones(B, device="cuda")
    out = torch.empty((B, D + 1), dtype=torch.int32, device="cuda")
    na = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = torch.empty(need - 1, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.MtpSpecError) as e:
        lib.spec_verify_sample(T, None, d, tau, None, None, 0, out, na, None, None, ws, None)
    assert e.value.code == -4   # MTPSPEC_ERR_WORKSPACE
