"""spec_verify_sample_static: sampling verification for callers that cannot allocate device
memory (a decode loop whose device memory belongs entirely to another allocator, or one
that must never risk the synchronisation an allocation can cause).  It keeps its scratch
in a fixed array inside the library, so this test passes no workspace.

Its results must equal those of spec_verify_sample with a caller workspace, and pass the
oracle's parity rule, on two calls in a row with different inputs (the second call must
not see the first call's leftovers).  A call leaves the device's free memory and torch's
allocator untouched.  At the largest batch the array holds, rows near its end are checked
against the oracle.  This file is collected last so that a run stopping at its first
failure has already run the rest."""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import WORKLOADS, Workload, make_verify_inputs

from sample_parity import check

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _dev(a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _outputs(B, D):
    return (torch.full((B, D + 1), -9, dtype=torch.int32, device=DEV),
            torch.full((B,), -9, dtype=torch.int32, device=DEV),
            torch.full((B, D), -1.0, device=DEV), torch.full((B, D), -1.0, device=DEV),
            torch.zeros(1, dtype=torch.int32, device=DEV))


def _args(x):
    B, D = x["d"].shape
    return (_dev(x["T"]), _dev(x["Q"]), _dev(x["d"]), _dev(x["tau"]), _dev(x.get("top_k")),
            _dev(x.get("top_p")), x["seed"]), _outputs(B, D)


def _run(x, static):
    B, D = x["d"].shape
    ins, (out, na, pt, pd, st) = _args(x)
    if static:
        lib.spec_verify_sample_static(*ins, out, na, pt, pd, status=st)
    else:
        ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, ins[0].shape[-1]),
                         dtype=torch.uint8, device=DEV)
        lib.spec_verify_sample(*ins, out, na, pt, pd, workspace=ws, status=st)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (out, na, pt, pd, st)]


def _as_dict(res):
    return dict(out=res[0], num_accepted=res[1], p_target=res[2], p_draft=res[3],
                status=int(res[4][0]))


def _oracle(x, rows=None):
    return oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], x.get("top_k"),
                                     x.get("top_p"), x["seed"], rows=rows)


def test_matches_workspace_entry_point_and_oracle_on_two_calls():
    first = make_verify_inputs(WORKLOADS["sample_b8_d3_v152k"])
    second = make_verify_inputs(Workload(
        name="second", B=40, D=2, V=30011, H=8, tau_range=(0.5, 1.2), greedy_frac=0.25,
        top_k=40, top_p=0.9, seed=21, philox_seed=22))
    for label, x in (("first call", first), ("second call", second)):
        got = _run(x, static=True)
        want = _run(x, static=False)
        for g, w in zip(got, want):
            np.testing.assert_array_equal(g, w)   # same kernels, deterministic: exact
        assert got[4][0] == 0
        check(_as_dict(got), _oracle(x), x, label=f"static {label}")


def test_a_call_allocates_nothing():
    x = make_verify_inputs(Workload(name="alloc", B=24, D=3, V=20011, H=8, tau=0.8, top_p=0.9,
                                    seed=5, philox_seed=5))
    ins, (out, na, pt, pd, st) = _args(x)
    lib.spec_verify_sample_static(*ins, out, na, pt, pd, status=st)  # set-up on this device
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(3):
        lib.spec_verify_sample_static(*ins, out, na, pt, pd, status=st)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert free1 == free0
    for key in ("allocation.all.allocated", "segment.all.allocated", "allocated_bytes.all.current"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key


def test_rejects_batches_beyond_the_fixed_scratch():
    # 65536 units is the limit: B * (D + 1) = 16385 * 4 is one row too many
    B, D, V = 16385, 3, 64
    T = torch.zeros((B, D + 1, V), device=DEV)
    Q = torch.zeros((B, D, V), device=DEV)
    d = torch.zeros((B, D), dtype=torch.int32, device=DEV)
    tau = torch.ones(B, device=DEV)
    out, na, pt, pd, st = _outputs(B, D)
    with pytest.raises(lib.MtpSpecError) as e:
        lib.spec_verify_sample_static(T, Q, d, tau, None, None, 0, out, na, pt, pd, st)
    assert e.value.code == -3
    # one row fewer fits: random rows fill every record of the array; rows at its end and a
    # seeded sample of the rest match the oracle
    x = make_verify_inputs(Workload(name="full", B=16384, D=3, V=64, H=8, tau_range=(0.5, 1.2),
                                    top_k=20, top_p=0.9, t_std=2.0, q_noise=1.0, seed=3,
                                    philox_seed=4))
    got = _as_dict(_run(x, static=True))
    assert got["status"] == 0
    rows = sorted(set(range(16384 - 64, 16384)) |
                  set(np.random.default_rng(0).choice(16384, 64, replace=False).tolist()))
    check(got, _oracle(x, rows=rows), x, rows=rows, label="static, 65536 units")
