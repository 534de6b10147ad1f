"""spec_verify_sample_static: sampling verification for callers that cannot allocate device
memory (a decode loop whose device memory belongs entirely to another allocator, or one
that must never risk the synchronisation an allocation can cause).  It keeps its scratch
in a fixed array inside the library, so this test passes no workspace.  Its results must
equal those of spec_verify_sample with a caller workspace, on two calls in a row with
different inputs (the second call must not see the first call's leftovers).  This file is
collected last so that a run stopping at its first failure has already run the rest."""
import numpy as np
import pytest
import torch

import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import WORKLOADS, Workload, make_verify_inputs

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


def _run(x, static):
    B, D = x["d"].shape
    T, Q = _dev(x["T"]), _dev(x["Q"])
    out, na, pt, pd, st = _outputs(B, D)
    args = (T, Q, _dev(x["d"]), _dev(x["tau"]), _dev(x["top_k"]), _dev(x["top_p"]), x["seed"],
            out, na, pt, pd)
    if static:
        lib.spec_verify_sample_static(*args, status=st)
    else:
        ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, T.shape[-1]), dtype=torch.uint8,
                         device=DEV)
        lib.spec_verify_sample(*args, workspace=ws, status=st)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in (out, na, pt, pd, st)]


def test_matches_workspace_entry_point_on_two_calls():
    first = make_verify_inputs(WORKLOADS["sample_b8_d3_v152k"])
    second = make_verify_inputs(Workload(
        name="second", B=40, D=2, V=30011, H=8, tau_range=(0.5, 1.2), greedy_frac=0.25,
        top_k=40, top_p=0.9, seed=21, philox_seed=22))
    for x in (first, second):
        got = _run(x, static=True)
        want = _run(x, static=False)
        for g, w in zip(got, want):
            np.testing.assert_array_equal(g, w)   # same kernels, deterministic: exact
        assert (got[1] >= 0).all()


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
    # one row fewer fits
    B = 16384
    res = _run(dict(T=np.zeros((B, D + 1, V), np.float32), Q=np.zeros((B, D, V), np.float32),
                    d=np.zeros((B, D), np.int32), tau=np.ones(B, np.float32), top_k=None,
                    top_p=None, seed=0), static=True)
    assert (res[1] == D).all()  # uniform p == q: every draft is kept
