"""GPU parity of mtp_state_snapshot / mtp_state_fixup against the CPU oracle: lengths,
recompute counts, the draft head's cut and every state byte bit-exact, including rows
with a bad accepted count; at the pages' size (19 MiB of memory tables and convolution
windows a row, 256 rows) the restored and kept rows are checked on the device."""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("B,D,row_bytes", [(1, 1, 16), (5, 3, 0), (37, 3, 4112), (64, 6, 65536),
                                           (300, 2, 1040), (3, 64, 1 << 20), (70000, 2, 16),
                                           (70000, 3, 0)])
def test_fixup_parity(B, D, row_bytes):
    rng = np.random.default_rng(B * 7 + D + row_bytes)
    a = rng.integers(0, D + 1, B).astype(np.int32)
    if B > 4:
        a[1], a[3] = -1, D + 1                            # bad counts: rows left alone
    kv0 = rng.integers(0, 5000, B).astype(np.int32)
    dk0 = (kv0 + rng.integers(-2, D + 3, B)).astype(np.int32)
    S0 = rng.integers(0, 256, (B, row_bytes), dtype=np.uint8)
    S1 = rng.integers(0, 256, (B, row_bytes), dtype=np.uint8)  # the state after the verify forward
    # snapshot on the GPU, compared with the oracle's
    st_d, bk_d = _t(S0), torch.empty((B, row_bytes), dtype=torch.uint8, device=DEV)
    if row_bytes:
        lib.mtp_state_snapshot(st_d, bk_d)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(bk_d.cpu().numpy(), oracle.state_snapshot(S0))
    st_d = _t(S1)
    kv_d = torch.full((B,), -9, dtype=torch.int32, device=DEV)
    rc_d = torch.full((B,), -9, dtype=torch.int32, device=DEV)
    dk_d = _t(dk0)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.mtp_state_fixup(_t(a), D, _t(kv0), kv_d, st_d if row_bytes else None,
                        bk_d if row_bytes else None, draft_kv_len=dk_d, recompute=rc_d,
                        status=status)
    torch.cuda.synchronize()
    kv, rc, S, dk, st = oracle.state_fixup(a, D, kv0, S1 if row_bytes else None,
                                           S0 if row_bytes else None, draft_kv_len=dk0)
    bad = (a < 0) | (a > D)
    got_kv, got_rc = kv_d.cpu().numpy(), rc_d.cpu().numpy()
    np.testing.assert_array_equal(got_kv[~bad], kv[~bad])
    np.testing.assert_array_equal(got_rc[~bad], rc[~bad])
    assert (got_kv[bad] == -9).all() and (got_rc[bad] == -9).all()   # untouched
    np.testing.assert_array_equal(dk_d.cpu().numpy(), dk)
    assert int(status.item()) == st
    if row_bytes:
        np.testing.assert_array_equal(st_d.cpu().numpy(), S)


def test_in_place_lengths():
    a = np.array([0, 2, 3], np.int32)
    kv = _t(np.array([10, 20, 30], np.int32))
    lib.mtp_state_fixup(_t(a), 3, kv, kv)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(kv.cpu().numpy(), [11, 23, 34])


def test_after_a_sampling_verify():
    # the accepted counts straight from spec_verify_sample on a small sampled workload
    from verify_spec_greedy_gb300.inputs import WORKLOADS, make_verify_inputs
    w = WORKLOADS["sample_b8_d3_v152k"].scaled(B=16, V=20011)
    x = make_verify_inputs(w)
    B, D = x["d"].shape
    out = torch.empty((B, D + 1), dtype=torch.int32, device=DEV)
    na = torch.empty(B, dtype=torch.int32, device=DEV)
    ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, w.V), dtype=torch.uint8, device=DEV)
    lib.spec_verify_sample(_t(x["T"]), _t(x["Q"]), _t(x["d"]), _t(x["tau"]), _t(x["top_k"]),
                           _t(x["top_p"]), x["seed"], out, na, None, None, ws)
    row_bytes = 8192
    rng = np.random.default_rng(3)
    S0 = rng.integers(0, 256, (B, row_bytes), dtype=np.uint8)
    S1 = rng.integers(0, 256, (B, row_bytes), dtype=np.uint8)
    st_d, bk_d = _t(S0), torch.empty((B, row_bytes), dtype=torch.uint8, device=DEV)
    lib.mtp_state_snapshot(st_d, bk_d)
    st_d.copy_(_t(S1))
    kv0 = np.full(B, 100, np.int32)
    kv_d, rc_d = torch.empty(B, dtype=torch.int32, device=DEV), torch.empty(B, dtype=torch.int32, device=DEV)
    lib.mtp_state_fixup(na, D, _t(kv0), kv_d, st_d, bk_d, recompute=rc_d)
    torch.cuda.synchronize()
    kv, rc, S, _, _ = oracle.state_fixup(na.cpu().numpy(), D, kv0, S1, S0)
    np.testing.assert_array_equal(kv_d.cpu().numpy(), kv)
    np.testing.assert_array_equal(rc_d.cpu().numpy(), rc)
    np.testing.assert_array_equal(st_d.cpu().numpy(), S)


def test_pages_size_on_device():
    # 256 rows of 19 MiB (the pages' copy of 18 memory tables and convolution windows):
    # restored rows equal the snapshot, kept rows the post-verify state
    B, D, rb = 256, 3, 19 << 20
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    S0 = torch.randint(0, 256, (B, rb), dtype=torch.uint8, device=DEV, generator=g)
    bk = torch.empty_like(S0)
    lib.mtp_state_snapshot(S0, bk)
    assert torch.equal(bk, S0)
    S1 = torch.randint(0, 256, (B, rb), dtype=torch.uint8, device=DEV, generator=g)
    ref_kept = S1.clone()
    a = torch.randint(0, D + 1, (B,), dtype=torch.int32, device=DEV, generator=g)
    kv0 = torch.arange(B, dtype=torch.int32, device=DEV)
    kv = torch.empty_like(kv0)
    lib.mtp_state_fixup(a, D, kv0, kv, S1, bk)
    torch.cuda.synchronize()
    miss = a < D
    assert torch.equal(S1[miss], S0[miss])
    assert torch.equal(S1[~miss], ref_kept[~miss])
    want, _, _, _, _ = oracle.state_fixup(a.cpu().numpy(), D, kv0.cpu().numpy(),
                                          np.zeros((B, 16), np.uint8), np.zeros((B, 16), np.uint8))
    np.testing.assert_array_equal(kv.cpu().numpy(), want)
