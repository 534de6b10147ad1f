"""The kernels' bounded waits give up and report it: every wait on a copy, a barrier or
another CTA polls a fixed number of times, then ORs MTPSPEC_STATUS_TIMEOUT into the status
word and lets the call end, so that the context stays usable.  No GPU fault is involved:
mtpspec_selftest_wait_timeout runs each kernel family's wait function on a barrier or a
counter that nothing completes (a barrier of two arrivals given one, a counter nothing
raises), with a short poll limit.  Afterwards a sampling verification on the same context
still matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import Workload, make_verify_inputs

from sample_parity import check

pytestmark = pytest.mark.gpu
TIMEOUT = 0x4


@pytest.mark.parametrize("which", [0, 1, 2])
@pytest.mark.parametrize("limit", [1, 4096])
def test_a_wait_that_nothing_completes_gives_up(which, limit):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib.mtpspec_selftest_wait_timeout(which, limit, st)
    torch.cuda.synchronize()
    assert int(st.item()) == TIMEOUT


def test_the_context_stays_usable():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for which in (0, 1, 2):
        lib.mtpspec_selftest_wait_timeout(which, 64, st)
    torch.cuda.synchronize()
    assert int(st.item()) == TIMEOUT
    w = Workload(name="after", B=6, D=2, V=4099, H=8, tau_range=(0.6, 1.2), top_p=0.9,
                 t_std=3.0, q_noise=1.0, seed=7, philox_seed=7)
    x = make_verify_inputs(w)
    B, D = x["d"].shape

    def dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    out = torch.empty((B, D + 1), dtype=torch.int32, device="cuda")
    na = torch.empty(B, dtype=torch.int32, device="cuda")
    pt = torch.empty((B, D), device="cuda")
    pd = torch.empty((B, D), device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, w.V), dtype=torch.uint8, device="cuda")
    lib.spec_verify_sample(dev(x["T"]), dev(x["Q"]), dev(x["d"]), dev(x["tau"]), None,
                           dev(x["top_p"]), x["seed"], out, na, pt, pd, ws, st2)
    torch.cuda.synchronize()
    g = dict(out=out.cpu().numpy(), num_accepted=na.cpu().numpy(), p_target=pt.cpu().numpy(),
             p_draft=pd.cpu().numpy(), status=int(st2.item()))
    assert g["status"] == 0
    o = oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], None, x["top_p"], x["seed"])
    check(g, o, x, label="after the timeouts")
