"""Every entry point can be captured into a CUDA graph: the library makes no call that a
stream capture forbids, allocates nothing and does not synchronise, so a replay gives the
direct call's results (bit for bit: the same inputs take the same path)."""
import numpy as np
import pytest
import torch

import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import WORKLOADS, make_verify_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _capture_and_compare(call, outs):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    direct = [o.clone() for o in outs]
    for o in outs:
        o.fill_(-3)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    for o, d in zip(outs, direct):
        assert torch.equal(o, d)


@pytest.mark.parametrize("mode", ["sample", "one_hot", "greedy"])
def test_verify_replays(mode):
    w = WORKLOADS["sample_b8_d3_v152k"].scaled(B=8, V=20011)
    x = make_verify_inputs(w)
    B, D = x["d"].shape
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    T, Q, d = t(x["T"]), t(x["Q"]), t(x["d"])
    tau, tk, tp = t(x["tau"]), t(x["top_k"]), t(x["top_p"])
    out = torch.empty((B, D + 1), dtype=torch.int32, device=DEV)
    na = torch.empty(B, dtype=torch.int32, device=DEV)
    pt = torch.empty((B, D), dtype=torch.float32, device=DEV)
    ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, w.V), dtype=torch.uint8, device=DEV)
    if mode == "greedy":
        call = lambda: lib.spec_verify_greedy(T, d, out, na)
        outs = [out, na]
    else:
        q = None if mode == "one_hot" else Q
        call = lambda: lib.spec_verify_sample(T, q, d, tau, tk, tp, x["seed"], out, na, pt, None, ws)
        outs = [out, na, pt]
    _capture_and_compare(call, outs)


def test_draft_side_replays():
    H, V, M = 256, 4000, 40
    g = torch.Generator(device=DEV)
    g.manual_seed(0)
    bf = lambda *s, sc=1.0: (torch.randn(s, device=DEV, generator=g) * sc).to(torch.bfloat16)
    h, e, we, wh = bf(M, H), bf(M, H), bf(H, sc=0.1) + 1, bf(H, sc=0.1) + 1
    Wp, L = bf(H, 2 * H, sc=0.02), bf(V, H, sc=0.02)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    wsd = torch.empty(max(1, lib.mtp_draft_input_workspace_bytes(M, H)), dtype=torch.uint8, device=DEV)
    ids = torch.empty(M, dtype=torch.int32, device=DEV)
    wsl = torch.empty(lib.mtp_lm_head_greedy_workspace_bytes(M, H, V), dtype=torch.uint8, device=DEV)
    logits = torch.randn((M, V), device=DEV)
    gids = torch.empty(M, dtype=torch.int32, device=DEV)

    def call():
        lib.mtp_draft_input(e, h, we, wh, Wp, y, 1e-6, wsd)
        lib.mtp_lm_head_greedy(y, L, ids, norm_w=we, eps=1e-6, workspace=wsl)
        lib.mtp_greedy_draft(logits, gids)
    _capture_and_compare(call, [y.view(torch.int16), ids, gids])
