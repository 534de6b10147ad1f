"""GPU parity of mtp_draft_input (RMSNorm x2, concat, eh_proj) against the CPU oracle:
every output within 2e-2 absolute of the oracle's double-precision value (bf16 inputs,
fp32 accumulation, bf16 output)."""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import (WORKLOADS, Workload, bf16_bits_to_f32,
                                             make_draft_input)

pytestmark = pytest.mark.gpu
DEV = "cuda"
ATOL = 2e-2


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def gpu_draft_input(e, h, we, wh, W, eps):
    M, H = e.shape
    y = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    nbytes = lib.mtp_draft_input_workspace_bytes(M, H)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=DEV) if nbytes else None
    lib.mtp_draft_input(_bf(e), _bf(h), _bf(we), _bf(wh), _bf(W), y, eps, ws)
    torch.cuda.synchronize()
    return bf16_bits_to_f32(y.view(torch.int16).cpu().numpy().view(np.uint16))


def _inputs(M, H, seed, wstd=0.02):
    w = Workload(name="d", B=1, D=1, V=16, H=H, M=M, seed=seed, w_std=wstd)
    x = make_draft_input(w)
    return x["e"][0], x["h"][0], x["we"], x["wh"], x["W"], x["eps"]


@pytest.mark.parametrize("M,H", [(1, 8), (1, 1024), (2, 64), (3, 520), (4, 2048),
                                 (5, 64), (16, 128), (24, 256), (33, 1024), (64, 512),
                                 (100, 384), (130, 264), (300, 1024)])
def test_draft_input_small(M, H):
    e, h, we, wh, W, eps = _inputs(M, H, seed=M * 1000 + H, wstd=0.5 / np.sqrt(2 * H))
    got = gpu_draft_input(e, h, we, wh, W, eps)
    want = oracle.draft_input(e, h, we, wh, W, eps)
    err = np.abs(got - want)
    assert err.max() <= ATOL, (err.max(), np.unravel_index(err.argmax(), err.shape))
    # well inside the bound on average: the bf16 output rounding dominates
    assert err.mean() <= 4e-3


@pytest.mark.parametrize("name", ["greedy_b1_d1_v32k", "sample_b8_d3_v152k"])
def test_draft_input_workloads_full(name):
    w = WORKLOADS[name]
    x = make_draft_input(w)
    for s in range(x["steps"]):
        got = gpu_draft_input(x["e"][s], x["h"][s], x["we"], x["wh"], x["W"], x["eps"])
        want = oracle.draft_input(x["e"][s], x["h"][s], x["we"], x["wh"], x["W"], x["eps"])
        assert np.abs(got - want).max() <= ATOL


def test_draft_input_six_sequential_steps():
    # the long-draft workload: six calls of one token, each call's output is the next
    # call's hidden state
    w = WORKLOADS["sample_b1_d6_v262k_bf16"]
    x = make_draft_input(w)
    h = x["h"][0]
    for s in range(x["steps"]):
        got = gpu_draft_input(x["e"][s], h, x["we"], x["wh"], x["W"], x["eps"])
        want = oracle.draft_input(x["e"][s], h, x["we"], x["wh"], x["W"], x["eps"])
        assert np.abs(got - want).max() <= ATOL
        h = np.ascontiguousarray(
            torch.from_numpy(got).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


@pytest.mark.parametrize("name", ["serve_b256_d3_v152k", "mtp_b64_d1_v129k_h7168"])
def test_draft_input_workloads_sampled(name):
    # full-size tensor-core path: 4000 outputs recomputed one by one by the oracle
    w = WORKLOADS[name]
    x = make_draft_input(w)
    e, h = x["e"][0], x["h"][0]
    got = gpu_draft_input(e, h, x["we"], x["wh"], x["W"], x["eps"])
    rng = np.random.default_rng(0)
    tok = np.sort(rng.integers(0, w.tokens, 4000))
    col = rng.integers(0, w.H, 4000)
    # include the corners of the output
    tok[:4] = [0, 0, w.tokens - 1, w.tokens - 1]
    col[:4] = [0, w.H - 1, 0, w.H - 1]
    order = np.argsort(tok, kind="stable")
    tok, col = tok[order], col[order]
    want = oracle.draft_input_at(e, h, x["we"], x["wh"], x["W"], x["eps"], tok, col)
    err = np.abs(got[tok, col] - want)
    assert err.max() <= ATOL, err.max()
    assert np.isfinite(got).all()
