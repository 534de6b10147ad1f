"""GPU parity of mtp_draft_steps (D serial greedy draft steps: embedding with the
position-0 mask, the input stage, a stub block, the output layer's pick) against the CPU
oracle, step by step: given the GPU's own inputs to step k (the previous ids and hidden
state), its hidden state must match the oracle's input stage within 2e-2 absolute and its
ids must pass the output layer's pick rule (the fp32-sum ambiguity bound); a head wired
to copy its token drafts exactly; the call replays from a CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300.inputs import (Workload, bf16_bits_to_f32, f32_to_bf16_bits,
                                             make_draft_input, make_lm_head_input)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _bf(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _inputs(M, H, V, seed):
    x = make_lm_head_input(M, H, V, seed=seed)
    E = make_lm_head_input(1, H, V, seed=seed + 1, w_std=0.5)["W"]
    di = make_draft_input(Workload(name="ds", B=1, D=1, V=16, H=H, M=M, seed=seed + 2, w_std=0.02))
    rng = np.random.default_rng(seed)
    ids0 = rng.integers(0, V, M).astype(np.int32)
    pos = rng.integers(0, 3, M).astype(np.int32)
    return dict(E=E, L=x["W"], nw=x["norm_w"], h=x["hidden"], we=di["we"], wh=di["wh"],
                Wp=di["W"], ids=ids0, pos=pos, eps=1e-6, M=M, H=H, V=V)


def gpu_steps(x, D, keep_hidden=True):
    M, H, V = x["M"], x["H"], x["V"]
    out = torch.full((M, D), -5, dtype=torch.int32, device=DEV)
    hout = torch.empty((D, M, H), dtype=torch.bfloat16, device=DEV) if keep_hidden else None
    ws = torch.empty(lib.mtp_draft_steps_workspace_bytes(M, H, V), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.mtp_draft_steps(_bf(x["E"]), torch.from_numpy(x["ids"]).to(DEV), _bf(x["h"]), _bf(x["we"]),
                        _bf(x["wh"]), _bf(x["Wp"]), _bf(x["L"]), out, x["eps"], norm_w=_bf(x["nw"]),
                        positions=torch.from_numpy(x["pos"]).to(DEV), hidden_out=hout, workspace=ws,
                        status=st)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (None if hout is None else _bits(hout)), int(st.item())


def check_steps(x, out, hout, toks):
    H, V, D = x["H"], x["V"], out.shape[1]
    ids_in, h_in = x["ids"], x["h"]
    for k in range(D):
        e = x["E"][ids_in].copy()
        e[(x["pos"] + k) == 0] = 0
        cols = np.tile(np.arange(H), len(toks))
        tk = np.repeat(toks, H)
        y = oracle.draft_input_at(e, h_in, x["we"], x["wh"], x["Wp"], x["eps"], tk, cols).reshape(len(toks), H)
        got = bf16_bits_to_f32(hout[k][toks])
        assert np.abs(got - y).max() <= 2e-2, (k, np.abs(got - y).max())
        ex, ad = oracle.lm_head_logits(hout[k], x["L"], toks, norm_w=x["nw"], eps=x["eps"],
                                       with_absdot=True)
        bound = H * 2.0 ** -23 * ad
        for i, t in enumerate(toks):
            a = int(np.argmax(ex[i]))
            amb = np.flatnonzero(ex[i] >= ex[i, a] - bound[i, a] - bound[i])
            g = int(out[t, k])
            assert g in amb, (k, t, g, a)
            if amb.size == 1:
                assert g == a
        ids_in, h_in = out[:, k], hout[k]


@pytest.mark.parametrize("M,H,V,D", [(1, 64, 500, 1), (3, 64, 500, 3), (4, 128, 1000, 2),
                                     (20, 256, 3001, 4), (33, 136, 2000, 3), (256, 512, 20000, 2),
                                     (2, 64, 500, 64)])
def test_steps_parity(M, H, V, D):
    x = _inputs(M, H, V, seed=M + H + D)
    out, hout, st = gpu_steps(x, D)
    assert st == 0
    assert ((out >= 0) & (out < V)).all()
    check_steps(x, out, hout, np.arange(M) if M <= 40 else np.linspace(0, M - 1, 12).astype(np.int64))
    # without keeping the hidden states the ids are the same
    out2, _, _ = gpu_steps(x, D, keep_hidden=False)
    np.testing.assert_array_equal(out2, out)


def test_copy_head_drafts_its_token():
    V, H, M, D = 48, 64, 7, 5
    one = f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    E = np.zeros((V, H), np.uint16)
    E[np.arange(V), np.arange(V)] = f32_to_bf16_bits(np.array([0.5], np.float32))[0]
    Wp = np.zeros((H, 2 * H), np.uint16)
    Wp[np.arange(H), np.arange(H)] = one
    ones = np.full(H, one, np.uint16)
    ids0 = np.array([3, 9, 47, 0, 12, 30, 5], np.int32)
    pos = np.array([4, 0, 2, 7, 0, 1, 9], np.int32)
    x = dict(E=E, L=E, nw=ones, h=np.zeros((M, H), np.uint16), we=ones, wh=ones, Wp=Wp,
             ids=ids0, pos=pos, eps=1e-6, M=M, H=H, V=V)
    out, _, st = gpu_steps(x, D)
    want, _, _ = oracle.draft_steps(E, ids0, x["h"], ones, ones, Wp, E, D, eps=1e-6, norm_w=ones,
                                    positions=pos)
    np.testing.assert_array_equal(out, want)
    assert (out[pos == 0] == 0).all() and (out[pos != 0] == ids0[pos != 0, None]).all()


def test_bad_ids_are_flagged():
    x = _inputs(4, 64, 300, seed=11)
    x["ids"] = np.array([5, -2, 300, 7], np.int32)
    x["pos"] = np.full(4, 3, np.int32)
    out, hout, st = gpu_steps(x, 2)
    assert st & lib.STATUS_BAD_DRAFT_ID
    e = x["E"][np.clip(x["ids"], 0, 299)].copy()
    e[[1, 2]] = 0
    y = oracle.draft_input(e, x["h"], x["we"], x["wh"], x["Wp"], x["eps"])
    assert np.abs(bf16_bits_to_f32(hout[0]) - y).max() <= 2e-2


def test_replays_from_a_cuda_graph():
    M, H, V, D = 64, 256, 5000, 3
    x = _inputs(M, H, V, seed=21)
    E, L, h = _bf(x["E"]), _bf(x["L"]), _bf(x["h"])
    we, wh, Wp, nw = _bf(x["we"]), _bf(x["wh"]), _bf(x["Wp"]), _bf(x["nw"])
    ids = torch.from_numpy(x["ids"]).to(DEV)
    pos = torch.from_numpy(x["pos"]).to(DEV)
    out = torch.empty((M, D), dtype=torch.int32, device=DEV)
    ws = torch.empty(lib.mtp_draft_steps_workspace_bytes(M, H, V), dtype=torch.uint8, device=DEV)
    call = lambda: lib.mtp_draft_steps(E, ids, h, we, wh, Wp, L, out, x["eps"], norm_w=nw,
                                       positions=pos, workspace=ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    direct = out.clone()
    g = torch.cuda.CUDAGraph()
    out.fill_(-1)
    n0 = lib.mtpspec_launch_count()
    with torch.cuda.graph(g):
        call()
    launches = lib.mtpspec_launch_count() - n0
    assert launches >= 3 * D
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, direct)
    # new inputs in the captured buffers
    ids.copy_(torch.flip(ids, [0]))
    g.replay()
    torch.cuda.synchronize()
    replayed = out.clone()
    call()
    torch.cuda.synchronize()
    assert torch.equal(out, replayed)


def test_serving_size_sampled_tokens():
    # 256 rows, H = 4096, V = 151,936, three steps: the serving workload's draft loop
    M, H, V, D = 256, 4096, 151936, 3
    x = _inputs(M, H, V, seed=4)
    out, hout, st = gpu_steps(x, D)
    assert st == 0
    check_steps(x, out, hout, np.array([0, 77, 255]))
