"""The Python binding's argument checks, on the host: a stand-in for the library records
the calls, and tensors wrapped to report a CUDA device stand in for device tensors.  Calls
shaped like the ones the GPU tests make go through with the right pointers and sizes;
host tensors, strided views, wrong element types, short buffers and mismatched draft
logits are refused before the library is called."""
import pytest
import torch

from verify_spec_greedy_gb300 import _binding as b


class _Dev(torch.Tensor):
    """A host tensor that reports a CUDA device (the binding only reads its pointer)."""

    @property
    def is_cuda(self):
        return True


def dev(*shape, dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype).as_subclass(_Dev)


class _FakeLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name == "mtpspec_status_string":
            return lambda code: b"MTPSPEC_ERR_TEST"

        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def lib(monkeypatch):
    fake = _FakeLib()
    monkeypatch.setattr(b, "_lib", fake)
    monkeypatch.setattr(b, "_stream", lambda s: 0)
    return fake


I32, F32, BF = torch.int32, torch.float32, torch.bfloat16


def verify_args(B=3, D=2, V=50, dtype=F32, draft=True):
    return dict(target_logits=dev(B, D + 1, V, dtype=dtype),
                draft_logits=dev(B, D, V, dtype=dtype) if draft else None,
                draft_ids=dev(B, D, dtype=I32), temperature=dev(B), top_k=dev(B, dtype=I32),
                top_p=dev(B), seed=5, out_tokens=dev(B, D + 1, dtype=I32),
                num_accepted=dev(B, dtype=I32), p_target=dev(B, D), p_draft=dev(B, D),
                workspace=dev(4096, dtype=torch.uint8), status=dev(1, dtype=I32))


def test_sampling_verify_passes_pointers_and_sizes(lib):
    a = verify_args()
    b.spec_verify_sample(**a)
    name, args = lib.calls[-1]
    assert name == "spec_verify_sample"
    assert args[0] == a["target_logits"].data_ptr() and args[1] == a["draft_logits"].data_ptr()
    assert args[2] == b.F32 and args[7] == 5 and args[8:11] == (3, 2, 50)
    assert args[16] == 4096                                   # workspace bytes
    # one-hot drafts, no filters, no optional outputs
    a.update(draft_logits=None, top_k=None, top_p=None, p_target=None, p_draft=None,
             status=None)
    b.spec_verify_sample(**a)
    args = lib.calls[-1][1]
    assert args[1] is None and args[5] is None and args[6] is None
    # the fixed-scratch variant takes the same checks, without a workspace
    a.pop("workspace")
    b.spec_verify_sample_static(**a)
    assert lib.calls[-1][0] == "spec_verify_sample_static"
    # bf16 logits (also as raw 16-bit views for the weights elsewhere)
    b.spec_verify_sample(**verify_args(dtype=BF))
    assert lib.calls[-1][1][2] == b.BF16


@pytest.mark.parametrize("field,value,err", [
    ("draft_logits", dev(3, 2, 50, dtype=BF), ValueError),     # dtype differs from target
    ("draft_logits", dev(3, 1, 50), ValueError),               # wrong shape
    ("draft_ids", dev(3, 2, dtype=torch.int64), TypeError),
    ("temperature", dev(3, dtype=torch.float64), TypeError),
    ("top_k", dev(3, dtype=torch.int64), TypeError),
    ("out_tokens", dev(3, 2, dtype=I32), ValueError),          # short: needs B x (D+1)
    ("num_accepted", dev(2, dtype=I32), ValueError),
    ("p_target", dev(3, 1), ValueError),
    ("status", dev(1, dtype=torch.int64), TypeError),
    ("temperature", torch.zeros(3), ValueError),               # a host tensor
    ("draft_ids", dev(2, 3, dtype=I32).t(), ValueError),       # a strided view
    ("num_accepted", None, ValueError),                        # required
])
def test_sampling_verify_refuses_bad_arguments(lib, field, value, err):
    a = verify_args()
    a[field] = value
    with pytest.raises(err):
        b.spec_verify_sample(**a)
    assert lib.calls == []


def test_greedy_paths(lib):
    T = dev(2, 4, 33)
    b.spec_verify_greedy(T, dev(2, 3, dtype=I32), dev(2, 4, dtype=I32), dev(2, dtype=I32))
    assert lib.calls[-1][1][3:6] == (2, 3, 33)
    b.mtp_greedy_draft(T.view(-1, 33), dev(8, dtype=I32))
    # an offset view into a larger buffer is contiguous and accepted
    buf = dev(1 + 8 * 30)
    b.mtp_greedy_draft(buf[1:].view(8, 30), dev(8, dtype=I32))
    assert lib.calls[-1][1][0] == buf.data_ptr() + 4
    with pytest.raises(ValueError):
        b.mtp_greedy_draft(T.view(-1, 33), dev(7, dtype=I32))
    with pytest.raises(TypeError):
        b.mtp_greedy_draft(dev(8, 33, dtype=torch.float16), dev(8, dtype=I32))
    with pytest.raises(ValueError):
        b.spec_verify_greedy(T, dev(2, 3, dtype=I32), dev(2, 3, dtype=I32), dev(2, dtype=I32))
    # an empty batch passes its (empty) tensors on
    b.spec_verify_greedy(dev(0, 2, 10), dev(0, 1, dtype=I32), dev(0, 2, dtype=I32),
                         dev(0, dtype=I32))


def test_draft_side(lib):
    M, H, V, D = 4, 16, 40, 3
    e, h, y = dev(M, H, dtype=BF), dev(M, H, dtype=BF), dev(M, H, dtype=BF)
    we, wh, W = dev(H, dtype=BF), dev(H, dtype=BF), dev(H, 2 * H, dtype=BF)
    b.mtp_draft_input(e, h, we, wh, W, y, 1e-6, dev(256, dtype=torch.uint8))
    b.mtp_draft_input(e, h, we, wh, W, y, 1e-6)                   # no workspace
    assert lib.calls[-1][1][10] == 0
    b.mtp_draft_input(e.view(torch.int16).as_subclass(_Dev), h, we, wh, W, y, 1e-6)
    with pytest.raises(TypeError):
        b.mtp_draft_input(dev(M, H), h, we, wh, W, y, 1e-6)       # fp32 where bf16 is read
    with pytest.raises(ValueError):
        b.mtp_draft_input(e, h, we, wh, dev(H, H, dtype=BF), y, 1e-6)
    L = dev(V, H, dtype=BF)
    b.mtp_lm_head_greedy(h, L, dev(M, dtype=I32), norm_w=we, eps=1e-6, out_logit=dev(M),
                         workspace=dev(512, dtype=torch.uint8), status=dev(1, dtype=I32))
    b.mtp_lm_head_greedy(dev(0, H, dtype=BF), dev(10, H, dtype=BF), dev(0, dtype=I32))
    with pytest.raises(TypeError):
        b.mtp_lm_head_greedy(h, L, dev(M, dtype=I32), out_logit=dev(M, dtype=BF))
    b.mtp_lm_head_topk(h, L, dev(M, 5, dtype=I32), out_logits=dev(M, 5))
    assert lib.calls[-1][1][7] == 5                               # k from the output's shape
    with pytest.raises(ValueError):
        b.mtp_lm_head_topk(h, L, dev(M, 5, dtype=I32), out_logits=dev(M, 4))
    b.mtp_draft_steps(dev(V, H, dtype=BF), dev(M, dtype=I32), h, we, wh, W, L,
                      dev(M, D, dtype=I32), 1e-6, norm_w=we, positions=dev(M, dtype=I32),
                      hidden_out=dev(D, M, H, dtype=BF), workspace=dev(64, dtype=torch.uint8),
                      status=dev(1, dtype=I32))
    assert lib.calls[-1][1][10:14] == (M, H, V, D)
    with pytest.raises(ValueError):
        b.mtp_draft_steps(dev(V, H, dtype=BF), dev(M, dtype=I32), h, we, wh, W, L,
                          dev(M, D, dtype=I32), 1e-6, hidden_out=dev(D - 1, M, H, dtype=BF))
    with pytest.raises(TypeError):
        b.mtp_draft_steps(dev(V, H, dtype=BF), dev(M, dtype=torch.int64), h, we, wh, W, L,
                          dev(M, D, dtype=I32), 1e-6)


def test_state(lib):
    B, rb = 5, 48
    S, Sb = dev(B, rb, dtype=torch.uint8), dev(B, rb, dtype=torch.uint8)
    b.mtp_state_snapshot(S, Sb)
    assert lib.calls[-1][1][2:4] == (B, rb)
    with pytest.raises(ValueError):
        b.mtp_state_snapshot(S, dev(B - 1, rb, dtype=torch.uint8))
    a, kv0, kv = dev(B, dtype=I32), dev(B, dtype=I32), dev(B, dtype=I32)
    b.mtp_state_fixup(a, 3, kv0, kv, S, Sb, draft_kv_len=dev(B, dtype=I32),
                      recompute=dev(B, dtype=I32), status=dev(1, dtype=I32))
    b.mtp_state_fixup(a, 3, kv, kv)                               # in place, no state
    assert lib.calls[-1][1][4] is None and lib.calls[-1][1][7] == 0
    b.mtp_state_snapshot(dev(B, 0, dtype=torch.uint8), dev(B, 0, dtype=torch.uint8))
    with pytest.raises(TypeError):
        b.mtp_state_fixup(dev(B, dtype=torch.int64), 3, kv0, kv)
    with pytest.raises(ValueError):
        b.mtp_state_fixup(a, 3, kv0, dev(B - 1, dtype=I32))


def test_a_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no fallback: without the built library every entry point raises
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "_stream", lambda s: 0)       # no CUDA stream on this host
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "libmtpspec.so"))
    with pytest.raises(ImportError):
        b.load()
    a = verify_args()
    with pytest.raises(ImportError):
        b.spec_verify_sample(**a)
    with pytest.raises(ImportError):
        b.spec_verify_workspace_bytes(1, 1, 10)
