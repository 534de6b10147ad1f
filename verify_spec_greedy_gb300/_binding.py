"""ctypes binding of libmtpspec: argument marshalling only.

Every function has the name of the C entry point it calls (include/libmtpspec.h) and
takes torch tensors that already live on the GPU; it passes their device pointers,
sizes and the current CUDA stream to the library and raises MtpSpecError on a non-zero
status.  All computation happens in the library's CUDA kernels.  There is no fallback:
if the library has not been built, loading it raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmtpspec.so")

F32, BF16 = 0, 1
STATUS_BAD_DRAFT_ID = 0x1
STATUS_BAD_PARAM = 0x2
STATUS_TIMEOUT = 0x4

_lib = None


class MtpSpecError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn}: {status_string(code)} ({code})")


def load():
    """Load libmtpspec.so (built by verify_spec_greedy_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmtpspec is not built ({LIB_PATH} missing); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = C.CDLL(LIB_PATH)
    p, i64, i32, u64, sz, f32 = (C.c_void_p, C.c_int64, C.c_int32, C.c_uint64, C.c_size_t,
                                 C.c_float)
    sigs = {
        "mtp_draft_input": ([p, p, p, p, p, p, i64, i64, f32, p, sz, p], C.c_int),
        "mtp_draft_input_workspace_bytes": ([i64, i64], sz),
        "mtp_greedy_draft": ([p, C.c_int, i64, i64, p, p], C.c_int),
        "spec_verify_greedy": ([p, C.c_int, p, i64, i32, i64, p, p, p, p], C.c_int),
        "spec_verify_sample": ([p, p, C.c_int, p, p, p, p, u64, i64, i32, i64, p, p, p, p, p, sz,
                                p, p], C.c_int),
        "spec_verify_workspace_bytes": ([i64, i32, i64], sz),
        "spec_verify_sample_static": ([p, p, C.c_int, p, p, p, p, u64, i64, i32, i64, p, p, p, p,
                                       p, p], C.c_int),
        "mtp_lm_head_greedy": ([p, p, f32, p, i64, i64, i64, p, p, p, sz, p, p], C.c_int),
        "mtp_lm_head_greedy_workspace_bytes": ([i64, i64, i64], sz),
        "mtp_state_snapshot": ([p, p, i64, i64, p], C.c_int),
        "mtp_state_fixup": ([p, i32, p, p, p, p, i64, i64, p, p, p, p], C.c_int),
        "mtp_lm_head_topk": ([p, p, f32, p, i64, i64, i64, i32, p, p, p, sz, p, p], C.c_int),
        "mtp_lm_head_topk_workspace_bytes": ([i64, i64, i64], sz),
        "mtp_draft_steps": ([p, p, p, p, p, p, p, p, p, f32, i64, i64, i64, i32, p, p, p, sz, p, p],
                            C.c_int),
        "mtp_draft_steps_workspace_bytes": ([i64, i64, i64], sz),
        "mtpspec_status_string": ([C.c_int], C.c_char_p),
        "mtpspec_launch_count": ([], C.c_uint64),
        "mtpspec_selftest_wait_timeout": ([C.c_int, C.c_uint32, C.c_void_p, C.c_void_p], C.c_int),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name, None)
        if fn is not None:
            fn.argtypes = args
            fn.restype = res
    _lib = lib
    return lib


def mtpspec_launch_count() -> int:
    """Kernel launches this library has enqueued since it was loaded."""
    return int(load().mtpspec_launch_count())


def status_string(code: int) -> str:
    return load().mtpspec_status_string(int(code)).decode()


def _stream(stream):
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# Argument checks.  The library reads and writes through raw device pointers with the
# sizes it is given, so a host tensor, a strided view, the wrong element type or a short
# buffer would be read or written out of bounds on the GPU; they are refused here.
_I32, _F32, _HALF = "int32", "float32", "16-bit"
_KINDS = None


def _kinds():
    """The accepted torch dtypes of each kind (built on first use: torch loads lazily)."""
    global _KINDS
    if _KINDS is None:
        import torch
        half = {torch.bfloat16, torch.float16, torch.int16}
        if hasattr(torch, "uint16"):
            half.add(torch.uint16)
        _KINDS = {_I32: frozenset([torch.int32]), _F32: frozenset([torch.float32]),
                  _HALF: frozenset(half), "tensor": torch.Tensor}
    return _KINDS


def _arg(t, name, kind=None, numel=0, optional=False):
    """Device pointer of tensor `t` after checking that it lives on a CUDA device, is
    contiguous, has the element type `kind` (int32, float32, or any 16-bit type for bf16
    bit patterns) and holds at least `numel` elements; None when `t` is None and allowed."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    kinds = _kinds()
    if not isinstance(t, kinds["tensor"]):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if kind is not None and t.dtype not in kinds[kind]:
        raise TypeError(f"{name} must hold {kind} values, got {t.dtype}")
    if numel and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements; {numel} are needed")
    return t.data_ptr()


def _ws(workspace):
    """(pointer, bytes) of an optional workspace tensor."""
    if workspace is None:
        return None, 0
    return _arg(workspace, "workspace"), workspace.numel() * workspace.element_size()


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _call(name, *args):
    rc = getattr(load(), name)(*args)
    if rc != 0:
        raise MtpSpecError(name, rc)


# ---------------------------------------------------------------- entry points

def mtpspec_selftest_wait_timeout(which: int, limit: int, status, stream=None):
    """Run one kernel family's bounded wait on a barrier that nothing completes (see
    include/libmtpspec.h); MTPSPEC_STATUS_TIMEOUT is OR-ed into `status` when it gives up."""
    _call("mtpspec_selftest_wait_timeout", int(which), int(limit),
          _arg(status, "status", _I32, 1), _stream(stream))


def mtp_draft_input_workspace_bytes(M: int, H: int) -> int:
    return int(load().mtp_draft_input_workspace_bytes(int(M), int(H)))


def mtp_draft_input(emb_next, hidden, enorm_w, hnorm_w, eh_proj_w, out, eps: float,
                    workspace=None, stream=None):
    """out[M, H] = eh_proj_w @ [enorm(emb_next); hnorm(hidden)] (all bf16 on the GPU)."""
    M, H = emb_next.shape
    wp, ws = _ws(workspace)
    _call("mtp_draft_input", _arg(emb_next, "emb_next", _HALF, M * H),
          _arg(hidden, "hidden", _HALF, M * H), _arg(enorm_w, "enorm_w", _HALF, H),
          _arg(hnorm_w, "hnorm_w", _HALF, H), _arg(eh_proj_w, "eh_proj_w", _HALF, 2 * H * H),
          _arg(out, "out", _HALF, M * H), M, H, float(eps), wp, ws, _stream(stream))
    return out


def mtp_greedy_draft(logits, out_ids, stream=None):
    """out_ids[M] = argmax of each row of logits[M, V] (lowest id on ties)."""
    M, V = logits.shape
    _call("mtp_greedy_draft", _arg(logits, "logits", numel=M * V), _dtype_code(logits), M, V,
          _arg(out_ids, "out_ids", _I32, M), _stream(stream))
    return out_ids


def mtp_lm_head_greedy_workspace_bytes(M: int, H: int, V: int) -> int:
    return int(load().mtp_lm_head_greedy_workspace_bytes(int(M), int(H), int(V)))


def mtp_lm_head_greedy(hidden, lm_head_w, out_ids, norm_w=None, eps: float = 0.0,
                       out_logit=None, workspace=None, status=None, stream=None):
    """out_ids[M] = argmax_v (lm_head_w @ x_t)_v, x_t = hidden[t] or its RMSNorm with norm_w
    (bf16 hidden [M, H] and lm_head_w [V, H] on the GPU; lowest id on ties)."""
    M, H = hidden.shape
    V = lm_head_w.shape[0]
    wp, ws = _ws(workspace)
    _call("mtp_lm_head_greedy", _arg(hidden, "hidden", _HALF, M * H),
          _arg(norm_w, "norm_w", _HALF, H, optional=True), float(eps),
          _arg(lm_head_w, "lm_head_w", _HALF, V * H), M, H, V,
          _arg(out_ids, "out_ids", _I32, M), _arg(out_logit, "out_logit", _F32, M, optional=True),
          wp, ws, _arg(status, "status", _I32, 1, optional=True), _stream(stream))
    return out_ids


def mtp_state_snapshot(state, backup, stream=None):
    """backup[b] = state[b] for device tensors of B rows (any dtype, same shape)."""
    B = state.shape[0]
    rb = state[0].numel() * state.element_size() if B else 0
    ps = _arg(state, "state")
    pb = _arg(backup, "backup")
    if backup.numel() * backup.element_size() < B * rb:
        raise ValueError("backup is smaller than state")
    _call("mtp_state_snapshot", ps, pb, B, rb, _stream(stream))
    return backup


def mtp_state_fixup(num_accepted, D: int, kv_len_before, kv_len, state=None, backup=None,
                    draft_kv_len=None, recompute=None, status=None, stream=None):
    """The post-verify fix-up of each row (see include/libmtpspec.h); state/backup are
    device tensors of B rows, or None for a model without recurrent state."""
    B = num_accepted.shape[0]
    rb = 0 if state is None else state[0].numel() * state.element_size()
    ps = _arg(state, "state", optional=True)
    pb = _arg(backup, "backup", optional=True)
    for t, n in ((state, "state"), (backup, "backup")):
        if t is not None and t.numel() * t.element_size() < B * rb:
            raise ValueError(f"{n} holds fewer than {B} rows of {rb} bytes")
    _call("mtp_state_fixup", _arg(num_accepted, "num_accepted", _I32, B), int(D),
          _arg(kv_len_before, "kv_len_before", _I32, B), _arg(kv_len, "kv_len", _I32, B),
          ps, pb, B, rb, _arg(draft_kv_len, "draft_kv_len", _I32, B, optional=True),
          _arg(recompute, "recompute", _I32, B, optional=True),
          _arg(status, "status", _I32, 1, optional=True), _stream(stream))
    return kv_len


def mtp_lm_head_topk_workspace_bytes(M: int, H: int, V: int) -> int:
    return int(load().mtp_lm_head_topk_workspace_bytes(int(M), int(H), int(V)))


def mtp_lm_head_topk(hidden, lm_head_w, out_ids, norm_w=None, eps: float = 0.0,
                     out_logits=None, workspace=None, status=None, stream=None):
    """out_ids[M, k]: the k largest logits' ids of each token (decreasing; ties by id)."""
    M, H = hidden.shape
    V = lm_head_w.shape[0]
    k = out_ids.shape[1]
    wp, ws = _ws(workspace)
    _call("mtp_lm_head_topk", _arg(hidden, "hidden", _HALF, M * H),
          _arg(norm_w, "norm_w", _HALF, H, optional=True), float(eps),
          _arg(lm_head_w, "lm_head_w", _HALF, V * H), M, H, V, k,
          _arg(out_ids, "out_ids", _I32, M * k),
          _arg(out_logits, "out_logits", _F32, M * k, optional=True), wp, ws,
          _arg(status, "status", _I32, 1, optional=True), _stream(stream))
    return out_ids


def mtp_draft_steps_workspace_bytes(M: int, H: int, V: int) -> int:
    return int(load().mtp_draft_steps_workspace_bytes(int(M), int(H), int(V)))


def mtp_draft_steps(embed_w, next_ids, hidden, enorm_w, hnorm_w, eh_proj_w, lm_head_w,
                    draft_ids, eps: float, norm_w=None, positions=None, hidden_out=None,
                    workspace=None, status=None, stream=None):
    """draft_ids[M, D] from D serial greedy steps of the draft head (stub block)."""
    M, H = hidden.shape
    V = embed_w.shape[0]
    D = draft_ids.shape[1]
    wp, ws = _ws(workspace)
    _call("mtp_draft_steps", _arg(embed_w, "embed_w", _HALF, V * H),
          _arg(next_ids, "next_ids", _I32, M),
          _arg(positions, "positions", _I32, M, optional=True),
          _arg(hidden, "hidden", _HALF, M * H), _arg(enorm_w, "enorm_w", _HALF, H),
          _arg(hnorm_w, "hnorm_w", _HALF, H), _arg(eh_proj_w, "eh_proj_w", _HALF, 2 * H * H),
          _arg(norm_w, "norm_w", _HALF, H, optional=True),
          _arg(lm_head_w, "lm_head_w", _HALF, V * H), float(eps), M, H, V, D,
          _arg(draft_ids, "draft_ids", _I32, M * D),
          _arg(hidden_out, "hidden_out", _HALF, D * M * H, optional=True), wp, ws,
          _arg(status, "status", _I32, 1, optional=True), _stream(stream))
    return draft_ids


def spec_verify_greedy(target_logits, draft_ids, out_tokens, num_accepted, status=None,
                       stream=None):
    """Greedy verification of draft_ids[B, D] against target_logits[B, D+1, V]."""
    B, D1, V = target_logits.shape
    D = D1 - 1
    _call("spec_verify_greedy", _arg(target_logits, "target_logits", numel=B * D1 * V),
          _dtype_code(target_logits), _arg(draft_ids, "draft_ids", _I32, B * D), B, D, V,
          _arg(out_tokens, "out_tokens", _I32, B * D1),
          _arg(num_accepted, "num_accepted", _I32, B),
          _arg(status, "status", _I32, 1, optional=True), _stream(stream))
    return out_tokens, num_accepted


def spec_verify_workspace_bytes(B: int, D: int, V: int) -> int:
    return int(load().spec_verify_workspace_bytes(int(B), int(D), int(V)))


def _verify_sample_args(target_logits, draft_logits, draft_ids, temperature, top_k, top_p,
                        seed, out_tokens, num_accepted, p_target, p_draft):
    """The checked arguments the two sampling entry points share, in their order: the
    logits, draft ids, per-row parameters, seed and sizes, then the outputs."""
    B, D1, V = target_logits.shape
    D = D1 - 1
    if draft_logits is not None and (draft_logits.dtype != target_logits.dtype or
                                     tuple(draft_logits.shape) != (B, D, V)):
        raise ValueError(f"draft_logits must be {target_logits.dtype} of shape {(B, D, V)}, "
                         f"got {draft_logits.dtype} {tuple(draft_logits.shape)}")
    head = (_arg(target_logits, "target_logits", numel=B * D1 * V),
            _arg(draft_logits, "draft_logits", numel=B * D * V, optional=True),
            _dtype_code(target_logits), _arg(draft_ids, "draft_ids", _I32, B * D),
            _arg(temperature, "temperature", _F32, B),
            _arg(top_k, "top_k", _I32, B, optional=True),
            _arg(top_p, "top_p", _F32, B, optional=True), int(seed) & 0xFFFFFFFFFFFFFFFF,
            B, D, V)
    tail = (_arg(out_tokens, "out_tokens", _I32, B * D1),
            _arg(num_accepted, "num_accepted", _I32, B),
            _arg(p_target, "p_target", _F32, B * D, optional=True),
            _arg(p_draft, "p_draft", _F32, B * D, optional=True))
    return head, tail


def spec_verify_sample(target_logits, draft_logits, draft_ids, temperature, top_k, top_p,
                       seed: int, out_tokens, num_accepted, p_target=None, p_draft=None,
                       workspace=None, status=None, stream=None):
    """Speculative-sampling verification (see include/libmtpspec.h)."""
    head, tail = _verify_sample_args(target_logits, draft_logits, draft_ids, temperature,
                                     top_k, top_p, seed, out_tokens, num_accepted, p_target,
                                     p_draft)
    wp, ws = _ws(workspace)
    _call("spec_verify_sample", *head, *tail, wp, ws,
          _arg(status, "status", _I32, 1, optional=True), _stream(stream))
    return out_tokens, num_accepted


def spec_verify_sample_static(target_logits, draft_logits, draft_ids, temperature, top_k, top_p,
                              seed: int, out_tokens, num_accepted, p_target=None, p_draft=None,
                              status=None, stream=None):
    """spec_verify_sample with the library's own fixed scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/libmtpspec.h)."""
    head, tail = _verify_sample_args(target_logits, draft_logits, draft_ids, temperature,
                                     top_k, top_p, seed, out_tokens, num_accepted, p_target,
                                     p_draft)
    _call("spec_verify_sample_static", *head, *tail,
          _arg(status, "status", _I32, 1, optional=True), _stream(stream))
    return out_tokens, num_accepted
