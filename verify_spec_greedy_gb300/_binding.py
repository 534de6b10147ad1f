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


def _ptr(t):
    return None if t is None else t.data_ptr()


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

def mtp_draft_input_workspace_bytes(M: int, H: int) -> int:
    return int(load().mtp_draft_input_workspace_bytes(int(M), int(H)))


def mtp_draft_input(emb_next, hidden, enorm_w, hnorm_w, eh_proj_w, out, eps: float,
                    workspace=None, stream=None):
    """out[M, H] = eh_proj_w @ [enorm(emb_next); hnorm(hidden)] (all bf16 on the GPU)."""
    M, H = emb_next.shape
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("mtp_draft_input", _ptr(emb_next), _ptr(hidden), _ptr(enorm_w), _ptr(hnorm_w),
          _ptr(eh_proj_w), _ptr(out), M, H, float(eps), _ptr(workspace), ws, _stream(stream))
    return out


def mtp_greedy_draft(logits, out_ids, stream=None):
    """out_ids[M] = argmax of each row of logits[M, V] (lowest id on ties)."""
    M, V = logits.shape
    _call("mtp_greedy_draft", _ptr(logits), _dtype_code(logits), M, V, _ptr(out_ids),
          _stream(stream))
    return out_ids


def mtp_lm_head_greedy_workspace_bytes(M: int, H: int, V: int) -> int:
    return int(load().mtp_lm_head_greedy_workspace_bytes(int(M), int(H), int(V)))


def mtp_lm_head_greedy(hidden, lm_head_w, out_ids, norm_w=None, eps: float = 0.0,
                       out_logit=None, workspace=None, status=None, stream=None):
    """out_ids[M] = argmax_v (lm_head_w @ x_t)_v, x_t = hidden[t] or its RMSNorm with norm_w
    (bf16 hidden [M, H] and lm_head_w [V, H] on the GPU; lowest id on ties)."""
    M, H = hidden.shape
    V = lm_head_w.shape[0]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("mtp_lm_head_greedy", _ptr(hidden), _ptr(norm_w), float(eps), _ptr(lm_head_w), M, H,
          V, _ptr(out_ids), _ptr(out_logit), _ptr(workspace), ws, _ptr(status), _stream(stream))
    return out_ids


def mtp_state_snapshot(state, backup, stream=None):
    """backup[b] = state[b] for device tensors of B rows (any dtype, same shape)."""
    B = state.shape[0]
    rb = state[0].numel() * state.element_size() if B else 0
    _call("mtp_state_snapshot", _ptr(state), _ptr(backup), B, rb, _stream(stream))
    return backup


def mtp_state_fixup(num_accepted, D: int, kv_len_before, kv_len, state=None, backup=None,
                    draft_kv_len=None, recompute=None, status=None, stream=None):
    """The post-verify fix-up of each row (see include/libmtpspec.h); state/backup are
    device tensors of B rows, or None for a model without recurrent state."""
    B = num_accepted.shape[0]
    rb = 0 if state is None else state[0].numel() * state.element_size()
    _call("mtp_state_fixup", _ptr(num_accepted), int(D), _ptr(kv_len_before), _ptr(kv_len),
          _ptr(state), _ptr(backup), B, rb, _ptr(draft_kv_len), _ptr(recompute), _ptr(status),
          _stream(stream))
    return kv_len


def mtp_lm_head_topk_workspace_bytes(M: int, H: int, V: int) -> int:
    return int(load().mtp_lm_head_topk_workspace_bytes(int(M), int(H), int(V)))


def mtp_lm_head_topk(hidden, lm_head_w, out_ids, norm_w=None, eps: float = 0.0,
                     out_logits=None, workspace=None, status=None, stream=None):
    """out_ids[M, k]: the k largest logits' ids of each token (decreasing; ties by id)."""
    M, H = hidden.shape
    V = lm_head_w.shape[0]
    k = out_ids.shape[1]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("mtp_lm_head_topk", _ptr(hidden), _ptr(norm_w), float(eps), _ptr(lm_head_w), M, H, V,
          k, _ptr(out_ids), _ptr(out_logits), _ptr(workspace), ws, _ptr(status), _stream(stream))
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
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("mtp_draft_steps", _ptr(embed_w), _ptr(next_ids), _ptr(positions), _ptr(hidden),
          _ptr(enorm_w), _ptr(hnorm_w), _ptr(eh_proj_w), _ptr(norm_w), _ptr(lm_head_w),
          float(eps), M, H, V, D, _ptr(draft_ids), _ptr(hidden_out), _ptr(workspace), ws,
          _ptr(status), _stream(stream))
    return draft_ids


def spec_verify_greedy(target_logits, draft_ids, out_tokens, num_accepted, status=None,
                       stream=None):
    """Greedy verification of draft_ids[B, D] against target_logits[B, D+1, V]."""
    B, D1, V = target_logits.shape
    _call("spec_verify_greedy", _ptr(target_logits), _dtype_code(target_logits), _ptr(draft_ids),
          B, D1 - 1, V, _ptr(out_tokens), _ptr(num_accepted), _ptr(status), _stream(stream))
    return out_tokens, num_accepted


def spec_verify_workspace_bytes(B: int, D: int, V: int) -> int:
    return int(load().spec_verify_workspace_bytes(int(B), int(D), int(V)))


def spec_verify_sample(target_logits, draft_logits, draft_ids, temperature, top_k, top_p,
                       seed: int, out_tokens, num_accepted, p_target=None, p_draft=None,
                       workspace=None, status=None, stream=None):
    """Speculative-sampling verification (see include/libmtpspec.h)."""
    B, D1, V = target_logits.shape
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _call("spec_verify_sample", _ptr(target_logits), _ptr(draft_logits),
          _dtype_code(target_logits), _ptr(draft_ids), _ptr(temperature), _ptr(top_k),
          _ptr(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF, B, D1 - 1, V, _ptr(out_tokens),
          _ptr(num_accepted), _ptr(p_target), _ptr(p_draft), _ptr(workspace), ws, _ptr(status),
          _stream(stream))
    return out_tokens, num_accepted


def spec_verify_sample_static(target_logits, draft_logits, draft_ids, temperature, top_k, top_p,
                              seed: int, out_tokens, num_accepted, p_target=None, p_draft=None,
                              status=None, stream=None):
    """spec_verify_sample with the library's own fixed scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/libmtpspec.h)."""
    B, D1, V = target_logits.shape
    _call("spec_verify_sample_static", _ptr(target_logits), _ptr(draft_logits),
          _dtype_code(target_logits), _ptr(draft_ids), _ptr(temperature), _ptr(top_k),
          _ptr(top_p), int(seed) & 0xFFFFFFFFFFFFFFFF, B, D1 - 1, V, _ptr(out_tokens),
          _ptr(num_accepted), _ptr(p_target), _ptr(p_draft), _ptr(status), _stream(stream))
    return out_tokens, num_accepted
