"""CPU oracle for the MTP speculative-decoding hot path (test infrastructure only).

The arithmetic lives in ``mtpspec_oracle.c`` (plain C, double precision); this module
compiles it with gcc and exposes it to Python through ctypes with numpy arrays.

Only the test suite, the package's ``smoke()`` check and the benchmark's CPU-baseline
leg and reference arm may import this package.  The product library (``verify_spec_greedy_gb300``) never
imports it and shares no code with it.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mtpspec_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmtpspec_oracle.so")

F32, BF16 = 0, 1
STATUS_BAD_DRAFT_ID = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmtpspec_oracle.so`` (gcc, no GPU)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = C.CDLL(build())
        p = C.c_void_p
        i64, i32, u64, u32, dbl = C.c_int64, C.c_int32, C.c_uint64, C.c_uint32, C.c_double
        lib.orc_philox4x32_10.argtypes = [p, p, p]
        lib.orc_philox4x32_10.restype = None
        lib.orc_uniforms.argtypes = [u64, u64, u32, p, p]
        lib.orc_uniforms.restype = None
        lib.orc_double_to_bf16.argtypes = [dbl]
        lib.orc_double_to_bf16.restype = C.c_uint16
        lib.orc_argmax.argtypes = [p, C.c_int, i64]
        lib.orc_argmax.restype = i64
        lib.orc_greedy_draft.argtypes = [p, C.c_int, i64, i64, p]
        lib.orc_greedy_draft.restype = C.c_int
        lib.orc_verify_greedy.argtypes = [p, C.c_int, p, i64, i32, i64, p, p, p]
        lib.orc_verify_greedy.restype = C.c_int
        lib.orc_filter.argtypes = [p, C.c_int, i64, dbl, i32, dbl, p, p]
        lib.orc_filter.restype = C.c_int
        lib.orc_verify_sample.argtypes = [p, p, C.c_int, p, p, p, p, u64, i64, i64, i32, i64,
                                          p, p, p, p, p, p]
        lib.orc_verify_sample.restype = C.c_int
        lib.orc_verify_unit.argtypes = [p, p, C.c_int, i64, i32, dbl, i32, dbl, dbl, dbl, i32, i32,
                                        i64, i64, dbl, p, p, p, p]
        lib.orc_verify_unit.restype = C.c_int
        lib.orc_draft_input.argtypes = [p, p, p, p, p, i64, i64, dbl, p, p]
        lib.orc_draft_input.restype = C.c_int
        lib.orc_draft_input_at.argtypes = [p, p, p, p, p, i64, i64, dbl, p, p, i64, p]
        lib.orc_draft_input_at.restype = C.c_int
        lib.orc_lm_head_logits.argtypes = [p, p, dbl, p, i64, i64, i64, p, i64, p, p]
        lib.orc_lm_head_logits.restype = C.c_int
        lib.orc_lm_head_greedy.argtypes = [p, p, dbl, p, i64, i64, i64, p, p]
        lib.orc_lm_head_greedy.restype = C.c_int
        lib.orc_state_snapshot.argtypes = [p, p, i64, i64]
        lib.orc_state_snapshot.restype = C.c_int
        lib.orc_state_fixup.argtypes = [p, i32, p, p, p, p, i64, i64, p, p, p]
        lib.orc_state_fixup.restype = C.c_int
        lib.orc_draft_steps.argtypes = [p, p, p, p, p, p, p, p, p, dbl, i64, i64, i64, i32, p, p, p]
        lib.orc_draft_steps.restype = C.c_int
        lib.orc_lm_head_topk.argtypes = [p, p, dbl, p, i64, i64, i64, i32, p, p]
        lib.orc_lm_head_topk.restype = C.c_int
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _logits(x):
    """(contiguous array, dtype code) for fp32 logits or bf16 logits stored as uint16 bits."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"logits must be float32 or bf16 bits (uint16), got {x.dtype}")


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- random numbers

def philox4x32_10(ctr, key):
    lib = _load()
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    lib.orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniforms(seed: int, row: int, pos: int):
    lib = _load()
    ua, us = C.c_double(), C.c_double()
    lib.orc_uniforms(seed, row, pos, C.byref(ua), C.byref(us))
    return ua.value, us.value


def double_to_bf16(v: float) -> int:
    return int(_load().orc_double_to_bf16(float(v)))


# ---------------------------------------------------------------- greedy

def argmax(x) -> int:
    x, dt = _logits(x)
    r = _load().orc_argmax(_ptr(x), dt, x.size)
    if r < 0:
        raise ValueError("argmax of an empty row or of a row holding NaN")
    return int(r)


def greedy_draft(logits):
    x, dt = _logits(logits)
    M, V = x.shape
    ids = np.zeros(M, np.int32)
    _check(_load().orc_greedy_draft(_ptr(x), dt, M, V, _ptr(ids)), "greedy_draft")
    return ids


def verify_greedy(T, d):
    """T [B, D+1, V], d [B, D] -> (out [B, D+1], num_accepted [B], status)."""
    x, dt = _logits(T)
    B, D1, V = x.shape
    d = np.ascontiguousarray(d, dtype=np.int32)
    assert d.shape == (B, D1 - 1)
    out = np.zeros((B, D1), np.int32)
    na = np.zeros(B, np.int32)
    st = np.zeros(1, np.int32)
    _check(_load().orc_verify_greedy(_ptr(x), dt, _ptr(d), B, D1 - 1, V, _ptr(out), _ptr(na),
                                     _ptr(st)), "verify_greedy")
    return out, na, int(st[0])


# ---------------------------------------------------------------- sampling

def filter_probs(x, tau: float, k: int = 0, p: float = 1.0, with_margin: bool = False):
    """Filtered, normalised probabilities of one logit row (temperature, top-k, top-p)."""
    x, dt = _logits(x)
    V = x.size
    prob = np.zeros(V, np.float64)
    m = C.c_double()
    _check(_load().orc_filter(_ptr(x), dt, V, float(tau), int(k), float(p), _ptr(prob),
                              C.byref(m)), "filter")
    return (prob, m.value) if with_margin else prob


def verify_sample(T, Q, d, tau, top_k=None, top_p=None, seed: int = 0, row0: int = 0):
    """Speculative-sampling verification of B rows.

    T [B, D+1, V], Q [B, D, V] (fp32, or bf16 bits as uint16) or None (a one-hot draft:
    the drafter's distribution is the point mass on its token), d [B, D] int32,
    tau [B] float32, top_k [B] int32 or None, top_p [B] float32 or None.
    Returns a dict: out, num_accepted, p_target, p_draft, status, margins [B, D+1, 4].
    """
    x, dt = _logits(T)
    B, D1, V = x.shape
    D = D1 - 1
    q = None
    if Q is not None:
        q, dq = _logits(Q)
        assert dt == dq
        assert q.shape == (B, D, V)
    d = np.ascontiguousarray(d, dtype=np.int32).reshape(B, D)
    tau = np.ascontiguousarray(tau, dtype=np.float32).reshape(B)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32).reshape(B)
    tp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32).reshape(B)
    out = np.zeros((B, D1), np.int32)
    na = np.zeros(B, np.int32)
    pt = np.zeros((B, D), np.float64)
    pd = np.zeros((B, D), np.float64)
    st = np.zeros(1, np.int32)
    mg = np.zeros((B, D1, 4), np.float64)
    _check(_load().orc_verify_sample(_ptr(x), _ptr(q), dt, _ptr(d), _ptr(tau), _ptr(tk), _ptr(tp),
                                     int(seed), int(row0), B, D, V, _ptr(out), _ptr(na), _ptr(pt),
                                     _ptr(pd), _ptr(st), _ptr(mg)), "verify_sample")
    return dict(out=out, num_accepted=na, p_target=pt, p_draft=pd, status=int(st[0]), margins=mg)


def verify_unit(t_row, q_row, d: int, tau: float, k: int = 0, p: float = 1.0,
                u_acc: float = 0.5, u_smp: float = 0.5, bonus: bool = False, draw: bool = True,
                gt: int = -1, gq: int = -1, delta: float = 0.0, with_weights: bool = False):
    """One verification unit with explicit uniforms (see orc_verify_unit).

    t_row [V] (and q_row [V], or None for a one-hot draft) fp32 or bf16 bits; bonus: the
    position after the last draft (a draw from p, no accept test).  gt / gq force the
    number of top-p groups kept in the target / draft row (-1: the rule); delta is the
    window of the reported alternative counts.  Returns a dict: accept, pt, pd, ratio,
    acc_margin, margin_t, margin_q, cdf_margin, token (-1 when nothing was drawn),
    cdf_lo / cdf_hi (the draw's distances to its cell's edges, relative to the total),
    tok_prev / tok_next (the neighbouring ids with positive draw weight, -1 if none),
    cut_t / cut_q = (groups the rule keeps, fewest, most within delta), w_draw [V] or None.
    """
    x, dt = _logits(t_row)
    V = x.size
    q = None
    if q_row is not None:
        q, dq = _logits(q_row)
        assert dq == dt and q.size == V
    dres = np.zeros(8, np.float64)
    dnb = np.zeros(4, np.float64)
    ires = np.zeros(7, np.int64)
    w = np.zeros(V, np.float64) if with_weights else None
    _check(_load().orc_verify_unit(_ptr(x), _ptr(q), dt, V, int(d), float(tau), int(k), float(p),
                                   float(u_acc), float(u_smp), int(bool(bonus)), int(bool(draw)),
                                   int(gt), int(gq), float(delta), _ptr(dres), _ptr(dnb),
                                   _ptr(ires), _ptr(w)), "verify_unit")
    return dict(accept=bool(dres[0]), pt=dres[1], pd=dres[2], ratio=dres[3], acc_margin=dres[4],
                margin_t=dres[5], margin_q=dres[6], cdf_margin=dres[7], token=int(ires[0]),
                cdf_lo=dnb[0], cdf_hi=dnb[1], tok_prev=int(dnb[2]), tok_next=int(dnb[3]),
                cut_t=tuple(int(v) for v in ires[1:4]), cut_q=tuple(int(v) for v in ires[4:7]),
                w_draw=w)


def verify_sample_rows(T, Q, d, tau, top_k=None, top_p=None, seed: int = 0, rows=None,
                       threads: int | None = None):
    """verify_sample on a subset of rows (each with its own Philox row counter), spread
    over host threads.  Returns the same dict restricted to ``rows`` (in that order)."""
    from concurrent.futures import ThreadPoolExecutor
    B = T.shape[0]
    rows = list(range(B)) if rows is None else [int(r) for r in rows]
    tk = None if top_k is None else np.asarray(top_k, dtype=np.int32)
    tp = None if top_p is None else np.asarray(top_p, dtype=np.float32)
    tau = np.asarray(tau, dtype=np.float32)

    def one(r):
        return verify_sample(T[r:r + 1], None if Q is None else Q[r:r + 1], d[r:r + 1], tau[r:r + 1],
                             None if tk is None else tk[r:r + 1],
                             None if tp is None else tp[r:r + 1], seed=seed, row0=r)

    nthr = threads or max(1, min(len(rows), os.cpu_count() or 1))
    with ThreadPoolExecutor(nthr) as ex:
        res = list(ex.map(one, rows))
    keys = ["out", "num_accepted", "p_target", "p_draft", "margins"]
    merged = {k: np.concatenate([r[k] for r in res]) if res else None for k in keys}
    merged["status"] = int(np.bitwise_or.reduce([r["status"] for r in res])) if res else 0
    return merged


# ---------------------------------------------------------------- draft input

def draft_input(e, h, we, wh, W, eps: float, return_xnorm: bool = False):
    """e, h [M, H] bf16 bits; we, wh [H]; W [H, 2H] -> y [M, H] float64 (before rounding)."""
    e = np.ascontiguousarray(e, dtype=np.uint16)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    we = np.ascontiguousarray(we, dtype=np.uint16)
    wh = np.ascontiguousarray(wh, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    M, H = e.shape
    y = np.zeros((M, H), np.float64)
    xn = np.zeros((M, 2 * H), np.uint16) if return_xnorm else None
    _check(_load().orc_draft_input(_ptr(e), _ptr(h), _ptr(we), _ptr(wh), _ptr(W), M, H,
                                   float(eps), _ptr(y), _ptr(xn)), "draft_input")
    return (y, xn) if return_xnorm else y


def draft_input_at(e, h, we, wh, W, eps: float, tok, col):
    """Selected outputs y[tok[i], col[i]] of draft_input (float64)."""
    e = np.ascontiguousarray(e, dtype=np.uint16)
    h = np.ascontiguousarray(h, dtype=np.uint16)
    we = np.ascontiguousarray(we, dtype=np.uint16)
    wh = np.ascontiguousarray(wh, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    M, H = e.shape
    tok = np.ascontiguousarray(tok, dtype=np.int64)
    col = np.ascontiguousarray(col, dtype=np.int64)
    y = np.zeros(tok.size, np.float64)
    _check(_load().orc_draft_input_at(_ptr(e), _ptr(h), _ptr(we), _ptr(wh), _ptr(W), M, H,
                                      float(eps), _ptr(tok), _ptr(col), tok.size, _ptr(y)),
           "draft_input_at")
    return y


# ---------------------------------------------------------------- draft output layer

def lm_head_logits(hidden, W, tok, norm_w=None, eps: float = 0.0, with_absdot: bool = False):
    """Logits [len(tok), V] (float64) of the draft head's output layer for tokens `tok`:
    hidden [M, H] and W [V, H] bf16 bits, norm_w [H] bf16 bits or None (no normalisation).
    With `with_absdot`, also sum_k |W[v, k] x_k| per logit."""
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    nw = None if norm_w is None else np.ascontiguousarray(norm_w, dtype=np.uint16)
    M, H = hidden.shape
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError("W must be [V, H]")
    tok = np.ascontiguousarray(tok, dtype=np.int64)
    lg = np.zeros((tok.size, V), np.float64)
    ad = np.zeros((tok.size, V), np.float64) if with_absdot else None
    _check(_load().orc_lm_head_logits(_ptr(hidden), _ptr(nw), float(eps), _ptr(W), M, H, V,
                                      _ptr(tok), tok.size, _ptr(lg), _ptr(ad)), "lm_head_logits")
    return (lg, ad) if with_absdot else lg


def lm_head_greedy(hidden, W, norm_w=None, eps: float = 0.0):
    """(ids int32 [M], max logit float64 [M]) of the greedy draft from the output layer."""
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    nw = None if norm_w is None else np.ascontiguousarray(norm_w, dtype=np.uint16)
    M, H = hidden.shape
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError("W must be [V, H]")
    ids = np.zeros(M, np.int32)
    mx = np.zeros(M, np.float64)
    _check(_load().orc_lm_head_greedy(_ptr(hidden), _ptr(nw), float(eps), _ptr(W), M, H, V,
                                      _ptr(ids), _ptr(mx)), "lm_head_greedy")
    return ids, mx


def lm_head_topk(hidden, W, k: int, norm_w=None, eps: float = 0.0):
    """(ids int32 [M, k], logits float64 [M, k]): the k largest logits of each token in
    decreasing order, equal logits by increasing id."""
    hidden = np.ascontiguousarray(hidden, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    nw = None if norm_w is None else np.ascontiguousarray(norm_w, dtype=np.uint16)
    M, H = hidden.shape
    V = W.shape[0]
    if W.shape[1] != H:
        raise ValueError("W must be [V, H]")
    ids = np.zeros((M, k), np.int32)
    vals = np.zeros((M, k), np.float64)
    _check(_load().orc_lm_head_topk(_ptr(hidden), _ptr(nw), float(eps), _ptr(W), M, H, V, int(k),
                                    _ptr(ids), _ptr(vals)), "lm_head_topk")
    return ids, vals


# ---------------------------------------------------------------- post-verify state

def state_snapshot(state):
    """backup = a copy of state [B, row_bytes] (uint8)."""
    state = np.ascontiguousarray(state, dtype=np.uint8)
    B, rb = state.shape
    backup = np.zeros_like(state)
    _check(_load().orc_state_snapshot(_ptr(state), _ptr(backup), B, rb), "state_snapshot")
    return backup


def state_fixup(num_accepted, D: int, kv_before, state=None, backup=None, draft_kv_len=None):
    """The post-verify fix-up of each row.  Returns (kv_len, recompute, state after,
    draft_kv_len after, status); state/backup are uint8 [B, row_bytes] or None (no
    recurrent state)."""
    na = np.ascontiguousarray(num_accepted, dtype=np.int32)
    B = na.size
    kvb = np.ascontiguousarray(kv_before, dtype=np.int32)
    if state is None:
        st_arr, bk, rb = None, None, 0
    else:
        st_arr = np.array(state, dtype=np.uint8, copy=True, order="C")
        bk = np.ascontiguousarray(backup, dtype=np.uint8)
        rb = st_arr.shape[1]
    dk = None if draft_kv_len is None else np.array(draft_kv_len, dtype=np.int32, copy=True)
    kv = np.zeros(B, np.int32)
    rc = np.zeros(B, np.int32)
    status = np.zeros(1, np.int32)
    _check(_load().orc_state_fixup(_ptr(na), int(D), _ptr(kvb), _ptr(kv), _ptr(st_arr), _ptr(bk),
                                   B, rb, _ptr(dk), _ptr(rc), _ptr(status)), "state_fixup")
    return kv, rc, st_arr, dk, int(status[0])


# ---------------------------------------------------------------- draft steps

def draft_steps(embed, next_ids, hidden, enorm_w, hnorm_w, eh_proj_w, lm_head_w, D: int,
                eps: float, norm_w=None, positions=None):
    """D serial greedy draft steps with a stub block.  Returns (draft_ids int32 [M, D],
    hidden_out bf16 bits [D, M, H], status)."""
    u16 = lambda a: np.ascontiguousarray(a, dtype=np.uint16)
    embed, hidden, enorm_w, hnorm_w = u16(embed), u16(hidden), u16(enorm_w), u16(hnorm_w)
    eh_proj_w, lm_head_w = u16(eh_proj_w), u16(lm_head_w)
    nw = None if norm_w is None else u16(norm_w)
    ids = np.ascontiguousarray(next_ids, dtype=np.int32)
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32)
    M, H = hidden.shape
    V = embed.shape[0]
    out = np.zeros((M, D), np.int32)
    hout = np.zeros((D, M, H), np.uint16)
    status = np.zeros(1, np.int32)
    _check(_load().orc_draft_steps(_ptr(embed), _ptr(ids), _ptr(pos), _ptr(hidden), _ptr(enorm_w),
                                   _ptr(hnorm_w), _ptr(eh_proj_w), _ptr(nw), _ptr(lm_head_w),
                                   float(eps), M, H, V, int(D), _ptr(out), _ptr(hout),
                                   _ptr(status)), "draft_steps")
    return out, hout, int(status[0])
