"""The C-ABI library loads on any host and exports every entry point its header
declares; host-side argument checks answer before any CUDA call (no GPU needed)."""
import ctypes as C
import os
import re

import pytest

import verify_spec_greedy_gb300 as lib
from verify_spec_greedy_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def so():
    cuda_build.build()
    return lib.load()


def _declared():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                            src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    assert _declared() == sorted([
        "mtp_draft_input", "mtp_draft_input_workspace_bytes", "mtp_greedy_draft",
        "mtp_lm_head_greedy", "mtp_lm_head_greedy_workspace_bytes", "mtp_lm_head_topk",
        "mtp_lm_head_topk_workspace_bytes",
        "mtp_state_snapshot", "mtp_state_fixup", "mtp_draft_steps",
        "mtp_draft_steps_workspace_bytes",
        "spec_verify_greedy", "spec_verify_sample", "spec_verify_workspace_bytes",
        "spec_verify_sample_static", "mtpspec_status_string", "mtpspec_launch_count",
        "mtpspec_selftest_wait_timeout"])


def test_every_declared_symbol_is_exported(so):
    for name in _declared():
        assert hasattr(so, name), name


def test_status_strings(so):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.status_string(code).startswith("MTPSPEC")
    assert "unknown" in lib.status_string(42)


def test_host_side_validation(so):
    nul = None
    assert so.mtp_greedy_draft(nul, 7, 1, 10, nul, nul) == -2           # dtype
    assert so.mtp_greedy_draft(nul, 0, 1, 0, nul, nul) == -3            # V < 1
    assert so.mtp_greedy_draft(nul, 0, 0, 10, nul, nul) == 0            # empty: no work
    assert so.mtp_greedy_draft(nul, 0, 1, 10, nul, nul) == -1           # null pointers
    assert so.mtp_greedy_draft(C.c_void_p(2), 0, 1, 10, C.c_void_p(16), nul) == -1  # misaligned
    assert so.spec_verify_greedy(nul, 0, nul, 1, 0, 10, nul, nul, nul, nul) == -3   # D < 1
    assert so.spec_verify_greedy(nul, 0, nul, 1, 65, 10, nul, nul, nul, nul) == -3  # D > 64
    assert so.spec_verify_greedy(nul, 0, nul, 0, 3, 10, nul, nul, nul, nul) == 0    # B == 0
    assert so.spec_verify_greedy(nul, 1, nul, 2, 3, 10, nul, nul, nul, nul) == -1
    assert so.spec_verify_greedy(nul, 0, nul, 1, 1, 2**31, nul, nul, nul, nul) == -3


def test_sampling_vocabulary_limit(so):
    # a cluster stages V up to 407,552 (fp32) or 815,104 (bf16) with draft logits, 651,776
    # or 1,303,552 one-hot; beyond that the chunked verifier takes V up to 256 chunks of
    # 32 KB of logits (2,097,152 fp32, 4,194,304 bf16) in either mode.  An empty batch
    # (B = 0) passes every check that does not touch device memory
    nul, draft = None, C.c_void_p(256)
    for dq, dtype, vmax in ((draft, 0, 2097152), (draft, 1, 4194304), (nul, 0, 2097152),
                            (nul, 1, 4194304)):
        args = lambda V: (nul, dq, dtype, nul, nul, nul, nul, 0, 0, 1, V, nul, nul, nul, nul,
                          nul, 0, nul, nul)
        assert so.spec_verify_sample(*args(407553)) == 0
        assert so.spec_verify_sample(*args(vmax)) == 0
        assert so.spec_verify_sample(*args(vmax + 1)) == -3
    # the workspace query knows neither the logit type nor the mode: it refuses what no
    # combination accepts, and past the cluster limits it counts the chunked verifier's
    # coordination slots
    assert so.spec_verify_workspace_bytes(1, 1, 4194304) > 0
    assert so.spec_verify_workspace_bytes(1, 1, 4194305) == 0
    assert so.spec_verify_workspace_bytes(8, 3, 407553) > so.spec_verify_workspace_bytes(8, 3, 407552)


def test_lm_head_greedy_host_checks(so):
    nul = None
    f = so.mtp_lm_head_greedy
    ok = (C.c_void_p(256), nul, 1e-6, C.c_void_p(512), 4, 64, 1000, C.c_void_p(1024), nul,
          C.c_void_p(4096), 1 << 20, nul, nul)
    def call(**kw):
        names = ["hidden", "norm_w", "eps", "W", "M", "H", "V", "ids", "logit", "ws", "wsb",
                 "status", "stream"]
        a = dict(zip(names, ok))
        a.update(kw)
        return f(*[a[n] for n in names])
    assert call(H=12) == -3                      # H % 8
    assert call(H=0) == -3
    assert call(V=0) == -3
    assert call(V=65535 * 128 + 1) == -3         # past the vocabulary tiles of one grid
    assert call(M=-1) == -3
    assert call(eps=-1.0) == -1
    assert call(M=0) == 0                        # nothing to do
    assert call(hidden=nul) == -1
    assert call(W=C.c_void_p(520)) == -1         # not 16-byte aligned
    assert call(ids=C.c_void_p(1026)) == -1
    assert call(ws=nul) == -4
    assert call(wsb=100) == -4
    assert call(ws=C.c_void_p(4100)) == -4       # not 256-byte aligned
    need = so.mtp_lm_head_greedy_workspace_bytes(4, 64, 1000)
    assert need == 256 + 1024 + 4 * 4 * 8   # keys: 4 tokens x 4 blocks of 256 ids
    assert so.mtp_lm_head_greedy_workspace_bytes(4, 12, 1000) == 0
    assert so.mtp_lm_head_greedy_workspace_bytes(0, 64, 1000) == 0


def test_lm_head_topk_host_checks(so):
    nul, p = None, C.c_void_p(4096)
    f = so.mtp_lm_head_topk
    args = lambda **kw: [kw.get(n, d) for n, d in (("h", p), ("nw", nul), ("eps", 1e-6), ("W", p),
                                                   ("M", 4), ("H", 64), ("V", 1000), ("k", 4),
                                                   ("ids", p), ("lg", nul), ("ws", p),
                                                   ("wsb", 1 << 30), ("st", nul), ("s", nul))]
    assert f(*args(k=0)) == -3
    assert f(*args(k=9)) == -3                   # at most 8
    assert f(*args(k=4, V=3)) == -3              # k <= V
    assert f(*args(M=0)) == 0
    assert f(*args(ids=nul)) == -1
    assert f(*args(wsb=64)) == -4
    assert so.mtp_lm_head_topk_workspace_bytes(4, 64, 1000) == 256 + 1024 + 4 * 4 * 8 * 8
    assert so.mtp_lm_head_topk_workspace_bytes(4, 60, 1000) == 0


def test_state_host_checks(so):
    nul, p16, q16 = None, C.c_void_p(4096), C.c_void_p(1 << 20)
    snap = so.mtp_state_snapshot
    assert snap(p16, q16, 2, 24, nul) == -3          # row_bytes % 16
    assert snap(p16, q16, -1, 32, nul) == -3
    assert snap(nul, nul, 0, 32, nul) == 0           # nothing to copy
    assert snap(nul, nul, 3, 0, nul) == 0
    assert snap(nul, q16, 2, 32, nul) == -1
    assert snap(C.c_void_p(4100), q16, 2, 32, nul) == -1   # misaligned
    assert snap(p16, C.c_void_p(4096 + 32), 2, 32, nul) == -1  # overlapping
    fix = so.mtp_state_fixup
    i4 = C.c_void_p(256)
    assert fix(i4, 0, i4, i4, nul, nul, 1, 0, nul, nul, nul, nul) == -3    # D < 1
    assert fix(i4, 65, i4, i4, nul, nul, 1, 0, nul, nul, nul, nul) == -3   # D > 64
    assert fix(i4, 3, i4, i4, p16, q16, 1, 40, nul, nul, nul, nul) == -3   # row_bytes % 16
    assert fix(nul, 3, nul, nul, nul, nul, 0, 0, nul, nul, nul, nul) == 0  # B == 0
    assert fix(nul, 3, i4, i4, nul, nul, 2, 0, nul, nul, nul, nul) == -1   # no counts
    assert fix(i4, 3, i4, i4, nul, q16, 2, 32, nul, nul, nul, nul) == -1   # state missing
    assert fix(i4, 3, i4, C.c_void_p(258), nul, nul, 2, 0, nul, nul, nul, nul) == -1


def test_draft_steps_host_checks(so):
    nul, p = None, C.c_void_p(4096)
    f = so.mtp_draft_steps
    names = ["E", "ids", "pos", "h", "we", "wh", "W", "nw", "L", "eps", "M", "H", "V", "D",
             "out", "hout", "ws", "wsb", "status", "stream"]
    ok = dict(E=p, ids=p, pos=nul, h=p, we=p, wh=p, W=p, nw=nul, L=p, eps=1e-6, M=4, H=64,
              V=100, D=3, out=p, hout=nul, ws=p, wsb=1 << 30, status=nul, stream=nul)
    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(*[a[n] for n in names])
    assert call(D=0) == -3
    assert call(D=65) == -3
    assert call(H=20) == -3
    assert call(V=0) == -3
    assert call(eps=-1.0) == -1
    assert call(M=0) == 0
    assert call(E=nul) == -1
    assert call(L=C.c_void_p(4104)) == -1
    assert call(out=C.c_void_p(4098)) == -1
    assert call(ws=nul) == -4
    assert call(wsb=16) == -4
    assert so.mtp_draft_steps_workspace_bytes(4, 64, 100) > 0
    assert so.mtp_draft_steps_workspace_bytes(4, 60, 100) == 0


def test_launch_count_starts_at_zero_on_the_host(so):
    assert lib.mtpspec_launch_count() >= 0


def test_wait_selftest_host_checks(so):
    f = so.mtpspec_selftest_wait_timeout
    st = C.c_void_p(256)
    assert f(3, 100, st, None) == -1        # which
    assert f(-1, 100, st, None) == -1
    assert f(0, 0, st, None) == -1          # limit
    assert f(0, (1 << 20) + 1, st, None) == -1
    assert f(0, 100, None, None) == -1      # status
    assert f(0, 100, C.c_void_p(258), None) == -1  # misaligned
