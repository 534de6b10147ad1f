"""The oracle's pins catch plausible mistakes.  Each case copies the oracle, the tests and
the input generator into a temporary directory, plants one mistake in the oracle's C
source (a dropped term, a wrong sign, index or word, a transposed operand, an off-by-one),
and runs the oracle's pin tests there: they must fail.  The product library is neither
built nor touched."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, text in oracle/mtpspec_oracle.c, the planted mistake)
MUTATIONS = [
    ("top-p boundary not strict", "int keep = S < p;", "int keep = S <= p;"),
    ("hidden half first in the concatenation",
     "orc_rmsnorm_bf16(e + t * H, we, H, eps, x);\n        orc_rmsnorm_bf16(h + t * H, wh, H, eps, x + H);",
     "orc_rmsnorm_bf16(h + t * H, wh, H, eps, x);\n        orc_rmsnorm_bf16(e + t * H, we, H, eps, x + H);"),
    ("argmax ties to the highest id", "if (v > bv) {", "if (v >= bv) {"),
    ("residual q - p", "double r = wp[i] / Zp - wq[i] / Zq;", "double r = wq[i] / Zq - wp[i] / Zp;"),
    ("accept test flipped", "accept = ua <= ratio;", "accept = ua >= ratio;"),
    ("top-k threshold off by one", "theta = s[k - 1].v;", "theta = s[k].v;"),
    ("Philox round word", "uint32_t n0 = hi1 ^ c1 ^ k0;", "uint32_t n0 = lo1 ^ c1 ^ k0;"),
    ("bonus drawn at position D-1",
     "rc = orc_unit(rowT + (size_t)D * (size_t)V * es, NULL,",
     "rc = orc_unit(rowT + (size_t)(D - 1) * (size_t)V * es, NULL,"),
    ("RMSNorm of the sum, not the mean", "double r = 1.0 / sqrt(ss / (double)H + eps);",
     "double r = 1.0 / sqrt(ss + eps);"),
    ("temperature dropped", "double wi = exp((s[kept].v - m) / tau);",
     "double wi = exp((s[kept].v - m));"),
    ("accept uniform from another word", "*u_acc = word_to_uniform(o[0]);",
     "*u_acc = word_to_uniform(o[2]);"),
    ("accept and draw share a word", "*u_smp = word_to_uniform(o[1]);",
     "*u_smp = word_to_uniform(o[0]);"),
    ("normalised activations not rounded to bf16",
     "out[i] = bf16_bits_to_double(orc_double_to_bf16(y));", "out[i] = y;"),
    ("draft outside q's support not accepted", "} else if (!inq[dj]) {", "} else if (0) {"),
    ("rejection draws from p, not the residual", "tok = orc_inverse_cdf_nb(wr, V, us, &dm, o->nb);",
     "tok = orc_inverse_cdf_nb(wp, V, us, &dm, o->nb);"),
    ("inverse CDF from the top id",
     "for (int64_t i = 0; i < V; ++i) {\n        double prev = c;",
     "for (int64_t i = V - 1; i >= 0; --i) {\n        double prev = c;"),
    ("output layer without its final norm",
     "if (norm_w)\n            orc_rmsnorm_bf16(h, norm_w, H, eps, x);",
     "if (0)\n            orc_rmsnorm_bf16(h, norm_w, H, eps, x);"),
    ("output-layer pick ties to the highest id", "if (lg[v] > lg[best])", "if (lg[v] >= lg[best])"),
    ("output-layer sum drops the last element",
     "for (int64_t k = 0; k < H; ++k) {\n                double pr",
     "for (int64_t k = 0; k < H - 1; ++k) {\n                double pr"),
    ("top-k of the output layer ties to the highest id", "(best < 0 || lg[v] > lg[best])",
     "(best < 0 || lg[v] >= lg[best])"),
    ("a hit keeps D positions", "kv = kv_before[b] + D + 1;", "kv = kv_before[b] + D;"),
    ("recompute omits the carried-in token", "rc = 1 + a;", "rc = a;"),
    ("a miss without recurrent state keeps a positions", "kv = kv_before[b] + 1 + a;",
     "kv = kv_before[b] + a;"),
    ("the draft head's KV is not cut on a miss",
     "if (draft_kv_len && miss && draft_kv_len[b] > kv)", "if (0)"),
    ("position-0 mask at every step", "positions[t] + k == 0", "positions[t] == 0"),
    ("a draft step's output not passed on as the next hidden state",
     "            h[i] = orc_double_to_bf16(y[i]);", "            (void)y[i];"),
    ("top-p alternatives: the upper end of the window on the wrong side",
     "if (S < p + delta)\n                ghi = gi;", "if (S < p - delta)\n                ghi = gi;"),
    ("top-p alternatives: a forced cut ignored", "keep = gi <= force_groups;", "keep = keep;"),
    ("draw neighbours: the next id skips one",
     "for (int64_t i = tok + 1; i < V; ++i)", "for (int64_t i = tok + 2; i < V; ++i)"),
    ("draw margins: the distances swapped", "lo = a;\n            hi = b;",
     "lo = b;\n            hi = a;"),
]


def _copy(dst):
    ignore = shutil.ignore_patterns("_build", "__pycache__", "*.so", "*.o")
    for d in ("oracle", "tests", "verify_spec_greedy_gb300"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d), ignore=ignore)
    for f in ("pytest.ini", "bench.py"):
        if os.path.exists(os.path.join(ROOT, f)):
            shutil.copy(os.path.join(ROOT, f), dst)


def _pin_run(dst, text=None, mistake=None):
    """Copy into dst, plant the mistake (if any), run the oracle's pin tests there; returns
    (exit code, the last lines of their output) or raises when the text is not unique."""
    _copy(dst)
    if text is not None:
        src = os.path.join(dst, "oracle", "mtpspec_oracle.c")
        s = open(src).read()
        if s.count(text) != 1:
            raise AssertionError("the text to change is not unique in the oracle")
        open(src, "w").write(s.replace(text, mistake))
    tests = sorted(os.path.join("tests", f) for f in os.listdir(os.path.join(dst, "tests"))
                   if f.startswith("test_oracle_") and f.endswith(".py")
                   and f != "test_oracle_mutations.py")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *tests], cwd=dst, capture_output=True, text=True, timeout=900)
    return r.returncode, r.stdout[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every case (and the unchanged control) run at once, one process each, spread over
    the host cores."""
    from concurrent.futures import ThreadPoolExecutor
    jobs = {None: (None, None)}
    jobs.update({name: (text, mistake) for name, text, mistake in MUTATIONS})
    base = tmp_path_factory.mktemp("pins")

    def run(item):
        i, (name, (text, mistake)) = item
        try:
            return name, _pin_run(str(base / f"case{i}"), text, mistake)
        except AssertionError as e:
            return name, (None, str(e))
    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        return dict(ex.map(run, enumerate(jobs.items())))


@pytest.mark.parametrize("name", [m[0] for m in MUTATIONS])
def test_a_planted_mistake_fails_a_pin(outcomes, name):
    code, out = outcomes[name]
    assert code == 1, f"{name}: no pin failed (exit code {code})\n{out}"


def test_the_copy_without_a_mistake_passes(outcomes):
    # the control: the same copy and command, unchanged, pass
    code, out = outcomes[None]
    assert code == 0, out
