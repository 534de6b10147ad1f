"""Host logic of bench.py, on the CPU: the algorithmic byte counts behind the roofline,
the ncu traffic lookup, the reference arm's row pool and the clock-sample parsing."""
import pytest

import bench
from verify_spec_greedy_gb300.inputs import WORKLOADS, make_verify_inputs


@pytest.fixture(scope="module")
def serve():
    w = WORKLOADS["serve_b256_d3_v152k"]
    return w, make_verify_inputs(w)


def test_verify_bytes_of_the_serving_call(serve):
    # 256 rows x 4 target rows, 192 sampled rows x 3 draft rows, 151,936 fp32 logits each;
    # then draft ids, the three per-row parameters, out_tokens, num_accepted and the two
    # probability outputs
    w, x = serve
    logits = (256 * 4 + 192 * 3) * 151936 * 4
    small = 256 * 3 * 4 + 256 * 3 * 4 + 256 * 4 * 4 + 256 * 4 + 2 * 256 * 3 * 4
    assert bench.verify_bytes(x) == logits + small == 972407808


def test_draft_input_bytes_of_the_serving_step(serve):
    w, _ = serve
    H, M = 4096, 768
    assert bench.draft_input_bytes(w) == H * 2 * H * 2 + 2 * M * H * 2 + 2 * H * 2 + M * H * 2
    assert round(bench.draft_input_bytes(w) / 1e6, 1) == 86.0


def test_whole_job_value_counts_every_rank():
    assert bench.whole_job_value(1024, 600, 4, 1000.0) == pytest.approx(4 * 1024 * 600)


def test_profiled_traffic_needs_the_same_kernel_source(monkeypatch, tmp_path):
    prof = tmp_path / "p.md"
    prof.write_text("x\nkernel_source_sha256: abc\n\ndram_bytes_per_launch: 12345\n")
    monkeypatch.setattr(bench, "PROFILE_FILE", str(prof))
    monkeypatch.setattr(bench, "kernel_hash", lambda: "abc")
    assert bench.profiled_traffic(bench.DEFAULT_WORKLOAD) == 12345.0
    assert bench.profiled_traffic("sample_b8_d3_v152k") is None     # another workload
    monkeypatch.setattr(bench, "kernel_hash", lambda: "def")
    assert bench.profiled_traffic(bench.DEFAULT_WORKLOAD) is None   # the kernel changed


def test_committed_profile_matches_the_committed_kernel(serve):
    # the verify summary records the source it was taken on; bench reports its traffic
    # only while that source is unchanged.  That traffic is at most 1 % above the
    # algorithmic bytes, and at least the bytes every call must read: the greedy rows
    # whole, and every sampled row's first position (target and draft), which no rejection
    # can skip
    _, x = serve
    t = bench.profiled_traffic(bench.DEFAULT_WORKLOAD)
    B, D, V = x["B"], x["D"], x["V"]
    greedy = int((x["tau"] == 0).sum())
    floor = (greedy * (D + 1) + (B - greedy) * 2) * V * 4
    assert t is None or floor <= t <= 1.01 * bench.verify_bytes(x)


def test_reference_pool_keeps_the_mix(serve):
    _, x = serve
    rows = bench.sample_rows(x, 16)
    greedy = [r for r in rows if x["tau"][r] == 0]
    assert len(rows) == 16 and len(set(rows)) == 16 and len(greedy) == 4


class _Proc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def _sampler(lines):
    c = bench.ClockSampler(0)
    c.proc = _Proc("\n".join(lines) + "\n")
    return c.stop()


def test_clock_samples_give_the_median_and_the_active_reasons():
    ok = "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1980, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active"
    r = _sampler([ok, ok, capped])
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["samples"] == 3
    assert r["reasons"] == ["sw_power_cap"]
    hot = "0, 1500, 2070, 1000.0, 0x40, Not Active, Active, Not Active, Not Active"
    assert _sampler([ok, hot])["reasons"] == ["hw_thermal_slowdown"]
    # unreadable lines are skipped; no samples at all is reported as such
    assert _sampler(["garbage", ok])["samples"] == 1
    assert _sampler(["garbage"])["reasons"] == ["no samples"]


def test_oracle_sample_on_one_core(serve):
    from verify_spec_greedy_gb300.inputs import make_draft_input
    w, x = serve
    v, cores, sample, dt = bench.oracle_sample(x, make_draft_input(w), w, rows=4, threads=1)
    assert cores == 1 and v > 0 and dt > 0
    assert sample.startswith("4 of 256 rows (1 greedy)")
    m = bench.cpu_model()
    assert m is None or (isinstance(m, str) and m)


def test_main_adds_the_cpu_baseline_after_the_gpu_step(monkeypatch, capsys):
    # the GPU step replaced by a stub: what main() does after it (the oracle on all host
    # cores and on one, the CPU model) runs as on a GPU machine
    import json
    import sys
    from verify_spec_greedy_gb300.inputs import make_draft_input
    w = WORKLOADS["sample_b8_d3_v152k"]
    x = make_verify_inputs(w)
    di = make_draft_input(w)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--workload", w.name])
    monkeypatch.setattr(bench, "run_gpu", lambda args, rank, world, dist: ({"metric": "m"}, x, di, w))
    monkeypatch.setattr(bench, "measure_per_config", lambda dev, cached=None: {"stub": {}})
    monkeypatch.setattr(bench, "_current_device", lambda: None)
    assert bench.main() == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["per_config"] == {"stub": {}}
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["seconds"] >= 10.0
    assert cb["single_thread"]["value"] > 0 and "cpu_model" in cb
