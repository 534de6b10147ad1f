"""Benchmark of the libmtpspec hot path on GB300.

One step = one pass of the whole hot path over one batch of a synthetic workload:
  1. mtp_draft_input     the draft head's input stage for the batch's M tokens
  2. mtp_greedy_draft    greedy drafts of the greedy rows (written into their draft ids)
  3. spec_verify_sample  verification of every row (greedy rows by the greedy rule)
The default workload is the batched-serving one: 256 rows x 3 drafts over a 151,936-id
vocabulary in fp32 (a quarter of the rows greedy, the rest sampled at temperatures
U[0.5, 1.2] with top-p 0.9), 768 draft-input tokens of hidden size 4096.  Its inputs
(1.2 GB per step) are larger than L2, so every step reads them from HBM.

Metric: verify rows per second (a row is one (b, j) logit row of V; B*(D+1) per step).
Prints one JSON line.  `--impl reference` times the CPU oracle instead (a bounded sample
of the same workload on the host cores).  Multi-GPU: one process per GPU, each running
an independent replica (the rows of a batch are independent; no collective).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "verify rows/s (B·(D+1)·V logits) & HBM GB/s vs 8 TB/s roofline; 1×GB300"
UNIT = "rows/s"
DEFAULT_WORKLOAD = "serve_b256_d3_v152k"
L2_BYTES = 129 * 1024 * 1024
PROFILE_FILE = os.path.join(ROOT, "profiles", "verify_sample_serve_b256_d3_v152k.md")
KERNEL_SOURCES = ["verify_spec_greedy_gb300/csrc/verify_sample.cu",
                  "verify_spec_greedy_gb300/csrc/common.cuh",
                  "verify_spec_greedy_gb300/csrc/philox.cuh"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=600)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["libmtpspec", "reference"], default="libmtpspec")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload timings added to the JSON line")
    ap.add_argument("--no-launch-count", action="store_true",
                    help="accepted for older command lines; launches are counted by the library")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's row count (profiling on a smaller case)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the verify and the draft-input calls alone on every workload "
                         "(one JSON line each) instead of the benchmark step")
    ap.add_argument("--graph-batch", action="store_true",
                    help="time the verify call of each small workload as a CUDA graph of 20 "
                         "back-to-back calls on distinct input copies (one JSON line each)")
    ap.add_argument("--lm-head", type=int, nargs=3, metavar=("M", "H", "V"), default=None,
                    help="time mtp_lm_head_greedy alone on seeded random inputs of this size "
                         "(--warmup, then --steps calls, each after an L2 flush)")
    return ap.parse_args()


# ---------------------------------------------------------------- distributed plumbing

def dist_init(n):
    if n <= 1 or "RANK" not in os.environ:
        return 0, 1, None
    import torch
    import torch.distributed as dist
    local = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(local)
    dist.init_process_group("nccl")
    return dist.get_rank(), dist.get_world_size(), dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_step, steps, world, ms_max):
    """Units per second of the whole job: every rank runs its own replica of the step, so
    the job processes world x units_per_step x steps units in the slowest rank's time."""
    return world * units_per_step * steps / (ms_max / 1e3)


# ---------------------------------------------------------------- workload bytes

def verify_bytes(x):
    """Algorithmic bytes of one spec_verify_sample call: each target row read once, each
    draft row of a sampled row read once (greedy rows need no draft logits), plus the
    per-row inputs and outputs."""
    B, D, V = x["B"], x["D"], x["V"]
    es = 4 if x["dtype"] == "f32" else 2
    n_greedy = int((x["tau"] == 0).sum())
    t_rows = B * (D + 1)
    q_rows = (B - n_greedy) * D
    small = B * D * 4 + B * 4 * 3 + B * (D + 1) * 4 + B * 4 + 2 * B * D * 4
    return (t_rows + q_rows) * V * es + small


def l2_flush(buf):
    """Evict L2: write a buffer of twice its size, then read it back.  The read writes the
    flush's own dirty lines back to HBM before the timed region, so that the kernel timed
    next starts on a clean L2 that holds none of its inputs (as after another kernel's
    reads), instead of paying for a full L2 of write-backs."""
    buf.fill_(1.0)
    buf.sum()


def draft_input_bytes(w):
    return 2 * w.H * 2 * w.H + 2 * w.tokens * w.H * 2 + 2 * w.H * 2 + w.tokens * w.H * 2


# ---------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- roofline inputs

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch of the verify kernel from the committed ncu summary, if it
    was taken on this workload with the current kernel source; else None."""
    if not os.path.exists(PROFILE_FILE) or workload != DEFAULT_WORKLOAD:
        return None
    src, traffic = None, None
    for line in open(PROFILE_FILE):
        if line.startswith("kernel_source_sha256:"):
            src = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            try:
                traffic = float(line.split(":", 1)[1].strip())
            except ValueError:
                traffic = None
    return traffic if src == kernel_hash() else None


# ---------------------------------------------------------------- CPU oracle baseline

def optional_top_p(x, to_dev):
    """The workload's per-row top-p on the device, or None when no row filters (every p is
    1): the call then runs without top-p values, as it does without top-k values."""
    return None if (x["top_p"] >= 1.0).all() else to_dev(x["top_p"])


def sample_rows(x, rows):
    """`rows` rows of the verify with the workload's mix of greedy rows (temperature 0,
    the first ones of the batch) and sampled rows."""
    B = x["B"]
    ng = int((x["tau"] == 0).sum())
    n_g = max(1, round(rows * ng / B)) if ng else 0
    return list(range(n_g)) + list(range(ng, ng + rows - n_g))


def cpu_model():
    """The host CPU's model name (lscpu), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
    except (OSError, subprocess.SubprocessError):
        return None
    for line in out.splitlines():
        if line.strip().lower().startswith("model name:"):
            return line.split(":", 1)[1].strip()
    return None


def oracle_sample(x, di, w, rows, min_seconds=0.0, sel=None, threads=None):
    """Time the oracle on a bounded sample: `rows` rows of the verify (the workload's mix
    of greedy and sampled rows; or the rows `sel`) plus the draft-input tokens of those
    rows and the greedy drafts of the greedy rows among them, spread over the host cores;
    the sample is repeated until at least `min_seconds` have passed."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    cores = threads or os.cpu_count() or 1
    B = x["B"]
    if sel is None:
        sel = sample_rows(x, rows)
    greedy = [r for r in sel if x["tau"][r] == 0]
    n_g = len(greedy)
    tok_per_row = max(1, w.tokens // B)
    ntok = tok_per_row * len(sel)
    e, h = di["e"][0][:ntok], di["h"][0][:ntok]
    chunks = [(i, min(ntok, i + 4)) for i in range(0, ntok, 4)]
    passes = 0
    t0 = time.perf_counter()
    while True:
        with ThreadPoolExecutor(cores) as ex:
            futs = [ex.submit(oracle.draft_input, e[a:b], h[a:b], di["we"], di["wh"], di["W"],
                              di["eps"]) for a, b in chunks]
            if n_g:
                futs.append(ex.submit(oracle.greedy_draft,
                                      x["Q"][greedy].reshape(-1, x["V"])))
            for f in futs:
                f.result()
        oracle.verify_sample_rows(x["T"], x["Q"], x["d"], x["tau"], x["top_k"], x["top_p"],
                                  x["seed"], rows=sel, threads=cores)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    rows_verified = passes * len(sel) * (x["D"] + 1)
    sample = (f"{len(sel)} of {B} rows ({n_g} greedy) of {w.name}: their verify, their "
              f"{ntok} draft-input tokens and the greedy drafts of the greedy rows"
              + (f"; {passes} passes" if passes > 1 else ""))
    return rows_verified / dt, cores, sample, dt


# ---------------------------------------------------------------- the GPU arm

def run_gpu(args, rank, world, dist):
    import torch
    import verify_spec_greedy_gb300 as lib
    from verify_spec_greedy_gb300.inputs import WORKLOADS, make_draft_input, make_verify_inputs

    dev = torch.device("cuda", torch.cuda.current_device())
    w = WORKLOADS[args.workload]
    if args.batch:
        w = w.scaled(B=args.batch, M=(w.tokens * args.batch) // w.B if w.M else 0)
    x = make_verify_inputs(w)
    di = make_draft_input(w)
    B, D, V = x["B"], x["D"], x["V"]
    ng = int((x["tau"] == 0).sum())
    assert (x["tau"][:ng] == 0).all() and (x["tau"][ng:] > 0).all()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    step_bytes = verify_bytes(x) + draft_input_bytes(w) + ng * D * V * (4 if x["dtype"] == "f32" else 2)
    copies = max(1, math.ceil(3 * L2_BYTES / step_bytes))
    T0, Q0 = to_dev(x["T"]), to_dev(x["Q"])
    sets = []
    for c in range(copies):
        sets.append(dict(
            T=T0 if c == 0 else T0.clone(), Q=Q0 if c == 0 else Q0.clone(),
            d=to_dev(x["d"]), e=to_dev(di["e"][0]), h=to_dev(di["h"][0]),
            W=to_dev(di["W"]) if c == 0 else sets[0]["W"].clone()))
    tau, top_p = to_dev(x["tau"]), optional_top_p(x, to_dev)
    top_k = to_dev(x["top_k"]) if (x["top_k"] > 0).any() else None
    we, wh = to_dev(di["we"]), to_dev(di["wh"])
    M, H = w.tokens, w.H
    y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
    ws_di = torch.empty(max(1, lib.mtp_draft_input_workspace_bytes(M, H)), dtype=torch.uint8, device=dev)
    out = torch.empty((B, D + 1), dtype=torch.int32, device=dev)
    na = torch.empty(B, dtype=torch.int32, device=dev)
    pt = torch.empty((B, D), dtype=torch.float32, device=dev)
    pd = torch.empty((B, D), dtype=torch.float32, device=dev)
    ws_v = torch.empty(lib.spec_verify_workspace_bytes(B, D, V), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    ev_v = []

    def run_step(s, timed=False):
        lib.mtp_draft_input(s["e"], s["h"], we, wh, s["W"], y, di["eps"], ws_di)
        if ng:
            lib.mtp_greedy_draft(s["Q"][:ng].view(ng * D, V), s["d"][:ng].view(-1))
        if timed:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
        # as a decode loop calls it: the tokens and accepted counts, no per-position
        # probabilities (so positions behind a row's first rejection need not be read)
        lib.spec_verify_sample(s["T"], s["Q"], s["d"], tau, top_k, top_p, x["seed"], out, na,
                               None, None, ws_v, status)
        if timed:
            b.record(stream)
            ev_v.append((a, b))

    def step(i, timed=False):
        run_step(sets[i % copies], timed)

    for i in range(max(3, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"status word {int(status.item())}"

    # launches of this library's kernels inside the timed region, counted by the library
    clocks = ClockSampler(dev.index)
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = lib.mtpspec_launch_count()
    t_start.record(stream)
    for i in range(args.steps):
        step(i, timed=True)
    t_end.record(stream)
    launches = lib.mtpspec_launch_count() - launches0
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(dist)
    ms = t_start.elapsed_time(t_end)
    ms_max = max_over_ranks(ms, dist)
    verify_ms = statistics.mean(a.elapsed_time(b) for a, b in ev_v)
    rows_per_step = B * (D + 1)
    value = whole_job_value(rows_per_step, args.steps, world, ms_max)
    # the same call with p_target and p_draft requested: every draft position is computed
    pev = []
    for i in range(max(3, min(args.steps, 20))):
        s_ = sets[i % copies]
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        lib.spec_verify_sample(s_["T"], s_["Q"], s_["d"], tau, top_k, top_p, x["seed"], out, na,
                               pt, pd, ws_v, status)
        b.record(stream)
        pev.append((a, b))
    torch.cuda.synchronize()
    verify_p_ms = statistics.median(a.elapsed_time(b) for a, b in pev[2:])

    # end to end through the C ABI with host buffers: pinned inputs copied in, results out
    host_in = {k: torch.from_numpy(np.ascontiguousarray(
        v if v.dtype != np.uint16 else v.view(np.int16))).pin_memory()
        for k, v in dict(T=x["T"], Q=x["Q"], d=x["d"], e=di["e"][0], h=di["h"][0],
                         W=di["W"]).items()}
    host_out = dict(out=torch.empty((B, D + 1), dtype=torch.int32).pin_memory(),
                    na=torch.empty(B, dtype=torch.int32).pin_memory(),
                    y=torch.empty((M, H), dtype=torch.bfloat16).pin_memory())
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    # two device input sets: step i's inputs are copied in on a side stream while step i - 1
    # computes on the other set (the copies run at the host link's rate, the compute on
    # the GPU: each step waits for its own copy, each copy for the step that last read
    # its set); the results go back on the compute stream after their step
    e2e_sets = [sets[0], {k: v.clone() for k, v in sets[0].items()}]
    copy_stream = torch.cuda.Stream()
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_free = [torch.cuda.Event(), torch.cuda.Event()]

    def e2e_step(i):
        s = e2e_sets[i % 2]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_free[i % 2])
            for k in ("T", "Q", "d", "e", "h", "W"):
                dst = s[k] if s[k].dtype != torch.bfloat16 else s[k].view(torch.int16)
                dst.copy_(host_in[k], non_blocking=True)
            ev_in[i % 2].record(copy_stream)
        stream.wait_event(ev_in[i % 2])
        run_step(s)
        ev_free[i % 2].record(stream)
        host_out["out"].copy_(out, non_blocking=True)
        host_out["na"].copy_(na, non_blocking=True)
        host_out["y"].copy_(y, non_blocking=True)

    for i in range(2):
        ev_free[i].record(stream)
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)
    for i in range(args.e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist)
    e2e_value = whole_job_value(rows_per_step, args.e2e_steps, world, e2e_ms)

    peak, peak_kind = measured_peaks()
    vb = verify_bytes(x)
    achieved = vb / (verify_ms / 1e3) / 1e9
    traffic = profiled_traffic(args.workload)
    # achieved counts every unit's logits (the call's algorithmic bytes); the call skips the
    # positions behind a row's first rejection once it knows of it, so the DRAM bytes it
    # reads (traffic, from the committed ncu summary) are fewer: their rate is given beside
    roofline = {"bound": "hbm", "kernel": "spec_verify_sample: k_verify_rr + k_argmax_verify_rows + k_verify_finalize",
                "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "frac_vs_nominal_8tbs": round(achieved / 8000.0, 4),
                "algorithmic_bytes_per_launch": vb,
                "launch_ms": round(verify_ms, 5), "traffic": traffic,
                "traffic_frac": (round(traffic / (verify_ms / 1e3) / 1e9 / peak, 4)
                                 if traffic else None),
                "with_probabilities": {"launch_ms": round(verify_p_ms, 5),
                                       "frac": round(vb / (verify_p_ms / 1e3) / 1e9 / peak, 4)}}

    res = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": max(3, args.warmup),
           "ms_per_step": round(ms_max / args.steps, 5), "logits_per_s": round(value * V, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": x["dtype"],
           "data": "synthetic",
           "config": {"workload": w.name, "B": B, "D": D, "V": V, "H": H, "draft_tokens": M,
                      "greedy_rows": ng, "top_k": int(w.top_k), "top_p": float(w.top_p),
                      "logits": x["dtype"], "step": "mtp_draft_input + mtp_greedy_draft + "
                      "spec_verify_sample", "verify_outputs": "out_tokens, num_accepted",
                      "parallelism": f"replicas x{world}",
                      "l2": ("inputs larger than L2" if copies == 1 else
                             f"{copies} rotating input copies, {copies * step_bytes / 1e6:.0f} MB")},
           "clocks": clk,
           "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h},
           "gpu_launches": launches,
           "roofline": roofline}
    return res, x, di, w


def _current_device():
    import torch
    return torch.device("cuda", torch.cuda.current_device())


def measure_per_config(dev, cached=None, graph_calls=20, reps=15):
    """Every workload's verify and draft-input calls, timed in this run: each call alone
    after an L2 flush (`l2_flush`: a write and a read of twice the L2), replayed from a CUDA
    graph of that one call (median of `reps` replays); the calls whose inputs fit L2 also as
    a CUDA graph of `graph_calls` back-to-back calls on distinct copies of the inputs (after
    a flush; per-call time = replay / calls); and the sampled workloads' verify once more
    with one-hot drafts.  Fractions are of the measured
    peaks (HBM copy bandwidth, or bf16 tensor throughput for a contraction whose
    arithmetic intensity is above the ridge).  `cached` maps a workload name to inputs
    already made (x, di)."""
    import torch
    import verify_spec_greedy_gb300 as lib
    from verify_spec_greedy_gb300.inputs import WORKLOADS, make_draft_input, make_verify_inputs
    hbm, _ = measured_peaks()
    tflops = 1881.1
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        tflops = float(json.load(open(pk)).get("bf16_tflops", tflops))
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    cached = cached or {}

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            l2_flush(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    def timed_call(fn):
        # one call captured in a CUDA graph and replayed: the device time of the call's
        # kernels without the host's argument marshalling, which a single small call would
        # otherwise expose (the GPU idles while the launch is prepared)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(2):
                fn()
        stream.wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ms = timed(g.replay)
        del g
        return ms

    def roof(nbytes, ms):
        ach = nbytes / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(ach / hbm, 4), "bytes": int(nbytes)}

    res = {}
    for name, w in WORKLOADS.items():
        x, di = cached.get(name) or (make_verify_inputs(w), make_draft_input(w))
        B, D, V = x["B"], x["D"], x["V"]
        es = 4 if x["dtype"] == "f32" else 2
        T, d = to_dev(x["T"]), to_dev(x["d"])
        Q = None if w.mode == "greedy" else to_dev(x["Q"])
        out = torch.empty((B, D + 1), dtype=torch.int32, device=dev)
        na = torch.empty(B, dtype=torch.int32, device=dev)
        entry = {"B": B, "D": D, "V": V, "H": w.H, "logits": x["dtype"]}
        if w.mode == "greedy":
            def call(Ti=T, Qi=None, o=out, n=na, one_hot=False):
                lib.spec_verify_greedy(Ti, d, o, n)
            vbytes = B * (D + 1) * V * es
            entry["verify_call"] = "spec_verify_greedy"
        else:
            tau, top_p = to_dev(x["tau"]), optional_top_p(x, to_dev)
            top_k = to_dev(x["top_k"]) if (x["top_k"] > 0).any() else None
            ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, V), dtype=torch.uint8,
                             device=dev)

            def call(Ti=T, Qi=Q, o=out, n=na, one_hot=False):
                lib.spec_verify_sample(Ti, None if one_hot else Qi, d, tau, top_k, top_p,
                                       x["seed"], o, n, None, None, ws)
            vbytes = verify_bytes(x)
            entry["verify_call"] = "spec_verify_sample"
        vms = timed_call(call)
        entry["verify_us"] = round(vms * 1e3, 2)
        entry["verify_rows_per_s"] = round(B * (D + 1) / (vms / 1e3), 1)
        entry["verify_roofline"] = roof(vbytes, vms)
        if w.mode != "greedy":
            # with p_target and p_draft requested: every draft position is computed
            ptp = torch.empty((B, D), device=dev)
            pdp = torch.empty((B, D), device=dev)
            pms = timed_call(lambda: lib.spec_verify_sample(T, Q, d, tau, top_k, top_p, x["seed"],
                                                            out, na, ptp, pdp, ws))
            entry["verify_with_probabilities_us"] = round(pms * 1e3, 2)
        if vbytes < L2_BYTES:
            # back-to-back calls as a decode loop issues them: a CUDA graph of calls, each on
            # its own copy of the logits
            Ts = [T] + [T.clone() for _ in range(graph_calls - 1)]
            Qs = None if Q is None else [Q] + [Q.clone() for _ in range(graph_calls - 1)]
            outs = [torch.empty_like(out) for _ in range(graph_calls)]
            nas = [torch.empty_like(na) for _ in range(graph_calls)]
            calls = [lambda i=i: call(Ts[i], None if Qs is None else Qs[i], outs[i], nas[i])
                     for i in range(graph_calls)]
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for c in calls:
                    c()
            stream.wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for c in calls:
                    c()
            gms = timed(graph.replay) / graph_calls
            entry["verify_graph_batch"] = {"calls": graph_calls, "us_per_call": round(gms * 1e3, 2),
                                           "rows_per_s": round(B * (D + 1) / (gms / 1e3), 1),
                                           "roofline": roof(vbytes, gms)}
            del graph, Ts, Qs
        if w.mode != "greedy":
            oms = timed_call(lambda: call(one_hot=True))
            ob = vbytes - (B - int((x["tau"] == 0).sum())) * D * V * es
            entry["one_hot_verify"] = {"us": round(oms * 1e3, 2),
                                       "rows_per_s": round(B * (D + 1) / (oms / 1e3), 1),
                                       "roofline": roof(ob, oms)}
        M, H = w.tokens, w.H
        e, h = to_dev(di["e"][0][:M]), to_dev(di["h"][0][:M])
        we, wh, W = to_dev(di["we"]), to_dev(di["wh"]), to_dev(di["W"])
        y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        wsd = torch.empty(max(1, lib.mtp_draft_input_workspace_bytes(M, H)), dtype=torch.uint8,
                          device=dev)
        dms = timed_call(lambda: lib.mtp_draft_input(e, h, we, wh, W, y, di["eps"], wsd))
        dbytes = draft_input_bytes(w)
        dflop = 2.0 * M * H * 2 * H
        if dflop / dbytes > tflops * 1e12 / (hbm * 1e9):
            ach = dflop / (dms / 1e3) / 1e12
            droof = {"bound": "tensor", "achieved": round(ach, 1), "peak": tflops,
                     "unit": "TFLOP/s", "frac": round(ach / tflops, 4), "flop": dflop}
        else:
            droof = roof(dbytes, dms)
        entry["draft_input"] = {"tokens": M, "us": round(dms * 1e3, 2),
                                "tokens_per_s": round(M / (dms / 1e3), 1), "roofline": droof}
        if droof["bound"] == "hbm" and dbytes < L2_BYTES:
            # back-to-back calls in a CUDA graph, each on its own copy of the weight (read
            # from HBM: the copies together exceed what one call leaves in L2 and the replay
            # starts after a flush)
            Ws = [W] + [W.clone() for _ in range(graph_calls - 1)]
            ys = [torch.empty_like(y) for _ in range(graph_calls)]
            wss = [torch.empty_like(wsd) for _ in range(graph_calls)]
            dcalls = [lambda i=i: lib.mtp_draft_input(e, h, we, wh, Ws[i], ys[i], di["eps"], wss[i])
                      for i in range(graph_calls)]
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for c in dcalls:
                    c()
            stream.wait_stream(side)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for c in dcalls:
                    c()
            gms = timed(graph.replay) / graph_calls
            entry["draft_input"]["graph_batch"] = {
                "calls": graph_calls, "us_per_call": round(gms * 1e3, 2),
                "tokens_per_s": round(M / (gms / 1e3), 1), "roofline": roof(dbytes, gms)}
            del graph, Ws
        res[name] = entry
        del T, Q
    return res


def run_sweep(args):
    """Per workload: one verify call (spec_verify_greedy for a greedy workload, else
    spec_verify_sample), one mtp_draft_input call of its draft-token count and one
    mtp_lm_head_greedy call of one token per row, the state snapshot and fix-up, and
    mtp_draft_steps (D steps, replayed from a CUDA graph), each timed
    alone with CUDA events after an L2 flush (`l2_flush`), median of the
    launches; rows/s, tokens/s and the fraction of the roofline that bounds each."""
    import numpy as np
    import torch
    import verify_spec_greedy_gb300 as lib
    from verify_spec_greedy_gb300.inputs import WORKLOADS, make_draft_input, make_verify_inputs
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm, hbm_kind = measured_peaks()
    tflops = 1881.1
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        tflops = float(json.load(open(pk)).get("bf16_tflops", tflops))
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def timed(fn, n):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(n):
            l2_flush(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    for name, w in WORKLOADS.items():
        x = make_verify_inputs(w)
        di = make_draft_input(w)
        B, D, V = x["B"], x["D"], x["V"]
        T, Q, d = to_dev(x["T"]), to_dev(x["Q"]), to_dev(x["d"])
        out = torch.empty((B, D + 1), dtype=torch.int32, device=dev)
        na = torch.empty(B, dtype=torch.int32, device=dev)
        if w.mode == "greedy":
            vfn = lambda: lib.spec_verify_greedy(T, d, out, na)
            vbytes = B * (D + 1) * V * (4 if x["dtype"] == "f32" else 2)
            vcall = "spec_verify_greedy"
        else:
            tau, top_p = to_dev(x["tau"]), optional_top_p(x, to_dev)
            top_k = to_dev(x["top_k"]) if (x["top_k"] > 0).any() else None
            ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, V), dtype=torch.uint8, device=dev)
            vfn = lambda: lib.spec_verify_sample(T, Q, d, tau, top_k, top_p, x["seed"], out, na,
                                                 None, None, ws)
            vbytes = verify_bytes(x)
            vcall = "spec_verify_sample"
            # the same rows with a one-hot draft (no draft logits are read)
            ofn = lambda: lib.spec_verify_sample(T, None, d, tau, top_k, top_p, x["seed"], out,
                                                 na, None, None, ws)
            ob = vbytes - (B - int((x["tau"] == 0).sum())) * D * V * (4 if x["dtype"] == "f32" else 2)
            oms = timed(ofn, 20)
            oach = ob / (oms / 1e3) / 1e9
            one_hot = {"ms": round(oms, 4), "rows_per_s": round(B * (D + 1) / (oms / 1e3), 1),
                       "roofline": {"bound": "hbm", "achieved": round(oach, 1), "peak": hbm,
                                    "unit": "GB/s", "frac": round(oach / hbm, 4), "bytes": ob}}
        vms = timed(vfn, 20)
        M, H = w.tokens, w.H  # tokens of one draft-input call
        e, h = to_dev(di["e"][0][:M]), to_dev(di["h"][0][:M])
        we, wh, W = to_dev(di["we"]), to_dev(di["wh"]), to_dev(di["W"])
        y = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        wsd = torch.empty(max(1, lib.mtp_draft_input_workspace_bytes(M, H)), dtype=torch.uint8, device=dev)
        dms = timed(lambda: lib.mtp_draft_input(e, h, we, wh, W, y, di["eps"], wsd), 20)
        dbytes = 2 * H * 2 * H + 2 * M * H * 2 + 2 * H * 2 + M * H * 2
        dflop = 2.0 * M * H * 2 * H
        tensor = dflop / dbytes > tflops * 1e12 / (hbm * 1e9)
        if tensor:
            droof = {"bound": "tensor", "achieved": round(dflop / (dms / 1e3) / 1e12, 1),
                     "peak": tflops, "unit": "TFLOP/s"}
        else:
            droof = {"bound": "hbm", "achieved": round(dbytes / (dms / 1e3) / 1e9, 1),
                     "peak": hbm, "unit": "GB/s"}
        droof["frac"] = round(droof["achieved"] / droof["peak"], 4)
        # the draft step's output layer with the greedy pick: one token per row, the
        # workload's hidden size and vocabulary (seeded random stand-ins for the weights);
        # beside it, the same pick through a cuBLAS product and torch.argmax, for context
        Ml, Hl = B, H
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed + 77)
        hl = torch.randn((Ml, Hl), device=dev, generator=gen).to(torch.bfloat16)
        Wl = (torch.randn((V, Hl), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
        nl = (1.0 + 0.1 * torch.randn((Hl,), device=dev, generator=gen)).to(torch.bfloat16)
        idl = torch.empty(Ml, dtype=torch.int32, device=dev)
        wsl = torch.empty(lib.mtp_lm_head_greedy_workspace_bytes(Ml, Hl, V), dtype=torch.uint8, device=dev)
        lms = timed(lambda: lib.mtp_lm_head_greedy(hl, Wl, idl, norm_w=nl, eps=1e-6, workspace=wsl), 20)

        def lib_pick():
            xf = hl.float()
            xn = (xf * torch.rsqrt((xf * xf).mean(-1, keepdim=True) + 1e-6) * nl.float()).to(torch.bfloat16)
            return torch.argmax(xn @ Wl.t(), dim=-1)
        cms = timed(lib_pick, 10)
        # the k = 8 largest logits of each token from the same layer
        idk = torch.empty((Ml, 8), dtype=torch.int32, device=dev)
        wsk = torch.empty(lib.mtp_lm_head_topk_workspace_bytes(Ml, Hl, V), dtype=torch.uint8, device=dev)
        kms = timed(lambda: lib.mtp_lm_head_topk(hl, Wl, idk, norm_w=nl, eps=1e-6, workspace=wsk), 20)
        # the serial draft loop: D steps of one token per row (embedding gather with the
        # position-0 mask, input stage, stub block, output-layer pick), replayed from one
        # CUDA graph
        El = (torch.randn((V, Hl), device=dev, generator=gen) * 0.5).to(torch.bfloat16)
        ids0 = torch.randint(0, V, (Ml,), dtype=torch.int32, device=dev, generator=gen)
        pos0 = torch.randint(0, 4, (Ml,), dtype=torch.int32, device=dev, generator=gen)
        dids = torch.empty((Ml, D), dtype=torch.int32, device=dev)
        wss = torch.empty(lib.mtp_draft_steps_workspace_bytes(Ml, Hl, V), dtype=torch.uint8, device=dev)
        we_s, wh_s = to_dev(di["we"]), to_dev(di["wh"])
        Wp_s = to_dev(di["W"])
        steps_call = lambda: lib.mtp_draft_steps(El, ids0, hl, we_s, wh_s, Wp_s, Wl, dids, 1e-6,
                                                 norm_w=nl, positions=pos0, workspace=wss)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            steps_call()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            steps_call()
        graph.replay()
        torch.cuda.synchronize()
        sms_ = timed(graph.replay, 10)
        sbytes_ = D * (V * Hl * 2 + 2 * Hl * 2 * Hl * 2 + 6 * Ml * Hl * 2)
        steps = {"M": Ml, "D": D, "ms": round(sms_, 4),
                 "draft_tokens_per_s": round(Ml * D / (sms_ / 1e3), 1), "graph": True,
                 "roofline": {"bound": "hbm", "achieved": round(sbytes_ / (sms_ / 1e3) / 1e9, 1),
                              "peak": hbm, "unit": "GB/s",
                              "frac": round(sbytes_ / (sms_ / 1e3) / 1e9 / hbm, 4), "bytes": sbytes_}}
        del Wl, El, graph
        lbytes = V * Hl * 2 + 2 * Ml * Hl * 2 + Hl * 2 + Ml * 4
        lflop = 2.0 * Ml * Hl * V
        if lflop / (tflops * 1e12) > lbytes / (hbm * 1e9):
            lroof = {"bound": "tensor", "achieved": round(lflop / (lms / 1e3) / 1e12, 1),
                     "peak": tflops, "unit": "TFLOP/s"}
        else:
            lroof = {"bound": "hbm", "achieved": round(lbytes / (lms / 1e3) / 1e9, 1),
                     "peak": hbm, "unit": "GB/s"}
        lroof["frac"] = round(lroof["achieved"] / lroof["peak"], 4)
        vach = vbytes / (vms / 1e3) / 1e9
        # the state around the verification: a snapshot of each row's recurrent state (the
        # pages' 19 MiB of memory tables and convolution windows) and the fix-up with this
        # workload's accepted counts (misses copy their row back)
        rb = 19 << 20
        S = torch.empty((B, rb), dtype=torch.uint8, device=dev)
        S.fill_(7)
        Sb = torch.empty_like(S)
        kv0 = torch.zeros(B, dtype=torch.int32, device=dev)
        kv1 = torch.empty_like(kv0)
        sms = timed(lambda: lib.mtp_state_snapshot(S, Sb), 10)
        fms = timed(lambda: lib.mtp_state_fixup(na, D, kv0, kv1, S, Sb), 10)
        nmiss = int((na < D).sum().item())
        del S, Sb
        sbytes, fbytes = 2 * B * rb, 2 * nmiss * rb + B * 12
        state = {"row_bytes": rb,
                 "snapshot": {"ms": round(sms, 4), "roofline": {
                     "bound": "hbm", "achieved": round(sbytes / (sms / 1e3) / 1e9, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(sbytes / (sms / 1e3) / 1e9 / hbm, 4), "bytes": sbytes}},
                 "fixup": {"ms": round(fms, 4), "rows_restored": nmiss, "roofline": {
                     "bound": "hbm", "achieved": round(fbytes / (fms / 1e3) / 1e9, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(fbytes / (fms / 1e3) / 1e9 / hbm, 4), "bytes": fbytes}}}
        print(json.dumps({
            "sweep": name, "dtype": x["dtype"], "B": B, "D": D, "V": V, "H": H,
            "verify": {"call": vcall, "ms": round(vms, 4),
                       "rows_per_s": round(B * (D + 1) / (vms / 1e3), 1),
                       "roofline": {"bound": "hbm", "achieved": round(vach, 1), "peak": hbm,
                                    "unit": "GB/s", "frac": round(vach / hbm, 4),
                                    "bytes": vbytes}},
            "verify_one_hot": None if w.mode == "greedy" else one_hot,
            "draft_input": {"M": M, "calls_per_step": w.draft_steps, "ms": round(dms, 4),
                            "tokens_per_s": round(M / (dms / 1e3), 1), "roofline": droof},
            "lm_head_greedy": {"M": Ml, "ms": round(lms, 4),
                               "tokens_per_s": round(Ml / (lms / 1e3), 1), "roofline": lroof,
                               "cublas_matmul_argmax_ms": round(cms, 4),
                               "top8_ms": round(kms, 4)},
            "state": state,
            "draft_steps": steps,
            "peaks": hbm_kind}), flush=True)
    return 0


def run_lm_head(args):
    """mtp_lm_head_greedy alone at (M, H, V): seeded random bf16 hidden states, final-norm
    and output-layer weights; prints one JSON line with the median time per call."""
    import numpy as np
    import torch
    import verify_spec_greedy_gb300 as lib
    M, H, V = args.lm_head
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm, hbm_kind = measured_peaks()
    gen = torch.Generator(device=dev)
    gen.manual_seed(1)
    h = torch.randn((M, H), device=dev, generator=gen).to(torch.bfloat16)
    W = (torch.randn((V, H), device=dev, generator=gen) * 0.02).to(torch.bfloat16)
    nw = (1.0 + 0.1 * torch.randn((H,), device=dev, generator=gen)).to(torch.bfloat16)
    ids = torch.empty(M, dtype=torch.int32, device=dev)
    ws = torch.empty(lib.mtp_lm_head_greedy_workspace_bytes(M, H, V), dtype=torch.uint8, device=dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(max(1, args.warmup)):
        lib.mtp_lm_head_greedy(h, W, ids, norm_w=nw, eps=1e-6, workspace=ws)
    ts = []
    for _ in range(max(1, args.steps)):
        l2_flush(flush)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        lib.mtp_lm_head_greedy(h, W, ids, norm_w=nw, eps=1e-6, workspace=ws)
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    ms = float(np.median(ts))
    nbytes = V * H * 2 + 2 * M * H * 2 + H * 2 + M * 4
    print(json.dumps({"lm_head_greedy": {"M": M, "H": H, "V": V}, "ms": round(ms, 4),
                      "tokens_per_s": round(M / (ms / 1e3), 1),
                      "hbm_gbs": round(nbytes / (ms / 1e3) / 1e9, 1), "hbm_peak": hbm,
                      "tflops": round(2.0 * M * H * V / (ms / 1e3) / 1e12, 1),
                      "peaks": hbm_kind}), flush=True)
    return 0


def run_graph_batch(args):
    """The verify call of each workload small enough to be bound by launch latency, as a
    CUDA graph of NB back-to-back calls, each on its own copy of the inputs (so that after
    an L2 flush every call reads its logits from HBM); per-call time = replay time / NB,
    median of 10 replays."""
    import numpy as np
    import torch
    import verify_spec_greedy_gb300 as lib
    from verify_spec_greedy_gb300.inputs import WORKLOADS, make_verify_inputs
    NB = 20
    dev = torch.device("cuda", torch.cuda.current_device())
    hbm, hbm_kind = measured_peaks()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    for name in ("greedy_b1_d1_v32k", "sample_b8_d3_v152k", "sample_b1_d6_v262k_bf16"):
        w = WORKLOADS[name]
        x = make_verify_inputs(w)
        B, D, V = x["B"], x["D"], x["V"]
        greedy = w.mode == "greedy"
        Ts = [to_dev(x["T"]) for _ in range(NB)]
        Qs = None if greedy else [to_dev(x["Q"]) for _ in range(NB)]
        d = to_dev(x["d"])
        outs = [torch.empty((B, D + 1), dtype=torch.int32, device=dev) for _ in range(NB)]
        nas = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(NB)]
        if greedy:
            calls = [lambda i=i: lib.spec_verify_greedy(Ts[i], d, outs[i], nas[i])
                     for i in range(NB)]
            vbytes = B * (D + 1) * V * (4 if x["dtype"] == "f32" else 2)
        else:
            tau, top_p = to_dev(x["tau"]), optional_top_p(x, to_dev)
            top_k = to_dev(x["top_k"]) if (x["top_k"] > 0).any() else None
            ws = torch.empty(lib.spec_verify_workspace_bytes(B, D, V), dtype=torch.uint8,
                             device=dev)
            calls = [lambda i=i: lib.spec_verify_sample(Ts[i], Qs[i], d, tau, top_k, top_p,
                                                        x["seed"], outs[i], nas[i], None, None,
                                                        ws)
                     for i in range(NB)]
            vbytes = verify_bytes(x)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for c in calls:
                c()
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for c in calls:
                c()
        for _ in range(3):
            graph.replay()
        ts = []
        for _ in range(10):
            l2_flush(flush)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        ms = statistics.median(ts) / NB
        ach = vbytes / (ms / 1e3) / 1e9
        # the outputs of the last replay equal those of a plain call
        ref_out = outs[0].clone()
        calls[0]()
        torch.cuda.synchronize()
        same = bool(all(torch.equal(o, ref_out) for o in outs))
        print(json.dumps({"graph_batch": name, "calls": NB, "ms_per_call": round(ms, 5),
                          "rows_per_s": round(B * (D + 1) / (ms / 1e3), 1),
                          "roofline": {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm,
                                       "unit": "GB/s", "frac": round(ach / hbm, 4),
                                       "bytes": vbytes, "peak_kind": hbm_kind},
                          "outputs_equal": same}), flush=True)
        del Ts, Qs, graph
    return 0


def main():
    args = parse_args()
    if args.sweep:
        return run_sweep(args)
    if args.graph_batch:
        return run_graph_batch(args)
    if args.lm_head:
        return run_lm_head(args)
    if args.impl == "reference":
        # host cores only: rank 0 runs the oracle, the other ranks exit without work (no
        # process group, so no GPU is touched)
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        return run_reference(args)
    rank, world, dist = dist_init(args.gpus)
    res, x, di, w = run_gpu(args, rank, world, dist)
    if rank == 0 and not args.no_per_config and not args.batch:
        res["per_config"] = measure_per_config(_current_device(), cached={w.name: (x, di)})
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            v, cores, sample, dt = oracle_sample(x, di, w, rows=x["B"], min_seconds=10.0)
            res["cpu_baseline"] = {"value": round(v, 2), "unit": UNIT, "cores": cores,
                                   "kind": "oracle", "sample": sample, "seconds": round(dt, 2),
                                   "cpu_model": cpu_model()}
            # the same oracle on one core, over a smaller sample of the same mix
            v1, _, sample1, dt1 = oracle_sample(x, di, w, rows=8, min_seconds=2.0, threads=1)
            res["cpu_baseline"]["single_thread"] = {"value": round(v1, 2), "unit": UNIT,
                                                    "sample": sample1, "seconds": round(dt1, 2)}
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_reference(args):
    """The reference arm: the CPU oracle on this arm's workload, metric and unit; each
    step a bounded sample of the workload on the host cores."""
    from verify_spec_greedy_gb300.inputs import WORKLOADS, make_draft_input, make_verify_inputs
    w = WORKLOADS[args.workload]
    x = make_verify_inputs(w)
    di = make_draft_input(w)
    # a pool of 16 rows in the workload's mix; warm-up steps verify all of it, and the
    # timed steps take turns through it, as many rows a step as keep the K steps near
    # two minutes on the host cores
    mixed = sample_rows(x, 16)
    g = [r for r in mixed if x["tau"][r] == 0]
    sp = [r for r in mixed if x["tau"][r] != 0]
    # interleaved, so that any run of consecutive rows keeps the mix
    pool = sorted(mixed, key=lambda r: (g.index(r) * len(mixed) / len(g)) if r in g
                  else (sp.index(r) + 0.5) * len(mixed) / len(sp))
    warm = max(3, min(args.warmup, 5))
    t_warm = []
    for _ in range(warm):
        t_warm.append(oracle_sample(x, di, w, len(pool), sel=pool)[3])
    steps = max(1, args.steps)
    per_row = min(t_warm) / len(pool)
    rows = int(min(len(pool), max(1, 120.0 / (steps * per_row))))
    # small samples use fewer cores: check the size with untimed steps and shrink it
    for _ in range(3):
        t_try = min(oracle_sample(x, di, w, rows, sel=pool[:rows])[3] for _ in range(2))
        if rows == 1 or steps * t_try <= 150.0:
            break
        rows = max(1, int(rows * 120.0 / (steps * t_try)))
    total_rows, t_sum, at = 0, 0.0, 0
    for _ in range(steps):
        sel = [pool[(at + i) % len(pool)] for i in range(rows)]
        at = (at + rows) % len(pool)
        v, cores, _, dt = oracle_sample(x, di, w, rows, sel=sel)
        total_rows += rows
        t_sum += dt
    value = total_rows * (x["D"] + 1) / t_sum
    n_greedy = sum(1 for r in pool if x["tau"][r] == 0)
    sample = (f"{rows} row(s) a step, taken in turn from {len(pool)} of {x['B']} rows "
              f"({n_greedy} greedy) of {w.name}: their verify, their draft-input tokens "
              f"and the greedy drafts of the greedy rows")
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": UNIT,
           "n_gpus": max(1, args.gpus), "device": "host cores", "steps": steps,
           "warmup": warm,
           "ms_per_step": round(1e3 * t_sum / steps, 2),
           "logits_per_s": round(value * x["V"], 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name, "B": x["B"], "D": x["D"], "V": x["V"], "H": w.H,
                      "draft_tokens": w.tokens},
           "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": cores,
                            "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
           "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
