"""Benchmark of the seq<->head re-layout (BASP and Ulysses) on GB300.

One step = one pass of the whole hot path over one batch of synthetic
attention activations: Q, K, V seq-sharded -> head-sharded (one call) and the
attention output O head-sharded -> seq-sharded (one call), through the C ABI.
GB/s counts algorithmic bytes: every element read once and written once,
2 * (bytes of Q + K + V + O) per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--layout basp|ulysses] [--algo fused|three_pass]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  The default workload is the largest one,
Llama-3.2-3B-shaped activations at B=2, S=32768.  With N > 1 every rank runs
an independent replica on its own GPU (the path has no cross-GPU step on one
box); ``value`` is all ranks' bytes over the slowest rank's time.  Launched
by torchrun, the ranks come from its environment; ``--gpus N`` alone starts N
local ranks itself.  ``--impl reference`` times the CPU oracle on the host
cores instead.
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime as _dt
import hashlib
import json
import math
import os
import socket
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("seq↔head re-layout GB/s (read+write) and % of GB300 HBM peak, "
          "BASP vs Ulysses")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "basp_relayout_kernel_all_workloads_dram_traffic.txt")
# the sources a traffic capture depends on: the kernel and the launch planning
# (tile order, grid, prefetch) in relayout.cu
KERNEL_SOURCES = tuple(os.path.join(ROOT, "sequence_re_layout_gb300", "csrc", f)
                       for f in ("relayout_kernel.cuh", "relayout.cu"))
# A kernel (or the rest of a step) reported above this multiple of the
# measured copy bandwidth is not believed: the copy peak is itself a
# read+write of the same bytes, so a permutation can match it, not exceed it
# by much.
PLAUSIBLE_FRACTION = 1.15
CONSISTENT_WITHIN = 0.05


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", default=None)
    p.add_argument("--layout", default="basp", choices=["basp", "ulysses"])
    p.add_argument("--algo", default="fused",
                   choices=["fused", "three_pass", "three_pass_elide"])
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--order", default="bshd", choices=["bshd", "sbhd"],
                   help="token order inside the shards (batch- or sequence-first)")
    p.add_argument("--qkv-packed", action="store_true",
                   help="seq2head reads one packed QKV projection output")
    p.add_argument("--dtype", default=None, choices=["bf16", "fp16", "fp32", "fp8"],
                   help="element type (default: the workload's, bf16)")
    p.add_argument("--graph", action="store_true",
                   help="capture the timed loop into one CUDA graph and replay it")
    p.add_argument("--soak-s", type=float, default=1.0,
                   help="untimed seconds at full load before the timed region "
                        "(so the clock samples see the loaded GPU)")
    p.add_argument("--window-ms", type=float, default=50.0,
                   help="shortest window for the per-kernel and steady-step "
                        "timings (each also spans >= --min-launches launches)")
    p.add_argument("--min-launches", type=int, default=200)
    p.add_argument("--cpu-baseline-s", type=float, default=8.0,
                   help="seconds of the one-thread oracle timing")
    p.add_argument("--cpu-all-s", type=float, default=4.0,
                   help="seconds of the all-core oracle timing")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the Ulysses / three-pass / foil / target / e2e / CPU legs")
    p.add_argument("--no-targets", action="store_true",
                   help="skip the per-target roofline legs")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks: torchrun's environment, or N local processes started here
# ---------------------------------------------------------------------------

def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_local_ranks(n: int, argv) -> int:
    """Run this script as n ranks on this node (RANK / LOCAL_RANK /
    WORLD_SIZE in each one's environment, rendezvous on 127.0.0.1), as
    torchrun would.  Returns the first non-zero exit code, else 0; when one
    rank fails, the others are stopped."""
    import signal
    port = _free_port()
    procs = []

    def stop_all(signum, frame):
        # a signal to this process (a timeout, ^C) ends the ranks too
        for q in procs:
            if q.poll() is None:
                q.terminate()
        for q in procs:
            try:
                q.wait(timeout=10)
            except subprocess.TimeoutExpired:
                q.kill()
        sys.exit(128 + signum)

    old = {sig: signal.signal(sig, stop_all) for sig in (signal.SIGTERM, signal.SIGINT)}
    try:
        for r in range(n):
            env = dict(os.environ, WORLD_SIZE=str(n), RANK=str(r), LOCAL_RANK=str(r),
                       LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1",
                       MASTER_PORT=str(port))
            procs.append(subprocess.Popen(
                [sys.executable, os.path.abspath(__file__)] + list(argv), env=env))
        rc = 0
        live = list(procs)
        while live:
            for p in list(live):
                code = p.poll()
                if code is None:
                    continue
                live.remove(p)
                if code != 0 and rc == 0:
                    rc = code
                    for q in live:
                        q.terminate()
            time.sleep(0.05)
        return rc
    finally:
        for sig, h in old.items():
            signal.signal(sig, h)


class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def hbm_peak():
    """The measured HBM copy bandwidth (GB/s) from MEASURED_PEAKS.json, else
    the fallback.  Accepts the number itself or a nested object holding it
    ("value", "burst" or "gbs")."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        v = d.get("hbm_gbs")
        if v is None and isinstance(d.get("hbm"), dict):
            v = d["hbm"]
        if isinstance(v, dict):
            v = next((v[k] for k in ("value", "burst", "gbs", "hbm_gbs") if k in v), None)
        if isinstance(v, (int, float)) and v > 0:
            return float(v), "measured"
    except (OSError, ValueError, AttributeError, TypeError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
             "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(device_index),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": "nvidia-smi unavailable"}
        rows = []
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
            except ValueError:
                continue
        win = [r for r in rows if t0 <= r[0] <= t1]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0, "note": "no sample inside the window"}
        reasons = sorted({n for r in win for n, v in zip(self.NAMES, r[4])
                          if v.lower().startswith("active")})
        power = []
        for r in win:
            try:
                power.append(float(r[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(r[1] for r in win),
                "sm_max_mhz": max(r[2] for r in win),
                "reasons": reasons, "samples": len(win),
                "power_w_median": statistics.median(power) if power else None,
                "window": "pre-timed soak at the same load + timed region"}


def source_digest():
    """Digest of the code of the kernel and its launch planning: comments and
    blank space removed, so a comment edit does not orphan a traffic record."""
    import re
    code = []
    for path in KERNEL_SOURCES:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            line = line.split("//", 1)[0].strip()
            if line:
                code.append(" ".join(line.split()))
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def ncu_traffic(workload: str, layout: str, kernel_role: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    try:
        with open(TRAFFIC_FILE) as f:
            lines = f.read().splitlines()
    except OSError:
        return None
    digest = source_digest()
    for l in lines:
        tok = l.split()
        if len(tok) >= 5 and tok[0] == "traffic" and tok[1] == workload \
                and tok[2] == layout and tok[3] == kernel_role:
            kv = dict(t.split("=", 1) for t in tok[4:] if "=" in t)
            if kv.get("source") != digest:
                return None
            return float(kv["bytes"])
    return None


def gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


def copy_rate_same_run(dev, n_elems=1 << 30, reps=10):
    """torch's copy_ of n_elems bf16 elements (read + write bytes), best of
    `reps`, CUDA events: the same kind of figure as the measured peak, taken
    in this run on this GPU, as a cross-check of the fractions."""
    import torch
    a = torch.empty(n_elems, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    b.copy_(a)
    best = math.inf
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        torch.cuda.synchronize(dev)
        best = min(best, e0.elapsed_time(e1))
    del a, b
    torch.cuda.empty_cache()
    return gbs(2 * 2 * n_elems, best)


def check_timings(s2h_bytes, s2h_ms, h2s_bytes, h2s_ms, step_ms, peak):
    """Cross-check the per-kernel launch times against the step time measured
    separately: the two kernels' times should add up to the step's (within
    CONSISTENT_WITHIN), and neither a kernel's own rate nor the rate it
    implies for the rest of the step may exceed PLAUSIBLE_FRACTION x peak."""
    total = s2h_ms + h2s_ms
    rest_after_s2h = step_ms - s2h_ms
    rest_after_h2s = step_ms - h2s_ms
    implied_h2s = gbs(h2s_bytes, rest_after_s2h) if rest_after_s2h > 0 else math.inf
    implied_s2h = gbs(s2h_bytes, rest_after_h2s) if rest_after_h2s > 0 else math.inf
    rates = [gbs(s2h_bytes, s2h_ms), gbs(h2s_bytes, h2s_ms), implied_h2s, implied_s2h]
    ratio = total / step_ms
    return {
        "s2h_plus_h2s_ms": round(total, 6),
        "step_ms": round(step_ms, 6),
        "ratio": round(ratio, 4),
        "consistent": abs(ratio - 1.0) <= CONSISTENT_WITHIN,
        "implied_head2seq_gbs": round(implied_h2s, 2) if math.isfinite(implied_h2s) else None,
        "implied_seq2head_gbs": round(implied_s2h, 2) if math.isfinite(implied_s2h) else None,
        "plausible": all(math.isfinite(r) and r <= PLAUSIBLE_FRACTION * peak for r in rates),
    }


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _alloc_sets(w, dtype, n_sets, dev, seed, packed=False):
    import torch
    import synth_inputs
    nq, nkv = w.tensor_elems(w.Hq), w.tensor_elems(w.Hkv)
    base = [synth_inputs.normal_device(n, seed + i, dtype, dev)
            for i, n in enumerate((nq, nkv, nkv, nq))]
    if packed:
        # ins[0] is the packed QKV buffer; ins[1], ins[2] are unused
        base[0] = synth_inputs.normal_device(nq + 2 * nkv, seed + 7, dtype, dev)
    sets = []
    for s in range(n_sets):
        ins = base if s == 0 else [t.clone() for t in base]
        outs = [torch.empty(n, dtype=ins[3].dtype, device=dev)
                for n in (nq, nkv, nkv, nq)]
        sets.append((ins, outs))
    return sets


def run_device(w, layout, algo, steps, warmup, dev, peak, soak_s=0.0, order="bshd",
               packed=False, graph=False, spread=0, window_ms=50.0, min_launches=200):
    """Time `steps` steps of the hot path, then each of the step's two calls
    alone and a steady window of steps, cross-checked; returns a dict."""
    import torch
    import sequence_re_layout_gb300 as basp

    K = w.K(layout)
    L = basp.Layout(w.B, w.S, w.Hq, w.Hkv, w.d, w.N, K, w.dtype, order=order)
    info = L.info
    T = info["bytes_q"] * 2 + info["bytes_kv"] * 2            # Q, K, V, O
    step_bytes = 2 * T
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = min(4096, max(2, -(-4 * l2 // step_bytes) + 1))   # >= 4x L2 per rotation
    sets = _alloc_sets(w, w.dtype, n_sets, dev, 1234, packed)
    ws = None
    if algo != "fused":
        ws = torch.empty(info["workspace_bytes"], dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    # raw addresses, so each call pays only the C ABI's own cost (the binding
    # checks tensor arguments, raw integers pass through as they are)
    ptrs = [([t.data_ptr() for t in ins], [t.data_ptr() for t in outs])
            for ins, outs in sets]
    wsp = ws.data_ptr() if ws is not None else None
    wsb = ws.numel() if ws is not None else 0
    passes = {"fused": 1, "three_pass": 3}.get(algo)
    if passes is None:                 # three_pass_elide
        passes = 2 if (info["seqs_per_group"] == 1 or order == "sbhd") else 3
    count = [0]

    def call(which, i):
        ins, outs = ptrs[i % n_sets]
        s = stream.cuda_stream
        count[0] += passes
        if which == "s2h" and packed:
            basp.basp_seq2head_qkv(L.handle, ins[0], outs[0], outs[1], outs[2], stream=s)
        elif which == "s2h":
            basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                               outs[0], outs[1], outs[2], wsp, wsb, stream=s)
        else:
            basp.basp_head2seq(L.handle, algo, ins[3], None, None,
                               outs[3], None, None, wsp, wsb, stream=s)

    def step(i):
        call("s2h", i)
        call("h2s", i)

    def timed(fn, n):
        """CUDA events around n back-to-back calls on the bench stream (events
        between launches would break programmatic dependent launch)."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1)

    def windowed(fn, est_ms):
        """ms per call over >= min_launches calls and >= window_ms, after a
        warm-up of that call alone."""
        timed(fn, 20)
        n = max(min_launches, int(math.ceil(window_ms / max(est_ms, 1e-4))))
        return timed(fn, n) / n, n

    timed_graph = None
    if graph:
        # the whole timed loop (`steps` steps, rotating buffers) captured as
        # one CUDA graph on a side stream, as capture requires, and replayed
        # once on the bench stream; the programmatic launches become
        # programmatic edges between the graph's kernel nodes
        for i in range(n_sets):
            step(i)                                    # first calls eagerly
        torch.cuda.synchronize(dev)
        cap = torch.cuda.Stream(dev)
        timed_graph = torch.cuda.CUDAGraph()
        stream = cap
        with torch.cuda.graph(timed_graph, stream=cap):
            for i in range(steps):
                step(i)
        stream = torch.cuda.current_stream(dev)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    soak_t0 = time.time()
    if soak_s > 0:
        i = 0
        while time.time() - soak_t0 < soak_s:
            for _ in range(50):
                step(i)
                i += 1
            torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    # the timed region: exactly `steps` whole steps back to back, events only
    # around the loop
    start.record(stream)
    if timed_graph is not None:
        timed_graph.replay()
    else:
        for i in range(steps):
            step(i)
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    total_ms = start.elapsed_time(end)
    est_step = total_ms / max(steps, 1)

    # per-call launch times and a steady window of whole steps, measured until
    # they agree (at most three attempts)
    attempts = []
    for _ in range(3):
        steady_ms, n_steady = windowed(step, est_step)
        s2h_ms, n_s2h = windowed(lambda i: call("s2h", i), est_step / 2)
        h2s_ms, n_h2s = windowed(lambda i: call("h2s", i), est_step / 2)
        chk = check_timings(2 * (info["bytes_q"] + 2 * info["bytes_kv"]), s2h_ms,
                            2 * info["bytes_q"], h2s_ms, steady_ms, peak)
        attempts.append((chk, steady_ms, n_steady, s2h_ms, n_s2h, h2s_ms, n_h2s))
        if chk["consistent"] and chk["plausible"]:
            break
    chk, steady_ms, n_steady, s2h_ms, n_s2h, h2s_ms, n_h2s = attempts[-1]
    chk["attempts"] = len(attempts)

    # distribution: 30 windows of whole steps back to back, events only
    # between windows (so programmatic launch overlaps every boundary but 29);
    # each window lasts >= 2 ms
    n_win = 30
    per_win = max(5, int(math.ceil(2.0 / max(est_step, 1e-4))))
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_win + 1)]
    timed(step, 20)
    evs[0].record(stream)
    i = 0
    for k in range(n_win):
        for _ in range(per_win):
            step(i)
            i += 1
        evs[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    win_ms = [evs[k].elapsed_time(evs[k + 1]) / per_win for k in range(n_win)]

    # spread: the same K-step loop repeated (only reported, never the value)
    repeats = [timed(step, steps) / steps for _ in range(spread)]
    launches_per_step = 2 * passes
    res = {
        "total_ms": total_ms, "ms_per_step": total_ms / steps,
        "step_bytes": step_bytes, "info": info, "n_sets": n_sets,
        "l2_bytes": l2, "s2h_ms_mean": s2h_ms, "h2s_ms_mean": h2s_ms,
        "s2h_launches_timed": n_s2h, "h2s_launches_timed": n_h2s,
        "steady_ms_per_step": steady_ms, "steady_steps": n_steady,
        "check": chk,
        "s2h_bytes": 2 * (info["bytes_q"] + 2 * info["bytes_kv"]),
        "h2s_bytes": 2 * info["bytes_q"],
        "launches_per_step": launches_per_step,
        "timed_launches": launches_per_step * steps,
        "total_launches": count[0],
        "repeat_ms_per_step": repeats,
        "window_ms_per_step": win_ms, "steps_per_window": per_win,
        "wall": (soak_t0 if soak_s > 0 else t0, t1),
    }
    del sets, ws
    L.close()
    torch.cuda.empty_cache()
    return res


def percentile(xs, q):
    """The q-th percentile (0..100) of xs, linear between closest ranks."""
    xs = sorted(xs)
    if not xs:
        return None
    pos = (len(xs) - 1) * q / 100.0
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(xs) - 1)
    return xs[lo] + (xs[hi] - xs[lo]) * (pos - lo)


def window_stats(r):
    """GB/s over the run's 30 step windows: median, p10 and p90."""
    g = [gbs(r["step_bytes"], ms) for ms in r["window_ms_per_step"]]
    return {"windows": len(g), "steps_per_window": r["steps_per_window"],
            "gbs_p10": round(percentile(g, 10), 2), "gbs_median": round(percentile(g, 50), 2),
            "gbs_p90": round(percentile(g, 90), 2),
            "note": "events only between windows; each window's first launch waits for the "
                    "last one's completion, so windows read a little below the back-to-back loop"}


def kernel_roofline(nbytes, ms, peak, traffic, plausible):
    """One call's roofline entry: algorithmic bytes over its mean launch time."""
    a = gbs(nbytes, ms)
    if not plausible:
        return {"achieved": None, "frac": None, "traffic": traffic,
                "algorithmic_bytes_per_launch": nbytes, "launch_ms_mean": round(ms, 6),
                "note": "withheld: the launch times and the step time disagree "
                        "beyond what the copy peak allows"}
    return {"achieved": round(a, 2), "frac": round(a / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": nbytes, "launch_ms_mean": round(ms, 6)}


def leg_summary(w, layout, r, peak, order="bshd", packed=False, algo="fused"):
    """Both directions' rooflines, the steady step and the cross-check of one
    (workload, layout) run."""
    traffic = {"s2h": None, "h2s": None}
    if order == "bshd" and not packed:
        traffic["s2h"] = ncu_traffic(w.name, layout, "seq2head_qkv_" + algo)
        traffic["h2s"] = ncu_traffic(w.name, layout, "head2seq_o_" + algo)
    ok = r["check"]["plausible"]
    s2h = kernel_roofline(r["s2h_bytes"], r["s2h_ms_mean"], peak, traffic["s2h"], ok)
    h2s = kernel_roofline(r["h2s_bytes"], r["h2s_ms_mean"], peak, traffic["h2s"], ok)
    steady = gbs(r["step_bytes"], r["steady_ms_per_step"])
    return {"workload": w.name, "layout": layout, "K": r["info"]["K"],
            "seq2head": s2h, "head2seq": h2s,
            "steady_step": {"gbs": round(steady, 2), "frac": round(steady / peak, 4),
                            "ms": round(r["steady_ms_per_step"], 6),
                            "steps": r["steady_steps"]},
            "distribution": window_stats(r),
            "check": r["check"]}


def run_e2e(w, layout, algo, steps, warmup, dev, mode="staged", order="bshd"):
    """Same step with the tensors in pinned host memory, inside the timed
    region every step.  mode "staged": basp_seq2head_host / basp_head2seq_host
    copy the inputs to device staging, re-lay out, copy the results back.
    mode "direct": the same calls without staging; the kernels read and write
    the pinned host buffers in place over the host link."""
    import torch
    import synth_inputs
    import sequence_re_layout_gb300 as basp

    K = w.K(layout)
    L = basp.Layout(w.B, w.S, w.Hq, w.Hkv, w.d, w.N, K, w.dtype, order=order)
    info = L.info
    nq, nkv = w.tensor_elems(w.Hq), w.tensor_elems(w.Hkv)
    hin = []
    for i, n in enumerate((nq, nkv, nkv, nq)):
        h = torch.empty(n, dtype=synth_inputs.DTYPES[w.dtype]).pin_memory()
        h.copy_(synth_inputs.normal_device(n, 1234 + i, w.dtype, dev))
        hin.append(h)
    hout = [torch.empty_like(t).pin_memory() for t in hin]
    staging = None
    if mode == "staged":
        staging = torch.empty(info["staging_bytes"], dtype=torch.uint8, device=dev)
    ws = None
    if algo != "fused":
        ws = torch.empty(info["workspace_bytes"], dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if mode == "direct":
            basp.basp_seq2head_host(L.handle, algo, hin[0], hin[1], hin[2],
                                    hout[0], hout[1], hout[2], None, 0,
                                    workspace=ws, stream=stream)
            basp.basp_head2seq_host(L.handle, algo, hin[3], None, None, hout[3],
                                    None, None, None, 0, workspace=ws, stream=stream)
            return
        basp.basp_seq2head_host(L.handle, algo, hin[0], hin[1], hin[2],
                                hout[0], hout[1], hout[2], staging,
                                workspace=ws, stream=stream)
        basp.basp_head2seq_host(L.handle, algo, hin[3], None, None, hout[3],
                                None, None, staging, workspace=ws, stream=stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    end.record(stream)
    torch.cuda.synchronize(dev)
    ms = start.elapsed_time(end) / steps
    T = sum(t.numel() * t.element_size() for t in hin)
    del staging, ws, hin, hout
    L.close()
    torch.cuda.empty_cache()
    return {"ms_per_step": ms, "bytes_in": T, "bytes_out": T, "step_bytes": 2 * T,
            "launches": (warmup + steps) * 2}


def _oracle_step(w, K, x, order, nthreads=None):
    """One step of the oracle: Q, K, V seq2head and O head2seq."""
    import oracle
    hs = (w.Hq, w.Hkv, w.Hkv, w.Hq)
    for i, (a, H) in enumerate(zip(x, hs)):
        fwd = i < 3
        if nthreads is None:
            f = oracle.seq2head if fwd else oracle.head2seq
            f(a, w.B, w.S, H, w.d, w.N, K, order=order)
        else:
            f = oracle.seq2head_threads if fwd else oracle.head2seq_threads
            f(a, w.B, w.S, H, w.d, w.N, K, nthreads, order=order)


def _oracle_inputs(w, on_gpu=False):
    """The step's four tensors as raw bits on the host, drawn by the CPU
    generator, or (on_gpu, which is much faster at full size) by the GPU's."""
    import torch
    import synth_inputs
    sizes = [w.B * w.S * h * w.d for h in (w.Hq, w.Hkv, w.Hkv, w.Hq)]
    if on_gpu:
        dev = torch.device("cuda", torch.cuda.current_device())
        return [synth_inputs.bits(synth_inputs.normal_device(n, 1234 + i, w.dtype, dev).cpu())
                for i, n in enumerate(sizes)]
    return [synth_inputs.bits(synth_inputs.normal(n, 1234 + i, w.dtype))
            for i, n in enumerate(sizes)]


def _time_oracle(w, K, x, order, budget_s, nthreads):
    reps, t0 = 0, time.perf_counter()
    while True:
        _oracle_step(w, K, x, order, nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            return reps, el


def cpu_baseline(w, layout, budget_1, budget_all, order="bshd"):
    """The oracle as it stands on the host cores, over whole steps of the same
    workload: the plain loop on one thread for about `budget_1` s, then the
    all-core form on every core this process may use for about `budget_all` s."""
    import oracle
    oracle.build()
    K = w.K(layout)
    x = _oracle_inputs(w, on_gpu=True)
    step_bytes = 2 * sum(a.nbytes for a in x)
    cores = oracle.host_cores()
    r1, e1 = _time_oracle(w, K, x, order, budget_1, None)
    ra, ea = _time_oracle(w, K, x, order, budget_all, cores)
    v1 = step_bytes * r1 / e1 / 1e9
    va = step_bytes * ra / ea / 1e9
    return {"value": round(va, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d whole steps of %s (%s, Q/K/V seq2head + O head2seq) on %d "
                      "threads, %.1f s" % (ra, w.name, layout, cores, ea),
            "threads_all": {"value": round(va, 3), "threads": cores, "steps": ra,
                            "seconds": round(ea, 2)},
            "threads_1": {"value": round(v1, 3), "threads": 1, "steps": r1,
                          "seconds": round(e1, 2)},
            "host_cores": cores}


def main_ours(args, dist):
    import torch
    import sequence_re_layout_gb300 as basp
    from sequence_re_layout_gb300.build import build_library
    from sequence_re_layout_gb300.workloads import (HEADLINE, TARGETS,
                                                    TARGET_FRACTION, WORKLOADS, Workload)

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    if dist.rank == 0:
        build_library()               # no-op when the library is up to date
    dist.barrier()
    basp.load_library()
    dev = torch.device("cuda", dist.local_rank % torch.cuda.device_count())
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.config or HEADLINE]
    if args.dtype:
        w = dataclasses.replace(w, dtype=args.dtype)
    peak, peak_kind = hbm_peak()
    kw = dict(window_ms=args.window_ms, min_launches=args.min_launches)

    sampler = ClockSampler(dev.index)
    dist.barrier()
    if args.qkv_packed and args.algo != "fused":
        raise SystemExit("--qkv-packed runs the fused path only")
    r = run_device(w, args.layout, args.algo, args.steps, args.warmup, dev, peak,
                   soak_s=args.soak_s, order=args.order, packed=args.qkv_packed,
                   graph=args.graph, spread=0 if args.no_extras else 5, **kw)
    sampler.stop()
    dist.barrier()
    t_max = dist.max(r["total_ms"])
    total_bytes = dist.sum(r["step_bytes"] * args.steps)
    value = total_bytes / (t_max * 1e-3) / 1e9
    clocks = sampler.summary(*r["wall"])
    launches_total = r["total_launches"]

    info = r["info"]
    head = leg_summary(w, args.layout, r, peak, args.order, args.qkv_packed, args.algo)
    s2h = head["seq2head"]
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps, 6), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic (~N(0,1) %s, seeded)" % w.dtype,
        "config": {
            "workload": w.name, "layout": args.layout, "algo": args.algo,
            "order": args.order, "qkv_packed": bool(args.qkv_packed),
            "cuda_graph": bool(args.graph),
            "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "N": w.N,
            "K": info["K"], "groups": info["groups"],
            "bytes_per_step": r["step_bytes"],
            "l2": "inputs rotate over %d buffer sets (%.0f MB per rotation, "
                  "L2 %.0f MB)" % (r["n_sets"], r["n_sets"] * r["step_bytes"] / 1e6,
                                   r["l2_bytes"] / 1e6),
            "parallelism": "replicas" if dist.world > 1 else "single GPU, %d virtual ranks" % w.N,
        },
        "pct_hbm_peak": round(100 * value / dist.world / peak, 2),
        "pct_hbm_nominal": round(100 * value / dist.world / NOMINAL_HBM_GBS, 2),
        "roofline": dict({
            "bound": "hbm", "kernel": "basp_relayout_kernel (seq2head Q,K,V)",
            "peak": peak, "unit": "GB/s",
            "launch_timing": "CUDA events around %d back-to-back launches of this "
                             "kernel alone on the bench stream, after 20 untimed "
                             "ones" % r["s2h_launches_timed"],
            "peak_kind": "of %s" % peak_kind}, **s2h),
        "head2seq": dict(head["head2seq"], launches_timed=r["h2s_launches_timed"]),
        "steady": dict(head["steady_step"],
                       note="the same step over a window of >= %g ms, after the "
                            "timed region; `value` is the timed region alone"
                            % args.window_ms),
        "timing_check": dict(head["check"], ratio_vs_timed_region=round(
            (r["s2h_ms_mean"] + r["h2s_ms_mean"]) / (t_max / args.steps), 4)),
        "distribution": head["distribution"],
        "context": {
            "pages_figures": "BASP vs Ulysses in training: 1.17-1.31x end-to-end step "
                             "speedup and 2.23-3.10x less all-to-all time (six Llama/Qwen "
                             "models, S=16K, B=2, N=8)",
            "pages_hardware": "2 nodes x 4 NVIDIA A100-40GB, 400 Gb/s InfiniBand, "
                              "modified DeepSpeed",
            "note": "the pages publish no GB/s for the re-layout itself; these are "
                    "context, not a baseline for this line"},
        "analytic": {"peers_per_rank": info["peers"],
                     "bytes_per_peer_q": info["bytes_per_peer_q"],
                     "bytes_per_peer_kv": info["bytes_per_peer_kv"],
                     "tokens_per_rank": info["tokens_per_rank"],
                     "foil_tokens_per_rank": info["foil_tokens_per_rank"]},
        "gpu_launches": r["timed_launches"],
        "clocks": clocks,
    }
    if r["repeat_ms_per_step"]:
        rg = sorted(gbs(r["step_bytes"], ms) for ms in r["repeat_ms_per_step"])
        out["spread"] = {"repeats": len(rg), "of": "the timed loop, run again after it",
                         "gbs_min": round(rg[0], 2), "gbs_median": round(statistics.median(rg), 2),
                         "gbs_max": round(rg[-1], 2)}
    if not args.no_extras:
        # end to end on every rank (replicas): all ranks' bytes over the
        # slowest rank's time, like `value`
        ne = max(3, min(args.steps, 50))
        dist.barrier()
        e = run_e2e(w, args.layout, args.algo, ne, 3, dev, mode="direct", order=args.order)
        dist.barrier()
        es = run_e2e(w, args.layout, args.algo, ne, 3, dev, mode="staged", order=args.order)
        e_ms, es_ms = dist.max(e["ms_per_step"]), dist.max(es["ms_per_step"])
        e_bytes, es_bytes = dist.sum(e["step_bytes"]), dist.sum(es["step_bytes"])
        out["e2e"] = {"value": round(gbs(e_bytes, e_ms), 2),
                      "unit": "GB/s", "h2d_bytes_per_step": e["bytes_in"] * dist.world,
                      "d2h_bytes_per_step": e["bytes_out"] * dist.world,
                      "ms_per_step": round(e_ms, 4),
                      "api": "basp_seq2head_host + basp_head2seq_host, direct mode "
                             "(no staging: kernels read and write the pinned host "
                             "buffers in place)",
                      "staged": {"value": round(gbs(es_bytes, es_ms), 2),
                                 "ms_per_step": round(es_ms, 4),
                                 "api": "basp_seq2head_host + basp_head2seq_host, "
                                        "staged mode (H2D copy, re-layout, D2H copy)"}}
        launches_total += e["launches"] * r["launches_per_step"] // 2
        launches_total += es["launches"] * r["launches_per_step"] // 2
    if not args.no_extras and dist.rank == 0:
        other = "ulysses" if args.layout == "basp" else "basp"
        ru = run_device(w, other, args.algo, args.steps, args.warmup, dev, peak,
                        order=args.order, packed=args.qkv_packed, **kw)
        lu = leg_summary(w, other, ru, peak, args.order, args.qkv_packed, args.algo)
        vu = gbs(ru["step_bytes"] * args.steps, ru["total_ms"])
        ou = ru["info"]
        out[other] = {"value": round(vu, 2), "ms_per_step": round(ru["ms_per_step"], 6),
                      "K": ou["K"], "pct_hbm_peak": round(100 * vu / peak, 2),
                      "peers_per_rank": ou["peers"],
                      "bytes_per_peer_q": ou["bytes_per_peer_q"],
                      "seq2head": lu["seq2head"], "head2seq": lu["head2seq"],
                      "steady": lu["steady_step"], "timing_check": lu["check"]}
        launches_total += ru["total_launches"]
        basp_r, uly_r = (r, ru) if args.layout == "basp" else (ru, r)
        out["basp_vs_ulysses"] = {
            "step_time_ratio": round(uly_r["steady_ms_per_step"] / basp_r["steady_ms_per_step"], 4),
            "peers_per_rank": {"basp": basp_r["info"]["peers"], "ulysses": uly_r["info"]["peers"]},
            "remote_bytes_per_rank": {
                lay: rr["info"]["peers"] * (rr["info"]["bytes_per_peer_q"] +
                                            2 * rr["info"]["bytes_per_peer_kv"])
                for lay, rr in (("basp", basp_r), ("ulysses", uly_r))},
            "note": "Ulysses step time over BASP's (steady windows). On one GPU both layouts "
                    "move the same bytes; BASP's rows are B times longer. The pages' gain "
                    "comes from keeping the K-way exchange inside a node."}
        legs = {(w.name, args.layout): head, (w.name, other): lu}
        if args.layout == "basp" and w.N % w.B == 0:
            # the review's "trivial alternative" (Strengths, Table I): Ulysses
            # with SP = N/B, every group of K = N/B ranks holding all B
            # sequences -- B*B*S/N tokens per rank, B times BASP's bytes
            wf = Workload(w.name + "_foil", w.B * w.B, w.S, w.Hq, w.Hkv, w.d,
                          w.N, w.N // w.B, w.dtype)
            rf = run_device(wf, "basp", args.algo, args.steps, args.warmup, dev, peak,
                            order=args.order, **kw)
            out["foil_ulysses_sp_n_over_b"] = {
                "tokens_per_rank": rf["info"]["tokens_per_rank"],
                "basp_tokens_per_rank": info["tokens_per_rank"],
                "bytes_per_step": rf["step_bytes"],
                "ms_per_step": round(rf["ms_per_step"], 6),
                "value": round(gbs(rf["step_bytes"] * args.steps, rf["total_ms"]), 2),
                "time_vs_basp": round(rf["ms_per_step"] / (r["total_ms"] / args.steps), 3),
                "steady_time_vs_basp": round(rf["steady_ms_per_step"] /
                                             r["steady_ms_per_step"], 3),
                "timing_check": rf["check"]}
            launches_total += rf["total_launches"]
        alts = [a for a in ("fused", "three_pass", "three_pass_elide") if a != args.algo]
        notes = {"three_pass": "same algorithmic bytes; the three passes move them 3x",
                 "three_pass_elide": "identity pass skipped when the receive chunks "
                                     "are already head-sharded (2 passes here: %s)"
                                     % ("yes" if info["seqs_per_group"] == 1 or
                                        args.order == "sbhd" else "no"),
                 "fused": "one pass"}
        for alt in alts:
            rt = run_device(w, args.layout, alt, args.steps, args.warmup, dev, peak,
                            order=args.order, **kw)
            vt = gbs(rt["step_bytes"] * args.steps, rt["total_ms"])
            out[alt] = {"value": round(vt, 2), "ms_per_step": round(rt["ms_per_step"], 6),
                        "pct_hbm_peak": round(100 * vt / peak, 2), "note": notes[alt]}
            launches_total += rt["total_launches"]
        if (not args.no_targets and args.algo == "fused" and args.order == "bshd"
                and not args.qkv_packed and not args.dtype):
            # every long-sequence target shape, both layouts, both directions
            for name in TARGETS:
                for lay in ("basp", "ulysses"):
                    if (name, lay) in legs:
                        continue
                    wt = WORKLOADS[name]
                    rt = run_device(wt, lay, "fused", args.steps, args.warmup, dev, peak, **kw)
                    legs[(name, lay)] = leg_summary(wt, lay, rt, peak)
                    launches_total += rt["total_launches"]
            tl = []
            for name in TARGETS:
                for lay in ("basp", "ulysses"):
                    leg = dict(legs[(name, lay)])
                    fr = [leg[k]["frac"] for k in ("seq2head", "head2seq")]
                    leg["meets_bar"] = all(f is not None and f >= TARGET_FRACTION for f in fr)
                    tl.append(leg)
            out["targets"] = {"bar": TARGET_FRACTION, "peak": peak,
                              "peak_kind": "of %s" % peak_kind,
                              "all_meet_bar": all(l["meets_bar"] for l in tl),
                              "legs": tl}
        cr = copy_rate_same_run(dev)
        out["roofline"]["copy_same_run"] = {
            "gbs": round(cr, 2), "kernel_vs_copy": round(s2h["achieved"] / cr, 4)
            if s2h["achieved"] else None,
            "how": "torch copy_ of 1 Gi bf16 elements, read + write bytes, best of 10, "
                   "in this run (the kind of copy MEASURED_PEAKS.json records)"}
        if dist.world == 1:
            out["cpu_baseline"] = cpu_baseline(w, args.layout, args.cpu_baseline_s,
                                               args.cpu_all_s, order=args.order)
    out["gpu_launches_total"] = launches_total
    if dist.rank == 0:
        print(json.dumps(out), flush=True)


def main_reference(args, dist):
    """The reference arm: the CPU oracle, as it stands, timed on the host
    cores (its all-core form, every core this process may use) over bounded
    samples of the same workload (rank 0 only)."""
    if dist.rank != 0:
        return
    import oracle
    from sequence_re_layout_gb300.workloads import HEADLINE, WORKLOADS
    oracle.build()
    w = WORKLOADS[args.config or HEADLINE]
    if args.dtype:
        w = dataclasses.replace(w, dtype=args.dtype)
    K = w.K(args.layout)
    o = args.order
    cores = oracle.host_cores()
    # bound the whole run to about two minutes: if one full-size step would
    # take longer than budget / (steps + warmup), shrink S (a multiple of K).
    # Inputs are drawn on the CPU: nothing on this arm touches the GPU.
    budget_s = 120.0
    probe_S = max(K, (w.S // 16) // K * K)
    wp = dataclasses.replace(w, S=probe_S)
    xp = _oracle_inputs(wp)
    t0 = time.perf_counter()
    _oracle_step(wp, K, xp, o, cores)
    per_token = (time.perf_counter() - t0) / probe_S
    per_step_budget = budget_s / max(1, args.steps + args.warmup)
    S = w.S
    if per_token * w.S > per_step_budget:
        S = max(K, int(per_step_budget / per_token) // K * K)
    ws = dataclasses.replace(w, S=S)
    x = _oracle_inputs(ws)
    for _ in range(args.warmup):
        _oracle_step(ws, K, x, o, cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(ws, K, x, o, cores)
    el = time.perf_counter() - t0
    step_bytes = 2 * sum(a.nbytes for a in x)
    value = step_bytes * args.steps / el / 1e9
    sample = ("%s at S=%d of %d (same B, heads, d, N, K), %d steps on %d threads, %.1f s"
              % (w.name, S, w.S, args.steps, cores, el))
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3),
        "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (~N(0,1) %s, seeded)" % w.dtype,
        "config": {"workload": w.name, "layout": args.layout, "algo": "oracle",
                   "order": o, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv,
                   "d": w.d, "N": w.N, "K": K},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse_args(argv)
    env_world = os.environ.get("WORLD_SIZE")
    if env_world is None and args.gpus > 1:
        sys.exit(launch_local_ranks(args.gpus, argv))
    if env_world is not None and int(env_world) != args.gpus:
        print("bench.py: --gpus %d but WORLD_SIZE=%s; they must agree"
              % (args.gpus, env_world), file=sys.stderr)
        sys.exit(2)
    dist = Dist()
    try:
        if args.impl == "reference":
            main_reference(args, dist)
        else:
            main_ours(args, dist)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
