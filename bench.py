"""Benchmark of the seq<->head re-layout (BASP and Ulysses) on GB300.

One step = one pass of the whole hot path over one batch of synthetic
attention activations: Q, K, V seq-sharded -> head-sharded (one call) and the
attention output O head-sharded -> seq-sharded (one call), through the C ABI.
GB/s counts algorithmic bytes: every element read once and written once,
2 * (bytes of Q + K + V + O) per step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--layout basp|ulysses] [--algo fused|three_pass]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs an
independent replica on its own GPU (the path has no cross-GPU step on one
box); ``value`` is all ranks' bytes over the slowest rank's time.
``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
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
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
KERNEL_SOURCE = os.path.join(ROOT, "sequence_re_layout_gb300", "csrc", "relayout_kernel.cuh")


def parse_args():
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
    p.add_argument("--cpu-baseline-s", type=float, default=10.0)
    p.add_argument("--no-extras", action="store_true",
                   help="skip the Ulysses / three-pass / e2e / CPU legs")
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: barrier and max-reduce on the host)
# ---------------------------------------------------------------------------

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
    """Digest of the kernel source's code: comments and blank space removed,
    so a comment edit does not orphan a traffic record."""
    import re
    with open(KERNEL_SOURCE) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    code = []
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


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _alloc_sets(w, K, dtype, n_sets, dev, seed, packed=False):
    import torch
    import synth_inputs
    nq, nkv = w.tensor_elems(w.Hq), w.tensor_elems(w.Hkv)
    base = [synth_inputs.normal(n, seed + i, dtype).to(dev)
            for i, n in enumerate((nq, nkv, nkv, nq))]
    if packed:
        # ins[0] is the packed QKV buffer; ins[1], ins[2] are unused
        base[0] = synth_inputs.normal(nq + 2 * nkv, seed + 7, dtype).to(dev)
    sets = []
    for s in range(n_sets):
        ins = base if s == 0 else [t.clone() for t in base]
        outs = [torch.empty(n, dtype=ins[3].dtype, device=dev)
                for n in (nq, nkv, nkv, nq)]
        sets.append((ins, outs))
    return sets


def run_device(w, layout, algo, steps, warmup, dev, soak_s=0.0, order="bshd",
               packed=False, graph=False, spread=0):
    """Time `steps` steps of the hot path; returns a dict of timings."""
    import torch
    import sequence_re_layout_gb300 as basp

    K = w.K(layout)
    L = basp.Layout(w.B, w.S, w.Hq, w.Hkv, w.d, w.N, K, w.dtype, order=order)
    info = L.info
    T = info["bytes_q"] * 2 + info["bytes_kv"] * 2            # Q, K, V, O
    step_bytes = 2 * T
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_sets = min(4096, max(2, -(-4 * l2 // step_bytes) + 1))   # >= 4x L2 per rotation
    sets = _alloc_sets(w, K, w.dtype, n_sets, dev, 1234, packed)
    ws = None
    if algo != "fused":
        ws = torch.empty(info["workspace_bytes"], dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(i):
        ins, outs = sets[i % n_sets]
        if packed:
            basp.basp_seq2head_qkv(L.handle, ins[0], outs[0], outs[1], outs[2],
                                   stream=stream)
        else:
            basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                               outs[0], outs[1], outs[2], ws, stream=stream)
        basp.basp_head2seq(L.handle, algo, ins[3], None, None,
                           outs[3], None, None, ws, stream=stream)

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
    # the timed region: `steps` whole steps back to back, events only around
    # the loop (events between launches would serialise them)
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

    # roofline: each kernel's average launch duration, `steps` launches of
    # that kernel alone back to back on the same stream
    def one_kernel(which):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            ins, outs = sets[i % n_sets]
            if which == "s2h" and packed:
                basp.basp_seq2head_qkv(L.handle, ins[0], outs[0], outs[1], outs[2],
                                       stream=stream)
            elif which == "s2h":
                basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                                   outs[0], outs[1], outs[2], ws, stream=stream)
            else:
                basp.basp_head2seq(L.handle, algo, ins[3], None, None,
                                   outs[3], None, None, ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / steps

    s2h_ms = one_kernel("s2h")
    h2s_ms = one_kernel("h2s")

    # spread: the same K-step loop repeated (only reported, never the value)
    repeats = []
    for _ in range(spread):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            step(i)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        repeats.append(e0.elapsed_time(e1) / steps)
    passes = {"fused": 1, "three_pass": 3}.get(algo)
    if passes is None:                 # three_pass_elide
        passes = 2 if (info["seqs_per_group"] == 1 or order == "sbhd") else 3
    launches_per_step = 2 * passes
    res = {
        "total_ms": total_ms, "ms_per_step": total_ms / steps,
        "step_bytes": step_bytes, "info": info, "n_sets": n_sets,
        "l2_bytes": l2, "s2h_ms_mean": s2h_ms, "h2s_ms_mean": h2s_ms,
        "s2h_bytes": 2 * (info["bytes_q"] + 2 * info["bytes_kv"]),
        "h2s_bytes": 2 * info["bytes_q"],
        "launches": (2 + spread) * launches_per_step * steps,  # step, roofline, spread loops
        "repeat_ms_per_step": repeats,
        "wall": (soak_t0 if soak_s > 0 else t0, t1),
    }
    del sets, ws
    L.close()
    torch.cuda.empty_cache()
    return res


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
    hin = [synth_inputs.normal(n, 1234 + i, w.dtype).pin_memory()
           for i, n in enumerate((nq, nkv, nkv, nq))]
    hout = [torch.empty_like(t).pin_memory() for t in hin]
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
    L.close()
    return {"ms_per_step": ms, "bytes_in": T, "bytes_out": T, "step_bytes": 2 * T}


def cpu_baseline(w, layout, budget_s, order="bshd"):
    """The oracle as it stands (plain C loop, one thread) on the host cores,
    over whole steps of the same workload, repeated until `budget_s`."""
    import oracle
    import synth_inputs
    oracle.build()
    K = w.K(layout)
    nq, nkv = w.tensor_elems(w.Hq), w.tensor_elems(w.Hkv)
    q, k, v, o = (synth_inputs.bits(synth_inputs.normal(n, 1234 + i, w.dtype))
                  for i, n in enumerate((nq, nkv, nkv, nq)))
    step_bytes = 2 * (q.nbytes + k.nbytes + v.nbytes + o.nbytes)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.seq2head(q, w.B, w.S, w.Hq, w.d, w.N, K, order=order)
        oracle.seq2head(k, w.B, w.S, w.Hkv, w.d, w.N, K, order=order)
        oracle.seq2head(v, w.B, w.S, w.Hkv, w.d, w.N, K, order=order)
        oracle.head2seq(o, w.B, w.S, w.Hq, w.d, w.N, K, order=order)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(step_bytes * reps / el / 1e9, 3), "unit": "GB/s",
            "cores": 1, "kind": "oracle",
            "sample": "%d whole steps of %s (%s, Q/K/V seq2head + O head2seq), "
                      "%.1f s" % (reps, w.name, layout, el)}


def gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


def main_ours(args, dist):
    import torch
    import sequence_re_layout_gb300 as basp
    from sequence_re_layout_gb300.build import build_library
    from sequence_re_layout_gb300.workloads import HEADLINE, WORKLOADS

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
        import dataclasses
        w = dataclasses.replace(w, dtype=args.dtype)
    peak, peak_kind = hbm_peak()

    sampler = ClockSampler(dev.index)
    dist.barrier()
    if args.qkv_packed and args.algo != "fused":
        raise SystemExit("--qkv-packed runs the fused path only")
    r = run_device(w, args.layout, args.algo, args.steps, args.warmup, dev,
                   soak_s=args.soak_s, order=args.order, packed=args.qkv_packed,
                   graph=args.graph, spread=0 if args.no_extras else 5)
    sampler.stop()
    dist.barrier()
    t_max = dist.max(r["total_ms"])
    total_bytes = dist.sum(r["step_bytes"] * args.steps)
    value = total_bytes / (t_max * 1e-3) / 1e9
    clocks = sampler.summary(*r["wall"])

    info = r["info"]
    s2h_gbs = gbs(r["s2h_bytes"], r["s2h_ms_mean"])
    traffic = None
    if args.order == "bshd" and not args.qkv_packed:
        traffic = ncu_traffic(w.name, args.layout, "seq2head_qkv_" + args.algo)
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
        "roofline": {
            "bound": "hbm", "kernel": "basp_relayout_kernel<16> (seq2head Q,K,V)",
            "achieved": round(s2h_gbs, 2), "peak": peak, "unit": "GB/s",
            "frac": round(s2h_gbs / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": r["s2h_bytes"],
            "launch_ms_mean": round(r["s2h_ms_mean"], 6),
            "launch_timing": "CUDA events around %d back-to-back launches of "
                             "this kernel alone on the bench stream" % args.steps,
            "peak_kind": "of %s" % peak_kind,
        },
        "head2seq": {"achieved_gbs": round(gbs(r["h2s_bytes"], r["h2s_ms_mean"]), 2),
                     "launch_ms_mean": round(r["h2s_ms_mean"], 6)},
        "analytic": {"peers_per_rank": info["peers"],
                     "bytes_per_peer_q": info["bytes_per_peer_q"],
                     "bytes_per_peer_kv": info["bytes_per_peer_kv"],
                     "tokens_per_rank": info["tokens_per_rank"],
                     "foil_tokens_per_rank": info["foil_tokens_per_rank"]},
        "gpu_launches": r["launches"],
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
        lps = r["launches"] // ((2 + len(r["repeat_ms_per_step"])) * args.steps)
        out["gpu_launches"] += 2 * ne * lps
    if not args.no_extras and dist.rank == 0:
        other = "ulysses" if args.layout == "basp" else "basp"
        ru = run_device(w, other, args.algo, args.steps, args.warmup, dev,
                        order=args.order, packed=args.qkv_packed)
        vu = gbs(ru["step_bytes"] * args.steps, ru["total_ms"])
        ou = ru["info"]
        out[other] = {"value": round(vu, 2), "ms_per_step": round(ru["ms_per_step"], 6),
                      "K": ou["K"], "pct_hbm_peak": round(100 * vu / peak, 2),
                      "peers_per_rank": ou["peers"],
                      "bytes_per_peer_q": ou["bytes_per_peer_q"],
                      "seq2head_gbs": round(gbs(ru["s2h_bytes"], ru["s2h_ms_mean"]), 2)}
        if args.layout == "basp" and w.N % w.B == 0:
            # the review's "trivial alternative" (Strengths, Table I): Ulysses
            # with SP = N/B, every group of K = N/B ranks holding all B
            # sequences -- B*B*S/N tokens per rank, B times BASP's bytes
            from sequence_re_layout_gb300.workloads import Workload
            wf = Workload(w.name + "_foil", w.B * w.B, w.S, w.Hq, w.Hkv, w.d,
                          w.N, w.N // w.B, w.dtype)
            rf = run_device(wf, "basp", args.algo, args.steps, args.warmup, dev,
                            order=args.order)
            out["foil_ulysses_sp_n_over_b"] = {
                "tokens_per_rank": rf["info"]["tokens_per_rank"],
                "basp_tokens_per_rank": info["tokens_per_rank"],
                "bytes_per_step": rf["step_bytes"],
                "ms_per_step": round(rf["ms_per_step"], 6),
                "value": round(gbs(rf["step_bytes"] * args.steps, rf["total_ms"]), 2),
                "time_vs_basp": round(rf["ms_per_step"] / (r["total_ms"] / args.steps), 3)}
            out["gpu_launches"] += rf["launches"]
        out["gpu_launches"] += ru["launches"]
        alts = [a for a in ("fused", "three_pass", "three_pass_elide") if a != args.algo]
        notes = {"three_pass": "same algorithmic bytes; the three passes move them 3x",
                 "three_pass_elide": "identity pass skipped when the receive chunks "
                                     "are already head-sharded (2 passes here: %s)"
                                     % ("yes" if info["seqs_per_group"] == 1 or
                                        args.order == "sbhd" else "no"),
                 "fused": "one pass"}
        for alt in alts:
            rt = run_device(w, args.layout, alt, args.steps, args.warmup, dev,
                            order=args.order)
            vt = gbs(rt["step_bytes"] * args.steps, rt["total_ms"])
            out[alt] = {"value": round(vt, 2), "ms_per_step": round(rt["ms_per_step"], 6),
                        "pct_hbm_peak": round(100 * vt / peak, 2), "note": notes[alt]}
            out["gpu_launches"] += rt["launches"]
        if dist.world == 1:
            out["cpu_baseline"] = cpu_baseline(w, args.layout, args.cpu_baseline_s,
                                               order=args.order)
    if dist.rank == 0:
        print(json.dumps(out), flush=True)


def main_reference(args, dist):
    """The reference arm: the CPU oracle, as it stands, timed on the host
    cores over bounded samples of the same workload (rank 0 only)."""
    if dist.rank != 0:
        return
    import oracle
    import synth_inputs
    from sequence_re_layout_gb300.workloads import HEADLINE, WORKLOADS
    oracle.build()
    w = WORKLOADS[args.config or HEADLINE]
    if args.dtype:
        import dataclasses
        w = dataclasses.replace(w, dtype=args.dtype)
    K = w.K(args.layout)
    o = args.order
    # bound the whole run to about two minutes: shrink S (a multiple of K) so
    # one step takes at most budget / (steps + warmup)
    budget_s = 120.0
    nq, nkv = w.tensor_elems(w.Hq), w.tensor_elems(w.Hkv)

    def make(S):
        ws = [w.B * S * h * w.d for h in (w.Hq, w.Hkv, w.Hkv, w.Hq)]
        return [synth_inputs.bits(synth_inputs.normal(n, 1234 + i, w.dtype))
                for i, n in enumerate(ws)]

    def one(S, x):
        oracle.seq2head(x[0], w.B, S, w.Hq, w.d, w.N, K, order=o)
        oracle.seq2head(x[1], w.B, S, w.Hkv, w.d, w.N, K, order=o)
        oracle.seq2head(x[2], w.B, S, w.Hkv, w.d, w.N, K, order=o)
        oracle.head2seq(x[3], w.B, S, w.Hq, w.d, w.N, K, order=o)

    S = w.S
    probe_S = max(K, (w.S // 16) // K * K)
    xp = make(probe_S)
    t0 = time.perf_counter()
    one(probe_S, xp)
    per_token = (time.perf_counter() - t0) / probe_S
    per_step_budget = budget_s / max(1, args.steps + args.warmup)
    if per_token * w.S > per_step_budget:
        S = max(K, int(per_step_budget / per_token) // K * K)
    x = make(S)
    for _ in range(args.warmup):
        one(S, x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one(S, x)
    el = time.perf_counter() - t0
    step_bytes = 2 * sum(a.nbytes for a in x)
    value = step_bytes * args.steps / el / 1e9
    sample = ("%s at S=%d of %d (same B, heads, d, N, K), %d steps, %.1f s"
              % (w.name, S, w.S, args.steps, el))
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3),
        "unit": "GB/s", "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * el / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (~N(0,1) %s, seeded)" % w.dtype,
        "config": {"workload": w.name, "layout": args.layout, "algo": "oracle",
                   "order": o, "B": w.B, "S": w.S, "Hq": w.Hq, "Hkv": w.Hkv,
                   "d": w.d, "N": w.N, "K": K},
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
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
