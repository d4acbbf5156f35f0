"""bench.py on the GPU, briefly: one JSON line with the fields the
measurement contract names, for the default (extras) run and a short
sequence-first run."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_default_line_has_the_contract_fields():
    d = _run("--steps", "20", "--warmup", "3", "--soak-s", "0.2", "--cpu-baseline-s", "1",
             "--cpu-all-s", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["steps"] == 20 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 1000 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "llama3.2-3b_B2_S32768"
    r = d["roofline"]
    assert r["bound"] == "hbm" and 0 < r["frac"] < 1.5 and r["achieved"] > 0
    # BASP against Ulysses on the same shape: peers K-1 = 3 against N-1 = 7
    bu = d["basp_vs_ulysses"]
    assert bu["peers_per_rank"] == {"basp": 3, "ulysses": 7} and bu["step_time_ratio"] > 0.9
    # the pages' own figures ride along as context, with their hardware
    assert "A100" in d["context"]["pages_hardware"]
    # a distribution over 30 step windows
    dd = d["distribution"]
    assert dd["windows"] == 30 and dd["gbs_p10"] <= dd["gbs_median"] <= dd["gbs_p90"]
    # the same-run copy rate sits beside the measured peak
    assert r["copy_same_run"]["gbs"] > 1000
    # the per-kernel times add up to the step time
    assert d["timing_check"]["consistent"] and d["timing_check"]["plausible"]
    assert 0.9 < d["timing_check"]["ratio_vs_timed_region"] < 1.1
    c = d["cpu_baseline"]
    assert set(("value", "unit", "cores", "kind", "sample")) <= set(c)
    assert c["threads_1"]["value"] > 0 and c["threads_all"]["threads"] == c["cores"] >= 1
    # every long-sequence target, both layouts, both directions
    t = d["targets"]
    got = {(l["workload"], l["layout"]) for l in t["legs"]}
    assert got == {(w, lay) for w in ("qwen1.5-1.8b_B2_S16384", "llama3.2-3b_B2_S16384",
                                      "llama3.2-3b_B2_S32768")
                   for lay in ("basp", "ulysses")}
    for l in t["legs"]:
        assert l["seq2head"]["frac"] > 0 and l["head2seq"]["frac"] > 0, l
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    for alt in ("ulysses", "three_pass", "three_pass_elide", "foil_ulysses_sp_n_over_b"):
        assert alt in d, alt


def test_sequence_first_packed_line():
    d = _run("--steps", "10", "--warmup", "3", "--soak-s", "0", "--no-extras",
             "--order", "sbhd", "--qkv-packed", "--config", "llama3.2-3b_B2_S4096")
    assert d["config"]["order"] == "sbhd" and d["config"]["qkv_packed"] is True
    assert d["value"] > 1000


def _two_rank_check(d):
    assert d["n_gpus"] == 2 and d["config"]["parallelism"] == "replicas"
    assert d["scaling"] == "weak" and d["value"] > 1000
    # value is both ranks' bytes over the slower rank's time
    assert abs(d["value"] - 2 * d["config"]["bytes_per_step"] / (d["ms_per_step"] * 1e6)) \
        < 0.01 * d["value"]


def test_two_replicas_started_by_the_gpus_flag():
    """--gpus 2 with no launcher: two local ranks (here both on cuda:0; their
    kernels never wait on each other, the ranks meet only at host barriers)."""
    _two_rank_check(_run("--gpus", "2", "--steps", "5", "--warmup", "2", "--soak-s", "0",
                         "--no-extras", "--config", "llama3.2-3b_B2_S4096"))


def test_two_replicas_under_torchrun():
    """The driver's multi-GPU launch: torchrun with --nproc-per-node 2."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--gpus", "2", "--steps", "5", "--warmup", "2", "--soak-s", "0",
                        "--no-extras", "--config", "llama3.2-3b_B2_S4096"],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    _two_rank_check(json.loads(lines[0]))
