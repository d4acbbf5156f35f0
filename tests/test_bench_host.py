"""Host logic of bench.py that needs no GPU: the replica barrier and the
max/sum reductions over gloo ranks (world size 2), the clock-sample parser,
the ncu traffic lookup, and the reference arm on a tiny budget."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _dist_worker(rank, world, port, result_dir):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank),
                       "LOCAL_RANK": str(rank), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    d = bench.Dist()
    d.barrier()
    mx = d.max(float(rank + 1) * 10.0)
    sm = d.sum(float(rank + 1))
    d.close()
    with open(os.path.join(result_dir, "r%d" % rank), "w") as f:
        json.dump({"max": mx, "sum": sm}, f)


def test_replica_reductions_over_gloo(tmp_path):
    mp.spawn(_dist_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        got = json.load(open(tmp_path / ("r%d" % r)))
        assert got == {"max": 20.0, "sum": 3.0}


def test_clock_summary_parses_nvidia_smi_lines():
    cs = bench.ClockSampler.__new__(bench.ClockSampler)
    cs.proc = object()
    cs.lines = [
        "2026/12/02 10:00:00.100, 2070, 2070, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.300, 1980, 2070, 800.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:05.000, 300, 2070, 90.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    import datetime as dt
    t0 = dt.datetime(2026, 12, 2, 10, 0, 0).timestamp()
    s = cs.summary(t0, t0 + 1.0)
    assert s["samples"] == 2 and s["sm_mhz"] == 2025.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"]


def test_traffic_lookup_tracks_the_kernel_source(tmp_path, monkeypatch):
    f = tmp_path / "t.txt"
    f.write_text("traffic wl basp seq2head_qkv_fused bytes=123 source=%s\n"
                 "traffic wl basp head2seq_o_fused bytes=7 source=0000\n"
                 % bench.source_digest())
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.ncu_traffic("wl", "basp", "seq2head_qkv_fused") == 123.0
    assert bench.ncu_traffic("wl", "basp", "head2seq_o_fused") is None   # stale
    assert bench.ncu_traffic("other", "basp", "seq2head_qkv_fused") is None


def test_reference_arm_prints_one_line():
    """--impl reference: the oracle on the host cores, one JSON line."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                        "reference", "--steps", "2", "--warmup", "1",
                        "--config", "llama3.2-3b_B2_S1024"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_under_two_ranks():
    """torchrun with 2 ranks: rank 0 alone prints the reference line, the other
    rank exits 0 without work."""
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--config", "llama3.2-3b_B2_S1024"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


@pytest.mark.parametrize("content,expect", [
    ('{"hbm_gbs": 6682.8}', (6682.8, "measured")),
    ('{"hbm_gbs": {"value": 6500}}', (6500.0, "measured")),
    ('{"hbm": {"burst": 6600}}', (6600.0, "measured")),
    ('{"bf16_tflops": 1900}', (bench.FALLBACK_HBM_GBS, "fallback")),
    ('not json', (bench.FALLBACK_HBM_GBS, "fallback")),
])
def test_peak_file_forms(tmp_path, monkeypatch, content, expect):
    (tmp_path / "MEASURED_PEAKS.json").write_text(content)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.hbm_peak() == expect


def test_peak_file_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")


def _run_bench(args, env_extra=None, timeout=600):
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "LOCAL_WORLD_SIZE", "MASTER_ADDR",
              "MASTER_PORT"):
        env.pop(k, None)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args,
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT,
                          env=env)


def test_gpus_flag_starts_that_many_ranks():
    """--gpus 2 with no launcher environment starts two local ranks (each
    with its own RANK / LOCAL_RANK), and rank 0's line reports both."""
    r = _run_bench(["--impl", "reference", "--gpus", "2", "--steps", "1",
                    "--warmup", "1", "--config", "tiny_B2_N4_S64_H4_d16_fp32"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout          # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["impl"] == "reference"


def test_gpus_flag_must_agree_with_the_launcher():
    """A launcher's WORLD_SIZE that disagrees with --gpus is an error, not a
    silent run at the launcher's size."""
    r = _run_bench(["--impl", "reference", "--gpus", "4", "--steps", "1",
                    "--warmup", "1", "--config", "tiny_B2_N4_S64_H4_d16_fp32"],
                   env_extra={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode != 0
    assert "must agree" in r.stderr


def test_timing_check_flags_impossible_kernel_times():
    """The cross-check of per-kernel launch times against the step time."""
    peak = 6700.0
    # 200 MB + 130 MB in 31 us + 20 us against a 51 us step: consistent
    ok = bench.check_timings(200e6, 0.031, 130e6, 0.020, 0.051, peak)
    assert ok["consistent"] and ok["plausible"]
    # a slow seq2head reading (43 us) leaves 10 us for 130 MB of head2seq:
    # 13 TB/s, above any copy peak
    bad = bench.check_timings(200e6, 0.043, 130e6, 0.020, 0.053, peak)
    assert not bad["plausible"] and not bad["consistent"]
    assert bad["implied_head2seq_gbs"] > 1.15 * peak


def test_percentiles():
    xs = [float(x) for x in range(1, 11)]          # 1..10
    assert bench.percentile(xs, 50) == 5.5
    assert bench.percentile(xs, 10) == 1.9
    assert bench.percentile(xs, 90) == 9.1
    assert bench.percentile([3.0], 90) == 3.0
    r = {"step_bytes": 1e9, "window_ms_per_step": [1.0, 2.0, 0.5], "steps_per_window": 7}
    st = bench.window_stats(r)
    assert st["gbs_median"] == 1000.0 and st["windows"] == 3 and st["steps_per_window"] == 7


def test_launcher_stops_its_ranks_on_sigterm(tmp_path):
    """A SIGTERM to the --gpus launcher ends the ranks it started (no orphans
    left holding GPUs after a timeout)."""
    import signal
    import time as _t
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    # a reference run long enough to be interrupted (many steps of a big shape)
    p = subprocess.Popen([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                          "reference", "--gpus", "2", "--steps", "100000", "--warmup", "0",
                          "--config", "llama3.2-1b_B2_S8192"],
                         cwd=ROOT, env=env, stdout=subprocess.DEVNULL,
                         stderr=subprocess.DEVNULL, start_new_session=True)
    _t.sleep(8)
    # rank 1 of the reference arm exits at once; rank 0 is still working
    kids = subprocess.run(["pgrep", "-P", str(p.pid)], capture_output=True, text=True).stdout.split()
    assert kids, "no rank running"
    p.send_signal(signal.SIGTERM)
    p.wait(timeout=60)
    _t.sleep(1)
    for k in kids:
        assert not os.path.exists("/proc/%s" % k) or \
            open("/proc/%s/stat" % k).read().split()[2] == "Z", "rank %s still running" % k


def test_committed_traffic_matches_the_current_kernel():
    """The ncu traffic record under profiles/ was taken on the kernel and
    launch planning that are in the tree now, for the headline and every
    target leg (else the bench would report traffic = null: recapture after
    changing relayout_kernel.cuh or relayout.cu)."""
    from sequence_re_layout_gb300.workloads import HEADLINE, TARGETS
    for wl in (HEADLINE,) + tuple(TARGETS):
        for lay in ("basp", "ulysses"):
            for role in ("seq2head_qkv_fused", "head2seq_o_fused"):
                assert bench.ncu_traffic(wl, lay, role) is not None, (wl, lay, role)
