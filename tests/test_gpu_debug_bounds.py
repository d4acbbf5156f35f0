"""The bounds-checking build (libbasp_debug.so) on the GPU: every access of
every kernel is checked against its buffer's extent.  Run over the fuzz cases
and the full-size workloads, it must find no access outside a buffer, and
its results must still match the oracle bit for bit.  Runs in a child process
because the library is chosen when the binding is first imported."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_no_access_outside_any_buffer():
    env = dict(os.environ, BASP_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "test_gpu_debug_bounds.py")],
                       env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "bounds ok" in r.stdout


def _child():
    sys.path.insert(0, HERE)
    sys.path.insert(0, os.path.dirname(HERE))
    import sequence_re_layout_gb300 as basp
    assert basp.binding.LIB_PATH.endswith("libbasp_debug.so")
    import test_gpu_fuzz
    from parity import assert_bits_equal, device_outputs, make_inputs, oracle_outputs
    from sequence_re_layout_gb300.workloads import WORKLOADS

    basp.basp_debug_bounds_violations()                   # start from zero
    for seed in range(60):
        test_gpu_fuzz.test_fuzz_against_oracle(seed)
    assert basp.basp_debug_bounds_violations() == 0
    for name in ("llama3.2-1b_B2_S8192", "llama3.2-3b_B2_S16384"):
        w = WORKLOADS[name]
        for layout in ("basp", "ulysses"):
            args = (w.B, w.S, w.Hq, w.Hkv, w.d, w.N, w.K(layout))
            q, k, v, o = make_inputs(w.B, w.S, w.Hq, w.Hkv, w.d, "bf16", 5, "bits")
            exp = oracle_outputs(q, k, v, o, *args)
            for algo in ("fused", "three_pass", "three_pass_elide"):
                got = device_outputs(q, k, v, o, *args, "bf16", algo)
                for nm, g, e in zip("qkvo", got, exp):
                    assert_bits_equal(g, e, "debug %s %s %s %s" % (name, layout, algo, nm))
    n = basp.basp_debug_bounds_violations()
    assert n == 0, "%d out-of-bounds accesses" % n
    print("bounds ok")


if __name__ == "__main__":
    _child()
