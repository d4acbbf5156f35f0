"""The all-core oracle (``basp_oracle_*_threads``) against the plain
single-thread element loop it restates.

The threaded form exists only so the benchmark can time the oracle on every
host core.  It must give the same bytes as the plain loop, which the other
pins fix: on every tiny shape of the brute-force enumeration, in both token
orders and both directions, for thread counts that do and do not divide the
row count (including more threads than rows), and on a workload-shaped case.
Outputs are pre-filled with a sentinel so a span that a thread skipped cannot
pass by reusing memory that happened to hold the right bytes.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth_inputs
from test_oracle_pins import CONFIG_SHAPES, tiny_shapes

SENTINEL = np.int32(-0x5A5A5A5B)


def _threads(direction, x, B, S, H, d, N, K, nthreads, order):
    """Call the C entry point directly on an output filled with a sentinel."""
    x = np.ascontiguousarray(x)
    out = np.full_like(x, SENTINEL if x.dtype == np.int32 else -1)
    if x.size == 0:
        return out
    fn = getattr(oracle._load(), "basp_oracle_%s_threads" % direction)
    rc = fn(B, S, H, d, N, K, x.itemsize, oracle.ORDERS[order], nthreads,
            x.ctypes.data_as(ctypes.c_void_p), out.ctypes.data_as(ctypes.c_void_p))
    assert rc == 0
    return out


@pytest.mark.parametrize("order", ["bshd", "sbhd"])
def test_threads_match_plain_loop_on_every_tiny_shape(order):
    shapes = tiny_shapes()
    assert len(shapes) > 300
    for (B, S, H, d, N, K) in shapes:
        x = np.arange(B * S * H * d, dtype=np.int32) * 5 + 11
        want_s2h = oracle.seq2head(x, B, S, H, d, N, K, order=order)
        want_h2s = oracle.head2seq(x, B, S, H, d, N, K, order=order)
        for nt in (1, 2, 3, 7, 64):
            np.testing.assert_array_equal(
                _threads("seq2head", x, B, S, H, d, N, K, nt, order), want_s2h)
            np.testing.assert_array_equal(
                _threads("head2seq", x, B, S, H, d, N, K, nt, order), want_h2s)


@pytest.mark.parametrize("name", ["llama1b", "llama3b", "llama1b_B1"])
def test_threads_match_plain_loop_on_workload_shapes(name):
    B, S, Hq, Hkv, d, N, K = CONFIG_SHAPES[name]
    for H, seed in ((Hq, 1), (Hkv, 2)):
        x = synth_inputs.bits(synth_inputs.normal(B * S * H * d, seed))
        for nt in (4, oracle.host_cores(), 13):
            np.testing.assert_array_equal(
                oracle.seq2head_threads(x, B, S, H, d, N, K, nt),
                oracle.seq2head(x, B, S, H, d, N, K))
            np.testing.assert_array_equal(
                oracle.head2seq_threads(x, B, S, H, d, N, K, nt),
                oracle.head2seq(x, B, S, H, d, N, K))


def test_threads_reject_what_the_plain_loop_rejects():
    x = np.zeros(2 * 6 * 4 * 2, dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.seq2head_threads(x, 2, 6, 4, 2, 4, 4, 4)     # S % K != 0
    with pytest.raises(ValueError):
        oracle.seq2head_threads(np.zeros(64, np.int32), 2, 8, 2, 2, 4, 2, 0)   # no threads


MUTATIONS = [
    ("a span starts one row late",
     "rows * i / nthreads, rows * (i + 1) / nthreads}",
     "rows * i / nthreads + (i > 0), rows * (i + 1) / nthreads}"),
    ("sequence and token digits of the source row swapped",
     "const int64_t bl   = (row / Sk) % Bg;",
     "const int64_t bl   = row % Bg;"),
    ("head block taken from the wrong modulus",
     "            const int64_t hl = h % Hk;\n            const int64_t r_out = g * K + jp;\n            for (int64_t e = 0; e < d; ++e) {\n                const int64_t src = r_in * P + (t_in * H + h) * d + e;\n                const int64_t dst = r_out * P + (t_out * Hk + hl) * d + e;\n                if (w->dir",
     "            const int64_t hl = h % K;\n            const int64_t r_out = g * K + jp;\n            for (int64_t e = 0; e < d; ++e) {\n                const int64_t src = r_in * P + (t_in * H + h) * d + e;\n                const int64_t dst = r_out * P + (t_out * Hk + hl) * d + e;\n                if (w->dir"),
]


@pytest.mark.parametrize("what,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_in_threaded_walk_is_caught(what, old, new, tmp_path):
    import os
    import subprocess
    src = os.path.join(os.path.dirname(oracle.__file__), "basp_oracle.c")
    text = open(src).read()
    assert text.count(old) == 1, "mutation anchor not found: " + what
    c = tmp_path / "mutant.c"
    c.write_text(text.replace(old, new))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(c)], check=True)
    lib = oracle.load_from(str(so))
    caught = False
    for (B, S, H, d, N, K) in tiny_shapes():
        x = np.arange(B * S * H * d, dtype=np.int32) * 5 + 11
        if x.size == 0:
            continue
        want = oracle.seq2head(x, B, S, H, d, N, K)
        out = np.full_like(x, SENTINEL)
        rc = lib.basp_oracle_seq2head_threads(B, S, H, d, N, K, 4, 0, 3,
                                              x.ctypes.data_as(ctypes.c_void_p),
                                              out.ctypes.data_as(ctypes.c_void_p))
        if rc != 0 or not np.array_equal(out, want):
            caught = True
            break
    assert caught, "no shape caught: " + what
