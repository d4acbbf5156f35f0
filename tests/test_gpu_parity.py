"""GPU parity: the CUDA path through the C ABI against the CPU oracle, bit for
bit (0 mismatching bits, bf16 and fp32 alike), on every workload shape at full
size, both layouts (BASP K = N/B, Ulysses K = N), both directions (Q, K, V
seq->head in one call; attention output O head->seq), both algorithms."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs
from parity import (assert_bits_equal, device_outputs, make_inputs,
                    oracle_outputs)
from sequence_re_layout_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu

ALGOS = ("fused", "three_pass", "three_pass_elide")


def _shapes():
    seen, out = set(), []
    for w in WORKLOADS.values():
        key = (w.B, w.S, w.Hq, w.Hkv, w.d, w.N, w.K_basp)
        if key in seen:
            continue
        seen.add(key)
        out.append(w)
    return out


def _check(w, dtype, layout, kind="normal", seed=1234):
    K = w.K(layout)
    args = (w.B, w.S, w.Hq, w.Hkv, w.d, w.N, K)
    q, k, v, o = make_inputs(w.B, w.S, w.Hq, w.Hkv, w.d, dtype, seed, kind)
    exp = oracle_outputs(q, k, v, o, *args)
    for algo in ALGOS:
        got = device_outputs(q, k, v, o, *args, dtype, algo)
        for name, g, e in zip(("q", "k", "v", "o"), got, exp):
            assert_bits_equal(g, e, "%s %s %s %s %s" % (w.name, layout, dtype, algo, name))
        del got
    torch.cuda.empty_cache()


@pytest.mark.parametrize("layout", ["basp", "ulysses"])
@pytest.mark.parametrize("w", _shapes(), ids=lambda w: w.name)
def test_full_size_bf16(w, layout):
    _check(w, "bf16", layout)


@pytest.mark.parametrize("layout", ["basp", "ulysses"])
@pytest.mark.parametrize("w", _shapes(), ids=lambda w: w.name)
def test_full_size_fp32(w, layout):
    _check(w, "fp32", layout)


@pytest.mark.parametrize("layout", ["basp", "ulysses"])
def test_tiny_index_valued(layout):
    """The tiny shape with every element set to its own index (distinct values
    across Q, K, V and O)."""
    w = WORKLOADS["tiny_B2_N4_S64_H4_d16_fp32"]
    _check(w, "fp32", layout, kind="index")


SMALL = [
    # (B, S, Hq, Hkv, d, N, K)  ragged tiles, odd rows, groups, K=1, K=3
    (2, 48, 6, 3, 24, 6, 3),      # K=3, rows of 2*24 and 1*24 elements
    (4, 36, 12, 6, 8, 6, 3),      # G=2 groups, Bg=2
    (6, 30, 6, 6, 40, 6, 3),      # G=2, Bg=3, rows of 80 elements
    (3, 1000, 8, 8, 8, 3, 1),     # K=1: local-only copy
    (1, 8, 8, 8, 8, 8, 8),        # one token per rank
    (2, 2056, 24, 8, 128, 8, 4),  # S/K = 514: ragged last tile of each block
    (2, 520, 12, 4, 72, 4, 4),    # vpr = 27 (bf16), not a power of two
    (8, 256, 32, 16, 16, 64, 8),  # 64 virtual ranks, 8 groups of 8
    (4, 512, 64, 32, 8, 128, 32), # 128 virtual ranks, 4 groups of 32
    (2, 96, 48, 48, 8, 48, 24),   # 48 ranks, K = 24 (not a power of two)
]


@pytest.mark.parametrize("shape", SMALL)
@pytest.mark.parametrize("dtype", ["bf16", "fp32", "fp16", "fp8"])
def test_small_shapes(shape, dtype):
    B, S, Hq, Hkv, d, N, K = shape
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, dtype, 99, kind="bits")
    exp = oracle_outputs(q, k, v, o, *shape)
    for algo in ALGOS:
        got = device_outputs(q, k, v, o, *shape, dtype, algo)
        for name, g, e in zip("qkvo", got, exp):
            assert_bits_equal(g, e, "%s %s %s %s" % (shape, dtype, algo, name))


@pytest.mark.parametrize("name", ["llama3.2-1b_B2_S8192", "llama3.2-3b_B2_S32768"])
@pytest.mark.parametrize("layout", ["basp", "ulysses"])
def test_full_size_fp8(name, layout):
    """1-byte elements (fp8 activations): the 1-byte word is never split."""
    _check(WORKLOADS[name], "fp8", layout)


@pytest.mark.parametrize("layout", ["basp", "ulysses"])
def test_full_size_fp16(layout):
    _check(WORKLOADS["llama3.2-1b_B2_S8192"], "fp16", layout)


@pytest.mark.parametrize("layout", ["basp", "ulysses"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_long_launch_ragged_tiles(layout, dtype):
    """A launch long enough for the 512-thread CTAs on 32 KiB tiles (about
    22K tiles of 16 KiB for Q, K, V), with S/K = 4098 tokens per block (the
    last tile of every block is ragged) and d = 136 (rows of 102 or 51
    vectors, not a power of two)."""
    from sequence_re_layout_gb300.workloads import Workload
    w = Workload("long_ragged", 2, 16392, 24, 8, 136, 8, 4)
    _check(w, dtype, layout, kind="bits", seed=4242)
