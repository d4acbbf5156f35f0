"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the oracle on the same seeded inputs, compare raw bits."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth_inputs
import sequence_re_layout_gb300 as basp


def make_inputs(B, S, Hq, Hkv, d, dtype, seed, kind="normal"):
    """CPU tensors q, k, v, o (flat virtual-rank buffers)."""
    n_q, n_kv = B * S * Hq * d, B * S * Hkv * d
    if kind == "index":
        # distinct values: every element of the four tensors a different integer
        q = synth_inputs.index_valued(n_q, 0)
        k = synth_inputs.index_valued(n_kv, n_q)
        v = synth_inputs.index_valued(n_kv, n_q + n_kv)
        o = synth_inputs.index_valued(n_q, n_q + 2 * n_kv)
        if dtype != "fp32":
            raise ValueError("index-valued inputs are fp32")
        return q, k, v, o
    gen = synth_inputs.normal if kind == "normal" else synth_inputs.random_bits
    return (gen(n_q, seed, dtype), gen(n_kv, seed + 1, dtype),
            gen(n_kv, seed + 2, dtype), gen(n_q, seed + 3, dtype))


def oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K):
    """Expected head-sharded Q, K, V and seq-sharded O, as raw-bit arrays."""
    bq, bk, bv, bo = (synth_inputs.bits(t) for t in (q, k, v, o))
    return (oracle.seq2head(bq, B, S, Hq, d, N, K),
            oracle.seq2head(bk, B, S, Hkv, d, N, K),
            oracle.seq2head(bv, B, S, Hkv, d, N, K),
            oracle.head2seq(bo, B, S, Hq, d, N, K))


def device_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K, dtype, algo,
                   stream=None):
    """Head-sharded Q, K, V and seq-sharded O from the CUDA path."""
    dev = torch.device("cuda:0")
    qd, kd, vd, od = (t.to(dev) for t in (q, k, v, o))
    outs = [torch.empty_like(t) for t in (qd, kd, vd, od)]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dtype) as L:
        ws = None
        if algo != "fused":
            ws = torch.empty(max(L.info["workspace_bytes"], 1), dtype=torch.uint8,
                             device=dev)
        s = stream or torch.cuda.current_stream()
        basp.basp_seq2head(L.handle, algo, qd, kd, vd, outs[0], outs[1], outs[2],
                           ws, stream=s)
        basp.basp_head2seq(L.handle, algo, od, None, None, outs[3], None, None,
                           ws, stream=s)
        torch.cuda.synchronize()
    return outs


def assert_bits_equal(dev_tensor, expected_bits, what):
    """0 mismatching bits, compared on the GPU."""
    got = dev_tensor.view(synth_inputs.BITS[dev_tensor.dtype])
    exp = torch.from_numpy(np.ascontiguousarray(expected_bits)).to(got.device)
    assert got.shape == exp.shape, what
    if not torch.equal(got, exp):
        bad = (got != exp).nonzero()
        n_bad = bad.numel()
        first = bad[:5].flatten().tolist()
        raise AssertionError("%s: %d mismatching elements, first at %s"
                             % (what, n_bad, first))
