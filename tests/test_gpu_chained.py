"""Chains of re-layouts on one stream, each call reading the buffer the call
before it wrote.

Every launch may be scheduled while the previous one drains, and its CTAs
prefetch their source lines into L2 before waiting for it.  In a chain, the
lines a launch prefetches are the ones the previous launch is still writing.
So a stale read anywhere would break these chains.  They check that each step
equals the oracle, and that seq2head followed by head2seq, repeated, gives
back the input bit for bit.  Both the fused and the three-pass paths run
(three-pass: pack -> exchange -> unpack, each pass reading the last one's
output).
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs
import sequence_re_layout_gb300 as basp

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

CHAINS = [
    # (B, S, Hq, Hkv, d, N, K, dtype): short launches (most of the grid is
    # resident while the previous launch drains), then a mid-size one
    (2, 1024, 24, 8, 128, 8, 4, "bf16"),
    (2, 1024, 24, 8, 128, 8, 8, "bf16"),
    (1, 2048, 32, 8, 64, 8, 8, "bf16"),
    (2, 4096, 32, 8, 64, 8, 4, "fp32"),
]


@pytest.mark.parametrize("shape", CHAINS, ids=lambda s: "B%d_S%d_K%d_%s" % (s[0], s[1], s[6], s[7]))
@pytest.mark.parametrize("algo", ["fused", "three_pass"])
def test_round_trip_chain_returns_the_input(shape, algo):
    B, S, Hq, Hkv, d, N, K, dt = shape
    nq, nkv = B * S * Hq * d, B * S * Hkv * d
    bits = synth_inputs.BITS[synth_inputs.DTYPES[dt]]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dt) as L:
        ws = torch.empty(max(1, L.info["workspace_bytes"]), dtype=torch.uint8, device=DEV)
        x0 = [synth_inputs.random_bits(n, 500 + i, dt) for i, n in enumerate((nq, nkv, nkv))]
        a = [t.to(DEV) for t in x0]
        b = [torch.empty_like(t) for t in a]
        rounds = 40
        for _ in range(rounds):
            # seq -> head into b, then head -> seq back into a: each launch
            # reads what the launch before it wrote
            basp.basp_seq2head(L.handle, algo, a[0], a[1], a[2], b[0], b[1], b[2], ws)
            basp.basp_head2seq(L.handle, algo, b[0], b[1], b[2], a[0], a[1], a[2], ws)
        # one more seq -> head, checked against the oracle
        basp.basp_seq2head(L.handle, algo, a[0], a[1], a[2], b[0], b[1], b[2], ws)
        torch.cuda.synchronize()
        for name, got, ref, H in zip("qkv", a, x0, (Hq, Hkv, Hkv)):
            assert torch.equal(got.cpu().view(bits), ref.view(bits)), \
                "%s not restored after %d round trips" % (name, rounds)
        for name, got, ref, H in zip("qkv", b, x0, (Hq, Hkv, Hkv)):
            want = oracle.seq2head(synth_inputs.bits(ref), B, S, H, d, N, K)
            assert np.array_equal(synth_inputs.bits(got.cpu()), want), name


def test_producer_kernel_then_relayout_each_step():
    """A torch kernel rewrites the input right before every re-layout on the
    same stream; every output must be the re-layout of that step's values."""
    B, S, Hq, Hkv, d, N, K = 2, 1024, 24, 8, 128, 8, 4
    n = B * S * Hq * d
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "fp32") as L:
        x = torch.empty(n, dtype=torch.float32, device=DEV)
        outs = [torch.empty_like(x) for _ in range(6)]
        for step, out in enumerate(outs):
            x.fill_(float(step + 1))          # producer: a torch kernel
            x[step::7] = -float(step)         # and a second one, strided
            basp.basp_seq2head(L.handle, "fused", x, None, None, out, None, None)
            basp.basp_head2seq(L.handle, "fused", out, None, None, x, None, None)
        torch.cuda.synchronize()
        for step, out in enumerate(outs):
            src = torch.full((n,), float(step + 1))
            src[step::7] = -float(step)
            want = oracle.seq2head(synth_inputs.bits(src), B, S, Hq, d, N, K)
            assert np.array_equal(synth_inputs.bits(out.cpu()), want), step


def test_qkv_projection_then_packed_seq2head():
    """The path as a model runs it: a GEMM (the fused QKV projection) writes
    the packed QKV activations, and basp_seq2head_qkv reads them right after,
    on the same stream, step after step with new weights."""
    B, S, Hq, Hkv, d, N, K = 2, 1024, 24, 8, 128, 8, 4
    hidden = 256
    W = (Hq + 2 * Hkv) * d
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    x = torch.randn(N, B * S // N, hidden, generator=g, device=DEV).to(torch.bfloat16)
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        nq, nkv = B * S * Hq * d, B * S * Hkv * d
        qkv = torch.empty(N, B * S // N, W, dtype=torch.bfloat16, device=DEV)
        outs = []
        for step in range(4):
            w = torch.randn(hidden, W, generator=g, device=DEV).to(torch.bfloat16)
            torch.matmul(x, w, out=qkv)                       # the producer GEMM
            o = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for n in (nq, nkv, nkv)]
            basp.basp_seq2head_qkv(L.handle, qkv, *o)
            outs.append((qkv.clone(), o))                     # snapshot after the call
        torch.cuda.synchronize()
        for step, (packed, o) in enumerate(outs):
            want = oracle.seq2head_qkv(synth_inputs.bits(packed.view(-1).cpu()),
                                       B, S, Hq, Hkv, d, N, K)
            for name, got, e in zip("qkv", o, want):
                assert np.array_equal(synth_inputs.bits(got.cpu()), e), (step, name)
