"""basp_seq2head_noalloc: the three-pass seq->head re-layout with the
library's built-in scratch, for callers that cannot allocate device memory
(a host framework's plugin interface whose allocator owns all device memory,
a serving loop that bans cudaMalloc on its hot path).

Two calls in a row through the C ABI, each on fresh inputs, must give the same
bits as the ordinary entry point basp_seq2head and as the CPU oracle; a call
whose scratch would exceed the built-in buffer is refused before any launch.
This file is collected last on purpose: it shares no state with the others
and passes alone or after them.
"""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs
import sequence_re_layout_gb300 as basp

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("shape,dtype,order", [
    # (B, S, Hq, Hkv, d, N, K): Llama-3.2-1B heads at S=1024 (24 MiB of
    # scratch for Q, K, V in bf16), BASP and Ulysses; then other element
    # types and the sequence-first order at sizes that fit the scratch
    ((2, 1024, 32, 8, 64, 8, 4), "bf16", "bshd"),
    ((2, 1024, 32, 8, 64, 8, 8), "bf16", "bshd"),
    ((2, 1024, 32, 8, 64, 8, 8), "bf16", "sbhd"),
    ((2, 512, 32, 8, 64, 8, 4), "fp32", "bshd"),
    ((2, 1024, 32, 8, 64, 8, 4), "fp8", "sbhd"),
])
def test_noalloc_matches_seq2head_on_two_calls(shape, dtype, order):
    B, S, Hq, Hkv, d, N, K = shape
    nq, nkv = B * S * Hq * d, B * S * Hkv * d
    bits = synth_inputs.BITS[synth_inputs.DTYPES[dtype]]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dtype, order=order) as L:
        assert 2 * (L.info["bytes_q"] + 2 * L.info["bytes_kv"]) <= basp.BASP_NOALLOC_SCRATCH_BYTES
        for call, seed in enumerate((101, 202)):
            ins = [synth_inputs.random_bits(n, seed + i, dtype).to(DEV)
                   for i, n in enumerate((nq, nkv, nkv))]
            want = [torch.empty_like(t) for t in ins]
            got = [torch.empty_like(t).view(bits).fill_(-1).view(t.dtype) for t in ins]
            basp.basp_seq2head(L.handle, "fused", *ins, *want)
            basp.basp_seq2head_noalloc(L.handle, *ins, *got)
            torch.cuda.synchronize()
            for name, g, w, x, H in zip("qkv", got, want, ins, (Hq, Hkv, Hkv)):
                assert torch.equal(g.view(bits), w.view(bits)), \
                    "call %d tensor %s differs from basp_seq2head" % (call, name)
                exp = oracle.seq2head(synth_inputs.bits(x.cpu()), B, S, H, d, N, K,
                                      order=order)
                assert np.array_equal(synth_inputs.bits(g.cpu()), exp), \
                    "call %d tensor %s differs from the oracle" % (call, name)


def test_noalloc_refuses_more_than_its_scratch():
    # S=2048: Q, K and V need 48 MiB of scratch, more than the 32 MiB built in
    B, S, Hq, Hkv, d, N, K = 2, 2048, 32, 8, 64, 8, 4
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        ins = [torch.zeros(B * S * h * d, dtype=torch.bfloat16, device=DEV)
               for h in (Hq, Hkv, Hkv)]
        outs = [torch.zeros_like(t) for t in ins]
        with pytest.raises(basp.BaspError) as e:
            basp.basp_seq2head_noalloc(L.handle, *ins, *outs)
        assert e.value.status == basp.BASP_ERR_WORKSPACE
        # Q alone (16 MiB of scratch) fits
        basp.basp_seq2head_noalloc(L.handle, ins[0], None, None, outs[0], None, None)
        torch.cuda.synchronize()
