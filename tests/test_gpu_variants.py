"""GPU parity for the two layout variants: sequence-first shards and the
packed QKV input/output.  Every bit is compared with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs
import sequence_re_layout_gb300 as basp
from parity import assert_bits_equal, make_inputs
from sequence_re_layout_gb300.workloads import WORKLOADS

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ALGOS = ("fused", "three_pass", "three_pass_elide")


def _run_sf(shape, dtype, seed=41, kind="bits"):
    B, S, Hq, Hkv, d, N, K = shape
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, dtype, seed, kind)
    bq, bk, bv, bo = (synth_inputs.bits(t) for t in (q, k, v, o))
    exp = (oracle.seq2head(bq, B, S, Hq, d, N, K, order="sbhd"),
           oracle.seq2head(bk, B, S, Hkv, d, N, K, order="sbhd"),
           oracle.seq2head(bv, B, S, Hkv, d, N, K, order="sbhd"),
           oracle.head2seq(bo, B, S, Hq, d, N, K, order="sbhd"))
    ins = [t.to(DEV) for t in (q, k, v, o)]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dtype, order="sbhd") as L:
        ws = torch.empty(max(1, L.info["workspace_bytes"]), dtype=torch.uint8, device=DEV)
        for algo in ALGOS:
            outs = [torch.empty_like(t) for t in ins]
            basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                               outs[0], outs[1], outs[2], ws)
            basp.basp_head2seq(L.handle, algo, ins[3], None, None, outs[3],
                               None, None, ws)
            torch.cuda.synchronize()
            for name, g, e in zip("qkvo", outs, exp):
                assert_bits_equal(g, e, "sbhd %s %s %s %s" % (shape, dtype, algo, name))


SF_SMALL = [
    (2, 64, 4, 4, 16, 4, 4),      # Ulysses, Bg = 2
    (4, 36, 12, 6, 8, 6, 3),      # G = 2, Bg = 2
    (6, 30, 6, 6, 40, 6, 3),      # Bg = 3
    (2, 2056, 24, 8, 128, 8, 8),  # Ulysses, ragged tiles
    (2, 520, 12, 4, 72, 4, 4),    # vpr = 27
    (4, 64, 8, 8, 16, 8, 2),      # BASP, Bg = 1
]


@pytest.mark.parametrize("shape", SF_SMALL)
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_seq_first_small(shape, dtype):
    _run_sf(shape, dtype)


@pytest.mark.parametrize("name", ["llama3.2-1b_B2_S8192", "llama3.2-3b_B2_S32768",
                                  "llama3.2-1b_S8192_B4"])
@pytest.mark.parametrize("layout", ["basp", "ulysses"])
def test_seq_first_full_size(name, layout):
    w = WORKLOADS[name]
    _run_sf((w.B, w.S, w.Hq, w.Hkv, w.d, w.N, w.K(layout)), "bf16", kind="normal")
    torch.cuda.empty_cache()


def _run_packed(shape, dtype, order, offset=0, seed=53, kind="bits"):
    B, S, Hq, Hkv, d, N, K = shape
    n_packed = B * S * (Hq + 2 * Hkv) * d
    gen = synth_inputs.normal if kind == "normal" else synth_inputs.random_bits
    packed = gen(n_packed, seed, dtype)
    hq, hk, hv = (gen(B * S * H * d, seed + i + 1, dtype)
                  for i, H in enumerate((Hq, Hkv, Hkv)))
    exp = oracle.seq2head_qkv(synth_inputs.bits(packed), B, S, Hq, Hkv, d, N, K, order)
    exp_back = oracle.head2seq_qkv(synth_inputs.bits(hq), synth_inputs.bits(hk),
                                   synth_inputs.bits(hv), B, S, Hq, Hkv, d, N, K, order)
    tdt = synth_inputs.DTYPES[dtype]
    esz = torch.tensor([], dtype=tdt).element_size()
    pad = 4096

    def padded(n, fill):
        raw = torch.full((pad + offset + n * esz + pad,), fill, dtype=torch.uint8, device=DEV)
        return raw[pad + offset:pad + offset + n * esz].view(tdt), raw

    pk, _ = padded(n_packed, 0x11)
    pk.copy_(packed.to(DEV))
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dtype, order=order) as L:
        outs = [padded(B * S * H * d, 0xEE) for H in (Hq, Hkv, Hkv)]
        basp.basp_seq2head_qkv(L.handle, pk, *[o for o, _ in outs])
        ins = [padded(t.numel(), 0x22)[0] for t in (hq, hk, hv)]
        for x, t in zip(ins, (hq, hk, hv)):
            x.copy_(t.to(DEV))
        back, back_raw = padded(n_packed, 0xEE)
        basp.basp_head2seq_qkv(L.handle, *ins, back)
        torch.cuda.synchronize()
    for name, (g, raw), e in zip("qkv", outs, exp):
        assert_bits_equal(g, e, "packed %s %s %s off %d %s" % (shape, dtype, order, offset, name))
        assert bool((raw[:pad + offset] == 0xEE).all()) and bool((raw[-pad:] == 0xEE).all())
    assert_bits_equal(back, exp_back, "packed back %s %s %s" % (shape, dtype, order))
    assert bool((back_raw[:pad + offset] == 0xEE).all()) and bool((back_raw[-pad:] == 0xEE).all())


PACKED_SMALL = [
    (2, 64, 4, 4, 16, 4, 2),
    (2, 64, 32, 8, 16, 8, 4),
    (2, 48, 24, 8, 8, 8, 8),
    (4, 36, 12, 6, 8, 6, 3),
    (2, 520, 12, 4, 72, 4, 4),
]


@pytest.mark.parametrize("shape", PACKED_SMALL)
@pytest.mark.parametrize("order", ["bshd", "sbhd"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_packed_qkv_small(shape, order, dtype):
    _run_packed(shape, dtype, order)


@pytest.mark.parametrize("offset", [2, 4, 8])
def test_packed_qkv_narrow_alignment(offset):
    _run_packed((2, 64, 32, 8, 16, 8, 4), "bf16", "bshd", offset=offset)


@pytest.mark.parametrize("name", ["llama3.2-1b_B2_S8192", "qwen1.5-1.8b_B2_S16384",
                                  "llama3.2-3b_B2_S16384", "llama3.2-1b_S8192_B8"])
@pytest.mark.parametrize("layout", ["basp", "ulysses"])
def test_packed_qkv_full_size(name, layout):
    w = WORKLOADS[name]
    _run_packed((w.B, w.S, w.Hq, w.Hkv, w.d, w.N, w.K(layout)), "bf16", "bshd",
                kind="normal")
    torch.cuda.empty_cache()
