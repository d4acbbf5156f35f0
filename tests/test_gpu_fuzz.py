"""Seeded fuzz of the CUDA path against the oracle: random small shapes that
meet the divisibility rules (any K dividing N, any group count), dtypes,
token orders, algorithms, packed-QKV entry points and pointer offsets that
select every vector width; and random long launches (150-300 MB of Q, K, V)
that take the 512-thread CTAs.  Every bit is compared."""
import random

import numpy as np
import pytest
import torch

import oracle
import synth_inputs
import sequence_re_layout_gb300 as basp

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _random_case(rng):
    N = rng.choice([1, 2, 3, 4, 6, 8, 12, 16])
    K = rng.choice([k for k in range(1, N + 1) if N % k == 0])
    G = N // K
    B = G * rng.randint(1, 3)
    S = K * rng.randint(1, 40)
    Hkv = K * rng.randint(1, 3)
    Hq = Hkv * rng.choice([1, 2, 3, 4])
    d = rng.choice([1, 2, 3, 8, 16, 24, 64, 80, 128])
    dtype = rng.choice(["bf16", "fp16", "fp32", "fp8"])
    order = rng.choice(["bshd", "sbhd"])
    algo = rng.choice(["fused", "three_pass", "three_pass_elide"])
    esz = {"fp32": 4, "fp8": 1}.get(dtype, 2)
    offset = rng.choice([0, 0, esz, 2 * esz, 8]) // esz * esz
    return (B, S, Hq, Hkv, d, N, K), dtype, order, algo, offset


def _buf(n, dtype, offset):
    t = synth_inputs.DTYPES[dtype]
    esz = torch.tensor([], dtype=t).element_size()
    raw = torch.empty(n * esz + offset + 64, dtype=torch.uint8, device=DEV)
    return raw[offset:offset + n * esz].view(t)


@pytest.mark.parametrize("seed", range(60))
def test_fuzz_against_oracle(seed):
    rng = random.Random(1000 + seed)
    (B, S, Hq, Hkv, d, N, K), dtype, order, algo, off = _random_case(rng)
    shape = (B, S, Hq, Hkv, d, N, K)
    tag = "%s %s %s %s off=%d" % (shape, dtype, order, algo, off)
    n_q, n_kv = B * S * Hq * d, B * S * Hkv * d
    host = [synth_inputs.random_bits(n, seed * 7 + i, dtype)
            for i, n in enumerate((n_q, n_kv, n_kv, n_q))]
    bits = [synth_inputs.bits(t) for t in host]
    exp = [oracle.seq2head(bits[0], B, S, Hq, d, N, K, order),
           oracle.seq2head(bits[1], B, S, Hkv, d, N, K, order),
           oracle.seq2head(bits[2], B, S, Hkv, d, N, K, order),
           oracle.head2seq(bits[3], B, S, Hq, d, N, K, order)]
    ins = []
    for t in host:
        x = _buf(t.numel(), dtype, off)
        x.copy_(t.to(DEV))
        ins.append(x)
    outs = [_buf(t.numel(), dtype, off) for t in host]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dtype, order=order) as L:
        ws = _buf(L.info["workspace_bytes"] // 4 + 1, "fp32", off if off % 4 == 0 else 0)
        basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                           outs[0], outs[1], outs[2], ws)
        basp.basp_head2seq(L.handle, algo, ins[3], None, None, outs[3], None, None, ws)
        # packed QKV forms on the same shape
        packed = synth_inputs.random_bits(B * S * (Hq + 2 * Hkv) * d, seed + 99, dtype)
        pexp = oracle.seq2head_qkv(synth_inputs.bits(packed), B, S, Hq, Hkv, d, N, K, order)
        pin = _buf(packed.numel(), dtype, off)
        pin.copy_(packed.to(DEV))
        pout = [_buf(n, dtype, off) for n in (n_q, n_kv, n_kv)]
        basp.basp_seq2head_qkv(L.handle, pin, *pout)
        pback = _buf(packed.numel(), dtype, off)
        basp.basp_head2seq_qkv(L.handle, *pout, pback)
        torch.cuda.synchronize()
    bt = synth_inputs.BITS[synth_inputs.DTYPES[dtype]]
    for name, g, e in zip("qkvo", outs, exp):
        got = g.view(bt).cpu().numpy()
        assert np.array_equal(got, e), "%s %s" % (tag, name)
    for name, g, e in zip("qkv", pout, pexp):
        assert np.array_equal(g.view(bt).cpu().numpy(), e), "%s packed %s" % (tag, name)
    assert np.array_equal(pback.view(bt).cpu().numpy(), synth_inputs.bits(packed)), \
        "%s packed round trip" % tag


def _random_long_case(rng):
    """A random shape whose seq2head launch is long enough (at least 8 waves
    of 16 KiB tiles) for the 512-thread CTAs on 32 KiB tiles, with 16-byte
    aligned rows so the 16-byte path runs."""
    N = rng.choice([2, 4, 8, 16])
    K = rng.choice([k for k in range(1, N + 1) if N % k == 0])
    G = N // K
    B = G * rng.randint(1, 2)
    Hkv = K * rng.randint(1, 2)
    Hq = Hkv * rng.choice([1, 2, 3])
    dtype = rng.choice(["bf16", "fp32", "fp8"])
    esz = {"fp32": 4, "fp8": 1}.get(dtype, 2)
    d = rng.choice([64, 80, 128, 144]) if esz > 1 else rng.choice([64, 128, 160])
    order = rng.choice(["bshd", "sbhd"])
    algo = rng.choice(["fused", "fused", "three_pass", "three_pass_elide"])
    target = rng.randint(150, 300) << 20            # bytes of Q, K and V
    per_token = B * (Hq + 2 * Hkv) * d * esz
    S = K * -(-target // (per_token * K))
    return (B, S, Hq, Hkv, d, N, K), dtype, order, algo


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_long_launches(seed):
    rng = random.Random(5000 + seed)
    (B, S, Hq, Hkv, d, N, K), dtype, order, algo = _random_long_case(rng)
    tag = "%s %s %s %s" % ((B, S, Hq, Hkv, d, N, K), dtype, order, algo)
    n_q, n_kv = B * S * Hq * d, B * S * Hkv * d
    host = [synth_inputs.random_bits(n, seed * 11 + i, dtype)
            for i, n in enumerate((n_q, n_kv, n_kv, n_q))]
    bits = [synth_inputs.bits(t) for t in host]
    exp = [oracle.seq2head(bits[0], B, S, Hq, d, N, K, order),
           oracle.seq2head(bits[1], B, S, Hkv, d, N, K, order),
           oracle.seq2head(bits[2], B, S, Hkv, d, N, K, order),
           oracle.head2seq(bits[3], B, S, Hq, d, N, K, order)]
    ins = [t.to(DEV) for t in host]
    outs = [torch.empty_like(t) for t in ins]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dtype, order=order) as L:
        ws = torch.empty(max(1, L.info["workspace_bytes"]), dtype=torch.uint8, device=DEV)
        basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                           outs[0], outs[1], outs[2], ws)
        basp.basp_head2seq(L.handle, algo, ins[3], None, None, outs[3], None, None, ws)
        torch.cuda.synchronize()
    bt = synth_inputs.BITS[synth_inputs.DTYPES[dtype]]
    for name, g, e in zip("qkvo", outs, exp):
        assert torch.equal(g.view(bt), torch.from_numpy(e).to(DEV)), "%s %s" % (tag, name)
