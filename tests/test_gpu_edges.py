"""GPU edge cases: empty shapes, narrower-than-16-byte alignment, guard bands
around every output, buffers above 2^31 elements, subsets of Q/K/V, streams,
and the host-buffer entry points."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs
import sequence_re_layout_gb300 as basp
from parity import (assert_bits_equal, device_outputs, make_inputs,
                    oracle_outputs)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ALGOS = ("fused", "three_pass", "three_pass_elide")


@pytest.mark.parametrize("shape", [
    (2, 0, 8, 8, 16, 4, 2),     # S = 0
    (0, 64, 8, 8, 16, 4, 4),    # B = 0 (Ulysses)
])
@pytest.mark.parametrize("algo", ALGOS)
def test_empty_shapes_launch_nothing(shape, algo):
    B, S, Hq, Hkv, d, N, K = shape
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        assert L.info["bytes_q"] == 0
        x = torch.empty(8, dtype=torch.bfloat16, device=DEV)
        y = torch.empty(8, dtype=torch.bfloat16, device=DEV)
        basp.basp_seq2head(L.handle, algo, x, None, None, y, None, None, None, 0)
        basp.basp_head2seq(L.handle, algo, x, None, None, y, None, None, None, 0)
        torch.cuda.synchronize()


def _padded(n, dtype, offset_bytes, fill_bits):
    """A view of n elements starting offset_bytes into a larger buffer whose
    other bytes hold a sentinel; returns (view, backing bytes)."""
    esz = torch.tensor([], dtype=dtype).element_size()
    pad = 4096
    raw = torch.full((pad + offset_bytes + n * esz + pad,), fill_bits,
                     dtype=torch.uint8, device=DEV)
    start = pad + offset_bytes
    view = raw[start:start + n * esz].view(dtype)
    return view, raw, start, start + n * esz


@pytest.mark.parametrize("offset", [0, 2, 4, 8, 256])
@pytest.mark.parametrize("algo", ALGOS)
def test_alignment_fallbacks_and_guard_bands(offset, algo):
    """Pointers 2/4/8 bytes past a 16-byte boundary take the narrower vector
    kernels; every byte outside the outputs and the workspace keeps its
    sentinel."""
    B, S, Hq, Hkv, d, N, K = 2, 96, 12, 4, 40, 4, 2
    dtype = "bf16"
    tdt = synth_inputs.DTYPES[dtype]
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, dtype, 5, kind="bits")
    exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
    ins, outs, raws = [], [], []
    for t in (q, k, v, o):
        xi, _, _, _ = _padded(t.numel(), tdt, offset, 0x5A)
        xi.copy_(t.to(DEV))
        xo, raw, a, b = _padded(t.numel(), tdt, offset, 0xA5)
        ins.append(xi)
        outs.append(xo)
        raws.append((raw, a, b))
    with basp.Layout(B, S, Hq, Hkv, d, N, K, dtype) as L:
        ws = wraw = None
        if algo != "fused":
            ws, wraw, wa, wb = _padded(L.info["workspace_bytes"], torch.uint8,
                                       offset, 0x3C)
        basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                           outs[0], outs[1], outs[2], ws)
        basp.basp_head2seq(L.handle, algo, ins[3], None, None, outs[3], None,
                           None, ws)
        torch.cuda.synchronize()
    for name, g, e in zip("qkvo", outs, exp):
        assert_bits_equal(g, e, "offset %d %s %s" % (offset, algo, name))
    for raw, a, b in raws:
        assert bool((raw[:a] == 0xA5).all()) and bool((raw[b:] == 0xA5).all())
    if wraw is not None:
        assert bool((wraw[:wa] == 0x3C).all()) and bool((wraw[wb:] == 0x3C).all())


@pytest.mark.parametrize("which", ["q", "kv", "k"])
def test_subsets_of_tensors(which):
    B, S, Hq, Hkv, d, N, K = 2, 128, 16, 8, 32, 8, 4
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 17, kind="bits")
    exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    outs = [torch.zeros_like(t) for t in (qd, kd, vd)]
    use = {"q": (1, 0, 0), "kv": (0, 1, 1), "k": (0, 1, 0)}[which]
    args = [t if u else None for t, u in zip((qd, kd, vd), use)]
    oargs = [t if u else None for t, u in zip(outs, use)]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        for algo in ALGOS:
            ws = torch.empty(L.info["workspace_bytes"], dtype=torch.uint8, device=DEV)
            for t in outs:
                t.zero_()
            basp.basp_seq2head(L.handle, algo, *args, *oargs, ws)
            torch.cuda.synchronize()
            for u, g, e, nm in zip(use, outs, exp[:3], "qkv"):
                if u:
                    assert_bits_equal(g, e, "%s %s %s" % (which, algo, nm))
                else:
                    assert int(g.view(torch.int16).abs().sum()) == 0


def test_side_stream():
    B, S, Hq, Hkv, d, N, K = 2, 1024, 32, 8, 64, 8, 4
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 23)
    exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
    s = torch.cuda.Stream()
    for algo in ALGOS:
        got = device_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K, "bf16", algo,
                             stream=s)
        for name, g, e in zip("qkvo", got, exp):
            assert_bits_equal(g, e, "side stream %s %s" % (algo, name))


@pytest.mark.parametrize("order", ["bshd", "sbhd"])
@pytest.mark.parametrize("algo", ALGOS)
def test_host_buffer_entry_points(algo, order):
    """basp_seq2head_host / basp_head2seq_host: pinned host in, pinned host
    out, device staging owned by the caller."""
    B, S, Hq, Hkv, d, N, K = 2, 2048, 32, 8, 64, 8, 8
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 31)
    bq, bk, bv, bo = (synth_inputs.bits(t) for t in (q, k, v, o))
    exp = (oracle.seq2head(bq, B, S, Hq, d, N, K, order=order),
           oracle.seq2head(bk, B, S, Hkv, d, N, K, order=order),
           oracle.seq2head(bv, B, S, Hkv, d, N, K, order=order),
           oracle.head2seq(bo, B, S, Hq, d, N, K, order=order))
    hin = [t.pin_memory() for t in (q, k, v, o)]
    hout = [torch.empty_like(t).pin_memory() for t in hin]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16", order=order) as L:
        staging = torch.empty(L.info["staging_bytes"], dtype=torch.uint8, device=DEV)
        ws = torch.empty(L.info["workspace_bytes"], dtype=torch.uint8, device=DEV)
        st = torch.cuda.current_stream()
        basp.basp_seq2head_host(L.handle, algo, hin[0], hin[1], hin[2],
                                hout[0], hout[1], hout[2], staging,
                                workspace=ws, stream=st)
        basp.basp_head2seq_host(L.handle, algo, hin[3], None, None, hout[3],
                                None, None, staging, workspace=ws, stream=st)
        st.synchronize()
    for name, g, e in zip("qkvo", hout, exp):
        np.testing.assert_array_equal(synth_inputs.bits(g), e, err_msg=name)


@pytest.mark.parametrize("algo", ALGOS)
def test_above_2_to_31_elements_sampled(algo):
    """A Q buffer of 2^31 bf16 elements (4 GiB; byte offsets past 2^32):
    round trip restores every bit, and 1<<14 sampled output elements match
    the oracle's single-element map."""
    B, S, H, d, N, K = 2, 262144, 32, 128, 8, 4
    n = B * S * H * d
    assert n == 1 << 31
    x = synth_inputs.random_bits_device(n, 77, "bf16", DEV)
    y = torch.empty_like(x)
    with basp.Layout(B, S, H, 8, d, N, K, "bf16") as L:
        ws = None
        if algo != "fused":
            ws = torch.empty(2 * L.info["bytes_q"] + 512, dtype=torch.uint8, device=DEV)
        basp.basp_seq2head(L.handle, algo, x, None, None, y, None, None, ws)
        torch.cuda.synchronize()
        g = torch.Generator().manual_seed(5)
        idx = torch.randint(0, n, (1 << 14,), generator=g)
        src = torch.tensor([oracle.head_to_seq_index(B, S, H, d, N, K, int(i))
                            for i in idx])
        got = y.view(torch.int16)[idx.to(DEV)].cpu()
        want = x.view(torch.int16)[src.to(DEV)].cpu()
        assert torch.equal(got, want)
        z = torch.empty_like(x)
        basp.basp_head2seq(L.handle, algo, y, None, None, z, None, None, ws)
        torch.cuda.synchronize()
        assert torch.equal(z.view(torch.int16), x.view(torch.int16))
    del x, y, z, ws
    torch.cuda.empty_cache()


@pytest.mark.parametrize("algo", ALGOS)
def test_pinned_host_buffers_direct(algo):
    """basp_seq2head / basp_head2seq on page-locked host buffers: the kernels
    read and write host memory in place (same pointer on the device under
    unified addressing)."""
    B, S, Hq, Hkv, d, N, K = 2, 2048, 32, 8, 64, 8, 4
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 37, kind="bits")
    exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
    hin = [t.pin_memory() for t in (q, k, v, o)]
    hout = [torch.empty_like(t).pin_memory() for t in hin]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        ws = torch.empty(L.info["workspace_bytes"], dtype=torch.uint8, device=DEV)
        basp.basp_seq2head(L.handle, algo, hin[0], hin[1], hin[2],
                           hout[0], hout[1], hout[2], ws)
        basp.basp_head2seq(L.handle, algo, hin[3], None, None, hout[3], None, None, ws)
        torch.cuda.synchronize()
    for name, g, e in zip("qkvo", hout, exp):
        np.testing.assert_array_equal(synth_inputs.bits(g), e, err_msg=name)


@pytest.mark.parametrize("algo", ALGOS)
def test_cuda_graph_capture_and_replay(algo):
    """The entry points allocate nothing and never synchronise, so a step
    (seq2head Q,K,V + head2seq O) can be captured into a CUDA graph and
    replayed; the programmatic launches become graph edges.  Replays on new
    input contents give the oracle's bits."""
    B, S, Hq, Hkv, d, N, K = 2, 1024, 32, 8, 64, 8, 4
    shapes = (B * S * Hq * d, B * S * Hkv * d, B * S * Hkv * d, B * S * Hq * d)
    ins = [torch.empty(n, dtype=torch.bfloat16, device=DEV) for n in shapes]
    outs = [torch.empty_like(t) for t in ins]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        ws = torch.empty(L.info["workspace_bytes"], dtype=torch.uint8, device=DEV)
        s = torch.cuda.Stream()

        def step():
            basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                               outs[0], outs[1], outs[2], ws, stream=s)
            basp.basp_head2seq(L.handle, algo, ins[3], None, None, outs[3],
                               None, None, ws, stream=s)

        with torch.cuda.stream(s):
            step()                                  # first call outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step()
        for seed in (3, 4):
            q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", seed, kind="bits")
            for dst, src in zip(ins, (q, k, v, o)):
                dst.copy_(src.to(DEV))
            torch.cuda.synchronize()
            g.replay()
            torch.cuda.synchronize()
            exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
            for name, got, e in zip("qkvo", outs, exp):
                assert_bits_equal(got, e, "graph %s seed %d %s" % (algo, seed, name))


@pytest.mark.parametrize("algo", ALGOS)
def test_host_entry_points_direct_mode(algo):
    """basp_*_host without staging: page-locked host buffers are re-laid out in
    place by the kernels; a pageable buffer is refused before any launch."""
    B, S, Hq, Hkv, d, N, K = 2, 2048, 32, 8, 64, 8, 4
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 43, kind="bits")
    exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
    hin = [t.pin_memory() for t in (q, k, v, o)]
    hout = [torch.empty_like(t).pin_memory() for t in hin]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        ws = torch.empty(L.info["workspace_bytes"], dtype=torch.uint8, device=DEV)
        st = torch.cuda.current_stream()
        basp.basp_seq2head_host(L.handle, algo, hin[0], hin[1], hin[2],
                                hout[0], hout[1], hout[2], None, 0,
                                workspace=ws, stream=st)
        basp.basp_head2seq_host(L.handle, algo, hin[3], None, None, hout[3],
                                None, None, None, 0, workspace=ws, stream=st)
        st.synchronize()
        pageable = torch.empty_like(q)
        with pytest.raises(basp.BaspError) as e:
            basp.basp_seq2head_host(L.handle, algo, hin[0], None, None, pageable,
                                    None, None, None, 0, workspace=ws, stream=st)
        assert e.value.status == basp.BASP_ERR_WORKSPACE
    for name, g, e in zip("qkvo", hout, exp):
        np.testing.assert_array_equal(synth_inputs.bits(g), e, err_msg=name)


def test_two_streams_at_once():
    """Two layouts (BASP and Ulysses) re-laid out concurrently on two streams,
    each several times back to back: both match the oracle."""
    B, S, Hq, Hkv, d, N = 2, 2048, 32, 8, 64, 8
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 61, kind="bits")
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    layouts = [basp.Layout(B, S, Hq, Hkv, d, N, 4, "bf16"),
               basp.Layout(B, S, Hq, Hkv, d, N, 8, "bf16")]
    ins = [t.to(DEV) for t in (q, k, v, o)]
    outs = [[torch.empty_like(t) for t in ins] for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(5):
        for L, s, out in zip(layouts, streams, outs):
            basp.basp_seq2head(L.handle, "fused", ins[0], ins[1], ins[2],
                               out[0], out[1], out[2], stream=s)
            basp.basp_head2seq(L.handle, "fused", ins[3], None, None, out[3],
                               None, None, stream=s)
    torch.cuda.synchronize()
    for L, out, K in zip(layouts, outs, (4, 8)):
        exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
        for name, g, e in zip("qkvo", out, exp):
            assert_bits_equal(g, e, "stream K=%d %s" % (K, name))
        L.close()


def test_host_threads_share_one_layout():
    """Four host threads, one shared layout handle, each thread on its own
    stream with its own buffers, 10 calls each: every result matches."""
    import threading
    B, S, Hq, Hkv, d, N, K = 2, 1024, 32, 8, 64, 8, 4
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 71, kind="bits")
    exp = oracle_outputs(q, k, v, o, B, S, Hq, Hkv, d, N, K)
    L = basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16")
    ins = [t.to(DEV) for t in (q, k, v, o)]
    results, errors = {}, []

    def work(idx):
        try:
            s = torch.cuda.Stream(device=DEV)
            outs = [torch.empty_like(t) for t in ins]
            algo = ALGOS[idx % len(ALGOS)]
            ws = torch.empty(L.info["workspace_bytes"], dtype=torch.uint8, device=DEV)
            for _ in range(10):
                basp.basp_seq2head(L.handle, algo, ins[0], ins[1], ins[2],
                                   outs[0], outs[1], outs[2], ws, stream=s)
                basp.basp_head2seq(L.handle, algo, ins[3], None, None, outs[3],
                                   None, None, ws, stream=s)
            s.synchronize()
            results[idx] = outs
        except Exception as e:          # collected and reported below
            errors.append(e)

    torch.cuda.synchronize()
    ts = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    L.close()
    assert not errors, errors[:3]
    for idx, outs in results.items():
        for name, g, e in zip("qkvo", outs, exp):
            assert_bits_equal(g, e, "thread %d %s" % (idx, name))


@pytest.mark.parametrize("order", ["bshd", "sbhd"])
@pytest.mark.parametrize("algo", ALGOS)
def test_head2seq_with_all_three_slots(algo, order):
    """head2seq of O, K and V in one call (the backward pass moves dQ, dK, dV
    this way), every algorithm, both token orders."""
    B, S, Hq, Hkv, d, N, K = 4, 256, 32, 8, 64, 8, 4       # G = 2, Bg = 2
    q, k, v, o = make_inputs(B, S, Hq, Hkv, d, "bf16", 83, kind="bits")
    ins = [t.to(DEV) for t in (o, k, v)]
    outs = [torch.empty_like(t) for t in ins]
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16", order=order) as L:
        ws = torch.empty(L.info["workspace_bytes"], dtype=torch.uint8, device=DEV)
        basp.basp_head2seq(L.handle, algo, *ins, *outs, ws)
        torch.cuda.synchronize()
    for name, t, g, H in zip("okv", (o, k, v), outs, (Hq, Hkv, Hkv)):
        e = oracle.head2seq(synth_inputs.bits(t), B, S, H, d, N, K, order=order)
        assert_bits_equal(g, e, "head2seq %s %s %s" % (algo, order, name))
