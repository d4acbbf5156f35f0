"""The autograd wrappers: forward values and gradients both match the oracle
(the gradient of seq2head is head2seq of the upstream gradient, and back)."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs
import sequence_re_layout_gb300 as basp
from sequence_re_layout_gb300.autograd import head2seq, seq2head

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _bits(t):
    return synth_inputs.bits(t.detach().cpu())


@pytest.mark.parametrize("K", [4, 8])
def test_seq2head_and_head2seq_gradients(K):
    B, S, Hq, Hkv, d, N = 2, 512, 32, 8, 64, 8
    nq, nkv = B * S * Hq * d, B * S * Hkv * d
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        q, k, v, o = (synth_inputs.normal(n, s, "bf16").to(DEV).requires_grad_()
                      for n, s in ((nq, 1), (nkv, 2), (nkv, 3), (nq, 4)))
        qh, kh, vh = seq2head(L, q, k, v)
        for x, y, H in ((q, qh, Hq), (k, kh, Hkv), (v, vh, Hkv)):
            assert np.array_equal(_bits(y), oracle.seq2head(_bits(x), B, S, H, d, N, K))
        gq, gk, gv = (synth_inputs.normal(n, s, "bf16").to(DEV)
                      for n, s in ((nq, 5), (nkv, 6), (nkv, 7)))
        torch.autograd.backward([qh, kh, vh], [gq, gk, gv])
        for x, g, H in ((q, gq, Hq), (k, gk, Hkv), (v, gv, Hkv)):
            assert np.array_equal(_bits(x.grad), oracle.head2seq(_bits(g), B, S, H, d, N, K))

        os_ = head2seq(L, o)
        assert np.array_equal(_bits(os_), oracle.head2seq(_bits(o), B, S, Hq, d, N, K))
        go = synth_inputs.normal(nq, 8, "bf16").to(DEV)
        os_.backward(go)
        assert np.array_equal(_bits(o.grad), oracle.seq2head(_bits(go), B, S, Hq, d, N, K))


def test_only_q_and_unused_outputs():
    """Q alone, and a loss that uses only some outputs (missing gradients)."""
    B, S, Hq, Hkv, d, N, K = 2, 256, 16, 8, 32, 8, 4
    nq, nkv = B * S * Hq * d, B * S * Hkv * d
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        q = synth_inputs.normal(nq, 11, "bf16").to(DEV).requires_grad_()
        qh, kh, vh = seq2head(L, q)
        assert kh is None and vh is None
        (qh.float() * 2).sum().backward()
        assert torch.equal(q.grad, torch.full_like(q, 2.0))
        k = synth_inputs.normal(nkv, 12, "bf16").to(DEV).requires_grad_()
        v = synth_inputs.normal(nkv, 13, "bf16").to(DEV).requires_grad_()
        q.grad = None
        qh, kh, vh = seq2head(L, q, k, v)
        kh.float().sum().backward()
        assert q.grad is None or torch.count_nonzero(q.grad) == 0
        assert torch.equal(k.grad, torch.ones_like(k))


@pytest.mark.parametrize("K", [4, 8])
def test_packed_qkv_forward_and_gradient(K):
    """seq2head_qkv: the head-sharded Q, K, V of a packed projection output,
    and the packed gradient (head2seq of each gradient, packed) -- with all
    three outputs used, and with only Q used (K and V gradients are zero)."""
    from sequence_re_layout_gb300.autograd import seq2head_qkv
    B, S, Hq, Hkv, d, N = 2, 256, 32, 8, 64, 8
    nq, nkv = B * S * Hq * d, B * S * Hkv * d
    with basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16") as L:
        qkv = synth_inputs.normal(nq + 2 * nkv, 21, "bf16").to(DEV).requires_grad_()
        qh, kh, vh = seq2head_qkv(L, qkv)
        want = oracle.seq2head_qkv(_bits(qkv), B, S, Hq, Hkv, d, N, K)
        for got, e in zip((qh, kh, vh), want):
            assert np.array_equal(_bits(got), e)
        gq, gk, gv = (synth_inputs.normal(n, s, "bf16").to(DEV)
                      for n, s in ((nq, 22), (nkv, 23), (nkv, 24)))
        torch.autograd.backward([qh, kh, vh], [gq, gk, gv])
        assert np.array_equal(_bits(qkv.grad), oracle.head2seq_qkv(
            _bits(gq), _bits(gk), _bits(gv), B, S, Hq, Hkv, d, N, K))

        qkv.grad = None
        qh, kh, vh = seq2head_qkv(L, qkv)
        qh.backward(gq)
        zeros = np.zeros(nkv, dtype=_bits(gq).dtype)
        assert np.array_equal(_bits(qkv.grad), oracle.head2seq_qkv(
            _bits(gq), zeros, zeros, B, S, Hq, Hkv, d, N, K))
