"""PyTorch autograd wrappers over the C ABI, for training loops.

The re-layout is a permutation, so its gradient is the inverse permutation:
the backward of seq2head is head2seq of the gradients, and the backward of
head2seq is seq2head.  Both directions run in the library's kernels; this
module only allocates the outputs with torch and routes the gradients.

    L = basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16")
    q_h, k_h, v_h = seq2head(L, q, k, v)     # before attention
    o_s = head2seq(L, o_h)                   # after attention
    q_h, k_h, v_h = seq2head_qkv(L, qkv)     # from a fused QKV projection

Inputs are virtual-rank buffers (flat, or any contiguous shape with the right
number of elements); outputs are flat tensors of the same dtype and device.
"""
from __future__ import annotations

import torch

from . import binding


def _stream():
    return torch.cuda.current_stream()


def _contig(t):
    return None if t is None else t.contiguous()


class _Seq2Head(torch.autograd.Function):
    @staticmethod
    def forward(ctx, layout, q, k, v):
        ctx.layout = layout
        ins = [_contig(t) for t in (q, k, v)]
        outs = [None if t is None else torch.empty_like(t).view(-1) for t in ins]
        binding.basp_seq2head(layout.handle, "fused", *ins, *outs, stream=_stream())
        return tuple(outs)

    @staticmethod
    def backward(ctx, dq, dk, dv):
        grads = [_contig(g) for g in (dq, dk, dv)]
        outs = [None if g is None else torch.empty_like(g) for g in grads]
        if any(g is not None for g in grads):
            binding.basp_head2seq(ctx.layout.handle, "fused", *grads, *outs,
                                  stream=_stream())
        return (None, *outs)


class _Head2Seq(torch.autograd.Function):
    @staticmethod
    def forward(ctx, layout, o):
        ctx.layout = layout
        o = o.contiguous()
        out = torch.empty_like(o).view(-1)
        binding.basp_head2seq(layout.handle, "fused", o, None, None, out, None, None,
                              stream=_stream())
        return out

    @staticmethod
    def backward(ctx, do):
        do = do.contiguous()
        out = torch.empty_like(do)
        binding.basp_seq2head(ctx.layout.handle, "fused", do, None, None, out, None,
                              None, stream=_stream())
        return None, out


def seq2head(layout, q, k=None, v=None):
    """seq-sharded Q (Hq heads) and optional K, V (Hkv heads) -> head-sharded,
    differentiable.  Returns a tuple (q_h, k_h, v_h) with None where an input
    was None."""
    return _Seq2Head.apply(layout, q, k, v)


def head2seq(layout, o):
    """head-sharded attention output O (Hq heads) -> seq-sharded,
    differentiable."""
    return _Head2Seq.apply(layout, o)


class _Seq2HeadQKV(torch.autograd.Function):
    @staticmethod
    def forward(ctx, layout, qkv):
        ctx.layout = layout
        qkv = qkv.contiguous()
        ctx.packed_shape = qkv.shape
        esz = qkv.element_size()
        i = layout.info
        outs = [torch.empty(n // esz, dtype=qkv.dtype, device=qkv.device)
                for n in (i["bytes_q"], i["bytes_kv"], i["bytes_kv"])]
        binding.basp_seq2head_qkv(layout.handle, qkv, *outs, stream=_stream())
        return tuple(outs)

    @staticmethod
    def backward(ctx, dq, dk, dv):
        i = ctx.layout.info
        ref = next(g for g in (dq, dk, dv) if g is not None)
        esz = ref.element_size()
        # the packed gradient has every head range: a missing one is zero
        grads = [torch.zeros(n // esz, dtype=ref.dtype, device=ref.device) if g is None
                 else g.contiguous()
                 for g, n in zip((dq, dk, dv), (i["bytes_q"], i["bytes_kv"], i["bytes_kv"]))]
        out = torch.empty(ctx.packed_shape, dtype=ref.dtype, device=ref.device)
        binding.basp_head2seq_qkv(ctx.layout.handle, *grads, out, stream=_stream())
        return None, out


def seq2head_qkv(layout, qkv):
    """seq-sharded packed QKV (each token row holds the Hq query heads, then
    the Hkv key heads, then the Hkv value heads: a fused QKV projection's
    output) -> head-sharded Q, K, V, differentiable.  The backward packs the
    three gradients into one seq-sharded gradient of the packed input."""
    return _Seq2HeadQKV.apply(layout, qkv)
