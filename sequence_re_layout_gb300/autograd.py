"""PyTorch autograd wrappers over the C ABI, for training loops.

The re-layout is a permutation, so its gradient is the inverse permutation:
the backward of seq2head is head2seq of the gradients, and the backward of
head2seq is seq2head.  Both directions run in the library's kernels; this
module only allocates the outputs with torch and routes the gradients.

    L = basp.Layout(B, S, Hq, Hkv, d, N, K, "bf16")
    q_h, k_h, v_h = seq2head(L, q, k, v)     # before attention
    o_s = head2seq(L, o_h)                   # after attention

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
