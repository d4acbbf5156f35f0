"""Pins for the oracle's two variants that the BASP review leaves open: the
sequence-first token order ([S, B, H, d], Megatron-style) and the packed QKV
input (one buffer of Hq + 2*Hkv heads per token row, as a fused QKV projection
writes it).  Each is checked against torch's permute of the logical tensors,
brute force against the slicing form, and the round trip."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs
from test_oracle_pins import LIB_SHAPES, tiny_shapes


def _sf_seq_from_X(X, N, K):
    """Library form of the sequence-first seq-sharded buffer of X[S,B,H,d]:
    X viewed [K, S/K, G, Bg, H, d], ranks (g, j) made the outer axes."""
    S, B, H, d = X.shape
    G = N // K
    return X.reshape(K, S // K, G, B // G, H, d).permute(2, 0, 1, 3, 4, 5).reshape(-1)


def _sf_head_from_X(X, N, K):
    """Library form of the sequence-first head-sharded buffer of X[S,B,H,d]:
    X viewed [S, G, Bg, K, H/K, d], ranks (g, j') made the outer axes."""
    S, B, H, d = X.shape
    G = N // K
    return X.reshape(S, G, B // G, K, H // K, d).permute(1, 3, 0, 2, 4, 5).reshape(-1)


@pytest.mark.parametrize("shape", LIB_SHAPES)
def test_seq_first_library_form(shape):
    B, S, H, d, N, K = shape
    X = synth_inputs.random_bits(B * S * H * d, seed=13).view(S, B, H, d)
    xs = synth_inputs.bits(_sf_seq_from_X(X, N, K))
    xh = synth_inputs.bits(_sf_head_from_X(X, N, K))
    np.testing.assert_array_equal(oracle.seq2head(xs, *shape, order="sbhd"), xh)
    np.testing.assert_array_equal(oracle.head2seq(xh, *shape, order="sbhd"), xs)


def test_seq_first_brute_force():
    """The sequence-first loop equals the sequence-first slicing form on every
    tiny shape, and round-trips."""
    for (B, S, H, d, N, K) in tiny_shapes():
        x = np.arange(B * S * H * d, dtype=np.int32) * 5 + 1
        y = oracle.seq2head(x, B, S, H, d, N, K, order="sbhd")
        np.testing.assert_array_equal(
            y, oracle.seq2head_by_slices(x, B, S, H, d, N, K, order="sbhd"))
        np.testing.assert_array_equal(
            oracle.head2seq(y, B, S, H, d, N, K, order="sbhd"), x)


def test_seq_first_equals_batch_first_when_one_sequence_per_group():
    """With Bg = 1 (every BASP layout) the two orders store the same bytes."""
    B, S, H, d, N, K = 4, 64, 8, 8, 8, 2
    x = synth_inputs.bits(synth_inputs.normal(B * S * H * d, 3))
    np.testing.assert_array_equal(oracle.seq2head(x, B, S, H, d, N, K, order="sbhd"),
                                  oracle.seq2head(x, B, S, H, d, N, K))


@pytest.mark.parametrize("shape", [
    # (B, S, Hq, Hkv, d, N, K)
    (2, 32, 32, 8, 8, 8, 4),
    (2, 32, 32, 8, 8, 8, 8),
    (2, 24, 24, 8, 4, 8, 4),
    (4, 12, 6, 3, 2, 6, 3),
])
@pytest.mark.parametrize("order", ["bshd", "sbhd"])
def test_packed_qkv_library_form(shape, order):
    """Packed QKV: the seq-sharded cut of cat([Xq, Xk, Xv], head axis) goes
    to the head-sharded cuts of Xq, Xk and Xv; and back."""
    B, S, Hq, Hkv, d, N, K = shape
    g = torch.Generator().manual_seed(29)
    mk = lambda H: torch.randint(-2 ** 15, 2 ** 15, (B, S, H, d), generator=g,
                                 dtype=torch.int16)
    Xq, Xk, Xv = mk(Hq), mk(Hkv), mk(Hkv)
    Xp = torch.cat([Xq, Xk, Xv], dim=2)
    if order == "bshd":
        from test_oracle_pins import _seq_sharded_from_X as seq_cut, \
            _head_sharded_from_X as head_cut
        prep = lambda X: X
    else:
        seq_cut, head_cut = _sf_seq_from_X, _sf_head_from_X
        prep = lambda X: X.transpose(0, 1).contiguous()
    packed = seq_cut(prep(Xp), N, K).numpy()
    q, k, v = oracle.seq2head_qkv(packed, B, S, Hq, Hkv, d, N, K, order)
    np.testing.assert_array_equal(q, head_cut(prep(Xq), N, K).numpy())
    np.testing.assert_array_equal(k, head_cut(prep(Xk), N, K).numpy())
    np.testing.assert_array_equal(v, head_cut(prep(Xv), N, K).numpy())
    np.testing.assert_array_equal(
        oracle.head2seq_qkv(q, k, v, B, S, Hq, Hkv, d, N, K, order), packed)
