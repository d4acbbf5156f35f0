"""Random mid-size shapes for the oracle's independent forms (hypothesis).

The brute-force pin covers every tiny shape; this draws larger ones (up to 16
ranks, 96 tokens, 16 heads, 8-wide heads, 1/2/4-byte elements, both token
orders) and checks that the plain element loop, the slicing of the logical
tensor and the all-core form agree byte for byte, and that head2seq undoes
seq2head.
"""
import numpy as np
import pytest

import oracle

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies


@st.composite
def shapes(draw):
    N = draw(st.sampled_from([1, 2, 3, 4, 6, 8, 12, 16]))
    K = draw(st.sampled_from([k for k in range(1, N + 1) if N % k == 0]))
    G = N // K
    B = G * draw(st.integers(1, 3))
    S = K * draw(st.integers(1, max(1, 96 // K)))
    H = K * draw(st.integers(1, max(1, 16 // K)))
    d = draw(st.integers(1, 8))
    dtype = draw(st.sampled_from([np.int8, np.int16, np.int32]))
    order = draw(st.sampled_from(["bshd", "sbhd"]))
    return B, S, H, d, N, K, dtype, order


@hypothesis.settings(max_examples=150, deadline=None)
@hypothesis.given(shapes(), st.integers(0, 2**31 - 1))
def test_forms_agree_on_random_shapes(shape, seed):
    B, S, H, d, N, K, dtype, order = shape
    n = B * S * H * d
    rng = np.random.default_rng(seed)
    info = np.iinfo(dtype)
    x = rng.integers(info.min, info.max, size=n, endpoint=True, dtype=np.int64).astype(dtype)
    y = oracle.seq2head(x, B, S, H, d, N, K, order=order)
    np.testing.assert_array_equal(y, oracle.seq2head_by_slices(x, B, S, H, d, N, K, order=order))
    np.testing.assert_array_equal(y, oracle.seq2head_threads(x, B, S, H, d, N, K, 5, order=order))
    z = oracle.head2seq(x, B, S, H, d, N, K, order=order)
    np.testing.assert_array_equal(z, oracle.head2seq_by_slices(x, B, S, H, d, N, K, order=order))
    np.testing.assert_array_equal(oracle.head2seq(y, B, S, H, d, N, K, order=order), x)
