"""Pins for the CPU oracle: what the BASP sources and the mathematics fix.

The review and abstract print no worked values for the re-layout, so the oracle is pinned by
(1) values worked by hand from the definitions, (2) library routines that reach
the same permutation another way (torch ``permute`` of the logical tensor), (3)
brute force over every tiny shape, and (4) the invariants the review states:
per-rank memory B*S/N tokens, K-1 instead of N-1 peers, groups that never talk
to each other, and B = 1 reducing to Ulysses ("BASP: Communication-Efficient
Batch-Aware Sequence Parallelism for LLM Training", evolve.pub review, sections
"Summary", "Key claims under review" and "Strengths").
"""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
import synth_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.txt")


def _read_golden():
    cases = []
    cur = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] in ("case", "qkvcase"):
                kv = dict(t.split("=") for t in tok[2:])
                cur = {"kind": tok[0], "name": tok[1], "order": kv.pop("order", "bshd"),
                       **{k: int(v) for k, v in kv.items()}}
                cases.append(cur)
            else:
                cur[tok[0]] = np.array([float(t) for t in tok[1:]], np.float32)
    return cases


GOLDEN_CASES = _read_golden()


@pytest.mark.parametrize("case", [c for c in GOLDEN_CASES if c["kind"] == "case"],
                         ids=lambda c: c["name"])
def test_hand_worked_values(case):
    c = case
    args = (c["B"], c["S"], c["H"], c["d"], c["N"], c["K"])
    o = c["order"]
    np.testing.assert_array_equal(oracle.seq2head(c["seq"], *args, order=o), c["head"])
    np.testing.assert_array_equal(oracle.head2seq(c["head"], *args, order=o), c["seq"])
    np.testing.assert_array_equal(oracle.seq2head_by_slices(c["seq"], *args, order=o), c["head"])
    np.testing.assert_array_equal(oracle.head2seq_by_slices(c["head"], *args, order=o), c["seq"])


@pytest.mark.parametrize("case", [c for c in GOLDEN_CASES if c["kind"] == "qkvcase"],
                         ids=lambda c: c["name"])
def test_hand_worked_packed_qkv(case):
    c = case
    args = (c["B"], c["S"], c["Hq"], c["Hkv"], c["d"], c["N"], c["K"])
    q, k, v = oracle.seq2head_qkv(c["packed"], *args)
    np.testing.assert_array_equal(q, c["q"])
    np.testing.assert_array_equal(k, c["k"])
    np.testing.assert_array_equal(v, c["v"])
    np.testing.assert_array_equal(oracle.head2seq_qkv(c["q"], c["k"], c["v"], *args),
                                  c["packed"])


def tiny_shapes():
    """Every tiny shape that meets the divisibility rules: B <= 4, N <= 8,
    S <= 16, H <= 8, d <= 4 (d in {1, 3, 4} to keep the count small)."""
    out = []
    for N in range(1, 9):
        for K in [k for k in range(1, N + 1) if N % k == 0]:
            G = N // K
            for B in [b for b in range(0, 5) if b % G == 0]:
                for S in sorted({0, K, 2 * K, 16 - 16 % K}):
                    if S > 16:
                        continue
                    for H in [h for h in (K, 2 * K) if h <= 8]:
                        for d in (1, 3):
                            out.append((B, S, H, d, N, K))
    return out


def test_brute_force_two_forms_agree():
    """P1: the element loop, the slicing of the logical tensor and the
    destination-driven single-element map agree on every tiny shape."""
    shapes = tiny_shapes()
    assert len(shapes) > 300
    for (B, S, H, d, N, K) in shapes:
        n = B * S * H * d
        x = np.arange(n, dtype=np.int32) * 7 + 3
        y = oracle.seq2head(x, B, S, H, d, N, K)
        np.testing.assert_array_equal(y, oracle.seq2head_by_slices(x, B, S, H, d, N, K))
        z = oracle.head2seq(x, B, S, H, d, N, K)
        np.testing.assert_array_equal(z, oracle.head2seq_by_slices(x, B, S, H, d, N, K))
        if n:
            src = [oracle.head_to_seq_index(B, S, H, d, N, K, o) for o in range(n)]
            np.testing.assert_array_equal(y, x[np.array(src)])


def _seq_sharded_from_X(X, N, K):
    """Library form of the seq-sharded layout: X[B,S,H,d] viewed as
    [G, Bg, K, S/K, H, d], ranks (g, j) made the outer axes."""
    B, S, H, d = X.shape
    G = N // K
    return X.reshape(G, B // G, K, S // K, H, d).permute(0, 2, 1, 3, 4, 5).reshape(-1)


def _head_sharded_from_X(X, N, K):
    """Library form of the head-sharded layout: X viewed as
    [G, Bg, S, K, H/K, d], ranks (g, j') made the outer axes."""
    B, S, H, d = X.shape
    G = N // K
    return X.reshape(G, B // G, S, K, H // K, d).permute(0, 3, 1, 2, 4, 5).reshape(-1)


LIB_SHAPES = [
    # (B, S, H, d, N, K)
    (2, 64, 4, 16, 4, 2),     # tiny config, BASP
    (2, 64, 4, 16, 4, 4),     # tiny config, Ulysses
    (2, 32, 32, 8, 8, 4),     # 1B-like heads, BASP
    (2, 32, 8, 8, 8, 8),      # 1B KV heads, Ulysses
    (2, 24, 24, 4, 8, 4),     # 3B-like 24 heads, H/K = 6
    (8, 16, 8, 4, 8, 1),      # B = N = 8: K = 1
    (4, 12, 6, 2, 6, 3),      # K = 3, non-power-of-two
    (6, 12, 6, 2, 6, 3),      # G = 2, Bg = 3
]


@pytest.mark.parametrize("shape", LIB_SHAPES)
def test_library_permute_form(shape):
    """P6: the oracle equals torch's permute of the logical tensor, both ways."""
    B, S, H, d, N, K = shape
    X = synth_inputs.random_bits(B * S * H * d, seed=11).view(B, S, H, d)
    xs = _seq_sharded_from_X(X, N, K)
    xh = _head_sharded_from_X(X, N, K)
    bs, bh = synth_inputs.bits(xs), synth_inputs.bits(xh)
    np.testing.assert_array_equal(oracle.seq2head(bs, *_args(shape)), bh)
    np.testing.assert_array_equal(oracle.head2seq(bh, *_args(shape)), bs)


def _args(shape):
    B, S, H, d, N, K = shape
    return (B, S, H, d, N, K)


@pytest.mark.parametrize("shape", LIB_SHAPES)
def test_index_values_decode_to_their_place(shape):
    """P2: with X[b,s,h,e] = its own flat index, every output value names the
    element that must sit there: same sequence of the rank's group, same token,
    head j'*H/K + hl, same e.  The output is a permutation of 0..T-1."""
    B, S, H, d, N, K = shape
    T = B * S * H * d
    X = torch.arange(T, dtype=torch.int64).view(B, S, H, d)
    xs = _seq_sharded_from_X(X, N, K).numpy()
    y = oracle.seq2head(xs, B, S, H, d, N, K)
    assert np.array_equal(np.sort(y), np.arange(T))           # bijection
    G, Bg, Hk = N // K, B // (N // K), H // K
    r, bl, s, hl, e = np.unravel_index(np.arange(T), (N, Bg, S, Hk, d))
    b_v, s_v, h_v, e_v = np.unravel_index(y, (B, S, H, d))
    np.testing.assert_array_equal(b_v, (r // K) * Bg + bl)
    np.testing.assert_array_equal(s_v, s)
    np.testing.assert_array_equal(h_v, (r % K) * Hk + hl)
    np.testing.assert_array_equal(e_v, e)


# The five workload families at a reduced sequence length (the layout rule does
# not depend on S beyond S % K == 0; the full lengths run in the GPU parity
# tests, where the oracle runs at full size).
CONFIG_SHAPES = {
    # name: (B, S, Hq, Hkv, d, N, K_basp)
    "tiny": (2, 64, 4, 4, 16, 4, 2),
    "llama1b": (2, 256, 32, 8, 64, 8, 4),
    "qwen1.8b": (2, 256, 16, 16, 128, 8, 4),
    "llama3b": (2, 256, 24, 8, 128, 8, 4),
    "llama1b_B1": (1, 256, 32, 8, 64, 8, 8),
    "llama1b_B4": (4, 256, 32, 8, 64, 8, 2),
    "llama1b_B8": (8, 256, 32, 8, 64, 8, 1),
}


@pytest.mark.parametrize("name", sorted(CONFIG_SHAPES))
@pytest.mark.parametrize("layout", ["basp", "ulysses"])
def test_round_trip_identity(name, layout):
    """P3: head2seq(seq2head(x)) is x, bit for bit, for Q (Hq) and K/V (Hkv)."""
    B, S, Hq, Hkv, d, N, Kb = CONFIG_SHAPES[name]
    K = Kb if layout == "basp" else N
    for H, seed in ((Hq, 1), (Hkv, 2)):
        x = synth_inputs.bits(synth_inputs.normal(B * S * H * d, seed))
        y = oracle.seq2head(x, B, S, H, d, N, K)
        assert not np.array_equal(y, x) or K == 1 or N == 1
        np.testing.assert_array_equal(oracle.head2seq(y, B, S, H, d, N, K), x)


def test_batch_one_is_ulysses():
    """P4: with B = 1 the BASP rule K = N/B gives K = N, the Ulysses layout
    (review "Strengths": the B = 1 case degenerates to standard Ulysses)."""
    B, S, H, d, N = 1, 64, 16, 8, 8
    K_basp = N // B
    x = synth_inputs.bits(synth_inputs.normal(B * S * H * d, 5))
    np.testing.assert_array_equal(oracle.seq2head(x, B, S, H, d, N, K_basp),
                                  oracle.seq2head(x, B, S, H, d, N, N))


@pytest.mark.parametrize("B", [2, 4, 8])
def test_each_group_is_an_independent_ulysses(B):
    """P4b: BASP with N = K*B is B independent K-way Ulysses exchanges, one per
    sequence (review "Summary": each group owns one sequence and runs its own
    K-way all-to-all)."""
    N, S, H, d = 8, 32, 8, 4
    K = N // B
    x = synth_inputs.bits(synth_inputs.normal(B * S * H * d, 7))
    y = oracle.seq2head(x, B, S, H, d, N, K)
    per_group = S * H * d            # one sequence per group in both layouts
    for g in range(B):
        xg = x[g * per_group:(g + 1) * per_group]
        yg = oracle.seq2head(xg, 1, S, H, d, K, K)
        np.testing.assert_array_equal(y[g * per_group:(g + 1) * per_group], yg)


def test_k_one_is_identity():
    """P5: K = 1 (B = N) keeps every element on its rank and in place."""
    B, S, H, d, N = 8, 32, 8, 4, 8
    x = synth_inputs.bits(synth_inputs.normal(B * S * H * d, 9))
    np.testing.assert_array_equal(oracle.seq2head(x, B, S, H, d, N, 1), x)
    np.testing.assert_array_equal(oracle.head2seq(x, B, S, H, d, N, 1), x)


@pytest.mark.parametrize("name", sorted(CONFIG_SHAPES))
@pytest.mark.parametrize("layout", ["basp", "ulysses"])
def test_memory_peers_and_group_locality(name, layout):
    """P8/P9: per-rank elements = B*S*H*d/N in both layouts; every element
    stays inside its group; each rank sends to exactly K-1 other ranks (N-1 for
    Ulysses), Bg*(S/K)*(H/K)*d elements to each (review "Summary": peers drop
    from N-1 to K-1 while every GPU keeps B*S/N tokens)."""
    B, S, Hq, Hkv, d, N, Kb = CONFIG_SHAPES[name]
    K = Kb if layout == "basp" else N
    S, d = 2 * K, 2                   # the counts below scale; keep it small
    H = Hq
    T = B * S * H * d
    P = T // N
    X = torch.arange(T, dtype=torch.int64).view(B, S, H, d)
    xs = _seq_sharded_from_X(X, N, K).numpy()
    # source position (flat, seq-sharded) of every head-sharded element
    where_src = np.empty(T, np.int64)
    where_src[xs] = np.arange(T)
    y = oracle.seq2head(xs, B, S, H, d, N, K)
    src_rank = where_src[y] // P
    dst_rank = np.arange(T) // P
    assert P * N == T and P == B * S * H * d // N
    assert np.all(src_rank // K == dst_rank // K)           # group locality
    G, Bg = N // K, B // (N // K)
    for r in range(N):
        sent = dst_rank[src_rank == r]
        peers, counts = np.unique(sent[sent != r], return_counts=True)
        assert len(peers) == K - 1
        assert np.all(counts == Bg * (S // K) * (H // K) * d)


def test_bad_shapes_rejected():
    x = np.zeros(2 * 8 * 4 * 2, np.int16)
    with pytest.raises(ValueError):
        oracle.seq2head(x, 2, 8, 4, 2, 4, 3)      # N % K
    with pytest.raises(ValueError):
        oracle.seq2head(x, 2, 8, 4, 2, 8, 2)      # B % (N/K)
    with pytest.raises(ValueError):
        oracle.seq2head(np.zeros(2 * 6 * 4 * 2, np.int16), 2, 6, 4, 2, 4, 4)  # S % K
    with pytest.raises(ValueError):
        oracle.seq2head(np.zeros(2 * 8 * 6 * 2, np.int16), 2, 8, 6, 2, 4, 4)  # H % K
