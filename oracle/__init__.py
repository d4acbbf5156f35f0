"""CPU oracle for the BASP / Ulysses sequence<->head re-layout.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The product
library never imports, links or calls it, and it imports nothing from the
product package.

Three forms of the same definition live here:

* ``seq2head`` / ``head2seq``: the plain element loop in ``basp_oracle.c``
  (source-driven; one ``memcpy`` of ``esz`` bytes per element), reached through
  ctypes.  It is the oracle the parity tests and the CPU baseline use.
* ``seq2head_threads`` / ``head2seq_threads``: the same element loop with its
  source rows split over host threads, for timing on every core.
* ``seq2head_by_slices`` / ``head2seq_by_slices``: the same definition written
  with numpy slicing of the logical tensor ``X[B, S, H, d]``: rebuild ``X``
  from the shards of one layout, cut it into the shards of the other.

What the layouts are (review "BASP: Communication-Efficient Batch-Aware
Sequence Parallelism for LLM Training", evolve.pub, sections "Summary",
"Strengths" and FAQ "What is Batch-Aware Sequence Parallelism (BASP)?"; the
fugumt.com related-papers entry "DeepSpeed Ulysses"):

* N ranks form G = N/K contiguous groups of K ranks; group g owns sequences
  ``g*Bg .. g*Bg+Bg-1`` with Bg = B/G.  BASP is K = N/B (Bg = 1, one sequence
  per group); Ulysses is K = N (one group owning all B sequences).
* seq-sharded: member j of group g holds tokens ``j*S/K .. (j+1)*S/K - 1`` of
  all H heads, stored ``[Bg, S/K, H, d]``.
* head-sharded: member j' holds all S tokens of heads
  ``j'*H/K .. (j'+1)*H/K - 1``, stored ``[Bg, S, H/K, d]``.
* Each rank shard has B*S*H*d/N elements in both layouts; shards lie back to
  back in rank order.

The elements are opaque words: pass any numpy dtype (bf16 travels as uint16).
The result is a bit copy, so tests compare raw bits.

Two variants, neither fixed by the BASP review or abstract (which give no
memory order and no projection layout):

* ``order="sbhd"``: sequence-first shards, the [S, B, H, d] activation order
  of Megatron-style stacks: seq-sharded ``[S/K, Bg, H, d]``, head-sharded
  ``[S, Bg, H/K, d]``.
* packed QKV: the seq-sharded input is one buffer whose every token row holds
  the Hq query heads, then the Hkv key heads, then the Hkv value heads (the
  output of a fused QKV projection).  ``seq2head_qkv`` splits each token row
  into those three head ranges and re-lays each out; ``head2seq_qkv`` is the
  inverse.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "basp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libbasp_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``basp_oracle.c`` with gcc into ``libbasp_oracle.so``."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                        "-o", tmp, _SRC], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_from(path):
    """Load a compiled copy of basp_oracle.c from `path` and declare its entry
    points (the tests use this to compile deliberately broken copies and
    check that the pins reject them)."""
    lib = ctypes.CDLL(path)
    _declare(lib)
    return lib


def _declare(lib):
    i64 = ctypes.c_int64
    for name in ("basp_oracle_seq2head", "basp_oracle_head2seq"):
        fn = getattr(lib, name)
        fn.argtypes = [i64] * 7 + [ctypes.c_void_p, ctypes.c_void_p]
        fn.restype = ctypes.c_int
    for name in ("basp_oracle_seq2head_ordered", "basp_oracle_head2seq_ordered"):
        fn = getattr(lib, name)
        fn.argtypes = [i64] * 7 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        fn.restype = ctypes.c_int
    fn = lib.basp_oracle_head_to_seq_index
    fn.argtypes = [i64] * 7
    fn.restype = i64
    for name in ("basp_oracle_seq2head_threads", "basp_oracle_head2seq_threads"):
        fn = getattr(lib, name, None)
        if fn is not None:
            fn.argtypes = [i64] * 7 + [ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_void_p]
            fn.restype = ctypes.c_int


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        _declare(lib)
        _lib = lib
    return _lib


def groups(N: int, K: int, B: int):
    """Return (G, Bg): number of groups and sequences per group."""
    G = N // K
    return G, B // G


def valid_shape(B, S, H, d, N, K) -> bool:
    """The divisibility rules the layouts need (review FAQ "What are BASP's
    main limitations?": N must be a multiple of the group count's batch split,
    heads must divide evenly across group members)."""
    if min(N, K, H, d) < 1 or B < 0 or S < 0:
        return False
    if N % K or (B % (N // K)) or S % K or H % K:
        return False
    return True


ORDERS = {"bshd": 0, "sbhd": 1}


def _run(fn_name, x, B, S, H, d, N, K, order="bshd"):
    x = np.ascontiguousarray(x)
    n = B * S * H * d
    if x.size != n:
        raise ValueError("input has %d elements, shape needs %d" % (x.size, n))
    out = np.empty_like(x)
    if n == 0:
        return out
    if order == "bshd":
        rc = getattr(_load(), fn_name)(B, S, H, d, N, K, x.itemsize,
                                       x.ctypes.data, out.ctypes.data)
    else:
        rc = getattr(_load(), fn_name + "_ordered")(
            B, S, H, d, N, K, x.itemsize, ORDERS[order], x.ctypes.data,
            out.ctypes.data)
    if rc != 0:
        raise ValueError("shape breaks a divisibility rule")
    return out


def seq2head(x, B, S, H, d, N, K, order="bshd"):
    """seq-sharded buffer (N shards of [Bg, S/K, H, d]) -> head-sharded buffer
    (N shards of [Bg, S, H/K, d]).  Plain C element loop.  ``order="sbhd"``
    takes sequence-first shards ([S/K, Bg, H, d] -> [S, Bg, H/K, d])."""
    return _run("basp_oracle_seq2head", x, B, S, H, d, N, K, order)


def head2seq(x, B, S, H, d, N, K, order="bshd"):
    """Inverse of :func:`seq2head`.  Plain C element loop."""
    return _run("basp_oracle_head2seq", x, B, S, H, d, N, K, order)


def _run_threads(fn_name, x, B, S, H, d, N, K, order, nthreads):
    x = np.ascontiguousarray(x)
    n = B * S * H * d
    if x.size != n:
        raise ValueError("input has %d elements, shape needs %d" % (x.size, n))
    out = np.empty_like(x)
    if n == 0:
        return out
    rc = getattr(_load(), fn_name)(B, S, H, d, N, K, x.itemsize, ORDERS[order],
                                   int(nthreads), x.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise ValueError("shape breaks a divisibility rule (or no threads)")
    return out


def seq2head_threads(x, B, S, H, d, N, K, nthreads, order="bshd"):
    """:func:`seq2head` on ``nthreads`` host threads: the same element loop,
    its source rows split into contiguous spans, one per thread (for timing
    the oracle on every host core; the tests check it against the plain
    loop)."""
    return _run_threads("basp_oracle_seq2head_threads", x, B, S, H, d, N, K,
                        order, nthreads)


def head2seq_threads(x, B, S, H, d, N, K, nthreads, order="bshd"):
    """:func:`head2seq` on ``nthreads`` host threads (see
    :func:`seq2head_threads`)."""
    return _run_threads("basp_oracle_head2seq_threads", x, B, S, H, d, N, K,
                        order, nthreads)


def host_cores() -> int:
    """Cores this process may run on (its CPU affinity set)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def split_packed_qkv(x, Hq, Hkv, d):
    """Cut a packed QKV buffer (token rows of Hq + 2*Hkv heads) into the
    Q, K and V buffers with the same token rows."""
    rows = x.reshape(-1, Hq + 2 * Hkv, d)
    return (np.ascontiguousarray(rows[:, :Hq]).reshape(-1),
            np.ascontiguousarray(rows[:, Hq:Hq + Hkv]).reshape(-1),
            np.ascontiguousarray(rows[:, Hq + Hkv:]).reshape(-1))


def join_packed_qkv(q, k, v, Hq, Hkv, d):
    """Inverse of :func:`split_packed_qkv`."""
    return np.concatenate([q.reshape(-1, Hq, d), k.reshape(-1, Hkv, d),
                           v.reshape(-1, Hkv, d)], axis=1).reshape(-1)


def seq2head_qkv(x, B, S, Hq, Hkv, d, N, K, order="bshd"):
    """Packed seq-sharded QKV -> head-sharded Q, K, V (three buffers)."""
    q, k, v = split_packed_qkv(x, Hq, Hkv, d)
    return (seq2head(q, B, S, Hq, d, N, K, order),
            seq2head(k, B, S, Hkv, d, N, K, order),
            seq2head(v, B, S, Hkv, d, N, K, order))


def head2seq_qkv(q, k, v, B, S, Hq, Hkv, d, N, K, order="bshd"):
    """Head-sharded Q, K, V -> one packed seq-sharded buffer."""
    return join_packed_qkv(head2seq(q, B, S, Hq, d, N, K, order),
                           head2seq(k, B, S, Hkv, d, N, K, order),
                           head2seq(v, B, S, Hkv, d, N, K, order), Hq, Hkv, d)


def head_to_seq_index(B, S, H, d, N, K, o):
    """Flat index in the seq-sharded buffer of the element that sits at flat
    index ``o`` of the head-sharded buffer (destination-driven form)."""
    r = _load().basp_oracle_head_to_seq_index(B, S, H, d, N, K, int(o))
    if r < 0:
        raise ValueError("bad shape or index")
    return r


# ---------------------------------------------------------------------------
# The definition through the logical tensor X[B, S, H, d] (numpy slicing).
# ---------------------------------------------------------------------------

def shard_seq(X, N, K):
    """Cut X[B, S, H, d] into the seq-sharded buffer (flat, rank order)."""
    B, S, H, d = X.shape
    G, Bg = groups(N, K, B)
    Sk = S // K
    parts = []
    for r in range(N):
        g, j = divmod(r, K)
        parts.append(X[g * Bg:(g + 1) * Bg, j * Sk:(j + 1) * Sk].reshape(-1))
    return np.concatenate(parts) if parts else X.reshape(-1)


def shard_head(X, N, K):
    """Cut X[B, S, H, d] into the head-sharded buffer (flat, rank order)."""
    B, S, H, d = X.shape
    G, Bg = groups(N, K, B)
    Hk = H // K
    parts = []
    for r in range(N):
        g, jp = divmod(r, K)
        parts.append(X[g * Bg:(g + 1) * Bg, :, jp * Hk:(jp + 1) * Hk].reshape(-1))
    return np.concatenate(parts) if parts else X.reshape(-1)


def unshard_seq(x, B, S, H, d, N, K):
    """Rebuild X[B, S, H, d] from a seq-sharded buffer."""
    G, Bg = groups(N, K, B)
    Sk = S // K
    X = np.empty((B, S, H, d), dtype=x.dtype)
    P = Bg * Sk * H * d
    for r in range(N):
        g, j = divmod(r, K)
        X[g * Bg:(g + 1) * Bg, j * Sk:(j + 1) * Sk] = \
            x[r * P:(r + 1) * P].reshape(Bg, Sk, H, d)
    return X


def unshard_head(x, B, S, H, d, N, K):
    """Rebuild X[B, S, H, d] from a head-sharded buffer."""
    G, Bg = groups(N, K, B)
    Hk = H // K
    X = np.empty((B, S, H, d), dtype=x.dtype)
    P = Bg * S * Hk * d
    for r in range(N):
        g, jp = divmod(r, K)
        X[g * Bg:(g + 1) * Bg, :, jp * Hk:(jp + 1) * Hk] = \
            x[r * P:(r + 1) * P].reshape(Bg, S, Hk, d)
    return X


def shard_seq_sf(X, N, K):
    """Cut X[S, B, H, d] (sequence-first logical tensor) into the
    sequence-first seq-sharded buffer: shard (g, j) = X[j-th token block,
    group g's sequences], stored [S/K, Bg, H, d]."""
    S, B, H, d = X.shape
    G, Bg = groups(N, K, B)
    Sk = S // K
    parts = []
    for r in range(N):
        g, j = divmod(r, K)
        parts.append(X[j * Sk:(j + 1) * Sk, g * Bg:(g + 1) * Bg].reshape(-1))
    return np.concatenate(parts) if parts else X.reshape(-1)


def shard_head_sf(X, N, K):
    """Cut X[S, B, H, d] into the sequence-first head-sharded buffer: shard
    (g, j') = X[all tokens, group g's sequences, j'-th head block], stored
    [S, Bg, H/K, d]."""
    S, B, H, d = X.shape
    G, Bg = groups(N, K, B)
    Hk = H // K
    parts = []
    for r in range(N):
        g, jp = divmod(r, K)
        parts.append(X[:, g * Bg:(g + 1) * Bg, jp * Hk:(jp + 1) * Hk].reshape(-1))
    return np.concatenate(parts) if parts else X.reshape(-1)


def unshard_seq_sf(x, B, S, H, d, N, K):
    G, Bg = groups(N, K, B)
    Sk = S // K
    X = np.empty((S, B, H, d), dtype=x.dtype)
    P = Sk * Bg * H * d
    for r in range(N):
        g, j = divmod(r, K)
        X[j * Sk:(j + 1) * Sk, g * Bg:(g + 1) * Bg] = \
            x[r * P:(r + 1) * P].reshape(Sk, Bg, H, d)
    return X


def unshard_head_sf(x, B, S, H, d, N, K):
    G, Bg = groups(N, K, B)
    Hk = H // K
    X = np.empty((S, B, H, d), dtype=x.dtype)
    P = S * Bg * Hk * d
    for r in range(N):
        g, jp = divmod(r, K)
        X[:, g * Bg:(g + 1) * Bg, jp * Hk:(jp + 1) * Hk] = \
            x[r * P:(r + 1) * P].reshape(S, Bg, Hk, d)
    return X


def seq2head_by_slices(x, B, S, H, d, N, K, order="bshd"):
    if not valid_shape(B, S, H, d, N, K):
        raise ValueError("shape breaks a divisibility rule")
    if order == "sbhd":
        return shard_head_sf(unshard_seq_sf(x, B, S, H, d, N, K), N, K)
    return shard_head(unshard_seq(x, B, S, H, d, N, K), N, K)


def head2seq_by_slices(x, B, S, H, d, N, K, order="bshd"):
    if not valid_shape(B, S, H, d, N, K):
        raise ValueError("shape breaks a divisibility rule")
    if order == "sbhd":
        return shard_seq_sf(unshard_head_sf(x, B, S, H, d, N, K), N, K)
    return shard_seq(unshard_head(x, B, S, H, d, N, K), N, K)
