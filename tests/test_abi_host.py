"""CPU checks of the C ABI: the library loads and exports every symbol that
include/basp.h declares; the layout descriptor applies the BASP review's rules
and derives its sizes; compute calls reject bad arguments before anything
touches a GPU (no call here reaches a CUDA API)."""
import os
import re

import pytest

import sequence_re_layout_gb300 as basp
from sequence_re_layout_gb300.build import build_library
from sequence_re_layout_gb300.workloads import WORKLOADS

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "basp.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_library()


def declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(basp_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    lib = basp.load_library()
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(basp.EXPORTS)


def test_debug_library_exports_its_extra_symbol():
    """libbasp_debug.so exports everything basp.h declares plus what
    basp_debug.h declares; the release library does not export the latter."""
    import ctypes
    from sequence_re_layout_gb300.build import DEBUG_LIB_PATH
    dbg = ctypes.CDLL(DEBUG_LIB_PATH)
    extra = declared_functions(HEADER.replace("basp.h", "basp_debug.h"))
    assert extra == ["basp_debug_bounds_violations"]
    for n in declared_functions() + extra:
        assert hasattr(dbg, n), n
    assert not hasattr(basp.load_library(), extra[0])


@pytest.mark.parametrize("args,status", [
    ((2, 64, 4, 4, 16, 4, 3), basp.BASP_ERR_DIVISIBILITY),     # N % K
    ((3, 64, 4, 4, 16, 4, 2), basp.BASP_ERR_DIVISIBILITY),     # B % (N/K)
    ((2, 62, 4, 4, 16, 4, 4), basp.BASP_ERR_DIVISIBILITY),     # S % K
    ((2, 64, 6, 4, 16, 4, 4), basp.BASP_ERR_DIVISIBILITY),     # Hq % K
    ((2, 64, 8, 2, 16, 4, 4), basp.BASP_ERR_DIVISIBILITY),     # Hkv % K (GQA)
    ((16, 64, 8, 8, 16, 8, 0), basp.BASP_ERR_BATCH_GT_RANKS),  # BASP rule, B > N
    ((3, 64, 8, 8, 16, 8, 0), basp.BASP_ERR_DIVISIBILITY),     # BASP rule, N % B
    ((2, 64, 0, 8, 16, 8, 8), basp.BASP_ERR_INVALID_ARG),
    ((2, 64, 8, 8, 0, 8, 8), basp.BASP_ERR_INVALID_ARG),
    ((-1, 64, 8, 8, 16, 8, 8), basp.BASP_ERR_INVALID_ARG),
    ((2, 1 << 40, 1 << 10, 8, 1 << 10, 8, 8), basp.BASP_ERR_TOO_LARGE),
])
def test_layout_rules(args, status):
    with pytest.raises(basp.BaspError) as e:
        basp.basp_layout_create(*args, "bf16")
    assert e.value.status == status


def test_bad_dtype():
    with pytest.raises(basp.BaspError) as e:
        basp.basp_layout_create(2, 64, 8, 8, 16, 8, 8, 7)
    assert e.value.status == basp.BASP_ERR_INVALID_ARG


def test_ulysses_accepts_batch_above_ranks():
    """B > N is only an error for the BASP rule; a Ulysses group (K = N) holds
    all B sequences."""
    with basp.Layout(16, 64, 8, 8, 16, 8, 8) as L:
        assert L.info["seqs_per_group"] == 16


@pytest.mark.parametrize("name", sorted(WORKLOADS))
@pytest.mark.parametrize("layout", ["basp", "ulysses", "rule"])
def test_derived_sizes(name, layout):
    """Per-rank tokens B*S/N in both layouts; K-1 peers; bytes per peer
    Bg*(S/K)*(H/K)*d*esz (review "Summary": peers N-1 -> K-1 with B*S/N tokens
    per GPU kept)."""
    w = WORKLOADS[name]
    K = 0 if layout == "rule" else w.K(layout)
    with basp.Layout(w.B, w.S, w.Hq, w.Hkv, w.d, w.N, K, w.dtype) as L:
        i = L.info
    Kx = w.K_basp if layout in ("basp", "rule") else w.N
    esz = 4 if w.dtype == "fp32" else 2
    G = w.N // Kx
    assert i["K"] == Kx and i["groups"] == G and i["seqs_per_group"] == w.B // G
    assert i["tokens_per_rank"] * w.N == w.B * w.S
    assert i["elems_per_rank_q"] * w.N == w.B * w.S * w.Hq * w.d
    assert i["elems_per_rank_kv"] * w.N == w.B * w.S * w.Hkv * w.d
    assert i["peers"] == Kx - 1
    assert i["bytes_per_peer_q"] * Kx == i["elems_per_rank_q"] * esz
    assert i["bytes_per_peer_kv"] * Kx == i["elems_per_rank_kv"] * esz
    assert i["bytes_q"] == w.B * w.S * w.Hq * w.d * esz
    assert i["workspace_bytes"] >= 2 * (i["bytes_q"] + 2 * i["bytes_kv"])
    if layout != "ulysses":
        # the review's "Strengths": Ulysses with SP = N/B would hold B^2 S/N
        assert i["foil_tokens_per_rank"] * w.N == w.B * w.B * w.S


def test_batch_one_rule_gives_ulysses():
    with basp.Layout(1, 8192, 32, 8, 64, 8, 0) as L:
        assert L.info["K"] == 8 and L.info["groups"] == 1


@pytest.fixture
def layout():
    with basp.Layout(2, 64, 8, 4, 16, 4, 2, "bf16") as L:
        yield L


FAKE = 1 << 40        # never dereferenced: each call below fails validation


def test_compute_rejects_before_launch(layout):
    h = layout.handle
    nq = layout.info["bytes_q"]
    nkv = layout.info["bytes_kv"]
    cases = [
        # unpaired input/output
        (lambda: basp.basp_seq2head(h, "fused", FAKE, None, None, None, None, None),
         basp.BASP_ERR_INVALID_ARG),
        # nothing to do
        (lambda: basp.basp_seq2head(h, "fused", None, None, None, None, None, None),
         basp.BASP_ERR_INVALID_ARG),
        # NULL layout
        (lambda: basp.basp_seq2head(0, "fused", FAKE, None, None, FAKE + nq, None, None),
         basp.BASP_ERR_INVALID_ARG),
        # misaligned for bf16
        (lambda: basp.basp_seq2head(h, "fused", FAKE + 1, None, None, FAKE + 2 * nq, None, None),
         basp.BASP_ERR_ALIGNMENT),
        # output overlaps its input
        (lambda: basp.basp_seq2head(h, "fused", FAKE, None, None, FAKE + nq - 2, None, None),
         basp.BASP_ERR_ALIASING),
        # output overlaps another tensor's input
        (lambda: basp.basp_seq2head(h, "fused", FAKE, FAKE + nq, None,
                                    FAKE + nq + nkv, FAKE + nq + 16, None),
         basp.BASP_ERR_ALIASING),
        # two outputs overlap
        (lambda: basp.basp_head2seq(h, "fused", FAKE, FAKE + nq, None,
                                    FAKE + 4 * nq, FAKE + 4 * nq + 64, None),
         basp.BASP_ERR_ALIASING),
        # three-pass without workspace / too small
        (lambda: basp.basp_seq2head(h, "three_pass", FAKE, None, None, FAKE + nq, None, None),
         basp.BASP_ERR_WORKSPACE),
        (lambda: basp.basp_seq2head(h, "three_pass", FAKE, None, None, FAKE + nq, None, None,
                                    FAKE + 8 * nq, 2 * nq - 1),
         basp.BASP_ERR_WORKSPACE),
        # workspace overlapping an input
        (lambda: basp.basp_seq2head(h, "three_pass", FAKE, None, None, FAKE + nq, None, None,
                                    FAKE + nq // 2, 4 * nq),
         basp.BASP_ERR_ALIASING),
        # unknown algorithm
        (lambda: basp.basp_seq2head(h, 9, FAKE, None, None, FAKE + nq, None, None),
         basp.BASP_ERR_INVALID_ARG),
        # host form: staging missing
        (lambda: basp.basp_seq2head_host(h, "fused", FAKE, None, None, FAKE + nq, None, None,
                                         None, 0),
         basp.BASP_ERR_WORKSPACE),
        # no-allocation form: unpaired, aliasing
        (lambda: basp.basp_seq2head_noalloc(h, FAKE, None, None, None, None, None),
         basp.BASP_ERR_INVALID_ARG),
        (lambda: basp.basp_seq2head_noalloc(h, FAKE, None, None, FAKE + 2, None, None),
         basp.BASP_ERR_ALIASING),
    ]
    for fn, status in cases:
        with pytest.raises(basp.BaspError) as e:
            fn()
        assert e.value.status == status, e.value


def test_status_strings():
    for s in range(9):
        assert basp.basp_status_string(s) not in ("", "unknown status")
    assert basp.basp_status_string(99) == "unknown status"


def test_noalloc_size_limit_checked_before_any_cuda_call():
    """A call needing more scratch than the built-in buffer is refused on the
    host (this CPU-only run has no CUDA device to fall back on)."""
    with basp.Layout(2, 4096, 32, 8, 64, 8, 4, "bf16") as L:
        nq = L.info["bytes_q"]
        with pytest.raises(basp.BaspError) as e:
            basp.basp_seq2head_noalloc(L.handle, FAKE, None, None, FAKE + nq, None, None)
        assert e.value.status == basp.BASP_ERR_WORKSPACE


def test_create_ex_orders_and_bad_order():
    h = basp.basp_layout_create_ex(2, 64, 8, 8, 16, 8, 8, "bf16", "sbhd")
    try:
        i = basp.basp_layout_query(h)
        assert i["order"] == basp.BASP_ORDER_SBHD
        assert i["bytes_qkv_packed"] == 2 * 64 * 24 * 16 * 2
    finally:
        basp.basp_layout_destroy(h)
    with pytest.raises(basp.BaspError) as e:
        basp.basp_layout_create_ex(2, 64, 8, 8, 16, 8, 8, "bf16", 5)
    assert e.value.status == basp.BASP_ERR_INVALID_ARG


def test_packed_qkv_rejects_before_launch(layout):
    h = layout.handle
    nq, nkv = layout.info["bytes_q"], layout.info["bytes_kv"]
    npk = layout.info["bytes_qkv_packed"]
    P = FAKE
    cases = [
        (lambda: basp.basp_seq2head_qkv(h, P, None, P + npk, P + 2 * npk), basp.BASP_ERR_INVALID_ARG),
        (lambda: basp.basp_seq2head_qkv(h, P + 1, P + npk, P + 2 * npk, P + 3 * npk), basp.BASP_ERR_ALIGNMENT),
        (lambda: basp.basp_seq2head_qkv(h, P, P + npk - 2, P + 2 * npk, P + 3 * npk), basp.BASP_ERR_ALIASING),
        (lambda: basp.basp_seq2head_qkv(h, P, P + npk, P + npk + 16, P + 3 * npk), basp.BASP_ERR_ALIASING),
        (lambda: basp.basp_head2seq_qkv(h, P, P + nq, P + nq + nkv, P + nq // 2), basp.BASP_ERR_ALIASING),
        (lambda: basp.basp_head2seq_qkv(h, P, P + nq, P + nq + nkv, None), basp.BASP_ERR_INVALID_ARG),
        (lambda: basp.basp_head2seq_qkv(0, P, P + nq, P + nq + nkv, P + 4 * npk), basp.BASP_ERR_INVALID_ARG),
    ]
    for fn, status in cases:
        with pytest.raises(basp.BaspError) as e:
            fn()
        assert e.value.status == status, e.value


def test_three_pass_elide_workspace_rule():
    """With one sequence per group the elided path needs one workspace region
    per tensor (not two) and refuses less."""
    with basp.Layout(2, 64, 8, 4, 16, 4, 2, "bf16") as L:      # BASP: Bg = 1
        nq = L.info["bytes_q"]
        h = L.handle
        with pytest.raises(basp.BaspError) as e:
            basp.basp_seq2head(h, "three_pass_elide", FAKE, None, None, FAKE + nq,
                               None, None, FAKE + 4 * nq, nq - 1)
        assert e.value.status == basp.BASP_ERR_WORKSPACE
        with pytest.raises(basp.BaspError) as e:
            basp.basp_seq2head(h, "three_pass_elide", FAKE, None, None, FAKE + nq,
                               None, None, FAKE + nq // 2, nq)
        assert e.value.status == basp.BASP_ERR_ALIASING


def test_layouts_from_many_threads():
    """Layout create / query / destroy from 8 host threads at once, and one
    shared handle queried concurrently (the handle is immutable)."""
    import threading
    shared = basp.Layout(2, 8192, 32, 8, 64, 8, 4, "bf16")
    errors = []

    def work(seed):
        try:
            for i in range(200):
                K = (1, 2, 4, 8)[(seed + i) % 4]
                with basp.Layout(8 // K * 2, 64 * K, 8 * K, 8 * K, 16, 8, K) as L:
                    assert L.info["K"] == K
                assert basp.basp_layout_query(shared.handle)["peers"] == 3
        except Exception as e:          # collected and reported below
            errors.append(e)

    ts = [threading.Thread(target=work, args=(s,)) for s in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    shared.close()
    assert not errors, errors[:3]


def test_binding_refuses_bad_tensors():
    """The binding checks tensor arguments before the C call: contiguity,
    size against the layout, and where the memory lives."""
    import torch
    with basp.Layout(2, 64, 8, 4, 16, 4, 2, "bf16") as L:
        nq = L.info["bytes_q"] // 2
        q = torch.empty(2 * nq, dtype=torch.bfloat16)[::2]          # strided view
        with pytest.raises(ValueError, match="contiguous"):
            basp.basp_seq2head(L.handle, "fused", q, None, None, FAKE, None, None)
        small = torch.empty(nq - 1, dtype=torch.bfloat16)
        with pytest.raises(ValueError, match="bytes"):
            basp.basp_seq2head(L.handle, "fused", small, None, None, FAKE, None, None)
        pageable = torch.empty(nq, dtype=torch.bfloat16)
        with pytest.raises(ValueError, match="CUDA tensor or page-locked"):
            basp.basp_seq2head(L.handle, "fused", pageable, None, None, FAKE, None, None)
        packed = torch.empty(L.info["bytes_qkv_packed"] // 2 - 1, dtype=torch.bfloat16)
        with pytest.raises(ValueError, match="bytes"):
            basp.basp_seq2head_qkv(L.handle, packed, FAKE, FAKE + 2 * nq, FAKE + 4 * nq)


def test_binding_refuses_a_tensor_on_another_device(monkeypatch):
    """A CUDA tensor on a device other than the current one is refused before
    the C call (the library launches on the current device).  A stand-in
    tensor plays cuda:1 so this runs without a GPU."""
    from sequence_re_layout_gb300 import binding

    class OnDevice1:
        is_cuda = True
        nbytes = 1 << 30
        device = type("Dev", (), {"index": 1})()

        def is_contiguous(self):
            return True

        def data_ptr(self):
            return FAKE

    monkeypatch.setattr(binding, "_current_device", lambda: 0)
    with basp.Layout(2, 64, 8, 4, 16, 4, 2, "bf16") as L:
        with pytest.raises(ValueError, match="current device is cuda:0"):
            basp.basp_seq2head(L.handle, "fused", OnDevice1(), None, None,
                               FAKE + (1 << 31), None, None)
