"""ctypes binding of ``libbasp.so`` (declared in ``include/basp.h``).

Argument marshalling only: every function here takes Python ints or torch
tensors, turns them into the C-ABI's pointers and sizes, calls the library and
raises :class:`BaspError` on a non-OK status.  The re-layout itself runs in the
library's CUDA kernels; there is no other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
# BASP_LIBRARY=debug selects the bounds-checking build (libbasp_debug.so);
# BASP_LIBRARY_PATH names any other build of the same sources explicitly
LIB_PATH = os.environ.get("BASP_LIBRARY_PATH") or os.path.join(
    PKG, "libbasp_debug.so" if os.environ.get("BASP_LIBRARY") == "debug" else "libbasp.so")

# enums of basp.h
BASP_DTYPE_BF16, BASP_DTYPE_FP32, BASP_DTYPE_FP16, BASP_DTYPE_FP8 = 0, 1, 2, 3
BASP_ALGO_FUSED, BASP_ALGO_THREE_PASS, BASP_ALGO_THREE_PASS_ELIDE = 0, 1, 2
BASP_ORDER_BSHD, BASP_ORDER_SBHD = 0, 1
(BASP_OK, BASP_ERR_INVALID_ARG, BASP_ERR_DIVISIBILITY, BASP_ERR_BATCH_GT_RANKS,
 BASP_ERR_ALIGNMENT, BASP_ERR_ALIASING, BASP_ERR_WORKSPACE, BASP_ERR_CUDA,
 BASP_ERR_TOO_LARGE) = range(9)

DTYPE_CODES = {"bf16": BASP_DTYPE_BF16, "fp32": BASP_DTYPE_FP32,
               "fp16": BASP_DTYPE_FP16, "fp8": BASP_DTYPE_FP8}
ALGO_CODES = {"fused": BASP_ALGO_FUSED, "three_pass": BASP_ALGO_THREE_PASS,
              "three_pass_elide": BASP_ALGO_THREE_PASS_ELIDE}
ORDER_CODES = {"bshd": BASP_ORDER_BSHD, "sbhd": BASP_ORDER_SBHD}

# every symbol include/basp.h declares
EXPORTS = ("basp_layout_create", "basp_layout_create_ex", "basp_layout_query",
           "basp_layout_destroy", "basp_seq2head", "basp_head2seq",
           "basp_seq2head_qkv", "basp_head2seq_qkv", "basp_seq2head_host",
           "basp_head2seq_host", "basp_seq2head_noalloc", "basp_status_string")

# size of the library's built-in scratch for basp_seq2head_noalloc
BASP_NOALLOC_SCRATCH_BYTES = 32 << 20


class basp_info(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "B", "S", "Hq", "Hkv", "d", "N", "K", "groups", "seqs_per_group",
        "tokens_per_rank", "elem_size", "elems_per_rank_q", "elems_per_rank_kv",
        "peers", "bytes_per_peer_q", "bytes_per_peer_kv", "bytes_q", "bytes_kv",
        "workspace_bytes", "staging_bytes", "foil_tokens_per_rank", "order",
        "bytes_qkv_packed")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class basp_layout_desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("B", "S", "Hq", "Hkv", "d", "N", "K")] + \
        [("dtype", ctypes.c_int), ("order", ctypes.c_int)]


class BaspError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, basp_status_string(status), status))


_lib = None


def load_library():
    """Load the in-tree ``libbasp.so``.  There is no fallback: a missing
    library is an error."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libbasp.so is not built (expected at %s); run "
            "sequence_re_layout_gb300.build.build_library()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    lib.basp_layout_create.argtypes = [i64] * 7 + [ctypes.c_int, ctypes.POINTER(vp)]
    lib.basp_layout_create.restype = ctypes.c_int
    lib.basp_layout_create_ex.argtypes = [ctypes.POINTER(basp_layout_desc),
                                          ctypes.POINTER(vp)]
    lib.basp_layout_create_ex.restype = ctypes.c_int
    lib.basp_layout_query.argtypes = [vp, ctypes.POINTER(basp_info)]
    lib.basp_layout_query.restype = ctypes.c_int
    lib.basp_layout_destroy.argtypes = [vp]
    lib.basp_layout_destroy.restype = None
    for name in ("basp_seq2head", "basp_head2seq"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, ctypes.c_int] + [vp] * 6 + [vp, sz, vp]
        fn.restype = ctypes.c_int
    for name in ("basp_seq2head_host", "basp_head2seq_host"):
        fn = getattr(lib, name)
        fn.argtypes = [vp, ctypes.c_int] + [vp] * 6 + [vp, sz, vp, sz, vp]
        fn.restype = ctypes.c_int
    lib.basp_seq2head_qkv.argtypes = [vp] * 6
    lib.basp_seq2head_qkv.restype = ctypes.c_int
    lib.basp_head2seq_qkv.argtypes = [vp] * 6
    lib.basp_head2seq_qkv.restype = ctypes.c_int
    lib.basp_seq2head_noalloc.argtypes = [vp] + [vp] * 6 + [vp]
    lib.basp_seq2head_noalloc.restype = ctypes.c_int
    if hasattr(lib, "basp_debug_bounds_violations"):
        lib.basp_debug_bounds_violations.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
        lib.basp_debug_bounds_violations.restype = ctypes.c_int
    lib.basp_status_string.argtypes = [ctypes.c_int]
    lib.basp_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _ptr(x):
    """A device/host address from None, an int or a tensor."""
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


# layout handle -> basp_info dict, so tensor arguments can be checked cheaply
_INFO = {}


def _info(layout):
    i = _INFO.get(layout)
    if i is None and layout:
        i = basp_layout_query(layout)
    return i


def _current_device() -> int:
    import torch
    return torch.cuda.current_device()


def _tptr(x, need, where, name, place, cur=None):
    """Address of a buffer argument.  Raw ints pass through unchecked; a tensor
    must be contiguous, hold at least `need` bytes, and live where the call
    reads it: "device" (a CUDA tensor on the current device, or page-locked
    host memory, which the kernels reach over the host link) or "host" (CPU
    memory)."""
    if x is None or isinstance(x, int):
        return _ptr(x)
    if not x.is_contiguous():
        raise ValueError("%s: %s must be contiguous" % (where, name))
    if need is not None and x.nbytes < need:
        raise ValueError("%s: %s holds %d bytes, the layout needs %d"
                         % (where, name, x.nbytes, need))
    if place == "device":
        if x.is_cuda:
            # the library launches on the current device (and takes its
            # built-in scratch there), so a tensor on another GPU would be
            # reached across devices: refuse it
            if cur is None:
                cur = _current_device()
            if x.device.index != cur:
                raise ValueError("%s: %s is on cuda:%s but the current device is "
                                 "cuda:%d; make its device current first"
                                 % (where, name, x.device.index, cur))
        elif not x.is_pinned():
            raise ValueError("%s: %s must be a CUDA tensor or page-locked host "
                             "memory" % (where, name))
    elif x.is_cuda:
        raise ValueError("%s: %s must be in host memory" % (where, name))
    return x.data_ptr() or None


def _triple(layout, where, names, bufs, place):
    """Check the (Hq, Hkv, Hkv) buffer triple of one call."""
    i = _info(layout)
    need = (i["bytes_q"], i["bytes_kv"], i["bytes_kv"]) if i else (None,) * 3
    # the current device, asked once for the whole triple
    cur = None
    if place == "device" and any(getattr(b, "is_cuda", False) for b in bufs):
        cur = _current_device()
    return [_tptr(b, n, where, nm, place, cur) for b, n, nm in zip(bufs, need, names)]


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _check(status, where):
    if status != BASP_OK:
        raise BaspError(status, where)


def basp_status_string(status: int) -> str:
    return load_library().basp_status_string(int(status)).decode()


def basp_layout_create(B, S, Hq, Hkv, d, N, K, dtype="bf16") -> int:
    """Create a layout handle (an opaque int).  ``K = 0`` asks for the BASP
    rule K = N/B.  ``dtype`` is "bf16", "fp16", "fp32" or the enum value."""
    code = DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype)
    h = ctypes.c_void_p()
    _check(load_library().basp_layout_create(B, S, Hq, Hkv, d, N, K, code,
                                             ctypes.byref(h)),
           "basp_layout_create")
    _INFO[h.value] = basp_layout_query(h.value)
    return h.value


def basp_layout_create_ex(B, S, Hq, Hkv, d, N, K, dtype="bf16", order="bshd") -> int:
    """Create a layout handle with a token order ("bshd" batch-first or
    "sbhd" sequence-first, or the enum value)."""
    desc = basp_layout_desc(
        B, S, Hq, Hkv, d, N, K,
        DTYPE_CODES[dtype] if isinstance(dtype, str) else int(dtype),
        ORDER_CODES[order] if isinstance(order, str) else int(order))
    h = ctypes.c_void_p()
    _check(load_library().basp_layout_create_ex(ctypes.byref(desc), ctypes.byref(h)),
           "basp_layout_create_ex")
    _INFO[h.value] = basp_layout_query(h.value)
    return h.value


def basp_layout_query(layout: int) -> dict:
    info = basp_info()
    _check(load_library().basp_layout_query(layout, ctypes.byref(info)),
           "basp_layout_query")
    return info.as_dict()


def basp_layout_destroy(layout: int) -> None:
    _INFO.pop(layout, None)
    load_library().basp_layout_destroy(layout)


def _algo(a):
    return ALGO_CODES[a] if isinstance(a, str) else int(a)


def _nbytes(x):
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.numel() * x.element_size()


def basp_seq2head(layout, algo, q, k, v, q_out, k_out, v_out,
                  workspace=None, workspace_bytes=None, stream=None):
    """seq-sharded -> head-sharded (device buffers); see ``basp.h``."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    w = "basp_seq2head"
    a = _triple(layout, w, ("q", "k", "v"), (q, k, v), "device")
    b = _triple(layout, w, ("q_out", "k_out", "v_out"), (q_out, k_out, v_out), "device")
    _check(load_library().basp_seq2head(
        layout, _algo(algo), *a, *b,
        _tptr(workspace, None, w, "workspace", "device"), wb, _stream(stream)), w)


def basp_head2seq(layout, algo, o, k, v, o_out, k_out, v_out,
                  workspace=None, workspace_bytes=None, stream=None):
    """head-sharded -> seq-sharded (device buffers); see ``basp.h``."""
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    w = "basp_head2seq"
    a = _triple(layout, w, ("o", "k", "v"), (o, k, v), "device")
    b = _triple(layout, w, ("o_out", "k_out", "v_out"), (o_out, k_out, v_out), "device")
    _check(load_library().basp_head2seq(
        layout, _algo(algo), *a, *b,
        _tptr(workspace, None, w, "workspace", "device"), wb, _stream(stream)), w)


def basp_seq2head_host(layout, algo, q, k, v, q_out, k_out, v_out, staging,
                       staging_bytes=None, workspace=None,
                       workspace_bytes=None, stream=None):
    """Host buffers in and out, device ``staging``; see ``basp.h``."""
    sb = _nbytes(staging) if staging_bytes is None else staging_bytes
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    w = "basp_seq2head_host"
    a = _triple(layout, w, ("q", "k", "v"), (q, k, v), "host")
    b = _triple(layout, w, ("q_out", "k_out", "v_out"), (q_out, k_out, v_out), "host")
    _check(load_library().basp_seq2head_host(
        layout, _algo(algo), *a, *b, _tptr(staging, None, w, "staging", "device"), sb,
        _tptr(workspace, None, w, "workspace", "device"), wb, _stream(stream)), w)


def basp_head2seq_host(layout, algo, o, k, v, o_out, k_out, v_out, staging,
                       staging_bytes=None, workspace=None,
                       workspace_bytes=None, stream=None):
    """Host buffers in and out, device ``staging``; see ``basp.h``."""
    sb = _nbytes(staging) if staging_bytes is None else staging_bytes
    wb = _nbytes(workspace) if workspace_bytes is None else workspace_bytes
    w = "basp_head2seq_host"
    a = _triple(layout, w, ("o", "k", "v"), (o, k, v), "host")
    b = _triple(layout, w, ("o_out", "k_out", "v_out"), (o_out, k_out, v_out), "host")
    _check(load_library().basp_head2seq_host(
        layout, _algo(algo), *a, *b, _tptr(staging, None, w, "staging", "device"), sb,
        _tptr(workspace, None, w, "workspace", "device"), wb, _stream(stream)), w)


def basp_debug_bounds_violations() -> int:
    """Debug build only: read and clear the count of out-of-bounds accesses
    the kernels skipped on the current device (synchronises it)."""
    lib = load_library()
    if not hasattr(lib, "basp_debug_bounds_violations"):
        raise RuntimeError("the loaded library is not the bounds-checking build "
                           "(set BASP_LIBRARY=debug before importing)")
    n = ctypes.c_ulonglong()
    _check(lib.basp_debug_bounds_violations(ctypes.byref(n)), "basp_debug_bounds_violations")
    return n.value


def basp_seq2head_qkv(layout, qkv, q_out, k_out, v_out, stream=None):
    """Packed seq-sharded QKV -> head-sharded Q, K, V; see ``basp.h``."""
    w = "basp_seq2head_qkv"
    i = _info(layout)
    p = _tptr(qkv, i["bytes_qkv_packed"] if i else None, w, "qkv", "device")
    b = _triple(layout, w, ("q_out", "k_out", "v_out"), (q_out, k_out, v_out), "device")
    _check(load_library().basp_seq2head_qkv(layout, p, *b, _stream(stream)), w)


def basp_head2seq_qkv(layout, q, k, v, qkv_out, stream=None):
    """Head-sharded Q, K, V -> packed seq-sharded QKV; see ``basp.h``."""
    w = "basp_head2seq_qkv"
    i = _info(layout)
    a = _triple(layout, w, ("q", "k", "v"), (q, k, v), "device")
    p = _tptr(qkv_out, i["bytes_qkv_packed"] if i else None, w, "qkv_out", "device")
    _check(load_library().basp_head2seq_qkv(layout, *a, p, _stream(stream)), w)


def basp_seq2head_noalloc(layout, q, k, v, q_out, k_out, v_out, stream=None):
    """seq-sharded -> head-sharded through the three-pass path, using the
    library's built-in scratch instead of a workspace: for callers that cannot
    allocate device memory.  See ``basp.h`` for the size limit and the rule
    that calls sharing the scratch must not overlap on the GPU."""
    w = "basp_seq2head_noalloc"
    a = _triple(layout, w, ("q", "k", "v"), (q, k, v), "device")
    b = _triple(layout, w, ("q_out", "k_out", "v_out"), (q_out, k_out, v_out), "device")
    _check(load_library().basp_seq2head_noalloc(layout, *a, *b, _stream(stream)), w)


class Layout:
    """Owns one layout handle; ``info`` holds the derived sizes."""

    def __init__(self, B, S, Hq, Hkv, d, N, K, dtype="bf16", order="bshd"):
        self.handle = basp_layout_create_ex(B, S, Hq, Hkv, d, N, K, dtype, order)
        self.info = basp_layout_query(self.handle)

    def close(self):
        if self.handle:
            basp_layout_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
