"""sequence_re_layout_gb300: the BASP / Ulysses sequence<->head re-layout of
attention activations as hand-written CUDA for sm_103a behind a C ABI
(``include/basp.h``), with a thin ctypes binding of the same names."""
from .binding import (  # noqa: F401
    ALGO_CODES, BASP_ALGO_FUSED, BASP_ALGO_THREE_PASS, BASP_ALGO_THREE_PASS_ELIDE, BASP_DTYPE_BF16,
    BASP_DTYPE_FP16, BASP_DTYPE_FP32, BASP_DTYPE_FP8, BASP_ERR_ALIASING, BASP_ERR_ALIGNMENT,
    BASP_ERR_BATCH_GT_RANKS, BASP_ERR_CUDA, BASP_ERR_DIVISIBILITY,
    BASP_ERR_INVALID_ARG, BASP_ERR_TOO_LARGE, BASP_ERR_WORKSPACE, BASP_OK,
    DTYPE_CODES, EXPORTS, ORDER_CODES, BASP_ORDER_BSHD, BASP_ORDER_SBHD,
    basp_layout_create_ex, basp_seq2head_qkv, basp_head2seq_qkv, BaspError, Layout, basp_head2seq, basp_head2seq_host,
    basp_layout_create, basp_layout_destroy, basp_layout_query, basp_seq2head,
    basp_seq2head_host, basp_seq2head_noalloc, basp_debug_bounds_violations, basp_status_string,
    BASP_NOALLOC_SCRATCH_BYTES, load_library)
