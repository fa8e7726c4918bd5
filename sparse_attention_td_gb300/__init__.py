"""GB300-native TidalDecode decode step (Position Persistent Sparse Attention).

A thin Python binding of ``libtd.so`` (C ABI in ``include/td.h``).  It only
marshals arguments -- tensor pointers, shapes and the current CUDA stream --
and checks that tensors are CUDA tensors of the declared shapes, so the C
library never sees a host pointer or a short buffer.  Every step of the
computation runs in the library's CUDA kernels; there is no fallback.

Entry points (same names as the C ABI):
  td_full_attn_select  one full-attention layer, optionally selecting top-k
  td_topk_select       the selection step alone, from given scores
  td_sparse_attn       one PPSA layer over a given index set
  td_decode_step       one decode step over an L-layer schedule
  Plan                 a decode step captured into a CUDA graph
"""
from ._lib import (  # noqa: F401
    MODE_FULL, MODE_FULL_SELECT, MODE_SPARSE, FLAG_INDEX_OUT_OF_RANGE,
    FLAG_SEQ_LEN_OUT_OF_RANGE, FLAG_WAIT_TIMEOUT, NOALLOC_SCRATCH_BYTES, TdError, Shape, Workspace, Plan, lib, lib_path,
    td_status_string, td_workspace_size, td_workspace_init, td_workspace_status,
    td_full_attn_select, td_full_attn_select_coverage, td_topk_select, td_index_overlap, td_kv_append, td_probe_layer_reads, td_sparse_attn, td_sparse_attn_noalloc, td_decode_step, td_set_tuning, td_query_splits, td_kernel_name,
    make_shape, default_scale,
)
