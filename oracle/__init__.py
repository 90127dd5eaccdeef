"""Float64 CPU oracle for sparse MLA decode under decode-context-parallel.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.
"""
from .smla_oracle import (  # noqa: F401
    E4M3_TABLE,
    bf16_bits_to_f64,
    dcp_filter_convert_index,
    dcp_local_seq_len,
    dcp_topk_merge,
    dense_mla_decode,
    e4m3_to_f64,
    flatten_lse_bhs,
    lse_merge,
    parse_rows,
    sparse_mla_decode,
    sparse_mla_decode_rows,
    topk_select,
)
