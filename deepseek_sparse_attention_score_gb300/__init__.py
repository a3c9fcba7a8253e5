"""GB300 (sm_103a) DeepSeek-Sparse-Attention hot path.

The compute lives in ``libdsa_gb300.so`` (hand-written CUDA, C ABI declared
in ``include/dsa.h``); :mod:`.abi` is its thin Python binding and
:mod:`.layer` chains the calls into one DSA layer step.
"""
from .abi import (  # noqa: F401
    DSAError,
    dsa_build_block_union,
    dsa_device_sm_count,
    dsa_launch_count,
    dsa_index_build_share_map,
    dsa_indexer_page_topk,
    dsa_indexer_topk,
    dsa_indexer_workspace_size,
    dsa_sparse_mla_decode,
    dsa_sparse_mla_decode_noalloc,
    dsa_paged_write_back,
    dsa_paged_write_back_pair,
    dsa_dense_mla,
    dsa_selftest_wait_timeout,
    dsa_indexer_topk_approx,
    dsa_topk_pages_from_tokens,
    dsa_sparse_mla_decode_workspace_size,
    dsa_sparse_mla_prefill_qblock,
    lib,
)
