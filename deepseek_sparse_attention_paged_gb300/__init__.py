"""DeepSeek Sparse Attention (DSA) decode path for one GB300 GPU (sm_103a).

The compute lives in the CUDA library ``libdsa_gb300.so`` behind the C ABI of ``include/dsa.h``;
this package is its Python binding (``capi``), a buffer-owning decode-step helper (``pipeline``),
the library build (``build``) and the seeded synthetic workloads (``workloads``).
"""
from .capi import (  # noqa: F401
    DSAError,
    dsa_indexer_logits,
    dsa_indexer_logits_workspace_size,
    dsa_read_device_error,
    dsa_sparse_mla_decode,
    dsa_sparse_mla_workspace_size,
    dsa_store_index_k,
    dsa_topk,
    dsa_topk_workspace_size,
)
