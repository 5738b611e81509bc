"""GB300 (sm_103a) library for the DSA decode/prefill hot path.

A fused lightning indexer with on-chip Top-K selection over a paged indexer K cache, followed by sparse
flash attention over the selected rows of a paged MLA latent-KV cache.  The compute lives in
``libdsa_gb300.so`` (hand-written CUDA behind the C ABI of ``include/dsa.h``); this package is the thin
ctypes binding with the same entry-point names.  PyTorch is used for device memory and streams only.
"""
from ._lib import (  # noqa: F401
    DSA_BF16,
    DSA_DEVERR_INDEX,
    DSA_DEVERR_PAGE,
    DSA_DEVERR_SEQ,
    DSA_DEVERR_TIMEOUT,
    DSA_ERR_CUDA,
    DSA_ERR_DEVICE,
    DSA_ERR_INVALID_ARG,
    DSA_ERR_TIMEOUT,
    DSA_ERR_UNSUPPORTED,
    DSA_FP8_E4M3,
    DSA_KV_FP8_ROW_BYTES,
    DSA_MXFP8_E4M3,
    DSA_OK,
    EXPORTED,
    LIB_PATH,
    DsaDims,
    DsaError,
    abi_version,
    append_rows,
    attn_combine,
    clear_device_error,
    fused_decode,
    fused_decode_launches,
    get_device_error,
    indexer_topk,
    indexer_topk_shard,
    indexer_topk_static,
    lib,
    set_wait_limit_ns,
    sparse_attn,
    sparse_attn_shard,
    status_string,
    topk_merge,
    workspace_size,
)
