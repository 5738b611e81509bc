"""ctypes binding of the C ABI in include/dsa.h (argument marshalling only).

Every compute step runs inside libdsa_gb300.so.  Tensors are passed as raw device pointers
(``tensor.data_ptr()``); the CUDA stream defaults to PyTorch's current stream.  A non-OK status raises
:class:`DsaError` carrying the library's own message.  There is no fallback: if the library is missing
or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdsa_gb300.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_CUDA, DSA_ERR_DEVICE, DSA_ERR_TIMEOUT = range(6)
DSA_BF16, DSA_FP8_E4M3, DSA_MXFP8_E4M3 = 0, 1, 2
DSA_KV_FP8_ROW_BYTES = 656
DSA_DEVERR_PAGE, DSA_DEVERR_SEQ, DSA_DEVERR_INDEX, DSA_DEVERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8

EXPORTED = (
    "dsa_abi_version",
    "dsa_status_string",
    "dsa_last_error_message",
    "dsa_workspace_size",
    "dsa_indexer_topk",
    "dsa_sparse_attn",
    "dsa_fused_decode",
    "dsa_fused_decode_launches",
    "dsa_get_device_error",
    "dsa_clear_device_error",
    "dsa_indexer_topk_static",
    "dsa_append_rows",
    "dsa_indexer_topk_shard",
    "dsa_sparse_attn_shard",
    "dsa_topk_merge",
    "dsa_attn_combine",
    "dsa_set_wait_limit_ns",
)


class DsaDims(ctypes.Structure):
    """Mirror of dsa_dims_t."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("total_q", ctypes.c_int32),
        ("max_q_len", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("idx_heads", ctypes.c_int32),
        ("idx_dim", ctypes.c_int32),
        ("idx_dtype", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("attn_heads", ctypes.c_int32),
        ("kv_dim", ctypes.c_int32),
        ("v_dim", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("kv_dtype", ctypes.c_int32),
    ]

    def __repr__(self):
        return "DsaDims(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class DsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} [status {status}]")
        self.status = status


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libdsa_gb300.so (built by ``sparse_attention_dsa_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m sparse_attention_dsa_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32p = ctypes.c_void_p, ctypes.c_void_p
            st = ctypes.c_int
            L.dsa_abi_version.restype = ctypes.c_int32
            L.dsa_abi_version.argtypes = []
            L.dsa_status_string.restype = ctypes.c_char_p
            L.dsa_status_string.argtypes = [st]
            L.dsa_last_error_message.restype = ctypes.c_char_p
            L.dsa_last_error_message.argtypes = []
            L.dsa_workspace_size.restype = ctypes.c_size_t
            L.dsa_workspace_size.argtypes = [ctypes.POINTER(DsaDims)]
            L.dsa_indexer_topk.restype = st
            L.dsa_indexer_topk.argtypes = [ctypes.POINTER(DsaDims)] + [vp] * 12
            L.dsa_indexer_topk_shard.restype = st
            L.dsa_indexer_topk_shard.argtypes = ([ctypes.POINTER(DsaDims)] + [vp] * 8 + [ctypes.c_int32] * 2 +
                                                 [vp] * 4)
            L.dsa_sparse_attn_shard.restype = st
            L.dsa_sparse_attn_shard.argtypes = ([ctypes.POINTER(DsaDims)] + [vp] * 6 + [ctypes.c_int32] * 2 +
                                                [vp] * 4)
            L.dsa_topk_merge.restype = st
            L.dsa_topk_merge.argtypes = [ctypes.c_int32] * 3 + [vp] * 5
            L.dsa_attn_combine.restype = st
            L.dsa_attn_combine.argtypes = [ctypes.c_int32] * 4 + [vp] * 5
            L.dsa_set_wait_limit_ns.restype = ctypes.c_uint64
            L.dsa_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
            L.dsa_sparse_attn.restype = st
            L.dsa_sparse_attn.argtypes = [ctypes.POINTER(DsaDims)] + [vp] * 10
            L.dsa_fused_decode.restype = st
            L.dsa_fused_decode.argtypes = [ctypes.POINTER(DsaDims)] + [vp] * 15
            L.dsa_fused_decode_launches.restype = ctypes.c_int32
            L.dsa_fused_decode_launches.argtypes = [ctypes.POINTER(DsaDims)]
            L.dsa_get_device_error.restype = st
            L.dsa_get_device_error.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int32)]
            L.dsa_clear_device_error.restype = st
            L.dsa_clear_device_error.argtypes = [vp, vp]
            L.dsa_indexer_topk_static.restype = st
            L.dsa_indexer_topk_static.argtypes = [ctypes.POINTER(DsaDims)] + [vp] * 12
            L.dsa_append_rows.restype = st
            L.dsa_append_rows.argtypes = [ctypes.POINTER(DsaDims)] + [vp] * 10
            _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != DSA_OK:
        msg = lib().dsa_last_error_message().decode() or lib().dsa_status_string(status).decode()
        raise DsaError(status, msg)


def abi_version() -> int:
    return int(lib().dsa_abi_version())


def status_string(status: int) -> str:
    return lib().dsa_status_string(status).decode()


def workspace_size(dims: DsaDims) -> int:
    return int(lib().dsa_workspace_size(ctypes.byref(dims)))


def indexer_topk(dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, topk_idx, workspace,
                 stream=None, topk_score=None):
    _check(lib().dsa_indexer_topk(ctypes.byref(dims), _ptr(q_idx), _ptr(q_scale), _ptr(w), _ptr(k_cache),
                                  _ptr(k_scale), _ptr(page_table), _ptr(seq_lens), _ptr(cu_q_lens), _ptr(topk_idx),
                                  _ptr(topk_score), _ptr(workspace), _stream(stream)))


def indexer_topk_shard(dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, pos_begin, pos_end,
                       topk_idx, topk_score, workspace, stream=None):
    """dsa_indexer_topk_shard: the Top-K of the positions in [pos_begin, pos_end) only, with their scores."""
    _check(lib().dsa_indexer_topk_shard(ctypes.byref(dims), _ptr(q_idx), _ptr(q_scale), _ptr(w), _ptr(k_cache),
                                        _ptr(k_scale), _ptr(page_table), _ptr(seq_lens), _ptr(cu_q_lens),
                                        int(pos_begin), int(pos_end), _ptr(topk_idx), _ptr(topk_score),
                                        _ptr(workspace), _stream(stream)))


def sparse_attn_shard(dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk_idx, pos_begin, pos_end, out, lse,
                      workspace, stream=None):
    """dsa_sparse_attn_shard: attention over the selected rows in [pos_begin, pos_end) (a partial out, lse)."""
    _check(lib().dsa_sparse_attn_shard(ctypes.byref(dims), _ptr(q), _ptr(kv_cache), _ptr(page_table),
                                       _ptr(seq_lens), _ptr(cu_q_lens), _ptr(topk_idx), int(pos_begin), int(pos_end),
                                       _ptr(out), _ptr(lse), _ptr(workspace), _stream(stream)))


def topk_merge(shards, total_q, top_k, topk_idx, topk_score, out_idx, out_score=None, stream=None):
    """dsa_topk_merge: the global Top-K of the shards' (position, score) lists, [shards, T, K] each."""
    _check(lib().dsa_topk_merge(int(shards), int(total_q), int(top_k), _ptr(topk_idx), _ptr(topk_score),
                                _ptr(out_idx), _ptr(out_score), _stream(stream)))


def attn_combine(shards, total_q, heads, v_dim, out_parts, lse_parts, out, lse=None, stream=None):
    """dsa_attn_combine: the shards' partial attention outputs joined by their log-sum-exp weights."""
    _check(lib().dsa_attn_combine(int(shards), int(total_q), int(heads), int(v_dim), _ptr(out_parts),
                                  _ptr(lse_parts), _ptr(out), _ptr(lse), _stream(stream)))


def set_wait_limit_ns(limit_ns: int) -> int:
    """dsa_set_wait_limit_ns: limit of the kernels' pipeline waits for later launches (0 = one second).
    Returns the previous limit."""
    return int(lib().dsa_set_wait_limit_ns(int(limit_ns)))


def sparse_attn(dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk_idx, out, lse, workspace, stream=None):
    _check(lib().dsa_sparse_attn(ctypes.byref(dims), _ptr(q), _ptr(kv_cache), _ptr(page_table), _ptr(seq_lens),
                                 _ptr(cu_q_lens), _ptr(topk_idx), _ptr(out), _ptr(lse), _ptr(workspace),
                                 _stream(stream)))


def fused_decode(dims, q_idx, q_scale, w, k_cache, k_scale, q, kv_cache, page_table, seq_lens, cu_q_lens, topk_idx,
                 out, lse, workspace, stream=None):
    _check(lib().dsa_fused_decode(ctypes.byref(dims), _ptr(q_idx), _ptr(q_scale), _ptr(w), _ptr(k_cache),
                                  _ptr(k_scale), _ptr(q), _ptr(kv_cache), _ptr(page_table), _ptr(seq_lens),
                                  _ptr(cu_q_lens), _ptr(topk_idx), _ptr(out), _ptr(lse), _ptr(workspace),
                                  _stream(stream)))


def fused_decode_launches(dims) -> int:
    """Kernel launches fused_decode makes for these dims on the current device (1, 2, or 0)."""
    n = int(lib().dsa_fused_decode_launches(ctypes.byref(dims)))
    if n < 0:
        raise DsaError(DSA_ERR_INVALID_ARG, lib().dsa_last_error_message().decode())
    return n


def indexer_topk_static(dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, topk_idx,
                        device_error=None, stream=None, topk_score=None):
    """dsa_indexer_topk_static: no workspace; the library's static device scratch is used instead."""
    _check(lib().dsa_indexer_topk_static(ctypes.byref(dims), _ptr(q_idx), _ptr(q_scale), _ptr(w), _ptr(k_cache),
                                         _ptr(k_scale), _ptr(page_table), _ptr(seq_lens), _ptr(cu_q_lens),
                                         _ptr(topk_idx), _ptr(topk_score), _ptr(device_error), _stream(stream)))


def get_device_error(workspace, stream=None) -> int:
    """Synchronises the stream and returns the device error word (0 = no error)."""
    code = ctypes.c_int32(0)
    status = lib().dsa_get_device_error(_ptr(workspace), _stream(stream), ctypes.byref(code))
    if status not in (DSA_OK, DSA_ERR_DEVICE, DSA_ERR_TIMEOUT):
        _check(status)
    return int(code.value)


def clear_device_error(workspace, stream=None):
    _check(lib().dsa_clear_device_error(_ptr(workspace), _stream(stream)))


def append_rows(dims, k_new, kv_new, page_table, seq_lens, cu_q_lens, k_cache, k_scale, kv_cache, workspace,
                stream=None):
    """dsa_append_rows: write every query token's new indexer key / latent-KV row at its position."""
    _check(lib().dsa_append_rows(ctypes.byref(dims), _ptr(k_new), _ptr(kv_new), _ptr(page_table), _ptr(seq_lens),
                                 _ptr(cu_q_lens), _ptr(k_cache), _ptr(k_scale), _ptr(kv_cache), _ptr(workspace),
                                 _stream(stream)))
