"""CPU oracle for the DSA hot path: lightning-indexer scores, Top-K selection, sparse flash attention.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's CPU-baseline leg are the
only callers.  The product library never loads it, and it shares no code with the CUDA path.

The arithmetic lives in ``dsa_oracle.c`` (plain C, double precision, OpenMP over query tokens only); this
module compiles it with gcc and marshals numpy arrays.  Every function follows the articles cited at the
top of ``dsa_oracle.c``; the readings taken where they are silent are listed there as well.

Parity status: the scoring formula, the causal/tie conventions and the attention are pinned by the hand
examples, closed forms and invariants in ``tests/test_oracle.py``.  Whether the articles' unnamed model
uses exactly this ReLU-weighted score cannot be pinned from the articles (they print no formula).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


_ERRORS = {-1: "bad argument", -2: "page id out of range", -3: "position out of range", -4: "out of memory"}


class _Dims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("total_q", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("idx_heads", ctypes.c_int32),
        ("idx_dim", ctypes.c_int32),
        ("idx_fp8", ctypes.c_int32),
        ("top_k", ctypes.c_int32),
        ("attn_heads", ctypes.c_int32),
        ("kv_dim", ctypes.c_int32),
        ("v_dim", ctypes.c_int32),
        ("kv_fp8", ctypes.c_int32),
        ("softmax_scale", ctypes.c_double),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle (gcc -O3 -fopenmp; no fast-math and no contraction into fused multiply-adds, so
    every product and sum is the IEEE double operation the C source writes)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            vp, i32 = ctypes.c_void_p, ctypes.c_int32
            L.oracle_bf16_value.restype = ctypes.c_double
            L.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            L.oracle_e4m3_value.restype = ctypes.c_double
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.oracle_index_scores.restype = ctypes.c_int64
            L.oracle_index_scores.argtypes = [ctypes.POINTER(_Dims)] + [vp] * 8 + [i32, vp]
            L.oracle_indexer_topk.restype = ctypes.c_int
            L.oracle_indexer_topk.argtypes = [ctypes.POINTER(_Dims)] + [vp] * 9 + [i32, vp, vp, vp]
            L.oracle_index_scores_batch.restype = ctypes.c_int
            L.oracle_index_scores_batch.argtypes = [ctypes.POINTER(_Dims)] + [vp] * 9 + [i32, ctypes.c_int64, vp]
            L.oracle_sparse_attn.restype = ctypes.c_int
            L.oracle_sparse_attn.argtypes = [ctypes.POINTER(_Dims)] + [vp] * 7 + [i32, vp, vp, vp]
            L.oracle_e8m0_value.restype = ctypes.c_double
            L.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_quantize_group.restype = None
            L.oracle_quantize_group.argtypes = [vp, i32, vp, vp]
            L.oracle_append_rows.restype = ctypes.c_int
            L.oracle_append_rows.argtypes = [ctypes.POINTER(_Dims)] + [vp] * 8
            L.oracle_set_threads.restype = ctypes.c_int
            L.oracle_set_threads.argtypes = [ctypes.c_int]
            _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be contiguous"
    return a.ctypes.data


def _dims(wl) -> _Dims:
    return _Dims(batch=wl.batch, total_q=wl.total_q, num_pages=wl.num_pages, page_size=wl.page_size,
                 max_pages_per_seq=wl.max_pages_per_seq, idx_heads=wl.idx_heads, idx_dim=wl.idx_dim,
                 idx_fp8=(2 if getattr(wl, "idx_mx", False) else 1) if wl.idx_fp8 else 0, top_k=wl.top_k, attn_heads=wl.attn_heads, kv_dim=wl.kv_dim,
                 v_dim=wl.v_dim, kv_fp8=1 if getattr(wl, "kv_fp8", False) else 0, softmax_scale=wl.softmax_scale)


def _check(rc):
    if rc < 0:
        raise OracleError(_ERRORS.get(int(rc), f"error {rc}"))


def bf16_value(bits: int) -> float:
    return float(lib().oracle_bf16_value(bits))


def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_value(code))


def _tl(tlist, total):
    if tlist is None:
        return None, total
    t = np.ascontiguousarray(tlist, dtype=np.int32)
    return t, int(t.shape[0])


def index_scores(wl, t: int) -> np.ndarray:
    """I[t, s] for s = 0..p_t (float64)."""
    pos = int(wl.query_positions()[t])
    out = np.empty(max(pos + 1, 1), dtype=np.float64)
    rc = lib().oracle_index_scores(ctypes.byref(_dims(wl)), _p(wl.q_idx), _p(wl.q_scale), _p(wl.w), _p(wl.k_cache),
                                   _p(wl.k_scale), _p(wl.page_table), _p(wl.seq_lens), _p(wl.cu_q_lens), int(t),
                                   _p(out))
    _check(rc)
    return out[: pos + 1]


def index_scores_batch(wl, tlist):
    """List of float64 score arrays I[t, 0..p_t] for the tokens in tlist (computed in parallel)."""
    tl = np.ascontiguousarray(tlist, dtype=np.int32)
    pos = wl.query_positions()[tl]
    stride = int(pos.max()) + 1 if len(tl) else 1
    buf = np.empty((len(tl), stride), dtype=np.float64)
    rc = lib().oracle_index_scores_batch(ctypes.byref(_dims(wl)), _p(wl.q_idx), _p(wl.q_scale), _p(wl.w),
                                         _p(wl.k_cache), _p(wl.k_scale), _p(wl.page_table), _p(wl.seq_lens),
                                         _p(wl.cu_q_lens), _p(tl), len(tl), stride, _p(buf))
    _check(rc)
    return [buf[i, : int(pos[i]) + 1] for i in range(len(tl))]


def indexer_topk(wl, tlist=None):
    """(topk int32 [nt, K] ascending with -1 padding, kth float64 [nt], nsel int32 [nt])."""
    tl, nt = _tl(tlist, wl.total_q)
    topk = np.empty((nt, wl.top_k), dtype=np.int32)
    kth = np.empty(nt, dtype=np.float64)
    nsel = np.empty(nt, dtype=np.int32)
    rc = lib().oracle_indexer_topk(ctypes.byref(_dims(wl)), _p(wl.q_idx), _p(wl.q_scale), _p(wl.w), _p(wl.k_cache),
                                   _p(wl.k_scale), _p(wl.page_table), _p(wl.seq_lens), _p(wl.cu_q_lens), _p(tl), nt,
                                   _p(topk), _p(kth), _p(nsel))
    _check(rc)
    return topk, kth, nsel


def sparse_attn(wl, topk, tlist=None, want_weights: bool = False):
    """(out float64 [nt, Hq, Dv], lse float64 [nt, Hq][, weights float64 [nt, Hq, K]])."""
    tl, nt = _tl(tlist, wl.total_q)
    topk = np.ascontiguousarray(topk, dtype=np.int32)
    assert topk.shape == (nt, wl.top_k)
    out = np.empty((nt, wl.attn_heads, wl.v_dim), dtype=np.float64)
    lse = np.empty((nt, wl.attn_heads), dtype=np.float64)
    wts = np.empty((nt, wl.attn_heads, wl.top_k), dtype=np.float64) if want_weights else None
    rc = lib().oracle_sparse_attn(ctypes.byref(_dims(wl)), _p(wl.q), _p(wl.kv_cache), _p(wl.page_table),
                                  _p(wl.seq_lens), _p(wl.cu_q_lens), _p(topk), _p(tl), nt, _p(out), _p(lse), _p(wts))
    _check(rc)
    return (out, lse, wts) if want_weights else (out, lse)


def e4m3_encode(y: float) -> int:
    """E4M3 code of the fp32 value y: nearest finite value, ties to the even code, saturating at 448."""
    return int(lib().oracle_e4m3_encode(float(y)))


def quantize_group(x) -> tuple:
    """(codes uint8 [n], scale float32) of one quantisation group: scale = absmax/448 (fp32), codes of x/scale."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.empty(x.shape[0], dtype=np.uint8)
    scale = np.empty(1, dtype=np.float32)
    lib().oracle_quantize_group(_p(x), int(x.shape[0]), _p(codes), _p(scale))
    return codes, np.float32(scale[0])


def append(wl, k_new=None, kv_new=None):
    """Copies of (k_cache, k_scale, kv_cache) after appending every query token's new rows at its position
    (k_new: bf16 bits [T, Di] or None; kv_new: bf16 bits [T, kv_dim] or None)."""
    k_cache = np.array(wl.k_cache, copy=True)
    k_scale = np.array(wl.k_scale, copy=True) if wl.k_scale is not None else None
    kv_cache = np.array(wl.kv_cache, copy=True) if wl.kv_cache is not None else None
    kn = np.ascontiguousarray(k_new, dtype=np.uint16) if k_new is not None else None
    kvn = np.ascontiguousarray(kv_new, dtype=np.uint16) if kv_new is not None else None
    if kn is not None:
        assert kn.shape == (wl.total_q, wl.idx_dim)
    if kvn is not None:
        assert kvn.shape == (wl.total_q, wl.kv_dim) and kv_cache is not None
    rc = lib().oracle_append_rows(ctypes.byref(_dims(wl)), _p(kn), _p(kvn), _p(wl.page_table), _p(wl.seq_lens),
                                  _p(wl.cu_q_lens), _p(k_cache), _p(k_scale), _p(kv_cache))
    _check(rc)
    return k_cache, k_scale, kv_cache


def e8m0_value(e: int) -> float:
    """OCP MX E8M0 scale byte: 2^(e - 127); 0xFF is NaN."""
    return float(lib().oracle_e8m0_value(e))


def set_threads(n: int) -> int:
    """Threads of the oracle's parallel loops from now on; returns the previous maximum."""
    return int(lib().oracle_set_threads(int(n)))
