"""The C-ABI library builds, loads and exports every entry point of include/dsa.h; host-side validation
answers before any launch.  No GPU needed: nothing here reaches a kernel."""
import ctypes
import os
import re

import pytest

import sparse_attention_dsa_gb300 as dsa
from sparse_attention_dsa_gb300 import build as dsa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    dsa_build.build()
    return dsa.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dsa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/dsa.h but not exported"
    assert set(names) == set(dsa.EXPORTED)


def test_abi_version_and_status_strings(L):
    assert dsa.abi_version() == 4
    for s in range(6):
        assert dsa.status_string(s).startswith("DSA_")
    assert "unknown" in dsa.status_string(99)


def _dims(**kw):
    d = dict(batch=2, total_q=2, max_q_len=1, num_pages=8, page_size=64, max_pages_per_seq=4, idx_heads=64,
             idx_dim=128, idx_dtype=0, top_k=16, attn_heads=128, kv_dim=576, v_dim=512, softmax_scale=1 / 24)
    d.update(kw)
    return dsa.DsaDims(**d)


def test_workspace_size(L):
    assert dsa.workspace_size(_dims()) >= 256
    assert L.dsa_workspace_size(None) == 0
    # few query tokens and K = 2048: the attention may split positions and needs merge scratch
    # (137 KiB per CTA of the largest grid it may use)
    # (decode shapes, one query token per sequence: plus T x K int32 for the single-launch kernel's rows)
    rows = lambda T, K: (T * K * 4 + 15) // 16 * 16
    ws = dsa.workspace_size(_dims(top_k=2048))
    assert ws - 256 - rows(2, 2048) > 0 and (ws - 256 - rows(2, 2048)) % (136 * 256 * 4 + 256 * 4) == 0
    # one 64-row tile per query (K = 16), or many query tokens: no splits
    assert dsa.workspace_size(_dims(top_k=16)) == 256 + rows(2, 16)
    assert dsa.workspace_size(_dims(batch=4096, total_q=4096, top_k=2048)) == 256 + rows(4096, 2048)
    # several query tokens per sequence: no single-launch kernel, so no rows area
    assert dsa.workspace_size(_dims(max_q_len=2, total_q=4, top_k=16)) == 256


def test_fused_decode_launches_host_cases(L):
    assert L.dsa_fused_decode_launches(None) == -1
    assert dsa.fused_decode_launches(_dims(batch=2, total_q=0)) == 0


FAKE = 0x10000  # an aligned non-null value; validation rejects the call before it is ever dereferenced


def _indexer(d, **ptrs):
    p = dict(q_idx=FAKE, q_scale=None, w=FAKE, k_cache=FAKE, k_scale=None, page_table=FAKE, seq_lens=FAKE,
             cu_q_lens=FAKE, topk=FAKE, score=None, ws=FAKE)
    p.update(ptrs)
    return dsa.lib().dsa_indexer_topk(ctypes.byref(d) if d is not None else None, p["q_idx"], p["q_scale"], p["w"],
                                      p["k_cache"], p["k_scale"], p["page_table"], p["seq_lens"], p["cu_q_lens"],
                                      p["topk"], p["score"], p["ws"], None)


def _indexer_shard(d, begin, end, **ptrs):
    p = dict(q_idx=FAKE, q_scale=None, w=FAKE, k_cache=FAKE, k_scale=None, page_table=FAKE, seq_lens=FAKE,
             cu_q_lens=FAKE, topk=FAKE, score=FAKE, ws=FAKE)
    p.update(ptrs)
    return dsa.lib().dsa_indexer_topk_shard(ctypes.byref(d), p["q_idx"], p["q_scale"], p["w"], p["k_cache"],
                                            p["k_scale"], p["page_table"], p["seq_lens"], p["cu_q_lens"], begin, end,
                                            p["topk"], p["score"], p["ws"], None)


def _static(d, **ptrs):
    p = dict(q_idx=FAKE, q_scale=None, w=FAKE, k_cache=FAKE, k_scale=None, page_table=FAKE, seq_lens=FAKE,
             cu_q_lens=FAKE, topk=FAKE, score=None, err=None)
    p.update(ptrs)
    return dsa.lib().dsa_indexer_topk_static(ctypes.byref(d) if d is not None else None, p["q_idx"], p["q_scale"],
                                             p["w"], p["k_cache"], p["k_scale"], p["page_table"], p["seq_lens"],
                                             p["cu_q_lens"], p["topk"], p["score"], p["err"], None)


def _sfa(d, **ptrs):
    p = dict(q=FAKE, kv=FAKE, page_table=FAKE, seq_lens=FAKE, cu_q_lens=FAKE, topk=FAKE, out=FAKE, lse=None, ws=FAKE)
    p.update(ptrs)
    return dsa.lib().dsa_sparse_attn(ctypes.byref(d), p["q"], p["kv"], p["page_table"], p["seq_lens"],
                                     p["cu_q_lens"], p["topk"], p["out"], p["lse"], p["ws"], None)


def _msg():
    return dsa.lib().dsa_last_error_message().decode()


@pytest.mark.parametrize("field,value,status", [
    ("batch", 0, dsa.DSA_ERR_INVALID_ARG),
    ("total_q", -1, dsa.DSA_ERR_INVALID_ARG),
    ("max_q_len", 0, dsa.DSA_ERR_INVALID_ARG),
    ("num_pages", 0, dsa.DSA_ERR_INVALID_ARG),
    ("page_size", 32, dsa.DSA_ERR_UNSUPPORTED),
    ("page_size", -64, dsa.DSA_ERR_INVALID_ARG),
    ("max_pages_per_seq", 0, dsa.DSA_ERR_INVALID_ARG),
    ("top_k", 0, dsa.DSA_ERR_INVALID_ARG),
    ("top_k", 1 << 20, dsa.DSA_ERR_UNSUPPORTED),
])
def test_indexer_rejects_bad_dims(L, field, value, status):
    assert _indexer(_dims(**{field: value})) == status
    assert field.split("_")[0] in _msg() or "page_size" in _msg()


def test_indexer_rejects_null_and_misaligned_pointers(L):
    assert _indexer(None) == dsa.DSA_ERR_INVALID_ARG
    assert _indexer(_dims(), q_idx=None) == dsa.DSA_ERR_INVALID_ARG and "q_idx" in _msg()
    assert _indexer(_dims(), k_cache=FAKE + 4) == dsa.DSA_ERR_INVALID_ARG and "aligned" in _msg()
    assert _indexer(_dims(), ws=None) == dsa.DSA_ERR_INVALID_ARG and "workspace" in _msg()
    # FP8 needs both scale arrays
    assert _indexer(_dims(idx_dtype=1)) == dsa.DSA_ERR_INVALID_ARG and "scale" in _msg()
    assert _indexer(_dims(idx_dtype=7)) != dsa.DSA_OK


def test_sfa_rejects_bad_arguments(L):
    assert _sfa(_dims(kv_dim=512)) == dsa.DSA_ERR_UNSUPPORTED
    assert _sfa(_dims(v_dim=600)) == dsa.DSA_ERR_INVALID_ARG
    assert _sfa(_dims(attn_heads=0)) == dsa.DSA_ERR_INVALID_ARG
    assert _sfa(_dims(attn_heads=256)) == dsa.DSA_ERR_UNSUPPORTED
    assert _sfa(_dims(softmax_scale=0.0)) == dsa.DSA_ERR_INVALID_ARG
    assert _sfa(_dims(), out=None) == dsa.DSA_ERR_INVALID_ARG
    assert _sfa(_dims(), lse=FAKE + 8) == dsa.DSA_ERR_INVALID_ARG


def test_mxfp8_indexer_shape_limits(L):
    # MXFP8 needs both scale arrays, and serves 64 heads of 128 dims only
    assert _indexer(_dims(idx_dtype=2)) == dsa.DSA_ERR_INVALID_ARG and "scale" in _msg()
    assert _indexer(_dims(idx_dtype=2, idx_heads=4, idx_dim=64), q_scale=FAKE, k_scale=FAKE) == dsa.DSA_ERR_UNSUPPORTED
    assert "MXFP8" in _msg()
    assert _indexer(_dims(idx_dtype=3), q_scale=FAKE, k_scale=FAKE) == dsa.DSA_ERR_INVALID_ARG
    assert _append(_dims(idx_dtype=2), k_scale=FAKE) == dsa.DSA_ERR_UNSUPPORTED and "MXFP8" in _msg()


def test_sfa_rejects_an_unknown_kv_dtype(L):
    assert _sfa(_dims(kv_dtype=7)) == dsa.DSA_ERR_INVALID_ARG and "kv_dtype" in _msg()


def _append(d, **ptrs):
    p = dict(k_new=FAKE, kv_new=FAKE, page_table=FAKE, seq_lens=FAKE, cu_q_lens=FAKE, k_cache=FAKE, k_scale=None,
             kv_cache=FAKE, ws=FAKE)
    p.update(ptrs)
    return dsa.lib().dsa_append_rows(ctypes.byref(d) if d is not None else None, p["k_new"], p["kv_new"],
                                     p["page_table"], p["seq_lens"], p["cu_q_lens"], p["k_cache"], p["k_scale"],
                                     p["kv_cache"], p["ws"], None)


def test_append_rejects_bad_arguments(L):
    assert _append(None) == dsa.DSA_ERR_INVALID_ARG
    assert _append(_dims(idx_dim=129)) == dsa.DSA_ERR_UNSUPPORTED and "idx_dim" in _msg()
    assert _append(_dims(idx_dim=63)) == dsa.DSA_ERR_UNSUPPORTED
    assert _append(_dims(idx_dtype=1)) == dsa.DSA_ERR_INVALID_ARG and "k_scale" in _msg()  # FP8 keys need scales
    assert _append(_dims(kv_dtype=5)) == dsa.DSA_ERR_INVALID_ARG and "kv_dtype" in _msg()
    assert _append(_dims(kv_dim=512)) == dsa.DSA_ERR_UNSUPPORTED
    assert _append(_dims(), kv_cache=None) == dsa.DSA_ERR_INVALID_ARG and "kv_cache" in _msg()
    assert _append(_dims(), k_new=FAKE + 2) == dsa.DSA_ERR_INVALID_ARG and "aligned" in _msg()
    # a NULL new-row pointer skips that cache (and its checks); nothing to do returns before any launch
    assert _append(_dims(), k_new=None, kv_new=None, k_cache=None, kv_cache=None) == dsa.DSA_OK
    assert _append(_dims(total_q=0)) == dsa.DSA_OK


def test_indexer_topk_score_pointer_is_checked(L):
    assert _indexer(_dims(), score=FAKE + 4) == dsa.DSA_ERR_INVALID_ARG and "topk_score" in _msg()


@pytest.mark.parametrize("begin,end", [(-64, 128), (32, 4096), (128, 128), (256, 64)])
def test_indexer_shard_rejects_bad_ranges(L, begin, end):
    assert _indexer_shard(_dims(), begin, end) == dsa.DSA_ERR_INVALID_ARG and "range" in _msg()


def test_sfa_shard_rejects_bad_ranges(L):
    def call(begin, end):
        return L.dsa_sparse_attn_shard(ctypes.byref(_dims()), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, begin, end, FAKE,
                                       None, FAKE, None)
    assert call(-1, 10) == dsa.DSA_ERR_INVALID_ARG and "range" in _msg()
    assert call(64, 64) == dsa.DSA_ERR_INVALID_ARG


def test_merge_and_combine_validate(L):
    assert L.dsa_topk_merge(0, 4, 16, FAKE, FAKE, FAKE, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_topk_merge(2, 4, 16, FAKE, None, FAKE, None, None) == dsa.DSA_ERR_INVALID_ARG and "score" in _msg()
    assert L.dsa_topk_merge(2, 4, 16, FAKE, FAKE, FAKE + 4, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_topk_merge(8, 4, 4096, FAKE, FAKE, FAKE, None, None) == dsa.DSA_ERR_UNSUPPORTED
    assert L.dsa_attn_combine(2, 4, 128, 511, FAKE, FAKE, FAKE, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_attn_combine(0, 4, 128, 512, FAKE, FAKE, FAKE, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_attn_combine(2, 4, 128, 512, FAKE, FAKE, None, None, None) == dsa.DSA_ERR_INVALID_ARG


def test_static_entry_rejects_before_touching_the_device(L):
    """The allocation-free indexer checks its host arguments before it looks anything up or enqueues: a NULL
    dims and a misaligned device_error pointer are rejected with no device at all."""
    assert _static(None) == dsa.DSA_ERR_INVALID_ARG and "dims" in _msg()
    assert _static(_dims(), err=FAKE + 2) == dsa.DSA_ERR_INVALID_ARG and "device_error" in _msg()


def test_wait_limit_setter_round_trips(L):
    old = dsa.set_wait_limit_ns(1234)
    try:
        assert dsa.set_wait_limit_ns(0) == 1234  # 0 restores the default of one second
        assert dsa.set_wait_limit_ns(old) == 10 ** 9
    finally:
        dsa.set_wait_limit_ns(old)


def test_device_error_helpers_validate(L):
    code = ctypes.c_int32(0)
    assert L.dsa_get_device_error(None, None, ctypes.byref(code)) == dsa.DSA_ERR_INVALID_ARG
    assert L.dsa_clear_device_error(None, None) == dsa.DSA_ERR_INVALID_ARG
