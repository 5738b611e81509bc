"""dsa_indexer_topk_static: the allocation-free variant of the indexer, for callers that cannot allocate
device memory (its scratch lives in a static device array inside the library).  Checked against the
workspace entry point on the same inputs, two calls in a row, through the C ABI.  This file is collected
last on purpose: it must pass both alone in a fresh process and after every other test."""
import numpy as np
import pytest
import torch

import sparse_attention_dsa_gb300 as dsa
from gen.workloads import make_workload

from _gpu import DeviceWorkload, check_topk, dims_for, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _static_call(dw, topk, err):
    dsa.indexer_topk_static(dw.dims, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table, dw.seq_lens,
                            dw.cu_q_lens, topk, err)
    torch.cuda.synchronize()
    return topk.cpu().numpy(), int(err.item())


@pytest.mark.parametrize("fp8", [False, True])
def test_static_scratch_matches_workspace_entry_two_calls(fp8):
    wl = make_workload("noalloc", 91, [5000, 777, 64], [1, 2, 1], idx_heads=64, idx_dim=128, idx_fp8=fp8,
                       top_k=512, attn_heads=128, with_sfa=False)
    dw = DeviceWorkload(wl).indexer()
    assert dw.error_word() == 0
    ref = dw.topk_host()
    for _ in range(2):
        topk = torch.full_like(dw.topk, -7)
        err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        got, code = _static_call(dw, topk, err)
        assert code == 0
        assert np.array_equal(got, ref)  # same kernels on the same inputs: identical selection
    check_topk(wl, ref)


def test_static_scratch_is_cleared_between_calls():
    wl = make_workload("noalloc", 92, [3000, 500], [1, 1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=64,
                       attn_heads=16, with_sfa=False)
    dw = DeviceWorkload(wl)
    good_pt = dw.page_table.clone()
    dw.page_table[0, 3] = 10 ** 6  # the first call sees a bad page id
    topk = torch.full_like(dw.topk, -7)
    err = torch.zeros((1,), dtype=torch.int32, device="cuda")
    _, code = _static_call(dw, topk, err)
    assert code & dsa.DSA_DEVERR_PAGE
    dw.page_table.copy_(good_pt)  # the second call is clean and must not inherit the old error
    got, code = _static_call(dw, topk, err)
    assert code == 0
    check_topk(wl, got)


def test_static_rejected_call_enqueues_nothing():
    """An argument the library rejects is reported before anything is put on the stream: the caller's
    device_error keeps its old value (a later clear of the scratch or copy of the word would change it)."""
    wl = make_workload("noalloc", 93, [2000], [1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=128,
                       attn_heads=128, with_sfa=False)
    dw = DeviceWorkload(wl)
    err = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    d = dims_for(wl, idx_heads=48)  # no kernel variant
    with pytest.raises(dsa.DsaError) as e:
        dsa.indexer_topk_static(d, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table, dw.seq_lens,
                                dw.cu_q_lens, dw.topk, err)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    with pytest.raises(dsa.DsaError) as e:
        dsa.indexer_topk_static(dw.dims, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table,
                                dw.seq_lens, dw.cu_q_lens, None, err)
    assert e.value.status == dsa.DSA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(err.item()) == 12345


def test_static_edge_calls():
    """No query token: nothing launches and the reported word is 0.  device_error NULL: the word is
    discarded and the selection is still written.  topk_score: the same scores as the workspace call."""
    wl = make_workload("noalloc", 94, [4000, 300], [1, 1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=256,
                       attn_heads=128, with_sfa=False)
    dw = DeviceWorkload(wl)
    ref_score = torch.empty((wl.total_q, wl.top_k), dtype=torch.float32, device="cuda")
    dsa.indexer_topk(dw.dims, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table, dw.seq_lens,
                     dw.cu_q_lens, dw.topk, dw.workspace, topk_score=ref_score)
    ref = dw.topk_host()
    err = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    d = dims_for(wl, total_q=0)
    topk = torch.full_like(dw.topk, -7)
    dsa.indexer_topk_static(d, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table, dw.seq_lens,
                            dw.cu_q_lens, topk, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and bool((topk == -7).all())
    score = torch.empty_like(ref_score)
    dsa.indexer_topk_static(dw.dims, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table, dw.seq_lens,
                            dw.cu_q_lens, topk, None, topk_score=score)
    torch.cuda.synchronize()
    assert np.array_equal(topk.cpu().numpy(), ref)
    assert torch.equal(score, ref_score)
