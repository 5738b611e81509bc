"""dsa_indexer_topk_static: the allocation-free variant of the indexer, for callers that cannot allocate
device memory (its scratch lives in a static device array inside the library).  Checked against the
workspace entry point on the same inputs, two calls in a row, through the C ABI.  This file is collected
last on purpose: it must pass both alone in a fresh process and after every other test."""
import numpy as np
import pytest
import torch

import sparse_attention_dsa_gb300 as dsa
from gen.workloads import make_workload

from _gpu import DeviceWorkload, check_topk, ensure_built

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
