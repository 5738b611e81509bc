"""Failure detection without faulting the GPU: bad inputs are planted on the host, the kernels' own
bounds checks turn them into bits of the device error word, the affected work is skipped, the rest of
the batch stays correct and the context stays usable."""
import numpy as np
import pytest
import torch

import sparse_attention_dsa_gb300 as dsa
from gen.workloads import make_workload

from _gpu import DeviceWorkload, check_attention, check_topk, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _wl(**kw):
    return make_workload("faults", 31, [3000, 500], [1, 1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=256,
                         attn_heads=128, **kw)


@pytest.mark.parametrize("bad", [10 ** 6, -5])
def test_out_of_range_page_id_is_reported_and_skipped(bad):
    wl = _wl()
    wl.page_table[0, 5] = bad  # a page sequence 0 needs
    dw = DeviceWorkload(wl).fused()
    code = dw.error_word()
    assert code & dsa.DSA_DEVERR_PAGE
    topk = dw.topk_host()
    check_topk(wl, topk, [1])  # the other sequence is untouched
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse, [1])
    # the selection of sequence 0 never names a position on the bad page
    sel = topk[0][topk[0] >= 0]
    assert not np.any(sel // 64 == 5)


def test_inconsistent_lengths_are_reported():
    wl = _wl()
    dw = DeviceWorkload(wl)
    dw.seq_lens[0] = wl.max_pages_per_seq * 64 + 1  # longer than its page-table row
    dw.fused()
    assert dw.error_word() & dsa.DSA_DEVERR_SEQ
    check_topk(wl, dw.topk_host(), [1])


def test_more_queries_than_cached_tokens_is_reported():
    wl = make_workload("faults", 32, [40, 300], [2, 1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=16,
                       attn_heads=16)
    dw = DeviceWorkload(wl)
    dw.seq_lens[0] = 1  # two query tokens but only one cached token
    dw.fused()
    assert dw.error_word() & dsa.DSA_DEVERR_SEQ
    check_topk(wl, dw.topk_host(), [2])


def test_topk_entry_beyond_causal_limit_is_reported_and_skipped():
    wl = _wl()
    dw = DeviceWorkload(wl).indexer()
    topk = dw.topk_host()
    bad = topk.copy()
    bad[0, 3] = wl.query_positions()[0] + 10
    dw.sfa(topk=torch.from_numpy(bad).cuda())
    assert dw.error_word() & dsa.DSA_DEVERR_INDEX
    cleaned = bad.copy()
    cleaned[0, 3] = -1
    out, lse = dw.out_host()
    check_attention(wl, cleaned, out, lse)


def test_clear_and_recover():
    wl = _wl()
    wl.page_table[1, 2] = -3
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() != 0
    dsa.clear_device_error(dw.workspace)
    assert dw.error_word() == 0
    good = _wl()
    dg = DeviceWorkload(good).fused()
    assert dg.error_word() == 0
    topk = dg.topk_host()
    check_topk(good, topk)
    out, lse = dg.out_host()
    check_attention(good, topk, out, lse)


def test_unsupported_shape_is_rejected_before_launch():
    wl = _wl()
    dw = DeviceWorkload(wl)
    d = dw.dims
    d.idx_heads = 48
    with pytest.raises(dsa.DsaError) as e:
        dw.indexer(dims=d)
    assert e.value.status == dsa.DSA_ERR_UNSUPPORTED
    assert dw.error_word() == 0
