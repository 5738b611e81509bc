"""Failure detection of the bounded device waits, without faulting or hanging the GPU.

With the pipeline-wait limit cut to a few hundred nanoseconds (dsa_set_wait_limit_ns), correct launches
have waits that run out: the kernels must set DSA_DEVERR_TIMEOUT, abandon their pipelines, still drain
their copies in flight and free their tensor memory (under the default limit), and return.  The host sees
DSA_ERR_TIMEOUT from dsa_get_device_error, the context stays usable, and once the default limit is back a
clean call on the same context is correct.  (No counterpart in the articles: this is the library's own
failure detection.)"""
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


@pytest.fixture
def short_waits():
    old = dsa.set_wait_limit_ns(200)
    try:
        yield
    finally:
        dsa.set_wait_limit_ns(old if old else 0)


CASES = {
    # one query token per sequence, 64 x 128 indexer: the single-launch decode kernel
    "single_launch": dict(lens=[5000, 3000], qls=[1, 1], hi=64, di=128, K=512, fp8=False),
    # several query tokens per sequence: the indexer, then the attention kernel (position splits merged)
    "two_kernels": dict(lens=[4000, 700], qls=[2, 3], hi=64, di=128, K=256, fp8=False),
    "fp8_keys": dict(lens=[6000], qls=[1], hi=64, di=128, K=1024, fp8=True),
}


def _wl(c, seed=61):
    return make_workload("timeout", seed, c["lens"], c["qls"], idx_heads=c["hi"], idx_dim=c["di"], idx_fp8=c["fp8"],
                         top_k=c["K"], attn_heads=128)


@pytest.mark.parametrize("name", list(CASES))
def test_short_wait_limit_reports_timeout_and_recovers(name, short_waits):
    c = CASES[name]
    wl = _wl(c)
    dw = DeviceWorkload(wl)
    dw.fused()
    torch.cuda.synchronize()  # the kernels returned: no hang, no fault
    code = dsa.get_device_error(dw.workspace)
    assert code & dsa.DSA_DEVERR_TIMEOUT, f"error word {code:#x}"
    status = dsa.lib().dsa_get_device_error(dw.workspace.data_ptr(), torch.cuda.current_stream().cuda_stream,
                                            __import__("ctypes").byref(__import__("ctypes").c_int32()))
    assert status == dsa.DSA_ERR_TIMEOUT
    # the standalone kernels take the same path
    dsa.clear_device_error(dw.workspace)
    dw.indexer()
    dw.sfa()
    torch.cuda.synchronize()
    assert dsa.get_device_error(dw.workspace) & dsa.DSA_DEVERR_TIMEOUT
    # back to the default limit: a clean call on the same context and workspace is correct
    dsa.set_wait_limit_ns(0)
    dsa.clear_device_error(dw.workspace)
    dw.fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)
