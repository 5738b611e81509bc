"""Zigzag context-parallel prefill of the prefill chunk (4096 new tokens after 61440 cached ones) with the
ranks' device work run one after another on the one GPU ("Day0 Inference Support and Performance
Optimization for New LLM Architectures", section 5.2; "Optimizing Inference for Hybrid Attention
Architectures: From Operator Fusion to Sequence Sharding", section "Sequence Sharding and Load Balancing
in the Prefill Phase").

Rank r's share is its two segments as a batch of two sequences on the same page-table row, run through
the library's fused call; the outputs are put back in chunk order with the same function the
multi-process path uses after its all-gather (the exchange itself is covered on gloo ranks in
tests/test_cp_gloo.py).  The reassembled selection must equal the single-GPU call's bit for bit and the
attention must agree with it within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import sparse_attention_dsa_gb300 as dsa
from gen.workloads import config
from sparse_attention_dsa_gb300 import cp

from _gpu import ATOL, RTOL, DeviceWorkload, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


@pytest.fixture(scope="module")
def prefill():
    wl = config(4)
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    out, lse = dw.out_host()
    return wl, dw, dw.topk_host(), out, lse


@pytest.mark.parametrize("world", [2, 4])
def test_zigzag_ranks_reassemble_to_the_single_gpu_result(prefill, world):
    wl, dw, topk_ref, out_ref, lse_ref = prefill
    n_new = wl.total_q
    cached = int(wl.seq_lens[0]) - n_new
    ws_bytes = cp.zigzag_workspace_size(dw.dims, cached, n_new, world)
    backend = cp.CudaBackend()
    tk, oo, ll, loads = [], [], [], []
    for r in range(world):
        rb = cp.zigzag_rank_batch(cached, n_new, world, r)
        d_r = cp.zigzag_rank_dims(dw.dims, cached, n_new, world, r)
        sel = torch.as_tensor(rb.queries, device="cuda")
        T_r = int(rb.cu_q_lens[-1])
        topk = torch.empty((T_r, wl.top_k), dtype=torch.int32, device="cuda")
        out = torch.empty((T_r, wl.attn_heads, wl.v_dim), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((T_r, wl.attn_heads), dtype=torch.float32, device="cuda")
        ws = torch.zeros((ws_bytes + 3) // 4, dtype=torch.int32, device="cuda")
        backend.step(d_r, dw.q_idx[sel].contiguous(), None, dw.w[sel].contiguous(), dw.k_cache, None,
                     dw.q[sel].contiguous(), dw.kv_cache, dw.page_table.expand(2, -1).contiguous(),
                     torch.as_tensor(rb.seq_lens, device="cuda"), torch.as_tensor(rb.cu_q_lens, device="cuda"), topk,
                     out, lse, ws)
        assert dsa.get_device_error(ws) == 0
        tk.append(topk.cpu().numpy())
        oo.append(out.float().cpu().numpy())
        ll.append(lse.cpu().numpy())
        loads.append(cp.causal_work(cached, rb.queries))
    topk = cp.zigzag_reassemble(n_new, world, tk)
    out = cp.zigzag_reassemble(n_new, world, oo).astype(np.float64)
    lse = cp.zigzag_reassemble(n_new, world, ll).astype(np.float64)
    assert np.array_equal(topk, topk_ref)
    assert np.all(np.abs(out - out_ref) <= ATOL + RTOL * np.abs(out_ref))
    assert np.all(np.abs(lse - lse_ref) <= ATOL + RTOL * np.abs(lse_ref))
    assert max(loads) / min(loads) < 1.0001  # the Zigzag pairing balances the causal scoring work
