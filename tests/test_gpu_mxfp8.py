"""GPU parity for the MXFP8 indexer (E4M3 codes, one E8M0 scale per 32 elements of q_idx and k_idx rows):
the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs, with the Top-K and
attention criteria of test_gpu_parity.  The kernel dequantises both operands to bf16 (a code times a power
of two, exact in bf16) before the tensor-core products; the oracle takes every element as code x scale."""
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


CASES = {
    # name: (seq_lens, q_lens, K, Hq, kv_fp8, extra)
    "one_query": ([5000, 2049, 130, 1], [1, 1, 1, 1], 512, 128, False, {}),
    "two_queries": ([3000, 700, 2], [2, 2, 2], 256, 128, False, {}),
    "salient_kv_fp8": ([4100, 8192], [1, 1], 2048, 128, True, dict(w_hi=0.125, salient_frac=0.01)),
    "fewer_than_k": ([100, 257, 3000], [1, 1, 1], 256, 16, False, {}),
}


def _wl(name, seed=55):
    lens, qls, k, hq, kv8, extra = CASES[name]
    return make_workload(name, seed, lens, qls, idx_heads=64, idx_dim=128, idx_fp8=True, idx_mx=True, top_k=k,
                         attn_heads=hq, kv_fp8=kv8, **extra)


@pytest.mark.parametrize("name", list(CASES))
def test_mxfp8_fused_matches_oracle(name):
    wl = _wl(name)
    assert wl.q_scale.dtype == np.uint8 and wl.k_scale.shape[-1] == 4
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


def test_mxfp8_standalone_indexer_matches_single_launch():
    wl = _wl("one_query")
    dw = DeviceWorkload(wl)
    assert dsa.fused_decode_launches(dw.dims) == 1
    dw.fused()
    topk1 = dw.topk_host().copy()
    dw.indexer()
    assert dw.error_word() == 0
    assert np.array_equal(dw.topk_host(), topk1)


def test_mxfp8_decode_32k_context_sampled():
    """The bench workload shape (32K context, K = 2048, salient rows) with MXFP8 indexer inputs, 8 sequences."""
    wl = make_workload("mx32k", 1002, [32768] * 8, [1] * 8, idx_heads=64, idx_dim=128, idx_fp8=True, idx_mx=True,
                       top_k=2048, attn_heads=128, w_hi=0.125, salient_frac=0.01)
    dw = DeviceWorkload(wl)
    assert dsa.fused_decode_launches(dw.dims) == 1
    dw.fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk, [0, 4, 7])
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse, [0, 7])


def test_mxfp8_subnormal_codes_and_extreme_scales():
    """Keys whose codes are all E4M3 subnormals under a scale of 2^30, and keys whose scale bytes are
    160..170 (factors beyond the bf16 range of a single product in the kernel's dequantisation), outrank
    every ordinary key by orders of magnitude: the Top-K holds all of them only if the kernel keeps
    subnormal codes and large scales exact.  The selection is checked against the oracle in full."""
    wl = make_workload("mx_extreme", 77, [300, 1000], [1, 1], idx_heads=64, idx_dim=128, idx_fp8=True,
                       idx_mx=True, top_k=64, attn_heads=16)
    rng = np.random.default_rng(5)
    special = []
    for b in range(wl.batch):
        L = int(wl.seq_lens[b])
        for j, pos in enumerate(rng.choice(L, 40, replace=False)):
            pg, r = int(wl.page_table[b, pos // 64]), int(pos % 64)
            if j < 20:  # codes 0x01..0x07 with random signs
                wl.k_cache[pg, r] = (rng.integers(1, 8, 128) | (rng.integers(0, 2, 128) << 7)).astype(np.uint8)
                wl.k_scale[pg, r] = 127 + 30
            else:
                wl.k_scale[pg, r] = rng.integers(160, 171, 4).astype(np.uint8)
            special.append((b, int(pos)))
    dw = DeviceWorkload(wl)
    dw.indexer()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    for b, pos in special:
        assert pos in set(topk[b].tolist()), f"sequence {b}: position {pos} not selected"
