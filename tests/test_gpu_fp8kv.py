"""GPU parity for the FP8 latent-KV cache and for appending a step's rows to the paged caches: the CUDA
path (through the C ABI) against the CPU oracle on the same seeded inputs.

FP8 latent-KV rows: Top-K exactly as in test_gpu_parity (the indexer does not read the latent-KV cache);
attention |gpu - oracle| <= 2e-2 + 1e-2 * |oracle| elementwise, the oracle taking every element as code x
scale exactly and the kernel rounding it to bf16 before the tensor-core products.
Appending: every cache byte and scale bit-exact (both sides quantise in fp32 with correctly rounded
divisions and nearest-even E4M3 rounding, so they take the same integer decisions).
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_dsa_gb300 as dsa
from gen.workloads import config, make_workload

from _gpu import DeviceWorkload, _dev, check_attention, check_topk, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


CASES = {
    # name: (seq_lens, q_lens, idx_fp8, K, Hq)
    "one_query": ([5000, 2049, 130, 1], [1, 1, 1, 1], False, 512, 128),
    "two_queries": ([3000, 700, 2], [2, 2, 2], False, 512, 128),
    "fp8_indexer_too": ([4100, 190, 1], [1, 2, 1], True, 256, 128),
    "few_heads_ragged": ([300, 1000, 64, 129], [1, 2, 1, 4], False, 64, 16),
}


def _wl(name, seed=91, kv_fp8=True, **kw):
    lens, qls, idx8, k, hq = CASES[name]
    return make_workload(name, seed, lens, qls, idx_heads=64, idx_dim=128, idx_fp8=idx8, top_k=k, attn_heads=hq,
                         kv_fp8=kv_fp8, **kw)


@pytest.mark.parametrize("name", list(CASES))
def test_fp8_kv_fused_matches_oracle(name):
    wl = _wl(name)
    assert wl.kv_cache.dtype == np.uint8 and wl.kv_cache.shape[-1] == dsa.DSA_KV_FP8_ROW_BYTES
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


def test_fp8_kv_takes_the_single_launch_and_matches_two_launches():
    wl = _wl("one_query")
    dw = DeviceWorkload(wl)
    assert dsa.fused_decode_launches(dw.dims) == 1
    dw.fused()
    topk1 = dw.topk_host().copy()
    out1, lse1 = dw.out_host()
    dw.indexer()
    dw.sfa()
    assert dw.error_word() == 0
    assert np.array_equal(dw.topk_host(), topk1)
    out2, lse2 = dw.out_host()
    np.testing.assert_allclose(out1, out2, rtol=0, atol=1e-2)
    np.testing.assert_allclose(lse1, lse2, rtol=0, atol=1e-5)


def test_fp8_kv_attention_on_oracle_selection_in_any_order():
    wl = _wl("two_queries")
    ref, _, _ = oracle.indexer_topk(wl)
    rng = np.random.default_rng(4)
    sel = np.stack([rng.permutation(r) for r in ref]).astype(np.int32)
    dw = DeviceWorkload(wl)
    dw.sfa(topk=torch.from_numpy(sel).cuda())
    assert dw.error_word() == 0
    out, lse = dw.out_host()
    check_attention(wl, sel, out, lse)


def test_fp8_kv_decode_32k_context_sampled():
    """The bench workload shape (32K context, K = 2048, 128 heads) with the FP8 latent-KV cache, on 8 of
    its sequences: full Top-K parity on every token, attention on a sample of tokens."""
    wl = config(2, batch=8, kv_fp8=True)
    dw = DeviceWorkload(wl)
    assert dsa.fused_decode_launches(dw.dims) == 1
    dw.fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk, [0, 3, 7])
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse, [0, 3, 7])


def _new_rows(wl, seed, spread=True):
    """Seeded new rows for every query token: normal values (at magnitudes 2^-6 .. 2^6 when `spread`),
    one all-zero key row, one all-zero latent tile, and a row whose values sit exactly at a quantisation
    tie."""
    rng = np.random.default_rng(seed)
    T = wl.total_q
    mags = np.float32(2.0) ** rng.integers(-6, 7, (T, 1)).astype(np.float32)
    if not spread:
        mags[:] = 1.0
    k = (rng.normal(0, 1, (T, wl.idx_dim)).astype(np.float32) * mags)
    kv = (rng.normal(0, 1, (T, wl.kv_dim)).astype(np.float32) * mags)
    k[0] = 0.0
    kv[min(1, T - 1), 128:256] = 0.0
    if T > 2:  # absmax 448 -> scale 1; 1.0625 lies halfway between the E4M3 values 1 and 1.125
        k[2, :] = 1.0625
        k[2, 0] = 448.0
    to_bf16 = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)  # truncation: exact bf16 values
    return to_bf16(k), to_bf16(kv)


@pytest.mark.parametrize("idx8,kv8", [(False, False), (True, True), (False, True), (True, False)])
def test_append_matches_oracle_bit_exactly(idx8, kv8):
    wl = make_workload("append", 5, [300, 129, 64, 1, 2000], [1, 3, 2, 1, 4], idx_heads=64, idx_dim=128,
                       idx_fp8=idx8, top_k=64, attn_heads=16, kv_fp8=kv8)
    k_new, kv_new = _new_rows(wl, 17 + 2 * idx8 + kv8)
    ref_k, ref_ks, ref_kv = oracle.append(wl, k_new, kv_new)
    dw = DeviceWorkload(wl)
    dsa.append_rows(dw.dims, _dev(k_new), _dev(kv_new), dw.page_table, dw.seq_lens, dw.cu_q_lens, dw.k_cache,
                    dw.k_scale, dw.kv_cache, dw.workspace)
    assert dw.error_word() == 0
    got_k = dw.k_cache.cpu().numpy().view(ref_k.dtype)
    got_kv = dw.kv_cache.cpu().numpy().view(ref_kv.dtype)
    assert np.array_equal(got_k, ref_k)
    assert np.array_equal(got_kv, ref_kv)
    if idx8:
        assert np.array_equal(dw.k_scale.cpu().numpy().view(np.uint32), ref_ks.view(np.uint32))


def test_append_then_fused_decode_matches_oracle():
    """One decode step end to end: the step's rows are appended (FP8 caches), then the fused call runs on
    the updated caches; both against the oracle doing the same two steps.  The new rows are N(0,1), the
    scale the attention tolerance is set for (larger values scale the kernel's bf16 rounding of the
    dequantised rows with them)."""
    wl = make_workload("step", 8, [5000, 2049, 130], [1, 1, 1], idx_heads=64, idx_dim=128, idx_fp8=True,
                       top_k=512, attn_heads=128, kv_fp8=True)
    k_new, kv_new = _new_rows(wl, 23, spread=False)
    wl.k_cache, wl.k_scale, wl.kv_cache = oracle.append(wl, k_new, kv_new)
    wl0 = make_workload("step", 8, [5000, 2049, 130], [1, 1, 1], idx_heads=64, idx_dim=128, idx_fp8=True,
                        top_k=512, attn_heads=128, kv_fp8=True)
    dw = DeviceWorkload(wl0)  # the caches before the step
    dsa.append_rows(dw.dims, _dev(k_new), _dev(kv_new), dw.page_table, dw.seq_lens, dw.cu_q_lens, dw.k_cache,
                    dw.k_scale, dw.kv_cache, dw.workspace)
    dw.fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


def test_append_with_a_bad_page_sets_the_error_and_writes_nothing():
    wl = make_workload("append", 5, [300, 129], [1, 1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=64,
                       attn_heads=16)
    k_new, kv_new = _new_rows(wl, 3)
    pt = wl.page_table.copy()
    pt[1, (129 - 1) // 64] = wl.num_pages + 5  # the second token's page is out of range
    dw = DeviceWorkload(wl)
    dw.page_table = _dev(pt)
    before_k, before_kv = dw.k_cache.clone(), dw.kv_cache.clone()
    dsa.append_rows(dw.dims, _dev(k_new), _dev(kv_new), dw.page_table, dw.seq_lens, dw.cu_q_lens, dw.k_cache,
                    dw.k_scale, dw.kv_cache, dw.workspace)
    assert dw.error_word() & dsa.DSA_DEVERR_PAGE
    # the first token's rows were written, the second token's were not
    b0 = int(wl.page_table[0, 299 // 64])
    assert np.array_equal(dw.k_cache.cpu().numpy().view(np.uint16)[b0, 299 % 64], k_new[0])
    changed = (dw.kv_cache != before_kv).reshape(dw.kv_cache.shape[0] * 64, -1).any(dim=1).sum().item()
    assert changed == 1
    changed_k = (dw.k_cache != before_k).reshape(dw.k_cache.shape[0] * 64, -1).any(dim=1).sum().item()
    assert changed_k == 1
