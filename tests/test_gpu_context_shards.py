"""Decode by context shards on one GPU ("Day0 Inference Support and Performance Optimization for New LLM
Architectures", section 5.1): every shard scores only its own positions and keeps a local Top-K of
(score, position); the shards' lists are merged with the same key; every shard attends over the selected
rows it holds and the partial (out, lse) are combined.  The shards run one after the other on the one
GPU, each with a page table that names only its own pages (every other entry is out of range, so a
read of one would set DSA_DEVERR_PAGE).

The merged selection must equal the unsharded call's bit for bit (positions and scores: the score of a
position does not depend on the range it is scored in), and the combined attention must match the
oracle on that selection within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import sparse_attention_dsa_gb300 as dsa
from gen.workloads import make_workload

from _gpu import DeviceWorkload, check_attention, check_topk, ensure_built

pytestmark = pytest.mark.gpu

BIG = 2 ** 31 - 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _ranges(max_ctx, n):
    """n contiguous page-aligned shards of [0, max_ctx); the last one open-ended."""
    per = -(-max_ctx // n)
    per = -(-per // 64) * 64
    return [(i * per, (i + 1) * per if i + 1 < n else BIG) for i in range(n)]


def _shard_table(pt, lo, hi):
    t = pt.clone()
    lp = torch.arange(pt.shape[1], device=pt.device)
    outside = (lp * 64 + 63 < lo) | (lp * 64 >= hi)
    t[:, outside] = 10 ** 6  # never read by a shard-restricted call
    return t


CASES = {
    "bf16_decode": dict(lens=[9000, 20000, 3000, 12345], qls=[1, 1, 1, 1], fp8=False, K=2048),
    "fp8_decode": dict(lens=[16384, 7000], qls=[1, 1], fp8=True, K=1024),
    "two_queries": dict(lens=[10000, 5000], qls=[2, 2], fp8=False, K=512),
}


@pytest.mark.parametrize("shards", [2, 3])
@pytest.mark.parametrize("name", list(CASES))
def test_sharded_decode_equals_unsharded(name, shards):
    c = CASES[name]
    wl = make_workload("cp", 71, c["lens"], c["qls"], idx_heads=64, idx_dim=128, idx_fp8=c["fp8"], top_k=c["K"],
                       attn_heads=128, w_hi=0.125, salient_frac=0.01)
    dw = DeviceWorkload(wl)
    T, K = wl.total_q, wl.top_k
    ref_idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    ref_score = torch.empty((T, K), dtype=torch.float32, device="cuda")
    dsa.indexer_topk(dw.dims, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table, dw.seq_lens,
                     dw.cu_q_lens, ref_idx, dw.workspace, topk_score=ref_score)
    assert dw.error_word() == 0
    rng = _ranges(wl.max_pages_per_seq * 64, shards)
    idx = torch.empty((shards, T, K), dtype=torch.int32, device="cuda")
    score = torch.empty((shards, T, K), dtype=torch.float32, device="cuda")
    for s, (lo, hi) in enumerate(rng):
        dsa.indexer_topk_shard(dw.dims, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale,
                               _shard_table(dw.page_table, lo, hi), dw.seq_lens, dw.cu_q_lens, lo, hi, idx[s],
                               score[s], dw.workspace)
    assert dw.error_word() == 0, "a shard read a page outside its range"
    # each shard's list: its own positions only, ascending, scores consistent with the full call
    for s, (lo, hi) in enumerate(rng):
        v = idx[s].cpu().numpy()
        ok = v >= 0
        assert np.all((v[ok] >= lo) & (v[ok] < hi))
    merged = torch.empty((T, K), dtype=torch.int32, device="cuda")
    merged_score = torch.empty((T, K), dtype=torch.float32, device="cuda")
    dsa.topk_merge(shards, T, K, idx, score, merged, merged_score)
    torch.cuda.synchronize()
    assert torch.equal(merged, ref_idx), "merged shard selection differs from the unsharded one"
    assert torch.equal(merged_score, ref_score)
    check_topk(wl, merged.cpu().numpy())
    # attention: per-shard partials, combined
    outs = torch.empty((shards, T, wl.attn_heads, wl.v_dim), dtype=torch.bfloat16, device="cuda")
    lses = torch.empty((shards, T, wl.attn_heads), dtype=torch.float32, device="cuda")
    for s, (lo, hi) in enumerate(rng):
        dsa.sparse_attn_shard(dw.dims, dw.q, dw.kv_cache, _shard_table(dw.page_table, lo, hi), dw.seq_lens,
                              dw.cu_q_lens, merged, lo, hi, outs[s], lses[s], dw.workspace)
    assert dw.error_word() == 0
    dsa.attn_combine(shards, T, wl.attn_heads, wl.v_dim, outs, lses, dw.out, dw.lse)
    out, lse = dw.out_host()
    check_attention(wl, merged.cpu().numpy(), out, lse)


def test_topk_scores_are_the_index_scores():
    """topk_score holds I[t, s] of each selected position (fp32 accumulation against the float64 oracle)
    and -inf on padding."""
    wl = make_workload("cp", 72, [3000, 100], [1, 1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=256,
                       attn_heads=128)
    dw = DeviceWorkload(wl)
    sc = torch.empty((wl.total_q, wl.top_k), dtype=torch.float32, device="cuda")
    dsa.indexer_topk(dw.dims, dw.q_idx, dw.q_scale, dw.w, dw.k_cache, dw.k_scale, dw.page_table, dw.seq_lens,
                     dw.cu_q_lens, dw.topk, dw.workspace, topk_score=sc)
    topk, sc = dw.topk_host(), sc.cpu().numpy()
    for t in range(wl.total_q):
        ref = oracle.index_scores(wl, t)
        sel = topk[t] >= 0
        np.testing.assert_allclose(sc[t][sel], ref[topk[t][sel]], rtol=1e-4, atol=1e-5)
        assert np.all(np.isneginf(sc[t][~sel]))


def test_merge_orders_ties_by_position():
    """Equal scores across shards: the lower position wins, and the output is ascending."""
    T, K = 2, 4
    idx = torch.tensor([[[0, 1, 2, 3], [4, 5, -1, -1]], [[10, 11, 12, 13], [20, 21, 22, 23]]],
                       dtype=torch.int32, device="cuda")
    score = torch.tensor([[[1.0, 2.0, 2.0, 0.5], [2.0, 3.0, -np.inf, -np.inf]],
                          [[7.0, 7.0, 7.0, 7.0], [7.0, 7.0, 9.0, 7.0]]], dtype=torch.float32, device="cuda")
    out = torch.empty((T, K), dtype=torch.int32, device="cuda")
    out_s = torch.empty((T, K), dtype=torch.float32, device="cuda")
    # shard-major input: [shards, T, K]
    dsa.topk_merge(2, T, K, idx.transpose(0, 1).contiguous(), score.transpose(0, 1).contiguous(), out, out_s)
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [[1, 2, 4, 5], [10, 11, 12, 22]]
    assert out_s.cpu().tolist() == [[2.0, 2.0, 2.0, 3.0], [7.0, 7.0, 7.0, 9.0]]


def test_combine_of_disjoint_halves_equals_whole():
    """Attention over a selection equals the log-sum-exp combine of the attention over its two halves."""
    wl = make_workload("cp", 73, [5000, 2500], [1, 1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=1024,
                       attn_heads=128)
    dw = DeviceWorkload(wl).indexer()
    T = wl.total_q
    outs = torch.empty((2, T, wl.attn_heads, wl.v_dim), dtype=torch.bfloat16, device="cuda")
    lses = torch.empty((2, T, wl.attn_heads), dtype=torch.float32, device="cuda")
    for s, (lo, hi) in enumerate([(0, 1500), (1500, BIG)]):
        dsa.sparse_attn_shard(dw.dims, dw.q, dw.kv_cache, dw.page_table, dw.seq_lens, dw.cu_q_lens, dw.topk, lo, hi,
                              outs[s], lses[s], dw.workspace)
    dsa.attn_combine(2, T, wl.attn_heads, wl.v_dim, outs, lses, dw.out, dw.lse)
    assert dw.error_word() == 0
    out, lse = dw.out_host()
    check_attention(wl, dw.topk_host(), out, lse)
