"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same seeded inputs.

Top-K: the selected sets must match exactly, except positions whose oracle score lies within 1e-3
(relative) of the K-th score, which may be swapped; the count, ordering and -1 padding are exact.
Attention: |gpu - oracle| <= 2e-2 + 1e-2 * |oracle| elementwise, evaluated on the GPU's own selection
(so that excused swaps do not leak into the output comparison).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_dsa_gb300 as dsa
from gen import bf16_to_f32, f32_to_bf16
from gen.workloads import config, make_workload

from _gpu import DeviceWorkload, check_attention, check_topk, dims_for, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


SMALL = {
    # name: (seq_lens, q_lens, Hi, Di, fp8, K, Hq, extra)
    "hi4_ragged": ([300, 1000, 64, 1, 129, 4096], [1, 2, 1, 1, 4, 3], 4, 64, False, 64, 16, {}),
    "hi4_fewer_than_k": ([100, 257, 256, 3000], [1, 1, 1, 1], 4, 64, False, 256, 16, {}),
    "hi64_bf16": ([5000, 2049, 130, 1], [1, 1, 1, 1], 64, 128, False, 512, 128, {}),
    "hi64_bf16_two_queries": ([3000, 700, 2], [2, 2, 2], 64, 128, False, 512, 128, {}),
    "hi64_bf16_prefill_block": ([2000], [37], 64, 128, False, 256, 128, {}),
    "hi64_fp8": ([5000, 190, 1], [1, 2, 1], 64, 128, True, 256, 128, {}),
    "hi64_salient": ([4100, 8192], [1, 1], 64, 128, False, 2048, 128, dict(w_hi=0.125, salient_frac=0.01)),
    "k_equals_one": ([700, 64], [1, 1], 64, 128, False, 1, 32, {}),
    # 32 query tokens: the attention splits each token's positions in two (the two-split merge path)
    "thirty_two_tokens": ([700 + 97 * i for i in range(32)], [1] * 32, 64, 128, False, 512, 128, {}),
    # the largest supported K (4096): one query per sequence (single launch), and FP8 keys with two
    # queries in a sequence (two launches); contexts below, just above and well above K
    "k_max_decode": ([9000, 4100, 3000], [1, 1, 1], 64, 128, False, 4096, 128, {}),
    "k_max_fp8_two_queries": ([9000, 4097], [2, 1], 64, 128, True, 4096, 128, {}),
}


def _small(name, seed=77, **kw):
    lens, qls, hi, di, fp8, k, hq, extra = SMALL[name]
    extra = dict(extra, **kw)
    return make_workload(name, seed, lens, qls, idx_heads=hi, idx_dim=di, idx_fp8=fp8, top_k=k, attn_heads=hq,
                         **extra)


@pytest.mark.parametrize("name", list(SMALL))
def test_fused_small(name):
    wl = _small(name)
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


@pytest.mark.parametrize("name", ["hi4_ragged", "hi64_bf16_two_queries", "hi64_fp8"])
def test_attention_on_oracle_selection_in_any_order(name):
    wl = _small(name)
    ref, _, _ = oracle.indexer_topk(wl)
    shuffled = np.ascontiguousarray(ref[:, ::-1])  # -1 entries first, positions descending
    dw = DeviceWorkload(wl)
    dw.sfa(topk=torch.from_numpy(shuffled).cuda())
    assert dw.error_word() == 0
    out, lse = dw.out_host()
    check_attention(wl, shuffled, out, lse)


def test_no_query_tokens_launches_nothing():
    """total_q = 0: every compute entry point returns OK, writes nothing and sets no device error."""
    wl = _small("hi64_bf16")
    dw = DeviceWorkload(wl)
    d = dims_for(wl, total_q=0)
    dw.topk.fill_(-7)
    dw.out.fill_(3)
    assert dsa.fused_decode_launches(d) == 0
    dw.fused(dims=d)
    dw.indexer(dims=d)
    dw.sfa(topk=dw.topk, dims=d)
    torch.cuda.synchronize()
    assert dw.error_word() == 0
    assert bool((dw.topk == -7).all()) and bool((dw.out == 3).all())


def test_attention_covering_whole_context_equals_dense():
    """K >= context: the selection is every visible row and the result is dense causal attention."""
    wl = make_workload("dense", 5, [200, 77], [2, 1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=256,
                       attn_heads=16)
    dw = DeviceWorkload(wl).fused()
    topk = dw.topk_host()
    pos = wl.query_positions()
    for t in range(wl.total_q):
        assert topk[t, : pos[t] + 1].tolist() == list(range(pos[t] + 1))
        assert np.all(topk[t, pos[t] + 1:] == -1)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


def test_hand_example_on_device():
    """The 3-position toy (scores 1.5, 2.0, 1.5; the tie at 1.5 goes to position 0) embedded in the
    smallest supported shape: 4 indexer heads of 64 dims, two of them with zero weight."""
    wl = make_workload("toy", 1, [3], [1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=2, attn_heads=16)
    q = np.zeros((1, 4, 64), np.float32)
    q[0, 0, 0] = 1
    q[0, 1, 1] = 1
    k = np.zeros((3, 64), np.float32)
    k[:, :2] = [[1, 1], [2, -1], [-1, 3]]
    wl.q_idx[:] = f32_to_bf16(q)
    pg = wl.page_table[0, 0]
    wl.k_cache[pg, :3] = f32_to_bf16(k)
    wl.w[:] = np.array([[1.0, 0.5, 0.0, 0.0]], np.float32)
    np.testing.assert_array_equal(oracle.index_scores(wl, 0), [1.5, 2.0, 1.5])
    dw = DeviceWorkload(wl).indexer()
    assert dw.topk_host()[0].tolist() == [0, 1]


def test_sfa_hand_example_on_device():
    """SFA toy: logits (0, ln 3) over rows {0, 1} -> weights (1/4, 3/4) -> out (0.5, 3.0), lse ln 4;
    a zero query gives (1, 2) and ln 2; the unselected row 2 has no influence."""
    wl = make_workload("toy", 2, [3], [1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=3, attn_heads=2,
                       softmax_scale=math.log(3.0))
    pg = wl.page_table[0, 0]
    kv = np.zeros((3, 576), np.float32)
    kv[0, :2] = [2, 0]
    kv[1, :2] = [0, 4]
    kv[1, 512] = 1  # a RoPE dim: counts for the logits, not part of V
    kv[2, :2] = [100, 100]
    wl.kv_cache[pg, :3] = f32_to_bf16(kv)
    q = np.zeros((1, 2, 576), np.float32)
    q[0, 0, 512] = 1
    wl.q[:] = f32_to_bf16(q)
    dw = DeviceWorkload(wl)
    dw.sfa(topk=torch.tensor([[1, -1, 0]], dtype=torch.int32, device="cuda"))
    out, lse = dw.out_host()
    np.testing.assert_allclose(out[0, :, :2], [[0.5, 3.0], [1.0, 2.0]], rtol=0, atol=1e-2)
    assert np.all(out[0, :, 2:] == 0)
    np.testing.assert_allclose(lse[0], [math.log(4), math.log(2)], rtol=0, atol=1e-3)


def test_topk_all_scores_tied_takes_lowest_positions():
    """Every position scores the same, so far more keys share every prefix than the select's candidate
    exchange holds and the exchanged per-byte passes run.  Ties are taken in ascending position order."""
    wl = make_workload("ties", 11, [5000], [1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=512,
                       attn_heads=128)
    wl.k_cache[:] = wl.k_cache[wl.page_table[0, 0], 0]
    scores = oracle.index_scores(wl, 0)
    assert np.all(scores == scores[0])
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    assert topk[0].tolist() == list(range(512))
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


def test_topk_scale_jump_across_the_context():
    """The second half of the context scores 16x higher (its indexer keys scaled exactly by 16), so the
    CTAs that score the first half guess the wrong top byte for the K-th key and the select runs its
    exchanged second-byte pass."""
    wl = make_workload("jump", 12, [8192], [1], idx_heads=64, idx_dim=128, idx_fp8=False, top_k=2048,
                       attn_heads=128)
    for lp in range(64, 128):
        pg = wl.page_table[0, lp]
        wl.k_cache[pg] = f32_to_bf16(bf16_to_f32(wl.k_cache[pg]) * np.float32(16.0))
    scores = oracle.index_scores(wl, 0)
    assert np.median(scores[4096:]) > 8 * np.median(scores[:4096])
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


def test_fused_decode_launch_count():
    """One query token per sequence with 64 x 128 indexer heads: one kernel per step; other shapes: two."""
    assert dsa.fused_decode_launches(DeviceWorkload(_small("hi64_bf16")).dims) == 1
    assert dsa.fused_decode_launches(DeviceWorkload(config(2, with_sfa=False)).dims) == 1
    assert dsa.fused_decode_launches(DeviceWorkload(_small("hi64_bf16_two_queries")).dims) == 2
    assert dsa.fused_decode_launches(DeviceWorkload(_small("hi4_ragged")).dims) == 2


@pytest.mark.parametrize("name", ["hi64_bf16", "hi64_fp8", "hi64_salient", "k_equals_one"])
def test_single_launch_matches_two_kernels(name):
    """The single-launch kernel selects exactly what the standalone indexer selects, and its attention
    agrees with the standalone attention kernel's (their position splits may differ, so the fp32
    summation order may too)."""
    wl = _small(name) if name != "hi64_fp8" else make_workload("fp8_single", 78, [5000, 190, 700], [1, 1, 1],
                                                              idx_heads=64, idx_dim=128, idx_fp8=True, top_k=256,
                                                              attn_heads=128)
    a = DeviceWorkload(wl)
    assert dsa.fused_decode_launches(a.dims) == 1
    a.fused()
    b = DeviceWorkload(wl).indexer().sfa()
    assert a.error_word() == 0 and b.error_word() == 0
    assert np.array_equal(a.topk_host(), b.topk_host())
    oa, la = a.out_host()
    ob, lb = b.out_host()
    np.testing.assert_allclose(oa.astype(np.float32), ob.astype(np.float32), rtol=1e-2, atol=1e-2)
    np.testing.assert_allclose(la, lb, rtol=1e-5, atol=1e-5)
    check_attention(wl, a.topk_host(), oa, la)


def test_page_permutation_gives_identical_results():
    a = _small("hi64_bf16", page_seed=1)
    b = _small("hi64_bf16", page_seed=2)
    assert not np.array_equal(a.page_table, b.page_table)
    da, db = DeviceWorkload(a).fused(), DeviceWorkload(b).fused()
    assert np.array_equal(da.topk_host(), db.topk_host())
    oa, la = da.out_host()
    ob, lb = db.out_host()
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_repeated_calls_are_deterministic():
    wl = _small("hi64_fp8")
    dw = DeviceWorkload(wl)
    dw.fused()
    t1, (o1, l1) = dw.topk_host().copy(), dw.out_host()
    dw.fused()
    assert np.array_equal(t1, dw.topk_host())
    o2, l2 = dw.out_host()
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_zero_query_tokens_is_a_no_op():
    wl = _small("hi4_ragged")
    dw = DeviceWorkload(wl)
    d = dw.dims
    d.total_q = 0
    dw.fused(dims=d)
    assert dw.error_word() == 0
    assert np.all(dw.topk_host() == -7)


# ---------------------------------------------------------------------------------------------------
# The five workload configurations at full size
# ---------------------------------------------------------------------------------------------------


@pytest.mark.parametrize("n", [1, 2, 3, 5])
def test_config_decode(n):
    wl = config(n)
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)


@pytest.mark.slow
def test_config_prefill():
    """4096 new tokens over 61440 cached ones (the prefill chunk): every one of the 4096 queries is checked
    against the oracle, the Top-K set (with the excusal band) and the attention output element by element."""
    wl = config(4)
    dw = DeviceWorkload(wl).fused()
    assert dw.error_word() == 0
    topk = dw.topk_host()
    check_topk(wl, topk)
    out, lse = dw.out_host()
    check_attention(wl, topk, out, lse)
    pos = wl.query_positions()
    valid = topk >= 0
    assert np.all(valid.sum(axis=1) == np.minimum(wl.top_k, pos + 1))
