"""Pins for the CPU oracle: hand-worked examples, closed forms, special cases and invariants.

None of these re-types the oracle's own formula: each checks it against something fixed independently
(a hand computation, dense softmax attention, a library decoder, or a property that must hold).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gen import bf16_to_f32, e4m3_encode_array
from gen.workloads import make_workload

from _util import workload_from_logical

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _val(x):
    return {"ln 3": math.log(3.0), "ln 4": math.log(4.0), "ln 2": math.log(2.0)}[x] if isinstance(x, str) else x


# ---------------------------------------------------------------------------------------------------
# Element decoders against the library's own conversions
# ---------------------------------------------------------------------------------------------------


def test_bf16_decoder_matches_torch_for_every_code():
    codes = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).double().numpy()
    ours = np.array([oracle.bf16_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decoder_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    ours = np.array([oracle.e4m3_value(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_generator_e4m3_encoder_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(-448, 448, 400_000),
        rng.normal(0, 1, 400_000),
        rng.uniform(-2.0 ** -5, 2.0 ** -5, 200_000),  # subnormal range
    ]).astype(np.float32)
    ours = e4m3_encode_array(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # saturation instead of NaN above the largest finite value
    assert np.all(e4m3_encode_array(np.array([449.0, 1e6, -500.0], dtype=np.float32)) == [0x7E, 0x7E, 0xFE])


# ---------------------------------------------------------------------------------------------------
# Hand-worked examples
# ---------------------------------------------------------------------------------------------------


def _indexer_toy():
    g = _load("indexer_toy.json")
    wl = workload_from_logical(seq_lens=[g["seq_len"]], q_lens=[1], page_size=g["page_size"],
                               page_table=g["page_table"], idx_q=np.array([g["q_idx"]]), w=np.array([g["w"]]),
                               idx_k_rows=[np.array(g["k"])], top_k=g["top_k"])
    return g, wl


def test_indexer_hand_example():
    g, wl = _indexer_toy()
    assert np.array_equal(oracle.index_scores(wl, 0), g["expected_scores"])
    topk, kth, nsel = oracle.indexer_topk(wl)
    assert topk[0].tolist() == g["expected_topk"]
    assert kth[0] == g["expected_kth"] and nsel[0] == 2


def test_indexer_hand_example_fp8_route():
    """Same toy through the FP8 route: codes chosen so code * scale reproduces the bf16 values."""
    g, _ = _indexer_toy()
    k = np.array(g["k"])
    q = np.array(g["q_idx"])
    # E4M3 of 1, 2, 3 and their halves are exact; store k/2 with scale 2 and q*1 with scale 1.
    k_codes = e4m3_encode_array((k / 2).astype(np.float32))
    q_codes = e4m3_encode_array(q.astype(np.float32))
    wl = workload_from_logical(seq_lens=[3], q_lens=[1], page_size=2, page_table=[[1, 0]], idx_q=q_codes[None],
                               w=np.array([g["w"]]), idx_k_rows=[k_codes], top_k=2, idx_fp8=True,
                               q_scale=np.ones((1, 2)), k_scale_rows=[[2.0, 2.0, 2.0]])
    assert np.array_equal(oracle.index_scores(wl, 0), g["expected_scores"])
    assert oracle.indexer_topk(wl)[0][0].tolist() == g["expected_topk"]


def _sfa_toy():
    g = _load("sfa_toy.json")
    wl = workload_from_logical(seq_lens=[g["seq_len"]], q_lens=[1], page_size=g["page_size"],
                               page_table=g["page_table"], idx_q=np.zeros((1, 1, 2)), w=np.zeros((1, 1)),
                               idx_k_rows=[np.zeros((3, 2))], top_k=len(g["topk"]), attn_q=np.array([g["q"]]),
                               kv_rows=[np.array(g["kv"])], v_dim=g["v_dim"], softmax_scale=_val(g["softmax_scale"]))
    return g, wl


def test_sparse_attention_hand_example():
    g, wl = _sfa_toy()
    out, lse, wts = oracle.sparse_attn(wl, np.array([g["topk"]]), want_weights=True)
    np.testing.assert_allclose(out[0], g["expected_out"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0], [_val(x) for x in g["expected_lse"]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(wts[0], g["expected_weights"], rtol=0, atol=1e-15)


def test_sparse_attention_no_selected_rows():
    _, wl = _sfa_toy()
    out, lse = oracle.sparse_attn(wl, np.array([[-1, -1, -1]]))
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------------------------------------------
# Closed forms / special cases on seeded workloads
# ---------------------------------------------------------------------------------------------------


def _small(idx_fp8=False, top_k=16, seq_lens=(37, 150, 5), q_lens=(1, 3, 2), page_size=64, seed=11, **kw):
    return make_workload("small", seed, list(seq_lens), list(q_lens), idx_heads=kw.pop("idx_heads", 3),
                         idx_dim=kw.pop("idx_dim", 8), idx_fp8=idx_fp8, top_k=top_k, attn_heads=kw.pop("hq", 4),
                         kv_dim=kw.pop("kv_dim", 24), v_dim=kw.pop("v_dim", 16), page_size=page_size, **kw)


def _dense_attention(wl, t):
    """Textbook causal softmax attention over ALL visible rows (float64, logical order)."""
    b = int(wl.query_seq()[t])
    p = int(wl.query_positions()[t])
    kv = bf16_to_f32(wl.logical_rows(wl.kv_cache, b)[: p + 1]).astype(np.float64)
    q = bf16_to_f32(wl.q[t]).astype(np.float64)
    z = wl.softmax_scale * q @ kv.T
    z = z - z.max(axis=1, keepdims=True)
    a = np.exp(z)
    lse = np.log(a.sum(axis=1)) + (wl.softmax_scale * q @ kv.T).max(axis=1)
    a /= a.sum(axis=1, keepdims=True)
    return a @ kv[:, : wl.v_dim], lse


@pytest.mark.parametrize("page_size", [4, 64])
def test_full_selection_equals_dense_causal_attention(page_size):
    wl = _small(top_k=160, page_size=page_size)  # K >= every context: Top-K keeps all visible rows
    topk, kth, nsel = oracle.indexer_topk(wl)
    pos = wl.query_positions()
    for t in range(wl.total_q):
        assert nsel[t] == pos[t] + 1
        assert topk[t, : nsel[t]].tolist() == list(range(pos[t] + 1))
        assert np.all(topk[t, nsel[t]:] == -1)
    out, lse = oracle.sparse_attn(wl, topk)
    for t in range(wl.total_q):
        ref, ref_lse = _dense_attention(wl, t)
        np.testing.assert_allclose(out[t], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[t], ref_lse, rtol=1e-12, atol=1e-12)


def test_scores_match_brute_force_over_logical_rows():
    """Paging and decoding: scores from the paged cache equal a direct evaluation on logical rows."""
    for fp8 in (False, True):
        wl = _small(idx_fp8=fp8, page_size=4)
        pos = wl.query_positions()
        for t in range(wl.total_q):
            b = int(wl.query_seq()[t])
            rows = wl.logical_rows(wl.k_cache, b)[: pos[t] + 1]
            if fp8:
                kk = torch.from_numpy(rows).view(torch.float8_e4m3fn).double().numpy()
                kk = kk * wl.logical_rows(wl.k_scale[..., None], b)[: pos[t] + 1]
                qq = torch.from_numpy(wl.q_idx[t]).view(torch.float8_e4m3fn).double().numpy() * wl.q_scale[t][:, None]
            else:
                kk = bf16_to_f32(rows).astype(np.float64)
                qq = bf16_to_f32(wl.q_idx[t]).astype(np.float64)
            per_head = np.maximum(qq @ kk.T, 0.0)  # [H, S]
            ref = wl.w[t].astype(np.float64) @ per_head
            np.testing.assert_allclose(oracle.index_scores(wl, t), ref, rtol=1e-12, atol=1e-12)


def test_topk_equals_lexsort_of_scores():
    wl = _small(top_k=16)
    topk, kth, nsel = oracle.indexer_topk(wl)
    for t in range(wl.total_q):
        sc = oracle.index_scores(wl, t)
        order = np.lexsort((np.arange(sc.shape[0]), -sc))[: wl.top_k]
        assert sorted(order.tolist()) == topk[t, : nsel[t]].tolist()
        assert kth[t] == sc[order[-1]]


def test_all_zero_scores_take_lowest_positions():
    """w = 0 makes every score 0: ties break toward the lower position."""
    wl = _small(top_k=8)
    wl.w[:] = 0.0
    topk, kth, nsel = oracle.indexer_topk(wl)
    for t in range(wl.total_q):
        n = nsel[t]
        assert topk[t, :n].tolist() == list(range(n)) and kth[t] == 0.0


# ---------------------------------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------------------------------


def test_topk_is_causal_unique_sorted_and_sized():
    wl = _small(top_k=16, seq_lens=(300, 17, 64), q_lens=(2, 17, 1))
    topk, _, nsel = oracle.indexer_topk(wl)
    pos = wl.query_positions()
    for t in range(wl.total_q):
        v = topk[t][topk[t] >= 0]
        assert v.shape[0] == nsel[t] == min(wl.top_k, pos[t] + 1)
        assert np.all(np.diff(v) > 0) and v.max() <= pos[t]
        assert np.all(topk[t, nsel[t]:] == -1)


def test_second_query_can_see_one_more_position():
    wl = _small(top_k=400, seq_lens=(300,), q_lens=(2,))
    topk, _, nsel = oracle.indexer_topk(wl)
    assert nsel.tolist() == [299, 300] and 299 not in topk[0] and 299 in topk[1]


def test_page_permutation_leaves_results_identical():
    a = _small(top_k=16, page_size=4, page_seed=1)
    b = _small(top_k=16, page_size=4, page_seed=2)
    assert not np.array_equal(a.page_table, b.page_table)
    ta, ka, _ = oracle.indexer_topk(a)
    tb, kb, _ = oracle.indexer_topk(b)
    assert np.array_equal(ta, tb) and np.array_equal(ka, kb)
    oa, la = oracle.sparse_attn(a, ta)
    ob, lb = oracle.sparse_attn(b, tb)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_head_weight_scaling_keeps_topk():
    wl = _small(top_k=16)
    ref, kref, _ = oracle.indexer_topk(wl)
    wl.w *= np.float32(2.0)  # exact: scores double exactly
    got, kgot, _ = oracle.indexer_topk(wl)
    assert np.array_equal(ref, got) and np.array_equal(2 * kref, kgot)


def test_fp8_scale_factors_out_of_relu():
    """Doubling every key scale doubles every score exactly (positive scales commute with ReLU)."""
    wl = _small(idx_fp8=True, top_k=16)
    s0 = [oracle.index_scores(wl, t) for t in range(wl.total_q)]
    wl.k_scale *= np.float32(2.0)
    for t in range(wl.total_q):
        assert np.array_equal(oracle.index_scores(wl, t), 2 * s0[t])


def test_attention_weights_sum_to_one_and_reconstruct_output():
    wl = _small(top_k=16)
    topk, _, _ = oracle.indexer_topk(wl)
    out, lse, wts = oracle.sparse_attn(wl, topk, want_weights=True)
    np.testing.assert_allclose(wts.sum(axis=2), 1.0, rtol=0, atol=1e-13)
    # out = sum_s exp(z_s - lse) v_s  with z recomputed from scratch
    for t in range(wl.total_q):
        b = int(wl.query_seq()[t])
        rows = wl.logical_rows(wl.kv_cache, b)
        sel = topk[t][topk[t] >= 0]
        kv = bf16_to_f32(rows[sel]).astype(np.float64)
        z = wl.softmax_scale * bf16_to_f32(wl.q[t]).astype(np.float64) @ kv.T
        rec = np.exp(z - lse[t][:, None]) @ kv[:, : wl.v_dim]
        np.testing.assert_allclose(out[t], rec, rtol=1e-12, atol=1e-12)


def test_selection_order_does_not_matter():
    wl = _small(top_k=16)
    topk, _, _ = oracle.indexer_topk(wl)
    rev = np.ascontiguousarray(topk[:, ::-1])
    o1, l1 = oracle.sparse_attn(wl, topk)
    o2, l2 = oracle.sparse_attn(wl, rev)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-13, atol=1e-13)


def test_bad_page_is_reported():
    wl = _small(top_k=16, page_size=4)
    wl.page_table[0, 0] = wl.num_pages + 3
    with pytest.raises(oracle.OracleError):
        oracle.indexer_topk(wl)


# ---------------------------------------------------------------------------------------------------
# FP8 latent-KV cache and appending a step's rows
# ---------------------------------------------------------------------------------------------------


def _torch_e4m3(x):
    """E4M3 codes of float32 values by torch's float8_e4m3fn conversion (finite range only)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _torch_e4m3_value(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn).double().numpy()


def test_oracle_e4m3_encoder_round_trips_every_finite_code():
    for c in list(range(0x7F)) + list(range(0x80, 0xFF)):
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c, hex(c)


def test_oracle_e4m3_encoder_matches_torch_and_ties_to_even():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(-448, 448, 6000), rng.normal(0, 1, 6000),
                        rng.uniform(-2.0 ** -5, 2.0 ** -5, 3000)]).astype(np.float32)
    ours = np.array([oracle.e4m3_encode(v) for v in x], dtype=np.uint8)
    assert np.array_equal(ours, _torch_e4m3(x))
    # midpoints between neighbouring finite values go to the even code (torch agrees)
    vals = _torch_e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    ours = np.array([oracle.e4m3_encode(v) for v in mids])
    lo = np.arange(0x7E)
    assert np.array_equal(ours, np.where(lo % 2 == 0, lo, lo + 1))
    assert np.array_equal(ours, _torch_e4m3(mids))
    assert oracle.e4m3_encode(449.0) == 0x7E and oracle.e4m3_encode(-1e6) == 0xFE
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def test_quantize_group_is_absmax_over_448_in_fp32():
    rng = np.random.default_rng(9)
    for mag in (1e-3, 1.0, 37.0, 3e4):
        x = (bf16_to_f32((rng.normal(0, 1, 128).astype(np.float32) * np.float32(mag)).view(np.uint32) >> 16)
             .astype(np.float32))
        codes, scale = oracle.quantize_group(x)
        amax = np.float32(np.max(np.abs(x)))
        assert scale == amax / np.float32(448.0)
        assert np.array_equal(codes, _torch_e4m3(x / scale))
        assert codes[np.argmax(np.abs(x))] & 0x7F == 0x7E
    codes, scale = oracle.quantize_group(np.zeros(128, dtype=np.float32))
    assert scale == 1.0 and np.all(codes == 0)


def _fp8_kv_rows(rng, n, v_dim=512, kv_dim=576):
    """Random FP8 latent-KV rows built byte by byte (codes, power-of-two tile scales, bf16 rope) and the
    same rows as exact bf16 values (e4m3 x 2^k has at most four significant bits)."""
    tiles = v_dim // 128
    codes = rng.integers(0, 0x7F, (n, v_dim)).astype(np.uint8) | (rng.integers(0, 2, (n, v_dim)) << 7).astype(np.uint8)
    scales = (2.0 ** rng.integers(-4, 5, (n, tiles))).astype(np.float32)
    rope_f = rng.normal(0, 1, (n, kv_dim - v_dim)).astype(np.float32)
    rope = (rope_f.view(np.uint32) >> 16).astype(np.uint16)
    fp8 = np.empty((n, v_dim + 4 * tiles + 2 * (kv_dim - v_dim)), dtype=np.uint8)
    fp8[:, :v_dim] = codes
    fp8[:, v_dim:v_dim + 4 * tiles] = scales.view(np.uint8).reshape(n, 4 * tiles)
    fp8[:, v_dim + 4 * tiles:] = rope.view(np.uint8).reshape(n, -1)
    vals = _torch_e4m3_value(codes) * np.repeat(scales.astype(np.float64), 128, axis=1)
    bf = np.empty((n, kv_dim), dtype=np.uint16)
    bf[:, :v_dim] = (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_to_f32(bf[:, :v_dim]).astype(np.float64), vals)  # exact in bf16
    bf[:, v_dim:] = rope
    return fp8, bf


def test_fp8_kv_attention_equals_bf16_attention_on_the_same_values():
    wl = _small(top_k=16, kv_dim=576, v_dim=512, hq=3)
    rng = np.random.default_rng(21)
    P = wl.kv_cache.shape[0] * wl.kv_cache.shape[1]
    fp8, bf = _fp8_kv_rows(rng, P)
    wl.kv_cache = bf.reshape(wl.kv_cache.shape)
    topk, _, _ = oracle.indexer_topk(wl)
    out_bf, lse_bf = oracle.sparse_attn(wl, topk)
    wl.kv_cache = fp8.reshape(wl.kv_cache.shape[0], wl.kv_cache.shape[1], -1)
    wl.kv_fp8 = True
    out_f8, lse_f8 = oracle.sparse_attn(wl, topk)
    assert np.array_equal(out_f8, out_bf) and np.array_equal(lse_f8, lse_bf)


@pytest.mark.parametrize("fp8", [False, True])
def test_append_writes_each_token_row_at_its_position(fp8):
    wl = _small(idx_fp8=fp8, top_k=16, kv_dim=576, v_dim=512, hq=2, kv_fp8=fp8)
    rng = np.random.default_rng(33 + fp8)
    T = wl.total_q
    k_new = (rng.normal(0, 2, (T, wl.idx_dim)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    kv_new = (rng.normal(0, 2, (T, wl.kv_dim)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    k_cache, k_scale, kv_cache = oracle.append(wl, k_new, kv_new)
    touched = set()
    for t, p in enumerate(wl.query_positions()):
        b = int(wl.query_seq()[t])
        page, slot = int(wl.page_table[b, p // wl.page_size]), int(p % wl.page_size)
        touched.add((page, slot))
        if not fp8:
            assert np.array_equal(k_cache[page, slot], k_new[t]) and np.array_equal(kv_cache[page, slot], kv_new[t])
            continue
        x = bf16_to_f32(k_new[t])
        s = np.float32(np.max(np.abs(x))) / np.float32(448.0)
        assert k_scale[page, slot] == s and np.array_equal(k_cache[page, slot], _torch_e4m3(x / s))
        row = kv_cache[page, slot]
        for tile in range(4):
            xt = bf16_to_f32(kv_new[t, 128 * tile:128 * (tile + 1)])
            st = np.float32(np.max(np.abs(xt))) / np.float32(448.0)
            assert row[512 + 4 * tile:516 + 4 * tile].view(np.float32)[0] == st
            assert np.array_equal(row[128 * tile:128 * (tile + 1)], _torch_e4m3(xt / st))
        assert np.array_equal(row[528:].view(np.uint16), kv_new[t, 512:])
    for page in range(k_cache.shape[0]):
        for slot in range(k_cache.shape[1]):
            if (page, slot) in touched:
                continue
            assert np.array_equal(k_cache[page, slot], wl.k_cache[page, slot])
            assert np.array_equal(kv_cache[page, slot], wl.kv_cache[page, slot])


# ---------------------------------------------------------------------------------------------------
# MXFP8 indexer inputs (E4M3 codes, one E8M0 scale per 32 elements)
# ---------------------------------------------------------------------------------------------------


def test_e8m0_decoder_matches_torch_for_every_byte():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).double().numpy()
    ours = np.array([oracle.e8m0_value(int(c)) for c in codes])
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])
    assert ours[127] == 1.0 and ours[0] == 2.0 ** -127 and ours[254] == 2.0 ** 127


def test_generator_mx_quantiser_follows_the_definition():
    from gen import quantize_mx_rows

    rng = np.random.default_rng(12)
    x = (rng.normal(0, 1, (40, 128)) * 2.0 ** rng.integers(-20, 20, (40, 1))).astype(np.float32)
    x[3, 32:64] = 0.0  # an all-zero group
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    codes, scales = quantize_mx_rows(bits)
    xf = bf16_to_f32(bits).reshape(40, 4, 32)
    amax = np.abs(xf).max(axis=-1)
    shared = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1))) - 8, 0).astype(np.int64)
    assert np.array_equal(scales.astype(np.int64) - 127, shared)
    # x / 2^shared can reach 512: the MX conversion saturates at the largest E4M3 value (torch gives NaN)
    y = (xf / np.float32(2.0) ** shared[..., None]).reshape(40, 128)
    ref = _torch_e4m3(np.clip(y, -448.0, 448.0))
    assert np.any(np.abs(y) > 448)
    assert np.array_equal(codes, ref)
    assert np.all(codes[3, 32:64] == 0) and scales[3, 1] == 127


def test_mx_scores_equal_bf16_scores_on_the_same_values():
    wl = _small(idx_fp8=True, idx_mx=True, idx_heads=3, idx_dim=64, top_k=16)
    assert wl.q_scale.shape == (wl.total_q, 3, 2) and wl.k_scale.shape[-1] == 2
    # the same values decoded by torch (codes as float8_e4m3fn, scales as float8_e8m0fnu), exact in bf16
    def decode(codes, scales):
        v = _torch_e4m3_value(codes.reshape(-1, codes.shape[-1]))
        s = torch.from_numpy(np.ascontiguousarray(scales.reshape(-1, scales.shape[-1]))).view(
            torch.float8_e8m0fnu).double().numpy()
        v = v * np.repeat(s, 32, axis=1)
        b = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        assert np.array_equal(bf16_to_f32(b).astype(np.float64), v)
        return b.reshape(codes.shape)
    scores_mx = [oracle.index_scores(wl, t) for t in range(wl.total_q)]
    top_mx = oracle.indexer_topk(wl)[0]
    wl.q_idx, wl.k_cache = decode(wl.q_idx, wl.q_scale), decode(wl.k_cache, wl.k_scale)
    wl.q_scale = wl.k_scale = None
    wl.idx_fp8, wl.idx_mx = False, False
    for t in range(wl.total_q):
        assert np.array_equal(oracle.index_scores(wl, t), scores_mx[t])
    assert np.array_equal(oracle.indexer_topk(wl)[0], top_mx)


def test_mx_scores_at_extreme_scales_match_a_direct_evaluation():
    """Keys made only of subnormal E4M3 codes under a scale of 2^30, and keys with scale bytes 160..170
    (factors near 2^43), against a float64 evaluation written from the definitions: codes decoded by
    torch's float8_e4m3fn, scale bytes as 2^(e - 127), then sum_h w * max(0, q . k) per position."""
    wl = _small(idx_fp8=True, idx_mx=True, idx_heads=3, idx_dim=64, top_k=16, seq_lens=(150, 70), q_lens=(1, 2))
    rng = np.random.default_rng(9)
    for b in range(wl.batch):
        for j, pos in enumerate(rng.choice(int(wl.seq_lens[b]), 12, replace=False)):
            pg, r = int(wl.page_table[b, pos // wl.page_size]), int(pos % wl.page_size)
            if j < 6:
                wl.k_cache[pg, r] = (rng.integers(1, 8, 64) | (rng.integers(0, 2, 64) << 7)).astype(np.uint8)
                wl.k_scale[pg, r] = 127 + 30
            else:
                wl.k_scale[pg, r] = rng.integers(160, 171, 2).astype(np.uint8)
    e8m0 = lambda e: np.ldexp(1.0, e.astype(np.int64) - 127)
    qv = _torch_e4m3_value(wl.q_idx.reshape(-1, 64)).reshape(wl.q_idx.shape) * np.repeat(e8m0(wl.q_scale), 32, axis=-1)
    got = oracle.index_scores_batch(wl, list(range(wl.total_q)))
    pos_all = wl.query_positions()
    for t in range(wl.total_q):
        b = int(wl.query_seq()[t])
        p = int(pos_all[t])
        rows = np.arange(p + 1)
        pages = wl.page_table[b, rows // wl.page_size]
        codes = wl.k_cache[pages, rows % wl.page_size]
        kv = _torch_e4m3_value(codes) * np.repeat(e8m0(wl.k_scale[pages, rows % wl.page_size]), 32, axis=-1)
        dots = kv @ qv[t].T  # [positions, heads]
        ref = (np.maximum(dots, 0.0) * wl.w[t].astype(np.float64)).sum(axis=1)
        np.testing.assert_allclose(got[t], ref, rtol=1e-12, atol=0.0)
        assert np.abs(ref).max() > 1e12  # the large scales are in play
