"""The seeded input generator: published SplitMix64 outputs, distributions, layouts, determinism."""
import numpy as np

import gen
from gen import workloads


def test_splitmix64_reference_outputs():
    # SplitMix64 seeded with 0: the first outputs of the published generator.
    assert gen.draw(0, 0) == 0xE220A8397B1DCDAF
    assert gen.draw(0, 1) == 0x6E789E6AA1B965F4
    assert gen.draw(0, 2) == 0x06C45D188009454F


def test_normal_moments_and_support():
    x = gen.bf16_to_f32(gen.normal_bf16(gen.stream_key(1, 2), 1_000_000)).astype(np.float64)
    assert abs(x.mean()) < 0.005 and abs(x.var() - 1.0) < 0.01
    assert x.min() >= -6.0 and x.max() <= 6.0


def test_uniform_range():
    u = gen.uniform_f32(gen.stream_key(3, 4), 100_000, 0.0, 0.125)
    assert u.min() >= 0.0 and u.max() < 0.125 and abs(u.mean() - 0.0625) < 0.001


def test_permutation_and_sampling():
    p = gen.permutation(gen.stream_key(5, 6), 1000)
    assert sorted(p.tolist()) == list(range(1000)) and not np.array_equal(p, np.arange(1000))
    s = gen.sample_without_replacement(gen.stream_key(5, 7), 32768, 327)
    assert np.unique(s).shape[0] == 327 and s.min() >= 0 and s.max() < 32768


def test_counter_based_offsets_are_consistent():
    k = gen.stream_key(9, 1)
    full = gen.normal_bf16(k, 1000)
    assert np.array_equal(full[400:700], gen.normal_bf16(k, 300, offset=400))


def test_workload_layout_and_determinism():
    a = workloads.make_workload("t", 5, [130, 64, 1], [2, 1, 1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=8,
                                attn_heads=4, salient_frac=0.05)
    b = workloads.make_workload("t", 5, [130, 64, 1], [2, 1, 1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=8,
                                attn_heads=4, salient_frac=0.05)
    assert np.array_equal(a.k_cache, b.k_cache) and np.array_equal(a.kv_cache, b.kv_cache)
    assert a.num_pages == 3 + 1 + 1
    used = a.page_table[a.page_table >= 0]
    assert sorted(used.tolist()) == list(range(a.num_pages))
    # tail slots of partial pages stay zero
    last = a.page_table[0, 2]
    assert np.all(a.k_cache[last, 2:] == 0) and np.all(a.kv_cache[last, 2:] == 0)
    assert a.notes["salient_rows"] == 6 + 3 + 0
    assert a.query_positions().tolist() == [128, 129, 63, 0]


def test_page_seed_changes_layout_not_content():
    a = workloads.make_workload("t", 5, [300], [1], idx_heads=2, idx_dim=64, idx_fp8=True, top_k=8, attn_heads=2,
                                page_seed=1)
    b = workloads.make_workload("t", 5, [300], [1], idx_heads=2, idx_dim=64, idx_fp8=True, top_k=8, attn_heads=2,
                                page_seed=2)
    assert not np.array_equal(a.page_table, b.page_table)
    assert np.array_equal(a.logical_rows(a.k_cache, 0), b.logical_rows(b.k_cache, 0))
    assert np.array_equal(a.logical_rows(a.k_scale, 0), b.logical_rows(b.k_scale, 0))
    assert np.array_equal(a.logical_rows(a.kv_cache, 0), b.logical_rows(b.kv_cache, 0))


def test_fp8_rows_use_absmax_over_448():
    a = workloads.make_workload("t", 6, [70], [1], idx_heads=2, idx_dim=128, idx_fp8=True, top_k=8, attn_heads=2,
                                with_sfa=False)
    k = a.logical_rows(a.k_cache, 0)
    s = a.logical_rows(a.k_scale, 0)
    # the largest magnitude of every row encodes to +-448 (code 0x7E / 0xFE)
    assert np.all(np.max(k & 0x7F, axis=1) == 0x7E)
    assert np.all(s > 0)


def test_config_lengths():
    assert workloads.config_lengths(2) == ([32768] * 32, [1] * 32)
    lens, q = workloads.config_lengths(5)
    assert len(lens) == 8 and q == [2] * 8 and min(lens) >= 16384 and max(lens) <= 131072
    assert workloads.config_lengths(5) == workloads.config_lengths(5)


def test_config1_shapes():
    wl = workloads.config(1)
    assert wl.q_idx.shape == (1, 4, 64) and wl.k_cache.shape == (64, 64, 64)
    assert wl.q.shape == (1, 16, 576) and wl.kv_cache.shape == (64, 64, 576)
    assert wl.top_k == 256 and abs(wl.softmax_scale - 1 / 24) < 1e-15
