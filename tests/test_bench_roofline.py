"""The algorithmic work bench.py divides by: score flops and byte counts of small workloads, against
counts written out by hand from the definitions (2*Hi*Di flops per query and visible position; every
visible key row read once per launch)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gen.workloads import config, make_workload  # noqa: E402


def test_indexer_flops_counts_every_visible_position_once():
    # two sequences: 300 cached positions with 3 queries (positions 297, 298, 299) and 64 with 1 (63)
    wl = make_workload("flops", 3, [300, 64], [3, 1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=16,
                       attn_heads=16, with_sfa=False)
    visible = (297 + 1) + (298 + 1) + (299 + 1) + (63 + 1)
    assert bench.indexer_flops(wl) == 2 * 4 * 64 * visible


def test_prefill_flops_match_the_closed_form():
    # the prefill chunk: 4096 queries at positions 61440 .. 65535, 64 heads of 128 dims
    wl = config(4, with_sfa=False)
    n = np.arange(61440, 65536, dtype=np.int64) + 1
    assert bench.indexer_flops(wl) == 2 * 64 * 128 * int(n.sum())
    assert abs(bench.indexer_flops(wl) / 1e12 - 4.2606) < 1e-3
    assert 4 in bench.TENSOR_BOUND_CONFIGS


def test_indexer_bytes_read_each_key_row_once():
    wl = make_workload("bytes", 5, [300, 64], [3, 1], idx_heads=4, idx_dim=64, idx_fp8=False, top_k=16,
                       attn_heads=16, with_sfa=False)
    keys = (300 + 64) * 64 * 2
    pages = (5 + 1) * 4
    q = 4 * 4 * (64 * 2 + 4)
    out = 4 * 16 * 4
    assert bench.indexer_bytes(wl) == keys + pages + q + out
