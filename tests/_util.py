"""Helpers shared by the tests: hand-built workloads from logical arrays, and Top-K set comparison."""
from __future__ import annotations

import math

import numpy as np

from gen import f32_to_bf16
from gen.workloads import Workload


def workload_from_logical(*, seq_lens, q_lens, page_size, page_table, idx_q, w, idx_k_rows, top_k,
                          attn_q=None, kv_rows=None, v_dim=None, softmax_scale=None, idx_fp8=False,
                          q_scale=None, k_scale_rows=None, num_pages=None) -> Workload:
    """Build a paged workload.  idx_k_rows / kv_rows are lists (per sequence) of logical rows.

    Float inputs are converted to bf16 bits and must be exactly representable (asserted).  With
    idx_fp8=True, idx_q / idx_k_rows are E4M3 codes (uint8) and the scales are given explicitly.
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    if num_pages is None:
        num_pages = int(pt.max()) + 1
    di = np.asarray(idx_k_rows[0]).shape[-1]

    def bf(x):
        x = np.asarray(x, dtype=np.float64)
        b = f32_to_bf16(x.astype(np.float32))
        back = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.array_equal(back, x), "toy values must be exact in bf16"
        return b

    if idx_fp8:
        k_cache = np.zeros((num_pages, page_size, di), dtype=np.uint8)
        k_scale = np.ones((num_pages, page_size), dtype=np.float32)
        qi = np.ascontiguousarray(idx_q, dtype=np.uint8)
    else:
        k_cache = np.zeros((num_pages, page_size, di), dtype=np.uint16)
        k_scale = None
        qi = bf(idx_q)
    for b, rows in enumerate(idx_k_rows):
        rows = np.asarray(rows)
        for s in range(int(seq_lens[b])):
            pg, sl = pt[b, s // page_size], s % page_size
            k_cache[pg, sl] = rows[s] if idx_fp8 else bf(rows[s])
            if idx_fp8:
                k_scale[pg, sl] = k_scale_rows[b][s]
    q = kv = None
    kv_dim = 576
    if kv_rows is not None:
        kv_dim = np.asarray(kv_rows[0]).shape[-1]
        kv = np.zeros((num_pages, page_size, kv_dim), dtype=np.uint16)
        for b, rows in enumerate(kv_rows):
            for s in range(int(seq_lens[b])):
                kv[pt[b, s // page_size], s % page_size] = bf(np.asarray(rows)[s])
        q = bf(attn_q)
    attn_heads = q.shape[1] if q is not None else 1
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(kv_dim)
    return Workload(name="toy", seed=0, seq_lens=seq_lens, cu_q_lens=cu, page_size=page_size, page_table=pt,
                    num_pages=num_pages, idx_heads=qi.shape[1], idx_dim=di, idx_fp8=idx_fp8, q_idx=qi,
                    q_scale=None if q_scale is None else np.ascontiguousarray(q_scale, dtype=np.float32),
                    w=np.ascontiguousarray(w, dtype=np.float32), k_cache=k_cache, k_scale=k_scale, top_k=top_k,
                    attn_heads=attn_heads, kv_dim=kv_dim, v_dim=v_dim if v_dim is not None else min(kv_dim, 512),
                    softmax_scale=float(softmax_scale), q=q, kv_cache=kv)


def topk_mismatch(gpu_row, ref_row, ref_scores, kth, nsel, rel_band=1e-3):
    """Compare a Top-K result with the oracle's, as sets, excusing positions within the band.

    gpu_row/ref_row: int arrays of length K with -1 padding.  ref_scores: oracle scores of every
    visible position (float64, index = position).  A position whose oracle score lies within
    rel_band * |kth| of the K-th score may be present or absent; every other position must agree,
    and the GPU must return exactly nsel valid, distinct positions.  Returns None when they agree,
    else a description of the first problem.
    """
    g = np.asarray(gpu_row)
    gv = g[g >= 0]
    if gv.shape[0] != nsel:
        return f"count {gv.shape[0]} != {nsel}"
    if np.unique(gv).shape[0] != gv.shape[0]:
        return "duplicate positions"
    if gv.shape[0] and (gv.max() >= ref_scores.shape[0]):
        return f"position {gv.max()} beyond the causal limit {ref_scores.shape[0] - 1}"
    r = np.asarray(ref_row)
    rv = r[r >= 0]
    sym = np.setxor1d(gv, rv)
    if sym.shape[0] == 0:
        return None
    band = rel_band * abs(kth)
    outside = [int(s) for s in sym if abs(ref_scores[s] - kth) > band]
    if outside:
        s = outside[0]
        return (f"{len(outside)} positions differ outside the band, e.g. {s} score {ref_scores[s]!r} vs "
                f"kth {kth!r} ({'gpu only' if s in gv else 'oracle only'})")
    return None
