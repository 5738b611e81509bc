"""Context parallelism across processes on CPU (gloo, world sizes 2 to 4): the Zigzag prefill layout and
decode by context shards of ``sparse_attention_dsa_gb300.cp``, with every device step done by the CPU
oracle (tests/_cp_oracle_backend.py), so that the partition, the all-gathers and the reassembly are
checked here; the same orchestration on the GPU library is in tests/test_gpu_zigzag.py.

Sources: "Day0 Inference Support and Performance Optimization for New LLM Architectures", section 5
(5.1 context parallelism for decode, 5.2 causal index load imbalance and the Zigzag layout);
"Optimizing Inference for Hybrid Attention Architectures: From Operator Fusion to Sequence Sharding",
section "Sequence Sharding and Load Balancing in the Prefill Phase".
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from sparse_attention_dsa_gb300 import cp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


# ---------------------------------------------------------------------------------------------------
# host logic
# ---------------------------------------------------------------------------------------------------


@pytest.mark.parametrize("n_new,world", [(4096, 2), (4096, 4), (4096, 8), (97, 3), (5, 4), (0, 2)])
def test_zigzag_partition_covers_every_query_once(n_new, world):
    segs = cp.zigzag_segments(n_new, world)
    lens = [e - s for s, e in segs]
    assert len(segs) == 2 * world and max(lens) - min(lens) <= 1 and sum(lens) == n_new
    allq = np.concatenate([cp.zigzag_rank_queries(n_new, world, r) for r in range(world)])
    assert np.array_equal(np.sort(allq), np.arange(n_new))
    for r in range(world):  # rank r: the r-th segment from the front and the r-th from the back
        a, b = cp.zigzag_rank_segments(n_new, world, r)
        assert a == segs[r] and b == segs[2 * world - 1 - r]


@pytest.mark.parametrize("world", [2, 4, 8])
def test_zigzag_balances_the_causal_work(world):
    """The prefill chunk of 4096 queries after 61440 cached tokens: per-rank causal work (sum of p + 1)
    under the Zigzag layout is equal to within one segment length's rounding, while the contiguous split
    gives the last rank the most."""
    zz = cp.rank_loads(61440, 4096, world, "zigzag")
    cont = cp.rank_loads(61440, 4096, world, "contiguous")
    assert sum(zz) == sum(cont) == cp.causal_work(61440, range(4096))
    assert max(zz) / min(zz) < 1.0001
    assert max(cont) / min(cont) > 1.0 + 0.9 * (4096 - 4096 / world) / (61440 + 4096)
    # without cached tokens (a first chunk) the imbalance of the contiguous split is extreme
    assert max(cp.rank_loads(0, 4096, world, "contiguous")) / min(cp.rank_loads(0, 4096, world, "contiguous")) > 2
    assert max(cp.rank_loads(0, 4096, world)) / min(cp.rank_loads(0, 4096, world)) < 1.01


def test_rank_batch_positions():
    """Each segment becomes a sequence whose newest tokens are exactly that segment's queries."""
    cached, n_new, world = 1000, 37, 3
    for r in range(world):
        rb = cp.zigzag_rank_batch(cached, n_new, world, r)
        pos = []
        for b in range(2):
            n = rb.cu_q_lens[b + 1] - rb.cu_q_lens[b]
            pos += list(rb.seq_lens[b] - n + np.arange(n))
        assert pos == list(cached + rb.queries)


def test_context_shards_cover_the_context():
    for max_ctx, world in [(32768, 2), (131072, 8), (1000, 3), (64, 4)]:
        rng = cp.context_shards(max_ctx, world)
        assert rng[0][0] == 0 and rng[-1][1] == cp.OPEN_END
        assert all(a[1] == b[0] for a, b in zip(rng, rng[1:]))
        assert all(lo % 64 == 0 for lo, _ in rng)


# ---------------------------------------------------------------------------------------------------
# gloo ranks
# ---------------------------------------------------------------------------------------------------

ZZ = dict(cached=900, n_new=61, hi=4, di=64, K=64, hq=16, seed=41)


def _zz_workload():
    from gen.workloads import make_workload

    c = ZZ
    return make_workload("zz", c["seed"], [c["cached"] + c["n_new"]], [c["n_new"]], idx_heads=c["hi"],
                         idx_dim=c["di"], idx_fp8=False, top_k=c["K"], attn_heads=c["hq"])


def _t(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a.copy())


def _dims(wl):
    import sparse_attention_dsa_gb300 as dsa

    return dsa.DsaDims(batch=wl.batch, total_q=wl.total_q, max_q_len=wl.max_q_len, num_pages=wl.num_pages,
                       page_size=wl.page_size, max_pages_per_seq=wl.max_pages_per_seq, idx_heads=wl.idx_heads,
                       idx_dim=wl.idx_dim, idx_dtype=0, top_k=wl.top_k, attn_heads=wl.attn_heads, kv_dim=wl.kv_dim,
                       v_dim=wl.v_dim, softmax_scale=wl.softmax_scale, kv_dtype=0)


def _zz_worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    from _cp_oracle_backend import OracleBackend

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    wl = _zz_workload()
    c = ZZ
    n_new, cached = c["n_new"], c["cached"]
    mine_q = cp.zigzag_rank_queries(n_new, world, rank)
    pos = cached + mine_q  # cache rows of this rank's tokens
    pt = wl.page_table[0]
    k_rows = np.stack([wl.k_cache[pt[p // 64], p % 64] for p in pos])
    kv_rows = np.stack([wl.kv_cache[pt[p // 64], p % 64] for p in pos])
    # this rank's cache holds the cached tokens only: the chunk's rows arrive through the all-gather
    k_cache, kv_cache = wl.k_cache.copy(), wl.kv_cache.copy()
    for p in range(cached, cached + n_new):
        k_cache[pt[p // 64], p % 64] = 0
        kv_cache[pt[p // 64], p % 64] = 0
    mine = dict(q_idx=_t(wl.q_idx[mine_q]), q_scale=None, w=_t(wl.w[mine_q]), q=_t(wl.q[mine_q]).view(torch.bfloat16),
                k_new=_t(k_rows), kv_new=_t(kv_rows))
    cache = dict(k_cache=_t(k_cache), k_scale=None, kv_cache=_t(kv_cache), page_table=_t(wl.page_table))
    topk, out, lse = cp.zigzag_prefill_rank(OracleBackend(), None, rank, world, _dims(wl), cached, n_new, mine, cache,
                                            None)
    complete = (np.array_equal(cache["k_cache"].numpy().view(np.uint16), wl.k_cache) and
                np.array_equal(cache["kv_cache"].numpy().view(np.uint16), wl.kv_cache))
    q.put((rank, complete, topk.numpy(), out.view(torch.int16).numpy(), lse.numpy()))
    dist.destroy_process_group()


def _spawn(target, world, *args):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for p in procs:
        p.start()
    import queue as _queue
    import time

    res, t0 = [], time.time()
    while len(res) < world:
        try:
            res.append(q.get(timeout=2))
        except _queue.Empty:
            dead = [p for p in procs if p.exitcode not in (None, 0)]
            if dead or time.time() - t0 > 600:
                for p in procs:
                    p.kill()
                raise AssertionError(f"a rank failed (exit codes {[p.exitcode for p in procs]})")
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(res, key=lambda x: x[0])


@pytest.mark.parametrize("world", [2, 4])
def test_zigzag_prefill_on_gloo_ranks_equals_one_process(world):
    """Every rank ends with the whole chunk in its caches, and the reassembled selection, output and lse
    equal those of one process computing the whole chunk (the same oracle arithmetic per query)."""
    import oracle
    from gen import f32_to_bf16

    res = _spawn(_zz_worker, world)
    wl = _zz_workload()
    wl.softmax_scale = float(np.float32(wl.softmax_scale))  # the ranks see it through the fp32 dims field
    sel, _, _ = oracle.indexer_topk(wl)
    o, l = oracle.sparse_attn(wl, sel)
    for rank, complete, topk, out, lse in res:
        assert complete, f"rank {rank}: cache incomplete after the all-gather"
        assert np.array_equal(topk, sel)
        assert np.array_equal(out.view(np.uint16), f32_to_bf16(o.astype(np.float32)))
        assert np.array_equal(lse, l.astype(np.float32))


CD = dict(lens=[700, 1500, 400], hi=4, di=64, K=128, hq=16, seed=42)


def _cd_workload():
    from gen.workloads import make_workload

    c = CD
    return make_workload("cd", c["seed"], c["lens"], [1] * len(c["lens"]), idx_heads=c["hi"], idx_dim=c["di"],
                         idx_fp8=False, top_k=c["K"], attn_heads=c["hq"])


def _cd_worker(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    from _cp_oracle_backend import OracleBackend

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    wl = _cd_workload()
    lo, hi = cp.context_shards(wl.max_pages_per_seq * 64, world)[rank]
    queries = dict(q_idx=_t(wl.q_idx), q_scale=None, w=_t(wl.w), q=_t(wl.q).view(torch.bfloat16),
                   seq_lens=_t(wl.seq_lens), cu_q_lens=_t(wl.cu_q_lens))
    cache = dict(k_cache=_t(wl.k_cache), k_scale=None, kv_cache=_t(wl.kv_cache), page_table=_t(wl.page_table))
    topk, out, lse = cp.context_decode_rank(OracleBackend(), None, rank, world, _dims(wl), lo, hi, queries, cache,
                                            None)
    q.put((rank, topk.numpy(), out.view(torch.int16).numpy(), lse.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_context_decode_on_gloo_ranks(world):
    """The merged selection equals the Top-K over the whole context by the same key; the combined attention
    matches the oracle's attention on that selection within the bf16 tolerance."""
    import oracle

    sys.path.insert(0, TESTS)
    from _cp_oracle_backend import OracleBackend
    from _gpu import ATOL, RTOL

    res = _spawn(_cd_worker, world)
    wl = _cd_workload()
    whole = torch.empty((wl.total_q, wl.top_k), dtype=torch.int32)
    OracleBackend().indexer_shard(_dims(wl), _t(wl.q_idx), None, _t(wl.w), _t(wl.k_cache), None, _t(wl.page_table),
                                  _t(wl.seq_lens), _t(wl.cu_q_lens), 0, cp.OPEN_END, whole,
                                  torch.empty((wl.total_q, wl.top_k)), None)
    ref_o, ref_l = oracle.sparse_attn(wl, whole.numpy())
    for rank, topk, out, lse in res:
        assert np.array_equal(topk, whole.numpy())
        o = (out.view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert np.all(np.abs(o - ref_o) <= ATOL + RTOL * np.abs(ref_o))
        assert np.all(np.abs(lse - ref_l) <= ATOL + RTOL * np.abs(ref_l))
