"""Context parallelism over several GPUs (one process per GPU) for the DSA path.

Two layouts, both from "Day0 Inference Support and Performance Optimization for New LLM Architectures",
section 5 (Context Parallelism), and "Optimizing Inference for Hybrid Attention Architectures: From
Operator Fusion to Sequence Sharding", section "Sequence Sharding and Load Balancing in the Prefill
Phase":

* Zigzag prefill (section 5.2).  A prefill chunk of n new query tokens is cut into 2W segments of nearly
  equal length; rank r takes segments r and 2W-1-r.  Under the causal mask a query at position p scores
  p+1 positions, so an early segment is cheap and a late one expensive: pairing the r-th cheapest with
  the r-th most expensive gives every rank about the same work.  Each rank holds the new indexer keys and
  latent-KV rows of its own tokens; they are all-gathered so that every rank's cache holds the whole
  chunk, each rank runs the indexer and the sparse attention for its own queries, and the outputs are
  all-gathered and put back in the original token order.
* Decode by context shards (section 5.1).  Rank r holds the cache positions [begin_r, end_r) of a long
  sequence.  It keeps a local Top-K of (score, position) over its positions; the lists are all-gathered
  and merged into the global Top-K with the same key; every rank attends over the selected rows it holds
  and the partial (out, lse) pairs are all-gathered and combined by their log-sum-exp weights.

The device work of a step goes through a backend object; :class:`CudaBackend` calls the library's C ABI
(``dsa_append_rows``, ``dsa_fused_decode``, ``dsa_indexer_topk_shard``, ``dsa_topk_merge``,
``dsa_sparse_attn_shard``, ``dsa_attn_combine``) on torch tensors of the current CUDA device.  The
exchanges are ``torch.distributed`` all-gathers (NCCL between GPUs; any backend works for the host
logic).  Everything here that is not a collective is a pure function of the sizes, so the per-rank steps
can also be run one after another in one process and reassembled with the same functions.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence, Tuple

import numpy as np

# ----------------------------------------------------------------------------------------------------
# Zigzag partition of a prefill chunk
# ----------------------------------------------------------------------------------------------------


def zigzag_segments(n_new: int, world: int) -> List[Tuple[int, int]]:
    """The 2*world segments [start, end) of query indices 0..n_new-1, lengths differing by at most one."""
    if world < 1 or n_new < 0:
        raise ValueError(f"need world >= 1 and n_new >= 0 (got {world}, {n_new})")
    m = 2 * world
    base, extra = divmod(n_new, m)
    segs, s = [], 0
    for i in range(m):
        e = s + base + (1 if i < extra else 0)
        segs.append((s, e))
        s = e
    return segs


def zigzag_rank_segments(n_new: int, world: int, rank: int) -> List[Tuple[int, int]]:
    """The two segments of rank `rank`: number rank (early, cheap) and number 2*world-1-rank (late)."""
    segs = zigzag_segments(n_new, world)
    return [segs[rank], segs[2 * world - 1 - rank]]


def zigzag_rank_queries(n_new: int, world: int, rank: int) -> np.ndarray:
    """Query indices (0..n_new-1) of one rank, in the order its outputs are laid out."""
    return np.concatenate([np.arange(s, e, dtype=np.int64) for s, e in zigzag_rank_segments(n_new, world, rank)])


def causal_work(cached: int, queries: Sequence[int]) -> int:
    """Positions scored by the given queries of a chunk appended after `cached` tokens: sum of (p + 1)."""
    q = np.asarray(queries, dtype=np.int64)
    return int(np.sum(cached + q + 1))


def rank_loads(cached: int, n_new: int, world: int, layout: str = "zigzag") -> List[int]:
    """Causal work of every rank under the zigzag layout or the plain contiguous split (for comparison)."""
    if layout == "zigzag":
        return [causal_work(cached, zigzag_rank_queries(n_new, world, r)) for r in range(world)]
    if layout == "contiguous":
        base, extra = divmod(n_new, world)
        out, s = [], 0
        for r in range(world):
            e = s + base + (1 if r < extra else 0)
            out.append(causal_work(cached, range(s, e)))
            s = e
        return out
    raise ValueError(layout)


@dataclass
class RankBatch:
    """A rank's share of a one-sequence prefill chunk, as the library's batch of sequences: each of its two
    segments is a sequence of its own whose newest tokens are that segment's queries (same page-table row,
    length up to the segment's last position)."""

    queries: np.ndarray     # query indices of the chunk, in output order
    seq_lens: np.ndarray    # int32 [2]
    cu_q_lens: np.ndarray   # int32 [3]
    max_q_len: int


def zigzag_rank_batch(cached: int, n_new: int, world: int, rank: int) -> RankBatch:
    segs = zigzag_rank_segments(n_new, world, rank)
    seq_lens = np.array([cached + e for _, e in segs], dtype=np.int32)
    lens = [e - s for s, e in segs]
    cu = np.array([0, lens[0], lens[0] + lens[1]], dtype=np.int32)
    return RankBatch(queries=zigzag_rank_queries(n_new, world, rank), seq_lens=seq_lens, cu_q_lens=cu,
                     max_q_len=max(max(lens), 1))


def zigzag_rank_dims(dims, cached: int, n_new: int, world: int, rank: int):
    """The library dims of one rank's share (dims: those of the whole chunk)."""
    rb = zigzag_rank_batch(cached, n_new, world, rank)
    return _dims_like(dims, batch=2, total_q=int(rb.cu_q_lens[-1]), max_q_len=rb.max_q_len)


def zigzag_workspace_size(dims, cached: int, n_new: int, world: int) -> int:
    """Workspace bytes a rank needs for zigzag_prefill_rank: the largest of the whole chunk's (the append)
    and every rank's share (fewer query tokens may let the attention split positions and use scratch)."""
    from ._lib import workspace_size

    return max([workspace_size(dims)] +
               [workspace_size(zigzag_rank_dims(dims, cached, n_new, world, r)) for r in range(world)])


def zigzag_reassemble(n_new: int, world: int, per_rank: Sequence[np.ndarray]) -> np.ndarray:
    """Rows of every rank's output (in that rank's output order) put back in chunk order."""
    first = np.asarray(per_rank[0])
    out = np.empty((n_new,) + first.shape[1:], dtype=first.dtype)
    for r in range(world):
        out[zigzag_rank_queries(n_new, world, r)] = np.asarray(per_rank[r])
    return out


# ----------------------------------------------------------------------------------------------------
# Context shards for decode
# ----------------------------------------------------------------------------------------------------

OPEN_END = 2 ** 31 - 1


def context_shards(max_ctx: int, world: int) -> List[Tuple[int, int]]:
    """world contiguous, page-aligned (64-position) ranges covering [0, max_ctx); the last one open-ended."""
    if world < 1 or max_ctx < 1:
        raise ValueError(f"need world >= 1 and max_ctx >= 1 (got {world}, {max_ctx})")
    per = -(-max_ctx // world)
    per = -(-per // 64) * 64
    return [(r * per, (r + 1) * per if r + 1 < world else OPEN_END) for r in range(world)]


# ----------------------------------------------------------------------------------------------------
# Collectives (torch.distributed); the sizes of a rank's rows may differ by one segment length
# ----------------------------------------------------------------------------------------------------


def all_gather_rows(group, tensor, counts: Sequence[int]):
    """All-gather a tensor whose leading dimension is counts[rank] on each rank (padded to the largest
    count for the exchange).  Returns the list of every rank's tensor, trimmed."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    m = max(int(c) for c in counts)
    shape = tuple(tensor.shape[1:])
    # rows travel as raw bytes, so any element type goes through any process-group backend
    raw = tensor.contiguous().reshape(tensor.shape[0], -1).view(torch.uint8)
    pad = torch.zeros((m, raw.shape[1]), dtype=torch.uint8, device=tensor.device)
    pad[: raw.shape[0]] = raw
    bufs = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(bufs, pad, group=group)
    return [b[: int(c)].view(tensor.dtype).reshape((int(c),) + shape) for b, c in zip(bufs, counts)]


# ----------------------------------------------------------------------------------------------------
# Backends: the device work of one rank
# ----------------------------------------------------------------------------------------------------


class CudaBackend:
    """The library's C ABI on torch tensors of the current CUDA device (dims: a DsaDims for the call)."""

    def __init__(self, stream=None):
        from . import _lib

        self.lib = _lib
        self.stream = stream

    def append(self, dims, k_new, kv_new, page_table, seq_lens, cu_q_lens, k_cache, k_scale, kv_cache, workspace):
        self.lib.append_rows(dims, k_new, kv_new, page_table, seq_lens, cu_q_lens, k_cache, k_scale, kv_cache,
                             workspace, self.stream)

    def step(self, dims, q_idx, q_scale, w, k_cache, k_scale, q, kv_cache, page_table, seq_lens, cu_q_lens, topk,
             out, lse, workspace):
        self.lib.fused_decode(dims, q_idx, q_scale, w, k_cache, k_scale, q, kv_cache, page_table, seq_lens, cu_q_lens,
                              topk, out, lse, workspace, self.stream)

    def indexer_shard(self, dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, lo, hi, topk,
                      score, workspace):
        self.lib.indexer_topk_shard(dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, lo,
                                    hi, topk, score, workspace, self.stream)

    def merge(self, shards, total_q, top_k, idx, score, out_idx, out_score):
        self.lib.topk_merge(shards, total_q, top_k, idx, score, out_idx, out_score, self.stream)

    def attn_shard(self, dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk, lo, hi, out, lse, workspace):
        self.lib.sparse_attn_shard(dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk, lo, hi, out, lse,
                                   workspace, self.stream)

    def combine(self, shards, total_q, heads, v_dim, outs, lses, out, lse):
        self.lib.attn_combine(shards, total_q, heads, v_dim, outs, lses, out, lse, self.stream)


def _dims_like(dims, **override):
    from ._lib import DsaDims

    d = DsaDims()
    for name, _ in DsaDims._fields_:
        setattr(d, name, getattr(dims, name))
    for k, v in override.items():
        setattr(d, k, v)
    return d


# ----------------------------------------------------------------------------------------------------
# Zigzag prefill step of one rank
# ----------------------------------------------------------------------------------------------------


def zigzag_prefill_rank(backend, group, rank: int, world: int, dims, cached: int, n_new: int, mine: dict,
                        cache: dict, workspace):
    """One rank's part of a Zigzag-parallel prefill of one sequence (cached tokens + n_new new ones).

    dims: the library dims of the whole chunk (batch 1, total_q = n_new, seq_lens [cached + n_new]).
    mine: this rank's query-side tensors in its output order (zigzag_rank_queries): q_idx, q_scale (or
      None), w, q, and its tokens' new cache rows k_new [T_r, Di] (bf16) and kv_new [T_r, D] (bf16).
    cache: this rank's paged caches and page table: k_cache, k_scale (or None), kv_cache, page_table
      [1, max_pages] (int32), on the device.
    workspace: zigzag_workspace_size(...) bytes, zero-filled before first use.
    Returns (topk [n_new, K], out [n_new, Hq, Dv], lse [n_new, Hq]) of the whole chunk in chunk order,
    the same on every rank.
    """
    import torch

    dev = mine["q"].device
    counts = [len(zigzag_rank_queries(n_new, world, r)) for r in range(world)]
    # 1. every rank's new rows, so that every cache holds the whole chunk (the indexer K cache all-gather)
    k_parts = all_gather_rows(group, mine["k_new"], counts)
    kv_parts = all_gather_rows(group, mine["kv_new"], counts)
    order = np.concatenate([zigzag_rank_queries(n_new, world, r) for r in range(world)])
    inv = torch.as_tensor(np.argsort(order), device=dev)
    k_new = torch.cat(k_parts)[inv].contiguous()
    kv_new = torch.cat(kv_parts)[inv].contiguous()
    seq_full = torch.tensor([cached + n_new], dtype=torch.int32, device=dev)
    cu_full = torch.tensor([0, n_new], dtype=torch.int32, device=dev)
    backend.append(dims, k_new, kv_new, cache["page_table"], seq_full, cu_full, cache["k_cache"],
                   cache.get("k_scale"), cache["kv_cache"], workspace)
    # 2. this rank's queries: two sequences sharing the page-table row
    rb = zigzag_rank_batch(cached, n_new, world, rank)
    T_r = int(rb.cu_q_lens[-1])
    d_r = zigzag_rank_dims(dims, cached, n_new, world, rank)
    pt2 = cache["page_table"].expand(2, -1).contiguous()
    seq_r = torch.as_tensor(rb.seq_lens, device=dev)
    cu_r = torch.as_tensor(rb.cu_q_lens, device=dev)
    K, Hq, Dv = dims.top_k, dims.attn_heads, dims.v_dim
    topk = torch.empty((T_r, K), dtype=torch.int32, device=dev)
    out = torch.empty((T_r, Hq, Dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((T_r, Hq), dtype=torch.float32, device=dev)
    backend.step(d_r, mine["q_idx"], mine.get("q_scale"), mine["w"], cache["k_cache"], cache.get("k_scale"), mine["q"],
                 cache["kv_cache"], pt2, seq_r, cu_r, topk, out, lse, workspace)
    # 3. every rank's outputs, back in chunk order
    res = []
    for t in (topk, out, lse):
        parts = all_gather_rows(group, t, counts)
        res.append(torch.cat(parts)[inv].contiguous())
    return tuple(res)


# ----------------------------------------------------------------------------------------------------
# Decode by context shards, one rank
# ----------------------------------------------------------------------------------------------------


def context_decode_rank(backend, group, rank: int, world: int, dims, lo: int, hi: int, queries: dict, cache: dict,
                        workspace):
    """One rank's part of a decode step whose sequences are sharded by position: this rank holds positions
    [lo, hi) in its caches (its page table names only those pages).

    queries: q_idx, q_scale (or None), w, q, seq_lens, cu_q_lens of the whole batch (replicated).
    Returns (topk [T, K], out [T, Hq, Dv], lse [T, Hq]), the same on every rank.
    """
    import torch
    import torch.distributed as dist

    dev = queries["q"].device
    T, K, Hq, Dv = dims.total_q, dims.top_k, dims.attn_heads, dims.v_dim
    idx = torch.empty((T, K), dtype=torch.int32, device=dev)
    score = torch.empty((T, K), dtype=torch.float32, device=dev)
    backend.indexer_shard(dims, queries["q_idx"], queries.get("q_scale"), queries["w"], cache["k_cache"],
                          cache.get("k_scale"), cache["page_table"], queries["seq_lens"], queries["cu_q_lens"], lo, hi,
                          idx, score, workspace)
    # local (position, score) lists of every shard, then the global Top-K with the same key
    idx_all = [torch.empty_like(idx) for _ in range(world)]
    score_all = [torch.empty_like(score) for _ in range(world)]
    dist.all_gather(idx_all, idx, group=group)
    dist.all_gather(score_all, score, group=group)
    topk = torch.empty((T, K), dtype=torch.int32, device=dev)
    backend.merge(world, T, K, torch.stack(idx_all).contiguous(), torch.stack(score_all).contiguous(), topk, None)
    # partial attention over the selected rows this shard holds, then the log-sum-exp combine
    out_p = torch.empty((T, Hq, Dv), dtype=torch.bfloat16, device=dev)
    lse_p = torch.empty((T, Hq), dtype=torch.float32, device=dev)
    backend.attn_shard(dims, queries["q"], cache["kv_cache"], cache["page_table"], queries["seq_lens"],
                       queries["cu_q_lens"], topk, lo, hi, out_p, lse_p, workspace)
    outs = [torch.empty_like(out_p) for _ in range(world)]
    lses = [torch.empty_like(lse_p) for _ in range(world)]
    dist.all_gather(outs, out_p, group=group)
    dist.all_gather(lses, lse_p, group=group)
    out = torch.empty_like(out_p)
    lse = torch.empty_like(lse_p)
    backend.combine(world, T, Hq, Dv, torch.stack(outs).contiguous(), torch.stack(lses).contiguous(), out, lse)
    return topk, out, lse
