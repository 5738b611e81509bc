"""The device steps of ``sparse_attention_dsa_gb300.cp`` computed by the CPU oracle on torch CPU tensors.

Test infrastructure only: it lets the multi-process (gloo) tests run the context-parallel orchestration
-- partition, all-gathers, reassembly -- on CPU ranks, with every step's arithmetic done by the oracle.
Tensors follow the library's conventions: bf16 data as int16 bit patterns or torch.bfloat16, positions
int32, scores and lse fp32.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from gen import f32_to_bf16
from gen.workloads import Workload


def _np(t):
    if t is None:
        return None
    a = t.detach().cpu()
    if a.dtype == torch.bfloat16:
        a = a.view(torch.int16)
    a = a.numpy()
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a)


def _workload(dims, *, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, q=None, kv_cache=None):
    fp8 = dims.idx_dtype != 0
    return Workload(name="cp", seed=0, seq_lens=_np(seq_lens).astype(np.int32), cu_q_lens=_np(cu_q_lens).astype(np.int32),
                    page_size=dims.page_size, page_table=_np(page_table).astype(np.int32), num_pages=dims.num_pages,
                    idx_heads=dims.idx_heads, idx_dim=dims.idx_dim, idx_fp8=fp8,
                    q_idx=_np(q_idx).astype(np.uint8 if fp8 else np.uint16), q_scale=_np(q_scale), w=_np(w),
                    k_cache=_np(k_cache).astype(np.uint8 if fp8 else np.uint16), k_scale=_np(k_scale),
                    top_k=dims.top_k, attn_heads=dims.attn_heads, kv_dim=dims.kv_dim, v_dim=dims.v_dim,
                    softmax_scale=float(dims.softmax_scale), q=_np(q), kv_cache=_np(kv_cache))


def _write_bf16(dst, x64):
    bits = f32_to_bf16(np.asarray(x64, dtype=np.float32))
    dst.copy_(torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(dst.shape))


def _select(scores, lo, hi, K):
    """Top-K of the positions in [lo, min(hi, n)) by (fp32 score desc, position asc), ascending; padded."""
    n = scores.shape[0]
    pos = np.arange(lo, max(lo, min(hi, n)))
    sc = scores[pos].astype(np.float32)
    order = np.lexsort((pos, -sc.astype(np.float64)))[:K]
    sel = np.sort(pos[order])
    idx = np.full(K, -1, np.int32)
    score = np.full(K, -np.inf, np.float32)
    idx[: sel.shape[0]] = sel
    score[: sel.shape[0]] = scores[sel].astype(np.float32)
    return idx, score


class OracleBackend:
    def append(self, dims, k_new, kv_new, page_table, seq_lens, cu_q_lens, k_cache, k_scale, kv_cache, workspace):
        wl = _workload(dims, q_idx=torch.zeros(1, dtype=torch.int16), q_scale=None, w=torch.zeros(1),
                       k_cache=k_cache, k_scale=k_scale, page_table=page_table, seq_lens=seq_lens,
                       cu_q_lens=cu_q_lens, kv_cache=kv_cache)
        kc, ks, kvc = oracle.append(wl, _np(k_new), _np(kv_new))
        k_cache.copy_(torch.from_numpy(kc.view(np.int16) if kc.dtype == np.uint16 else kc))
        if k_scale is not None:
            k_scale.copy_(torch.from_numpy(ks))
        kv_cache.copy_(torch.from_numpy(kvc.view(np.int16)))

    def step(self, dims, q_idx, q_scale, w, k_cache, k_scale, q, kv_cache, page_table, seq_lens, cu_q_lens, topk, out,
             lse, workspace):
        wl = _workload(dims, q_idx=q_idx, q_scale=q_scale, w=w, k_cache=k_cache, k_scale=k_scale,
                       page_table=page_table, seq_lens=seq_lens, cu_q_lens=cu_q_lens, q=q, kv_cache=kv_cache)
        sel, _, _ = oracle.indexer_topk(wl)
        o, l = oracle.sparse_attn(wl, sel)
        topk.copy_(torch.from_numpy(sel))
        _write_bf16(out, o)
        lse.copy_(torch.from_numpy(l.astype(np.float32)))

    def indexer_shard(self, dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, lo, hi, topk,
                      score, workspace):
        wl = _workload(dims, q_idx=q_idx, q_scale=q_scale, w=w, k_cache=k_cache, k_scale=k_scale,
                       page_table=page_table, seq_lens=seq_lens, cu_q_lens=cu_q_lens)
        T, K = wl.total_q, wl.top_k
        pos = wl.query_positions()
        for t in range(T):
            # every rank of these CPU tests holds the whole cache; the shard range restricts the candidates
            i, s = _select(oracle.index_scores(wl, t), lo, hi, K)
            topk[t] = torch.from_numpy(i)
            score[t] = torch.from_numpy(s)

    def merge(self, shards, total_q, top_k, idx, score, out_idx, out_score):
        I, S = _np(idx), _np(score)
        for t in range(total_q):
            cand_i = I[:, t, :].reshape(-1)
            cand_s = S[:, t, :].reshape(-1).astype(np.float64)
            ok = cand_i >= 0
            ci, cs = cand_i[ok], cand_s[ok]
            keep = np.lexsort((ci, -cs))[:top_k]
            mask = np.zeros(ci.shape[0], bool)
            mask[keep] = True
            chosen = ci[mask]  # candidate order
            out_idx[t] = -1
            out_idx[t, : chosen.shape[0]] = torch.from_numpy(chosen.astype(np.int32))
            if out_score is not None:
                out_score[t] = -np.inf
                out_score[t, : chosen.shape[0]] = torch.from_numpy(cs[mask].astype(np.float32))

    def attn_shard(self, dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk, lo, hi, out, lse, workspace):
        wl = _workload(dims, q_idx=torch.zeros(1, dtype=torch.int16), q_scale=None, w=torch.zeros(1),
                       k_cache=torch.zeros((dims.num_pages, 64, dims.idx_dim), dtype=torch.int16), k_scale=None,
                       page_table=page_table, seq_lens=seq_lens, cu_q_lens=cu_q_lens, q=q, kv_cache=kv_cache)
        sel = _np(topk).copy()
        sel[(sel < lo) | (sel >= hi)] = -1
        o, l = oracle.sparse_attn(wl, sel)
        _write_bf16(out, o)
        lse.copy_(torch.from_numpy(l.astype(np.float32)))

    def combine(self, shards, total_q, heads, v_dim, outs, lses, out, lse):
        O = _np(outs)
        Ov = (O.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        L = _np(lses).astype(np.float64)
        m = L.max(axis=0)
        wgt = np.where(np.isneginf(L), 0.0, np.exp(L - np.where(np.isneginf(m), 0.0, m)[None]))
        tot = wgt.sum(axis=0)
        res = np.where(tot[..., None] > 0, (wgt[..., None] * Ov).sum(axis=0) / np.where(tot > 0, tot, 1.0)[..., None],
                       0.0)
        _write_bf16(out, res)
        lse.copy_(torch.from_numpy(np.where(tot > 0, m + np.log(np.where(tot > 0, tot, 1.0)), -np.inf).astype(np.float32)))

