"""Device-side helpers for the GPU tests: upload a workload, call the library through the C ABI, compare
with the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_attention_dsa_gb300 as dsa
from sparse_attention_dsa_gb300 import build as dsa_build

from _util import topk_mismatch

ATOL, RTOL = 2e-2, 1e-2  # attention outputs: |gpu - oracle| <= ATOL + RTOL * |oracle| (bf16 out, fp32 accumulation)


def ensure_built():
    dsa_build.build()
    dsa.lib()


def dims_for(wl, **override) -> dsa.DsaDims:
    d = dsa.DsaDims(batch=wl.batch, total_q=wl.total_q, max_q_len=wl.max_q_len, num_pages=wl.num_pages,
                    page_size=wl.page_size, max_pages_per_seq=wl.max_pages_per_seq, idx_heads=wl.idx_heads,
                    idx_dim=wl.idx_dim,
                    idx_dtype=(dsa.DSA_MXFP8_E4M3 if getattr(wl, "idx_mx", False) else dsa.DSA_FP8_E4M3)
                    if wl.idx_fp8 else dsa.DSA_BF16,
                    top_k=wl.top_k, attn_heads=wl.attn_heads, kv_dim=wl.kv_dim, v_dim=wl.v_dim,
                    softmax_scale=wl.softmax_scale,
                    kv_dtype=dsa.DSA_FP8_E4M3 if getattr(wl, "kv_fp8", False) else dsa.DSA_BF16)
    for k, v in override.items():
        setattr(d, k, v)
    return d


def _dev(a, device="cuda"):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


class DeviceWorkload:
    """A workload resident on the GPU, plus output buffers and a zeroed workspace."""

    def __init__(self, wl, device="cuda"):
        self.wl = wl
        self.dims = dims_for(wl)
        self.q_idx = _dev(wl.q_idx, device)
        self.q_scale = _dev(wl.q_scale, device)
        self.w = _dev(wl.w, device)
        self.k_cache = _dev(wl.k_cache, device)
        self.k_scale = _dev(wl.k_scale, device)
        self.q = _dev(wl.q, device)
        self.kv_cache = _dev(wl.kv_cache, device)
        self.page_table = _dev(wl.page_table, device)
        self.seq_lens = _dev(wl.seq_lens, device)
        self.cu_q_lens = _dev(wl.cu_q_lens, device)
        T = max(wl.total_q, 1)
        self.topk = torch.full((T, wl.top_k), -7, dtype=torch.int32, device=device)
        self.out = torch.zeros((T, wl.attn_heads, wl.v_dim), dtype=torch.bfloat16, device=device)
        self.lse = torch.zeros((T, wl.attn_heads), dtype=torch.float32, device=device)
        ws = dsa.workspace_size(self.dims)
        self.workspace = torch.zeros((ws + 3) // 4, dtype=torch.int32, device=device)

    def indexer(self, dims=None):
        dsa.indexer_topk(dims or self.dims, self.q_idx, self.q_scale, self.w, self.k_cache, self.k_scale,
                         self.page_table, self.seq_lens, self.cu_q_lens, self.topk, self.workspace)
        return self

    def sfa(self, topk=None, dims=None):
        t = self.topk if topk is None else topk
        dsa.sparse_attn(dims or self.dims, self.q, self.kv_cache, self.page_table, self.seq_lens, self.cu_q_lens, t,
                        self.out, self.lse, self.workspace)
        return self

    def fused(self, dims=None):
        dsa.fused_decode(dims or self.dims, self.q_idx, self.q_scale, self.w, self.k_cache, self.k_scale, self.q,
                         self.kv_cache, self.page_table, self.seq_lens, self.cu_q_lens, self.topk, self.out, self.lse,
                         self.workspace)
        return self

    def error_word(self) -> int:
        return dsa.get_device_error(self.workspace)

    def topk_host(self):
        torch.cuda.synchronize()
        return self.topk.cpu().numpy()

    def out_host(self):
        torch.cuda.synchronize()
        return self.out.float().cpu().numpy().astype(np.float64), self.lse.cpu().numpy().astype(np.float64)


def check_topk(wl, gpu_topk, tlist=None):
    """Top-K parity for the listed tokens (default: all).  Returns the number of excused positions.

    The oracle's scores of every visible position are computed only for the tokens whose selection differs
    from the oracle's as a set (they decide whether the difference lies inside the excusal band)."""
    tlist = list(range(wl.total_q)) if tlist is None else list(tlist)
    ref, kth, nsel = oracle.indexer_topk(wl, tlist)
    differ = [i for i, t in enumerate(tlist)
              if np.setxor1d(gpu_topk[t][gpu_topk[t] >= 0], ref[i][ref[i] >= 0]).shape[0] > 0]
    scores = dict(zip(differ, oracle.index_scores_batch(wl, [tlist[i] for i in differ]))) if differ else {}
    pos = wl.query_positions()
    excused = 0
    for i, t in enumerate(tlist):
        sc = scores[i] if i in scores else np.zeros(int(pos[t]) + 1)  # unused when the sets agree
        msg = topk_mismatch(gpu_topk[t], ref[i], sc, kth[i], nsel[i])
        assert msg is None, f"token {t}: {msg}"
        g = gpu_topk[t][gpu_topk[t] >= 0]
        excused += int(np.setxor1d(g, ref[i][ref[i] >= 0]).shape[0])
        assert np.all(np.diff(g) > 0), f"token {t}: selection not in ascending order"
        assert np.all(gpu_topk[t][nsel[i]:] == -1), f"token {t}: padding is not -1"
    return excused


def check_attention(wl, topk_rows, gpu_out, gpu_lse, tlist=None):
    """Attention parity for the listed tokens, evaluated by the oracle on the given selections."""
    tlist = list(range(wl.total_q)) if tlist is None else list(tlist)
    sel = np.ascontiguousarray(np.asarray(topk_rows)[tlist], dtype=np.int32)
    ref_out, ref_lse = oracle.sparse_attn(wl, sel, tlist)
    go, gl = gpu_out[tlist], gpu_lse[tlist]
    err = np.abs(go - ref_out)
    bad = err > ATOL + RTOL * np.abs(ref_out)
    assert not bad.any(), (f"{int(bad.sum())} output elements out of tolerance; worst abs err {err.max():.4g} "
                           f"at {np.unravel_index(np.argmax(err), err.shape)}")
    finite = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(gl), finite)
    lerr = np.abs(gl[finite] - ref_lse[finite])
    assert np.all(lerr <= ATOL + RTOL * np.abs(ref_lse[finite])), f"lse worst abs err {lerr.max():.4g}"
    return float(err.max())
