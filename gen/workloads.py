"""Seeded synthetic DSA workloads: paged indexer K cache, paged latent-KV cache, queries, head weights.

Shapes follow the five decode/prefill configurations of the fused-indexer + sparse-flash-attention path:

====  ==============================================================================================
cfg   workload
====  ==============================================================================================
1     decode, B=1, ctx 4096, 1 query; indexer 4 heads x 64-d bf16, w ~ U(0,1); K=256; SFA 16 x 576
2     decode, B=32, ctx 32768, 1 query; indexer 64 x 128-d bf16, w ~ U(0,1)/8, 1% of k rows x4;
      K=2048; SFA 128 x 576
3     as 2 with the indexer q/k in FP8 E4M3 and per-row fp32 scales (absmax/448)
4     prefill chunk: B=1, 61440 cached + 4096 new = 65536, causal; indexer 64 x 128 bf16; K=2048
5     varlen decode: B=8, ctx ~ U{16384..131072}, 2 causal queries; indexer 64 x 128 FP8; K=2048
====  ==============================================================================================

Recipe (identical for every config and for the small test cases):

* seed = 1000 + config number; each tensor draws from its own SplitMix64 stream (seed, tensor id).
* Activations ~ N(0,1) (Irwin-Hall 12) rounded to bf16; head weights ~ U(0, w_hi) in fp32.
* Page table: physical page ids are a Fisher-Yates permutation of [0, sum_b ceil(L_b/64)), dealt in
  (sequence, logical page) order; unused entries are -1.  Tail slots of a partial last page are zero.
* Logical row (b, s) of a cache draws the same numbers whatever page holds it, so permuting pages
  leaves the logical content unchanged.
* Salient positions (configs 2/3): floor(1% of L_b) rows per sequence, drawn without replacement,
  have their indexer key multiplied by 4 (exact in bf16).
* FP8 inputs: bf16 values quantised per row (one row = one token's 128-d key, or one (token, head)
  query row) with scale = absmax/448.
* MXFP8 indexer inputs (idx_mx): the same bf16 rows quantised with one E8M0 scale per 32 elements
  (shared exponent floor(log2(absmax)) - 8); scales are bytes [..., Di / 32].
* FP8 latent-KV cache (kv_fp8): the same bf16 rows, each 128-dim tile of the leading Dv dims quantised
  with its own absmax/448 scale; row layout 656 bytes = Dv codes, Dv/128 fp32 scales, the remaining
  (rotary) dims as bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

from . import (
    f32_to_bf16,
    bf16_to_f32,
    normal_bf16,
    paged_normal_bf16,
    permutation,
    quantize_e4m3_rows,
    quantize_mx_rows,
    sample_without_replacement,
    stream_key,
    uniform_f32,
    uniform_int,
)

PAGE_SIZE = 64

T_QIDX, T_W, T_KIDX, T_Q, T_KV, T_PT, T_LEN, T_SALIENT = 1, 2, 3, 4, 5, 6, 7, 8


@dataclass
class Workload:
    name: str
    seed: int
    seq_lens: np.ndarray  # int32 [B]
    cu_q_lens: np.ndarray  # int32 [B+1]
    page_size: int
    page_table: np.ndarray  # int32 [B, max_pages_per_seq]
    num_pages: int
    idx_heads: int
    idx_dim: int
    idx_fp8: bool
    q_idx: np.ndarray  # bf16 bits uint16 [T, Hi, Di] or E4M3 codes uint8
    q_scale: Optional[np.ndarray]  # f32 [T, Hi] (FP8 only)
    w: np.ndarray  # f32 [T, Hi]
    k_cache: np.ndarray  # bf16 bits uint16 [P, 64, Di] or E4M3 codes uint8
    k_scale: Optional[np.ndarray]  # f32 [P, 64] (FP8 only)
    top_k: int
    attn_heads: int
    kv_dim: int
    v_dim: int
    softmax_scale: float
    q: Optional[np.ndarray] = None  # bf16 bits uint16 [T, Hq, kv_dim]
    kv_cache: Optional[np.ndarray] = None  # bf16 bits uint16 [P, 64, kv_dim], or uint8 [P, 64, 656] (kv_fp8)
    notes: dict = field(default_factory=dict)
    kv_fp8: bool = False
    idx_mx: bool = False  # with idx_fp8: q/k scales are E8M0 bytes per 32 elements (MXFP8)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.cu_q_lens[-1])

    @property
    def max_q_len(self) -> int:
        return int(np.max(np.diff(self.cu_q_lens))) if self.batch else 0

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.page_table.shape[1])

    def query_positions(self) -> np.ndarray:
        """Absolute cache position of every query token (the newest tokens of each sequence)."""
        pos = np.empty(self.total_q, dtype=np.int64)
        for b in range(self.batch):
            lo, hi = int(self.cu_q_lens[b]), int(self.cu_q_lens[b + 1])
            n = hi - lo
            pos[lo:hi] = int(self.seq_lens[b]) - n + np.arange(n)
        return pos

    def query_seq(self) -> np.ndarray:
        out = np.empty(self.total_q, dtype=np.int64)
        for b in range(self.batch):
            out[self.cu_q_lens[b]:self.cu_q_lens[b + 1]] = b
        return out

    def logical_rows(self, cache: np.ndarray, b: int) -> np.ndarray:
        """Rows 0..L_b-1 of sequence b gathered from a paged cache (for inspection and tests)."""
        L = int(self.seq_lens[b])
        s = np.arange(L)
        pages = self.page_table[b, s // self.page_size]
        return cache[pages, s % self.page_size]


def build_page_table(seed: int, seq_lens: Sequence[int], page_size: int = PAGE_SIZE, max_pages: Optional[int] = None):
    seq_lens = [int(x) for x in seq_lens]
    need = [max(0, math.ceil(L / page_size)) for L in seq_lens]
    total = sum(need)
    mp = max(need) if max_pages is None else max_pages
    mp = max(mp, 1)
    perm = permutation(stream_key(seed, T_PT), total)
    pt = np.full((len(seq_lens), mp), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[off:off + n]
        off += n
    return pt, max(total, 1)


def make_workload(name: str, seed: int, seq_lens: Sequence[int], q_lens: Sequence[int], *, idx_heads: int,
                  idx_dim: int, idx_fp8: bool, top_k: int, attn_heads: int, kv_dim: int = 576, v_dim: int = 512,
                  w_hi: float = 1.0, salient_frac: float = 0.0, salient_mult: float = 4.0,
                  page_size: int = PAGE_SIZE, softmax_scale: Optional[float] = None, with_sfa: bool = True,
                  page_seed: Optional[int] = None, kv_fp8: bool = False, idx_mx: bool = False) -> Workload:
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    q_lens = np.asarray(q_lens, dtype=np.int32)
    assert seq_lens.shape == q_lens.shape
    assert np.all(q_lens <= seq_lens), "each sequence must already hold its query tokens"
    cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(q_lens)
    T = int(cu[-1])
    pt, num_pages = build_page_table(seed if page_seed is None else page_seed, seq_lens, page_size)
    row_stride_b = pt.shape[1] * page_size

    q_idx = normal_bf16(stream_key(seed, T_QIDX), T * idx_heads * idx_dim).reshape(T, idx_heads, idx_dim)
    w = uniform_f32(stream_key(seed, T_W), T * idx_heads, 0.0, w_hi).reshape(T, idx_heads)
    k_cache = paged_normal_bf16(stream_key(seed, T_KIDX), seq_lens, pt, page_size, idx_dim, row_stride_b, num_pages)
    notes = {}
    if salient_frac > 0:
        sal_key = stream_key(seed, T_SALIENT)
        n_sal = 0
        for b, L in enumerate(seq_lens):
            m = int(math.floor(salient_frac * int(L)))
            if m == 0:
                continue
            rows = sample_without_replacement(sal_key ^ (b * 0x9E3779B97F4A7C15 & (2**64 - 1)), int(L), m)
            pages = pt[b, rows // page_size]
            slots = rows % page_size
            vals = bf16_to_f32(k_cache[pages, slots]) * np.float32(salient_mult)
            k_cache[pages, slots] = f32_to_bf16(vals)
            n_sal += m
        notes["salient_rows"] = n_sal
    q_scale = k_scale = None
    if idx_fp8 and idx_mx:
        q_idx, q_scale = quantize_mx_rows(q_idx)
        k_cache, k_scale = quantize_mx_rows(k_cache)
    elif idx_fp8:
        q_idx, q_scale = quantize_e4m3_rows(q_idx)
        k_cache, k_scale = quantize_e4m3_rows(k_cache)
    q = kv = None
    if with_sfa:
        q = normal_bf16(stream_key(seed, T_Q), T * attn_heads * kv_dim).reshape(T, attn_heads, kv_dim)
        kv = paged_normal_bf16(stream_key(seed, T_KV), seq_lens, pt, page_size, kv_dim, row_stride_b, num_pages)
        if kv_fp8:
            kv = kv_rows_to_fp8(kv, v_dim)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(kv_dim)
    return Workload(name=name, seed=seed, seq_lens=seq_lens, cu_q_lens=cu, page_size=page_size, page_table=pt,
                    num_pages=num_pages, idx_heads=idx_heads, idx_dim=idx_dim, idx_fp8=idx_fp8, q_idx=q_idx,
                    q_scale=q_scale, w=w, k_cache=k_cache, k_scale=k_scale, top_k=top_k, attn_heads=attn_heads,
                    kv_dim=kv_dim, v_dim=v_dim, softmax_scale=float(softmax_scale), q=q, kv_cache=kv, notes=notes,
                    kv_fp8=bool(kv_fp8 and with_sfa), idx_mx=bool(idx_fp8 and idx_mx))


def kv_fp8_row_bytes(kv_dim: int = 576, v_dim: int = 512) -> int:
    return v_dim + 4 * (v_dim // 128) + 2 * (kv_dim - v_dim)


def kv_rows_to_fp8(kv_bf16: np.ndarray, v_dim: int = 512) -> np.ndarray:
    """bf16-bits rows [..., kv_dim] -> uint8 rows [..., 656] in the FP8 latent-KV layout (input synthesis)."""
    kv = np.ascontiguousarray(kv_bf16, dtype=np.uint16)
    lead, kv_dim = kv.shape[:-1], kv.shape[-1]
    n = int(np.prod(lead)) if lead else 1
    flat = kv.reshape(n, kv_dim)
    tiles = np.ascontiguousarray(flat[:, :v_dim]).reshape(n * (v_dim // 128), 128)
    codes, scales = quantize_e4m3_rows(tiles)
    out = np.empty((n, kv_fp8_row_bytes(kv_dim, v_dim)), dtype=np.uint8)
    out[:, :v_dim] = codes.reshape(n, v_dim)
    out[:, v_dim:v_dim + 4 * (v_dim // 128)] = scales.reshape(n, v_dim // 128).view(np.uint8).reshape(n, -1)
    out[:, v_dim + 4 * (v_dim // 128):] = np.ascontiguousarray(flat[:, v_dim:]).view(np.uint8).reshape(n, -1)
    return out.reshape(*lead, out.shape[-1])


CONFIG_NAMES = {
    1: "decode_b1_ctx4096_hi4x64_bf16_k256_hq16",
    2: "decode_b32_ctx32768_hi64x128_bf16_k2048_hq128",
    3: "decode_b32_ctx32768_hi64x128_fp8_k2048_hq128",
    4: "prefill_b1_ctx65536_q4096_hi64x128_bf16_k2048_hq128",
    5: "varlen_decode_b8_ctx16k-128k_q2_hi64x128_fp8_k2048_hq128",
}


def config_lengths(n: int, seed: Optional[int] = None):
    """(seq_lens, q_lens) of configuration n."""
    seed = 1000 + n if seed is None else seed
    if n == 1:
        return [4096], [1]
    if n in (2, 3):
        return [32768] * 32, [1] * 32
    if n == 4:
        return [65536], [4096]
    if n == 5:
        lens = uniform_int(stream_key(seed, T_LEN), 8, 16384, 131072)
        return [int(x) for x in lens], [2] * 8
    raise ValueError(n)


def config(n: int, seed: Optional[int] = None, with_sfa: bool = True, batch: Optional[int] = None,
           kv_fp8: bool = False, idx_mx: bool = False) -> Workload:
    """Workload of configuration n (1..5).  `batch` truncates to the first sequences (same data);
    `kv_fp8` stores the latent-KV cache in the FP8 layout (same bf16 rows, quantised); `idx_mx` makes
    the indexer inputs MXFP8 (the same bf16 rows with one E8M0 scale per 32 elements)."""
    seed = 1000 + n if seed is None else seed
    lens, qls = config_lengths(n, seed)
    if batch is not None:
        lens, qls = lens[:batch], qls[:batch]
    common = dict(with_sfa=with_sfa, kv_fp8=kv_fp8)
    if idx_mx:
        return make_workload(CONFIG_NAMES[n] + "_mxfp8", seed, lens, qls, idx_heads=64, idx_dim=128, idx_fp8=True,
                             idx_mx=True, top_k=2048, attn_heads=128, w_hi=0.125,
                             salient_frac=0.01 if n in (2, 3) else 0.0, **common)
    if n == 1:
        return make_workload(CONFIG_NAMES[1], seed, lens, qls, idx_heads=4, idx_dim=64, idx_fp8=False, top_k=256,
                             attn_heads=16, w_hi=1.0, **common)
    if n == 2:
        return make_workload(CONFIG_NAMES[2], seed, lens, qls, idx_heads=64, idx_dim=128, idx_fp8=False,
                             top_k=2048, attn_heads=128, w_hi=0.125, salient_frac=0.01, **common)
    if n == 3:
        return make_workload(CONFIG_NAMES[3], seed, lens, qls, idx_heads=64, idx_dim=128, idx_fp8=True,
                             top_k=2048, attn_heads=128, w_hi=0.125, salient_frac=0.01, **common)
    if n == 4:
        return make_workload(CONFIG_NAMES[4], seed, lens, qls, idx_heads=64, idx_dim=128, idx_fp8=False,
                             top_k=2048, attn_heads=128, w_hi=0.125, **common)
    if n == 5:
        return make_workload(CONFIG_NAMES[5], seed, lens, qls, idx_heads=64, idx_dim=128, idx_fp8=True,
                             top_k=2048, attn_heads=128, w_hi=0.125, **common)
    raise ValueError(n)
