"""Attention edge cases that random N(0,1) inputs never reach, against the oracle on the same selection
(|gpu - oracle| <= 2e-2 + 1e-2 |oracle| elementwise, lse likewise):

* logits that jump by far more than the online softmax's rescale threshold late in a split's rows, so
  the running maximum is raised and the partial output rescaled mid-stream;
* position splits whose maxima differ by tens of natural-log units, the edge case of the split merge's
  weights (a split whose rows all but vanish next to another's);
* a Top-K that is not a multiple of the 64-row tile, with -1 entries inside a split's tiles.

The logits are made extreme by scaling the 64 rotary dims of selected latent-KV rows by a power of two
(exact in bf16): those dims count in the logits but are not part of V, so the softmax sees jumps of tens
to hundreds of natural-log units while the outputs stay at the scale of N(0,1) values.  (Scaling the V
part as well would make the outputs large, and the bf16 rounding of the softmax weights, a property of
the bf16 path rather than an error, would then exceed the output tolerance wherever large values of
opposite sign cancel.)  Sources: "Optimizing Inference for Hybrid Attention Architectures: From
Operator Fusion to Sequence Sharding", section "Breaking Down the Computational Path of Hybrid
Attention", step 2 (softmax over the selected positions); "Day0 Inference Support and Performance
Optimization for New LLM Architectures", section 3.2.
"""
import numpy as np
import pytest
import torch

from gen import bf16_to_f32, f32_to_bf16
from gen.workloads import make_workload

from _gpu import DeviceWorkload, check_attention, ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    ensure_built()


def _scale_rows(wl, b, positions, factor):
    """Multiply the rotary dims (512..575) of the latent-KV rows of sequence b at the given logical positions
    by `factor` (a power of 2): their logits move, their values do not."""
    for s in positions:
        pg, sl = wl.page_table[b, s // 64], s % 64
        row = wl.kv_cache[pg, sl]
        row[512:] = f32_to_bf16(bf16_to_f32(row[512:]) * np.float32(factor))


def _run(wl, topk):
    dw = DeviceWorkload(wl)
    dw.sfa(topk=torch.from_numpy(np.ascontiguousarray(topk, dtype=np.int32)).cuda())
    assert dw.error_word() == 0
    out, lse = dw.out_host()
    return check_attention(wl, topk, out, lse)


def _wl(lens, qls, K, seed=21):
    return make_workload("edges", seed, lens, qls, idx_heads=4, idx_dim=64, idx_fp8=False, top_k=K, attn_heads=128)


@pytest.mark.parametrize("factor", [16.0, 64.0, 256.0])
def test_late_logit_jump_rescales_the_running_max(factor):
    """One token, K = 2048 over positions 0..2047 (eight position splits of 256 rows).  Rows late in every
    split get rotary parts scaled so that their logits jump by about factor/3 standard deviations (10 to
    over 100 natural-log units above the rows before them) after several tiles have accumulated."""
    wl = _wl([4096], [1], 2048)
    topk = np.arange(2048, dtype=np.int32)[None, :]
    late = [s for s in range(2048) if (s % 256) >= 200 and s % 3 == 0]
    _scale_rows(wl, 0, late, factor)
    _run(wl, topk)


def test_split_maxima_differ_strongly():
    """The rows of one position split have logits tens of units above the others': the merge weights of
    the other splits all but vanish next to it, and the split with the huge maximum dominates every head."""
    wl = _wl([4096], [1], 2048)
    topk = np.arange(2048, dtype=np.int32)[None, :]
    _scale_rows(wl, 0, range(768, 1024), 32.0)
    _run(wl, topk)
    # and the opposite skew: one split far below the others
    wl2 = _wl([4096], [1], 2048, seed=22)
    _scale_rows(wl2, 0, [s for s in range(2048) if not (256 <= s < 512)], 8.0)
    _run(wl2, topk)


def test_two_split_merge_with_skewed_maxima():
    """32 tokens: every token's positions are split in two (the compact two-split merge).  For even
    tokens the second split's rows are scaled up, for odd tokens the first split's."""
    lens = [2500 + 13 * i for i in range(32)]
    wl = _wl(lens, [1] * 32, 1024, seed=23)
    topk = np.stack([np.arange(1024, dtype=np.int32) * 2 for _ in range(32)])
    for b in range(32):
        half = range(1024, 2048, 2) if b % 2 == 0 else range(0, 1024, 2)
        _scale_rows(wl, b, [s for s in half if s % 4 == 0], 16.0)
    _run(wl, topk)


@pytest.mark.parametrize("K", [1000, 777, 65])
def test_ragged_top_k_with_holes(K):
    """K not a multiple of 64, the list in descending order, -1 entries scattered through every split."""
    lens = [3000, 1500, 900]
    wl = _wl(lens, [1, 1, 1], K, seed=24)
    rng = np.random.default_rng(K)
    topk = np.full((3, K), -1, dtype=np.int32)
    for b, L in enumerate(lens):
        sel = np.sort(rng.choice(L, size=min(K, L), replace=False))[::-1]
        topk[b, : sel.shape[0]] = sel
        topk[b, rng.choice(K, size=K // 7, replace=False)] = -1
    _scale_rows(wl, 0, [int(s) for s in topk[0][topk[0] >= 0][-40:]], 16.0)  # a jump in the last rows
    _run(wl, topk)


def test_a_split_with_no_selected_row():
    """Every entry of one position split is -1: that split contributes weight 0 (its O is never read)."""
    wl = _wl([4096], [1], 2048, seed=25)
    topk = np.arange(2048, dtype=np.int32)[None, :].copy()
    topk[0, 512:768] = -1
    _run(wl, topk)
