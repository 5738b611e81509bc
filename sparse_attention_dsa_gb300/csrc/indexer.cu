// Fused lightning indexer + Top-K for sm_103a.
//
// Computes, for every query token t, I[t,s] = sum_h w[t,h] * max(0, q_idx[t,h,:] . k[s,:]) over the
// visible positions s <= p_t, and writes only the K best positions ("Optimizing Inference for Hybrid
// Attention Architectures: From Operator Fusion to Sequence Sharding", section "Breaking Down the
// Computational Path of Hybrid Attention", step 1; "Day0 Inference Optimization for Next-Generation
// Hybrid-Architecture LLMs Based on CANN", section 2.1: scoring, head weighting and Top-K fused in one
// kernel that reads the paged K cache; "Day0 Inference Support and Performance Optimization for New LLM
// Architectures", section 3.1: no score tensor leaves the chip).
//
// Work decomposition: one thread-block cluster of C CTAs per (sequence, block of up to QB query tokens).
// CTA r of the cluster scores positions [r*chunk, (r+1)*chunk) of that sequence and keeps the scores as
// order-preserving uint32 keys in its own shared memory.  A cluster-wide radix select (4 passes of 8
// bits; histograms exchanged through distributed shared memory) then finds the K-th key, and every CTA
// writes its selected positions in ascending order at an offset derived from the per-CTA counts.
//
// Scoring pipeline inside a CTA (warp-specialised):
//   warp 0  : TMA producer.  Each 128-position tile is two 64-token pages of the indexer K cache,
//             fetched with 3-D tensor-map loads (page id from the page table) into 128B-swizzled smem.
//   warp 1  : tcgen05 issuer.  D[128 positions, N] = K_tile[128, Di] * Qblk[N, Di]^T with
//             N = QB*Hi (padded to 16), accumulated in fp32 in tensor memory (two buffers).
//   warps 2-5: epilogue.  Each thread owns one TMEM lane (= one position), reads its N columns and
//             reduces sum_h w*max(0, acc) per query (FP8: times the key row scale), then stores the key.
//   warps 6-7: idle during scoring; all 8 warps run the selection.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kTileM = 128;  // positions per tile (two pages)
constexpr int kPage = 64;
constexpr int kMaxCluster = 16;

template <int HI, int DI, int QB, bool FP8>
struct IdxCfg {
    static constexpr int kNReal = HI * QB;
    static constexpr int kN = kNReal < 16 ? 16 : ((kNReal + 15) / 16) * 16;  // UMMA N for M = 128
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kRowBytes = DI * kElem;
    static constexpr int kAtoms = kRowBytes / 128;  // 128-byte swizzle atoms along K
    static constexpr int kStageBytes = kTileM * kRowBytes;
    static constexpr int kQBytes = kN * kRowBytes;
    static constexpr int kMmaK = FP8 ? 32 : 16;  // elements per UMMA
    static constexpr int kKSteps = DI / kMmaK;
    // accumulator buffers in TMEM: enough that the MMA issuer rarely waits for the epilogue
    static constexpr int kAccBufs = (4 * kN) <= 512 ? 4 : 2;
    static constexpr int kTmemCols = (kAccBufs * kN) <= 32 ? 32 : (kAccBufs * kN) <= 64 ? 64
                                     : (kAccBufs * kN) <= 128 ? 128 : (kAccBufs * kN) <= 256 ? 256 : 512;
    static constexpr uint32_t kIdesc = make_idesc(128, kN, FP8 ? 0u : 1u, FP8 ? 0u : 1u, 0u, 0u);
    static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle atoms");
    static_assert(kN <= 256, "UMMA N limit");
};

struct SelectSmem {
    uint32_t hist[2][256];
    uint32_t totals[256];
    uint32_t gt[kMaxCluster];
    uint32_t ecnt[kMaxCluster];
    uint32_t scan_e[kThreads / 32];
    uint32_t scan_s[kThreads / 32];
    uint32_t take_me;
    uint32_t off_me;
};

struct CtrlSmem {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[4];
    uint64_t tempty[4];
    uint64_t qbar;
    uint32_t tmem_base;
    int32_t consumed;  // tiles consumed by the MMA warp (drain bookkeeping)
    int32_t issued;    // tiles issued by the producer
    int32_t qwaited;
};

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Cluster-wide Top-K of one query.  keys: this CTA's n local keys (position range_start + i);
// hist0: this CTA's histogram of the keys' top byte, built while scoring; allh: 2 x C x 256 scratch for
// the gathered per-CTA histograms.  visible = p + 1 positions exist in total.  All CTAs of the cluster
// call this with identical (K, visible), so the cluster barriers inside match up.
__device__ void cluster_select(const uint32_t* keys, const uint32_t* hist0, uint32_t* allh, int n, int K,
                               int64_t visible, int32_t* out_row, int range_start, uint32_t rank, uint32_t C,
                               SelectSmem& S) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (visible <= K) {  // every visible position is kept: 0..p in order, then -1
        const int per = (K + (int)C - 1) / (int)C;
        const int lo = (int)rank * per, hi = min(K, lo + per);
        for (int s = lo + tid; s < hi; s += kThreads) out_row[s] = (int64_t)s < visible ? s : -1;
        return;
    }
    uint32_t prefix = 0, remaining = (uint32_t)K;
    if (tid < kMaxCluster) S.gt[tid] = 0;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        const uint32_t hmask = pass == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
        const int buf = pass & 1;
        uint32_t* ah = allh + buf * C * 256;  // this pass's gathered histograms, [C][256]
        if (pass > 0) {  // the top-byte histogram (pass 0) was built while scoring
            S.hist[buf][tid] = 0;
            __syncthreads();
            // plain shared atomics: the keys spread over many bins here, where a warp-level match would
            // cost one round per distinct bin
            for (int i = tid; i < n; i += kThreads) {
                const uint32_t key = keys[i];
                if (((key ^ prefix) & hmask) == 0) atomicAdd(&S.hist[buf][(key >> shift) & 255u], 1u);
            }
            __syncthreads();
        }
        {
            // push this CTA's bin count into slot [rank] of every CTA's buffer (posted remote stores);
            // the cluster barrier below makes them visible
            const uint32_t v = pass == 0 ? hist0[tid] : S.hist[buf][tid];
            const uint32_t slot = smem_u32(ah + rank * 256 + tid);
            for (uint32_t r = 0; r < C; ++r) st_dsmem_u32(mapa_shared(slot, r), v);
        }
        cluster_sync();
        {
            uint32_t tot = 0;
            for (uint32_t r = 0; r < C; ++r) tot += ah[r * 256 + tid];
            S.totals[tid] = tot;
        }
        __syncthreads();
        // every warp finds the bin that holds the remaining-th largest key itself (no broadcast barrier)
        uint32_t bstar = 0, rem_in = 0;
        {
            uint32_t v[8], lsum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                v[j] = S.totals[lane * 8 + j];
                lsum += v[j];
            }
            uint32_t incl = lsum;  // sum over lanes >= this one (bins at or above lane*8)
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t t = __shfl_down_sync(0xFFFFFFFFu, incl, off);
                if (lane + off < 32) incl += t;
            }
            uint32_t above = incl - lsum;
            uint32_t found = 0, fb = 0, fr = 0;
#pragma unroll
            for (int j = 7; j >= 0; --j) {
                if (above < remaining && remaining <= above + v[j]) {
                    found = 1;
                    fb = (uint32_t)(lane * 8 + j);
                    fr = remaining - above;
                }
                above += v[j];
            }
            const uint32_t who = __ballot_sync(0xFFFFFFFFu, found != 0);
            const int src_lane = who ? __ffs(who) - 1 : 0;
            bstar = __shfl_sync(0xFFFFFFFFu, fb, src_lane);
            rem_in = __shfl_sync(0xFFFFFFFFu, fr, src_lane);
        }
        // keys above the boundary bin, per source CTA (warp r handles CTA r, r + 8, ...)
        for (uint32_t r = (uint32_t)warp; r < C; r += kThreads / 32) {
            uint32_t s = 0;
            for (int i = lane; i < 256; i += 32) s += (uint32_t)i > bstar ? ah[r * 256 + i] : 0u;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
            if (lane == 0) S.gt[r] += s;
        }
        if (pass == 3 && tid < (int)C) S.ecnt[tid] = ah[tid * 256 + bstar];
        remaining = rem_in;
        prefix |= bstar << shift;
    }
    const uint32_t T = prefix;
    __syncthreads();  // the per-CTA counts (gt, ecnt) are complete
    if (tid == 0) {
        uint32_t ties_before = 0, running = 0;
        for (uint32_t r = 0; r < C; ++r) {
            const uint32_t need = remaining > ties_before ? remaining - ties_before : 0u;
            const uint32_t take = need < S.ecnt[r] ? need : S.ecnt[r];
            if (r == rank) {
                S.take_me = take;
                S.off_me = running;
            }
            ties_before += S.ecnt[r];
            running += S.gt[r] + take;
        }
    }
    __syncthreads();
    const uint32_t take_me = S.take_me, off_me = S.off_me;
    // Ordered compaction.  Warp w owns the contiguous segment [w*seg, (w+1)*seg) of the local keys:
    // one pass counts its keys above T and its ties, a block barrier turns the counts into per-warp
    // offsets, a second pass writes the selected positions in order.
    const int nw = kThreads / 32;
    const int seg = ((n + nw - 1) / nw + 31) / 32 * 32;
    const int lo = warp * seg, hi = min(n, lo + seg);
    uint32_t cnt_gt = 0, cnt_tie = 0;
    for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < hi ? keys[i] : 0u;
        cnt_gt += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, key > T));
        cnt_tie += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, key == T && i < hi));
    }
    if (lane == 0) {
        S.scan_e[warp] = cnt_tie;
        S.scan_s[warp] = cnt_gt;
    }
    __syncthreads();
    uint32_t tie_base = 0, out_base = off_me;
    for (int k = 0; k < warp; ++k) {
        const uint32_t ties_k = S.scan_e[k];
        const uint32_t take_k = take_me > tie_base ? min(ties_k, take_me - tie_base) : 0u;
        out_base += S.scan_s[k] + take_k;
        tie_base += ties_k;
    }
    if (cnt_gt == 0 && (cnt_tie == 0 || tie_base >= take_me)) return;  // nothing selected in this segment
    uint32_t run_tie = tie_base, run_sel = 0;
    for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < hi ? keys[i] : 0u;
        const bool e = key == T && i < hi, g = key > T;
        const uint32_t be = __ballot_sync(0xFFFFFFFFu, e);
        const uint32_t tie_rank = run_tie + (uint32_t)__popc(be & lanemask_lt());
        const bool sel = g || (e && tie_rank < take_me);
        const uint32_t bs = __ballot_sync(0xFFFFFFFFu, sel);
        if (sel) out_row[out_base + run_sel + (uint32_t)__popc(bs & lanemask_lt())] = range_start + i;
        run_tie += (uint32_t)__popc(be);
        run_sel += (uint32_t)__popc(bs);
    }
}

template <int HI, int DI, int QB, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_topk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                        const IndexerParams p) {
    using Cfg = IdxCfg<HI, DI, QB, FP8>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled operand tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    uint8_t* a_tiles = smem;                                   // S * kStageBytes
    uint8_t* q_tile = a_tiles + (size_t)S * Cfg::kStageBytes;  // kQBytes
    uint32_t* keys = reinterpret_cast<uint32_t*>(q_tile + Cfg::kQBytes);  // QB * chunk
    float* w_s = reinterpret_cast<float*>(keys + (size_t)QB * p.chunk);   // kN
    int32_t* pages_s = reinterpret_cast<int32_t*>(w_s + Cfg::kN);         // chunk / 64
    uint32_t* hist0 = reinterpret_cast<uint32_t*>(pages_s + p.chunk / kPage);  // QB x 256
    uint32_t* allh = hist0 + QB * 256;                                      // 2 x C x 256
    SelectSmem* sel = reinterpret_cast<SelectSmem*>(allh + 2 * cluster_nctarank() * 256);
    CtrlSmem* ctl = reinterpret_cast<CtrlSmem*>((reinterpret_cast<uintptr_t>(sel + 1) + 15) & ~uintptr_t(15));

    // the attention kernel queued behind this one may be scheduled now: it waits on the device before it
    // reads the Top-K this kernel writes
    allow_dependent_launch();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t C = cluster_nctarank();
    const uint32_t rank = cluster_ctarank();
    const int item = blockIdx.x / (int)C;
    const int b = item / p.blocks_per_seq;
    const int jb = item % p.blocks_per_seq;
    if (b >= p.batch) return;  // uniform over the cluster
    const int cu0 = p.cu_q_lens[b];
    const int n_b = p.cu_q_lens[b + 1] - cu0;
    const int j0 = jb * p.qb;
    const int L = p.seq_lens[b];
    if (cu0 < 0 || n_b < 0 || cu0 + n_b > p.total_q) {
        if (jb == 0 && rank == 0 && tid == 0) raise_error(p.err, DSA_DEVERR_SEQ);
        return;
    }
    if (j0 >= n_b) return;  // uniform over the cluster
    if (n_b > L || L > p.max_pages * kPage || L < 0) {
        if (rank == 0 && tid == 0) raise_error(p.err, DSA_DEVERR_SEQ);
        return;
    }
    const int nq = min(p.qb, n_b - j0);
    const int t0 = cu0 + j0;
    const int64_t p_last = (int64_t)L - n_b + j0 + nq - 1;  // position of the block's last query
    const int range_start = (int)rank * p.chunk;
    const int64_t range_end = (int64_t)range_start + p.chunk;
    const int64_t hi = range_end < p_last + 1 ? range_end : p_last + 1;
    const int n_pos = hi > range_start ? (int)(hi - range_start) : 0;
    const int ntiles = (n_pos + kTileM - 1) / kTileM;
    const int n_keys = ntiles * kTileM;

    // ---- set-up: page list, head weights, barriers, tensor memory --------------------------------------
    const int32_t* pt_row = p.page_table + (int64_t)b * p.max_pages;
    for (int i = tid; i < ntiles * 2; i += kThreads) {
        const int lp = range_start / kPage + i;
        int32_t pg = -1;
        if ((int64_t)lp * kPage < hi) {
            pg = pt_row[lp];
            if (pg < 0 || pg >= p.num_pages) {
                raise_error(p.err, DSA_DEVERR_PAGE);
                pg = -1;
            }
        }
        pages_s[i] = pg;
    }
    for (int i = tid; i < QB * 256; i += kThreads) hist0[i] = 0;
    for (int c = tid; c < Cfg::kN; c += kThreads) {
        float wv = 0.f;
        if (c < nq * HI) {
            const int64_t idx = (int64_t)(t0 + c / HI) * HI + (c % HI);
            wv = p.w[idx];
            if (FP8) wv *= p.q_scale[idx];
        }
        w_s[c] = wv;
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], 1);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&ctl->tfull[i], 1);
            mbar_init(&ctl->tempty[i], 4);
        }
        mbar_init(&ctl->qbar, 1);
        ctl->consumed = 0;
        ctl->issued = 0;
        ctl->qwaited = 0;
        fence_mbar_init();
    }
    if (warp == 1 && ntiles > 0) {
        tmem_alloc(&ctl->tmem_base, Cfg::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- scoring pipeline -----------------------------------------------------------------------------
    if (ntiles > 0) {
        // The producer and MMA warps run their loops with all 32 lanes (every lane waits on the barriers,
        // one lane issues), so no lane of these warps sits at the block barrier while the loop runs.
        if (warp == 0) {
            if (lane == 0) {
                prefetch_tensormap(&kmap);
                prefetch_tensormap(&qmap);
                mbar_arrive_expect_tx(&ctl->qbar, Cfg::kQBytes);
#pragma unroll
                for (int a = 0; a < Cfg::kAtoms; ++a)
                    tma_load_2d(q_tile + a * Cfg::kN * 128, &qmap, &ctl->qbar, a * (128 / Cfg::kElem), t0 * HI);
            }
            int issued = 0;
            int s = 0;  // ring slot and its phase, advanced without a division by the runtime depth
            uint32_t ph = 0;
            for (int i = 0; i < ntiles; ++i, s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->empty[s], ph ^ 1u, p.err))) break;
                if (lane == 0) {
                    const int32_t pg0 = pages_s[2 * i], pg1 = pages_s[2 * i + 1];
                    const uint32_t bytes = (uint32_t)((pg0 >= 0) + (pg1 >= 0)) * (kPage * Cfg::kRowBytes);
                    if (bytes == 0) {
                        mbar_arrive(&ctl->full[s]);
                    } else {
                        mbar_arrive_expect_tx(&ctl->full[s], bytes);
                        uint8_t* dst = a_tiles + (size_t)s * Cfg::kStageBytes;
#pragma unroll
                        for (int a = 0; a < Cfg::kAtoms; ++a) {
                            if (pg0 >= 0)
                                tma_load_3d(dst + a * (kTileM * 128), &kmap, &ctl->full[s], a * (128 / Cfg::kElem),
                                            0, pg0);
                            if (pg1 >= 0)
                                tma_load_3d(dst + a * (kTileM * 128) + kPage * 128, &kmap, &ctl->full[s],
                                            a * (128 / Cfg::kElem), 0, pg1);
                        }
                    }
                }
                __syncwarp();
                issued = i + 1;
            }
            if (lane == 0) ctl->issued = issued;
        } else if (warp == 1) {
            const uint32_t tmem = ctl->tmem_base;
            const uint32_t q_base = smem_u32(q_tile);
            int consumed = 0;
            bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&ctl->qbar, 0, p.err));
            if (lane == 0) ctl->qwaited = ok ? 1 : 0;
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; ok && i < ntiles; ++i, s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                const int ab = i % Cfg::kAccBufs;
                const uint32_t aph = (uint32_t)(i / Cfg::kAccBufs) & 1u;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->tempty[ab], aph ^ 1u, p.err))) break;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->full[s], ph, p.err))) break;
                consumed = i + 1;
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t a_base = smem_u32(a_tiles + (size_t)s * Cfg::kStageBytes);
#pragma unroll
                    for (int k = 0; k < Cfg::kKSteps; ++k) {
                        const int kb = k * Cfg::kMmaK * Cfg::kElem;  // byte offset along K
                        const int atom = kb / 128, off = kb % 128;
                        const uint64_t ad = smem_desc(a_base + atom * (kTileM * 128) + off, 16, 1024, kSwizzle128B);
                        const uint64_t bd = smem_desc(q_base + atom * (Cfg::kN * 128) + off, 16, 1024, kSwizzle128B);
                        if (FP8)
                            umma_f8_ss(tmem + ab * Cfg::kN, ad, bd, Cfg::kIdesc, k > 0);
                        else
                            umma_f16_ss(tmem + ab * Cfg::kN, ad, bd, Cfg::kIdesc, k > 0);
                    }
                    umma_commit(&ctl->empty[s]);
                    umma_commit(&ctl->tfull[ab]);
                }
                __syncwarp();
            }
            if (lane == 0) ctl->consumed = consumed;
        } else if (warp >= 2 && warp < 6) {
            const uint32_t quad = (uint32_t)(warp & 3);  // TMEM lanes this warp may access
            const int row = (int)quad * 32 + lane;       // position within the tile
            const uint32_t tmem = ctl->tmem_base + ((quad * 32u) << 16);
            int64_t pq[QB];
#pragma unroll
            for (int q = 0; q < QB; ++q) pq[q] = (int64_t)L - n_b + j0 + q;
            for (int i = 0; i < ntiles; ++i) {
                const int ab = i % Cfg::kAccBufs;
                const uint32_t aph = (uint32_t)(i / Cfg::kAccBufs) & 1u;
                const int local = i * kTileM + row;
                const int pos = range_start + local;
                const int32_t pg = pages_s[2 * i + (row >> 6)];
                float ksc = 1.f;
                if (FP8 && pg >= 0) ksc = __ldg(p.k_scale + (int64_t)pg * kPage + (row & 63));
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->tfull[ab], aph, p.err))) break;
                tc_fence_after();
                float acc[QB];
#pragma unroll
                for (int q = 0; q < QB; ++q) acc[q] = 0.f;
                if constexpr (HI % 32 == 0) {
                    // One query's heads, 32 columns per TMEM wait, in a rolled loop: the code stays small
                    // (it shares the instruction cache with the MMA warp), eight independent partial sums
                    // keep the FMA chains short, and the weights come four at a time.
#pragma unroll
                    for (int q = 0; q < QB; ++q) {
                        float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
                        for (int c0 = q * HI; c0 < (q + 1) * HI; c0 += 32) {
                            float v0[16], v1[16];
                            tmem_ld16(tmem + ab * Cfg::kN + c0, v0);
                            tmem_ld16(tmem + ab * Cfg::kN + c0 + 16, v1);
                            tmem_ld_wait();
                            tmem_regs_ready(v0);
                            tmem_regs_ready(v1);
                            const float4* w4 = reinterpret_cast<const float4*>(w_s + c0);
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4) {
                                const float4 wv = w4[j4];
                                const float* v = j4 < 4 ? v0 + 4 * j4 : v1 + 4 * (j4 - 4);
                                part[(2 * j4) & 7] = fmaf(wv.x, fmaxf(v[0], 0.f), part[(2 * j4) & 7]);
                                part[(2 * j4 + 1) & 7] = fmaf(wv.y, fmaxf(v[1], 0.f), part[(2 * j4 + 1) & 7]);
                                part[(2 * j4) & 7] = fmaf(wv.z, fmaxf(v[2], 0.f), part[(2 * j4) & 7]);
                                part[(2 * j4 + 1) & 7] = fmaf(wv.w, fmaxf(v[3], 0.f), part[(2 * j4 + 1) & 7]);
                            }
                        }
                        acc[q] = ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
                    }
                } else
#pragma unroll
                for (int c0 = 0; c0 < Cfg::kNReal; c0 += 32) {
                    float v0[16], v1[16];
                    tmem_ld16(tmem + ab * Cfg::kN + c0, v0);
                    if (c0 + 16 < Cfg::kNReal) tmem_ld16(tmem + ab * Cfg::kN + c0 + 16, v1);
                    tmem_ld_wait();
                    tmem_regs_ready(v0);
                    if (c0 + 16 < Cfg::kNReal) tmem_regs_ready(v1);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int c = c0 + j;
                        if (c < Cfg::kNReal) acc[c / HI] += w_s[c] * fmaxf(v0[j], 0.f);
                    }
                    if (c0 + 16 < Cfg::kNReal) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int c = c0 + 16 + j;
                            if (c < Cfg::kNReal) acc[c / HI] += w_s[c] * fmaxf(v1[j], 0.f);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->tempty[ab]);
#pragma unroll
                for (int q = 0; q < QB; ++q) {
                    uint32_t key = 0;
                    if (q < nq && pg >= 0 && (int64_t)pos <= pq[q]) key = score_key(FP8 ? acc[q] * ksc : acc[q]);
                    keys[q * p.chunk + local] = key;
                    // top-byte histogram for the first radix pass (warp-aggregated)
                    const uint32_t bin = key >> 24;
                    const uint32_t peers = __match_any_sync(0xFFFFFFFFu, bin);
                    if (lane == __ffs(peers) - 1) atomicAdd(&hist0[q * 256 + bin], (uint32_t)__popc(peers));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (ntiles > 0) {
        // Drain: copies that were issued but never consumed (only after a timeout) must land before exit.
        if (warp == 0 && lane == 0) {
            if (!ctl->qwaited) mbar_wait(&ctl->qbar, 0, p.err);
            for (int i = ctl->consumed; i < ctl->issued; ++i) mbar_wait(&ctl->full[i % S], (uint32_t)(i / S) & 1u, p.err);
        }
        if (warp == 1) tmem_dealloc(ctl->tmem_base, Cfg::kTmemCols);
    }

    // ---- cluster-wide Top-K per query -------------------------------------------------------------------
    for (int q = 0; q < nq; ++q) {
        const int64_t visible = (int64_t)L - n_b + j0 + q + 1;
        cluster_select(keys + (size_t)q * p.chunk, hist0 + q * 256, allh, n_keys, p.top_k, visible,
                       p.topk + (int64_t)(t0 + q) * p.top_k, range_start, rank, C, *sel);
    }
    // No cluster barrier here: every remote access is a histogram push, and the pushes of a pass complete
    // before that pass's barrier, so after the last pass no CTA touches another's shared memory.
}

template <int HI, int DI, int QB, bool FP8>
size_t indexer_smem_bytes(int stages, int chunk, int cluster) {
    using Cfg = IdxCfg<HI, DI, QB, FP8>;
    return 1024 + (size_t)stages * Cfg::kStageBytes + Cfg::kQBytes + (size_t)QB * chunk * 4 + Cfg::kN * 4 +
           (size_t)(chunk / kPage) * 4 + (size_t)(QB + 2 * cluster) * 256 * 4 + sizeof(SelectSmem) + sizeof(CtrlSmem) +
           64;
}

template <int HI, int DI, int QB, bool FP8>
cudaError_t launch_variant(const IndexerLaunch& L, cudaStream_t stream) {
    using Cfg = IdxCfg<HI, DI, QB, FP8>;
    auto kern = indexer_topk_kernel<HI, DI, QB, FP8>;
    const int chunk = L.params.chunk;
    // choose the number of pipeline stages from the shared-memory budget
    int stages = kMaxStages;
    while (stages > 2 && indexer_smem_bytes<HI, DI, QB, FP8>(stages, chunk, L.cluster) > (size_t)L.smem_limit) --stages;
    const size_t smem = indexer_smem_bytes<HI, DI, QB, FP8>(stages, chunk, L.cluster);
    if (smem > (size_t)L.smem_limit) return cudaErrorInvalidConfiguration;
    IndexerParams prm = L.params;
    prm.stages = stages;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)L.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(L.items * L.cluster));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.check_occupancy) {
        int nclusters = 0;
        e = cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (nclusters < 1) return cudaErrorInvalidClusterSize;
    }
    return cudaLaunchKernelEx(&cfg, kern, L.kmap, L.qmap, prm);
}

}  // namespace

int indexer_variant_n(int idx_heads, int idx_dim, int fp8, int qb) {
    // UMMA N of the variant that serves these shapes (0 = unsupported)
    if (!fp8 && idx_heads == 4 && idx_dim == 64 && qb >= 1 && qb <= 4) return 16;
    if (idx_heads == 64 && idx_dim == 128 && (qb == 1 || qb == 2 || (qb == 4 && !fp8))) return 64 * qb;
    return 0;
}

size_t indexer_smem_estimate(int idx_heads, int idx_dim, int fp8, int qb, int stages, int chunk, int cluster) {
    if (!fp8 && idx_heads == 4 && idx_dim == 64) return indexer_smem_bytes<4, 64, 4, false>(stages, chunk, cluster);
    if (idx_heads == 64 && idx_dim == 128) {
        if (fp8) {
            if (qb == 1) return indexer_smem_bytes<64, 128, 1, true>(stages, chunk, cluster);
            if (qb == 2) return indexer_smem_bytes<64, 128, 2, true>(stages, chunk, cluster);
        } else {
            if (qb == 1) return indexer_smem_bytes<64, 128, 1, false>(stages, chunk, cluster);
            if (qb == 2) return indexer_smem_bytes<64, 128, 2, false>(stages, chunk, cluster);
            if (qb == 4) return indexer_smem_bytes<64, 128, 4, false>(stages, chunk, cluster);
        }
    }
    return ~size_t(0);
}

cudaError_t launch_indexer(const IndexerLaunch& L, cudaStream_t stream) {
    const int qb = L.params.qb;
    if (!L.fp8 && L.idx_heads == 4 && L.idx_dim == 64) return launch_variant<4, 64, 4, false>(L, stream);
    if (L.idx_heads == 64 && L.idx_dim == 128) {
        if (L.fp8) {
            if (qb == 1) return launch_variant<64, 128, 1, true>(L, stream);
            if (qb == 2) return launch_variant<64, 128, 2, true>(L, stream);
        } else {
            if (qb == 1) return launch_variant<64, 128, 1, false>(L, stream);
            if (qb == 2) return launch_variant<64, 128, 2, false>(L, stream);
            if (qb == 4) return launch_variant<64, 128, 4, false>(L, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace dsa
