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
// order-preserving uint32 keys in its own shared memory.  A cluster-wide radix select (8-bit digits,
// most significant first; histograms and, for the last two bytes, the surviving candidate keys
// exchanged through distributed shared memory, usually in two rounds) then finds the K-th key, and
// every CTA writes its selected positions in ascending order at an offset derived from the per-CTA
// counts.
//
// Scoring pipeline inside a CTA (warp-specialised):
//   warp 0  : TMA producer.  Each 128-position tile is two 64-token pages of the indexer K cache,
//             fetched with 3-D tensor-map loads (page id from the page table) into 128B-swizzled smem.
//   warp 1  : tcgen05 issuer.  D[128 positions, N] = K_tile[128, Di] * Qblk[N, Di]^T with
//             N = QB*Hi (padded to 16), accumulated in fp32 in tensor memory (two or four buffers).
//   warps 2-5 and 6-9: two epilogue groups (even and odd tiles).  Each thread owns one TMEM lane
//             (= one position), reads its N columns and reduces sum_h w*max(0, acc) per query (FP8:
//             times the key row scale), then stores the key.
//   MXFP8 keys: warps 6-9 instead dequantise each landed tile to bf16 into tensor memory (the MMA's A
//             operand), and warps 2-5 are the only epilogue group.
//   other warps: idle during scoring; every warp takes part in the selection.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 384;  // threads of the standalone indexer kernel (warps 10-11 only join the select)
constexpr int kMaxWarps = 16;  // select scratch sized for up to 512 threads
constexpr int kTileM = 128;  // positions per tile (two pages)
constexpr int kPage = 64;
constexpr int kMaxCluster = 16;

// MX: FP8 codes with one E8M0 scale per 32 elements of a row (MXFP8).  A code times its group's power of
// two is exact in bf16, so the K tiles are dequantised to bf16 by converter warps (the query once at
// set-up) and scored by the bf16 MMA: one accumulator, and the epilogue of the other variants.
template <int HI, int DI, int QB, bool FP8, bool MX = false>
struct IdxCfg {
    static_assert(!MX || (FP8 && QB == 1 && DI == 128), "MXFP8: FP8 codes of 128 dims, one query per work item");
    static constexpr int kNReal = HI * QB;
    static constexpr int kN = kNReal < 16 ? 16 : ((kNReal + 15) / 16) * 16;  // UMMA N for M = 128
    static constexpr int kAccCols = kN;                  // TMEM columns of one tile's accumulator
    static constexpr int kElem = FP8 ? 1 : 2;            // bytes per element of the cached K tiles
    static constexpr int kRowBytes = DI * kElem;
    static constexpr int kAtoms = kRowBytes / 128;  // 128-byte swizzle atoms along K (of the loaded tiles)
    static constexpr int kStageBytes = kTileM * kRowBytes;
    static constexpr bool kMmaBf16 = !FP8 || MX;         // the MMA reads bf16 tiles
    static constexpr int kMmaElem = kMmaBf16 ? 2 : 1;
    static constexpr int kQBytes = kN * DI * kMmaElem;   // the query tile as the MMA reads it
    static constexpr int kScaleStageBytes = MX ? kTileM * (DI / 32) : 0;  // a tile's E8M0 key scales (MX)
    static constexpr int kMmaK = kMmaBf16 ? 16 : 32;  // elements per UMMA
    static constexpr int kKSteps = DI / kMmaK;
    // accumulator buffers in TMEM: enough that the MMA issuer rarely waits for the epilogue
    static constexpr int kAccBufs = (4 * kAccCols) <= 512 ? 4 : 2;
    // MX: two dequantised K tiles in TMEM after the accumulators (the MMA's A operand; lane = key row,
    // column j = dims 2j and 2j + 1 as a bf16 pair)
    static constexpr int kACol = kAccBufs * kAccCols;
    static constexpr int kACols = MX ? DI / 2 : 0;
    static constexpr int kUsedCols = kACol + 2 * kACols;
    static constexpr int kTmemCols = kUsedCols <= 32 ? 32 : kUsedCols <= 64 ? 64 : kUsedCols <= 128 ? 128
                                     : kUsedCols <= 256 ? 256 : 512;
    static_assert(kUsedCols <= 512, "TMEM columns");
    static constexpr uint32_t kIdesc = make_idesc(128, kN, kMmaBf16 ? 1u : 0u, kMmaBf16 ? 1u : 0u, 0u, 0u);
    static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle atoms");
    // the select's fallback exchange space (2 x C x 256 words) lives in the stage ring (at least 2 stages)
    static_assert(2 * kStageBytes >= 2 * kMaxCluster * 256 * 4, "stage ring too small for the select");
    static_assert(kN <= 256, "UMMA N limit");
    static_assert(QB <= 4, "per-query select state is sized for four queries");
};

constexpr int kCandCap = 256;  // second-round candidates one CTA may send (a power of two)
// Up to this many candidates the K-th key is found by ranking them directly (quadratic work); more take two
// histogram rounds over their low bytes.
constexpr int kRankPick = 128;

// Words of the per-CTA page list: one per 64-position page, rounded up to whole 16-byte units.
__host__ __device__ constexpr int page_words(int chunk) { return ((chunk / kPage) + 3) & ~3; }

struct SelectSmem {
    alignas(16) uint32_t hist[2][256];
    alignas(16) uint32_t totals[256];
    uint32_t res[8];                 // results broadcast from the warp that finds a boundary bin
    uint32_t gt[kMaxCluster];        // keys above the boundary found so far, per CTA of the cluster
    uint32_t ecnt[kMaxCluster];      // keys equal to the K-th key, per CTA
    uint32_t guess_in[kMaxCluster];  // round A: every CTA's guess of the top byte (pushed by that CTA)
    uint32_t ncand_in[kMaxCluster];  // round B: every CTA's candidate count (pushed by that CTA)
    uint32_t sure_in[kMaxCluster];   // round B: every CTA's keys above the 16-bit prefix (pushed by that CTA)
    uint32_t scan_e[kMaxWarps];
    uint32_t scan_s[kMaxWarps];
    uint32_t ncand;
    uint32_t take_me;
    uint32_t off_me;
    uint8_t cwarp[kCandCap];  // round B: the warp segment each of this CTA's candidates came from
};

struct CtrlSmem {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[4];
    uint64_t tempty[4];
    uint64_t bfull[2];   // MX: a dequantised K tile is ready (converter warps)
    uint64_t bempty[2];  // MX: its MMAs are done
    uint64_t qbar;
    uint64_t mma_done;   // every MMA the issuer made has completed (before tensor memory is released)
    uint32_t tmem_base;
    int32_t consumed;  // tiles consumed by the MMA warp (drain bookkeeping)
    int32_t issued;    // tiles issued by the producer
    int32_t qwaited;
};

// MX key dequantisation without conversion instructions.  An E4M3 code c placed in a bf16 as
// (c & 0x80) << 8 | (c & 0x7F) << 4 (its exponent field in the low four exponent bits, its mantissa in
// the top three mantissa bits) is exactly 2^-120 times the code's value, subnormal codes included
// (they land on bf16 subnormals with the same spacing); the group scale 2^(e - 127) then makes it a
// product by 2^(e - 7), exact in bf16 for every finite result.  Returns the bf16x2 word of the codes
// in bytes b0 and b1 of w (b0 in the low half): a byte permute (sel = 0x1804 for bytes 0 and 1, 0x3A24
// for bytes 2 and 3) builds [b1 | sign(b0) x 8 | b0 | 0], and one arithmetic shift by four then leaves
// each code's sign at its half's bit 15 and its low seven bits at bits 4..10; the mask clears the
// sign copies in between.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_unscaled(uint32_t w, uint32_t sel) {
    uint32_t t;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(w), "r"(0u), "r"(sel));
    return (uint32_t)((int32_t)t >> 4) & 0x87F087F0u;
}

// bf16x2 a * b, nearest-even, subnormals kept (as a fused multiply-add with -0)
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(0x80008000u));
    return d;
}

// The factor 2^(e - 7) of E8M0 byte e as a bf16x2 pair, split in two when it exceeds the bf16 range:
// lo = 2^min(e - 7, 127) (NaN for e = 255), hi = 2^max(e - 134, 0).
__device__ __forceinline__ uint32_t mx_factor_lo(uint32_t e) {
    const uint32_t b = e == 255u ? 0x7FC0u : (min(e + 120u, 254u) << 7);
    return b | (b << 16);
}
__device__ __forceinline__ uint32_t mx_factor_hi(uint32_t e) {
    const uint32_t b = (max(e, 134u) - 7u) << 7;
    return b | (b << 16);
}

// E8M0 scale byte e as the float 2^(e - 127) (e = 0: 2^-127, a subnormal; e = 255: NaN).
__device__ __forceinline__ float e8m0_factor(uint32_t e) {
    if (e == 0u) return __uint_as_float(0x00400000u);
    if (e == 255u) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(e << 23);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// The bin of `totals` (256 bins, ascending key order, 16-byte aligned) that holds the remaining-th largest
// key, and that key's rank inside the bin.  Called by one warp; every lane gets the result.
__device__ __forceinline__ void boundary_bin(const uint32_t* totals, uint32_t remaining, uint32_t& bstar,
                                             uint32_t& rem) {
    const int lane = threadIdx.x & 31;
    uint32_t v[8], lsum = 0;
    {
        const uint4 a = reinterpret_cast<const uint4*>(totals)[2 * lane];
        const uint4 b = reinterpret_cast<const uint4*>(totals)[2 * lane + 1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) lsum += v[j];
    uint32_t incl = lsum;  // keys in the bins at or above lane*8
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
    const int src = who ? __ffs(who) - 1 : 0;
    bstar = __shfl_sync(0xFFFFFFFFu, fb, src);
    rem = __shfl_sync(0xFFFFFFFFu, fr, src);
}

// S.gt[r] += the keys of CTA r in bins above bstar (its histogram: ah[r * stride + bin]).
template <int NT>
__device__ __forceinline__ void add_above(const uint32_t* ah, int stride, uint32_t bstar, uint32_t C, SelectSmem& S) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (uint32_t r = (uint32_t)warp; r < C; r += NT / 32) {
        uint32_t s = 0;
        for (int i = lane; i < 256; i += 32) s += (uint32_t)i > bstar ? ah[r * stride + i] : 0u;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
        if (lane == 0) S.gt[r] += s;
    }
}

// One radix pass with a cluster-wide histogram: this CTA's keys that match `prefix` above bit shift+8 are
// counted by their byte at `shift`, every CTA's histogram is pushed into slot [rank] of `buf` ([C][256]) in
// every CTA of the cluster, and all CTAs find the same boundary bin.
template <int NT>
__device__ void exchange_pass(const uint32_t* keys, int n, uint32_t prefix, int shift, uint32_t* buf, uint32_t rank,
                              uint32_t C, uint32_t& remaining, uint32_t& bstar, SelectSmem& S) {
    const int tid = threadIdx.x;
    const uint32_t hmask = 0xFFFFFFFFu << (shift + 8);
    if (tid < 256) S.hist[0][tid] = 0;
    __syncthreads();
    // plain shared atomics: a warp-level match would cost one round per distinct bin
    for (int i = tid; i < n; i += NT) {
        const uint32_t key = keys[i];
        if (((key ^ prefix) & hmask) == 0) atomicAdd(&S.hist[0][(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 256) {
        const uint32_t slot = smem_u32(buf + rank * 256 + tid);
        for (uint32_t r = 0; r < C; ++r) st_dsmem_u32(mapa_shared(slot, r), S.hist[0][tid]);
    }
    cluster_sync();
    if (tid < 256) {
        uint32_t tot = 0;
        for (uint32_t r = 0; r < C; ++r) tot += buf[r * 256 + tid];
        S.totals[tid] = tot;
    }
    __syncthreads();
    if (tid < 32) {
        uint32_t b, rem;
        boundary_bin(S.totals, remaining, b, rem);
        if (tid == 0) {
            S.res[0] = b;
            S.res[1] = rem;
        }
    }
    __syncthreads();
    bstar = S.res[0];
    remaining = S.res[1];
    add_above<NT>(buf, 256, bstar, C, S);
    __syncthreads();  // S.totals, S.hist and S.res are reused next
}

// Cluster-wide Top-K of one query: the K largest of the cluster's keys, as positions in ascending order.
//   keys: this CTA's n keys (position range_start + i); hist0: their top-byte histogram, built while
//   scoring; allh: C x 768 words of exchange space that nothing but this function touches; sbuf:
//   2 x C x 256 words of further exchange space that peers may write once every CTA of the cluster has
//   finished scoring.
// The K-th key is found radix-fashion, most significant byte first, with two cluster rounds in the usual
// case: round A exchanges the top-byte histograms together with a second-byte histogram of the bin each
// CTA guesses will hold the K-th key (the bin where its own count from the top reaches its share of K);
// when every guess is the agreed top byte, the second byte is settled in the same round.  Round B sends
// every key that still matches
// the 16-bit prefix (usually a few dozen per CTA) to every CTA, which finds the exact K-th key among them.
// A wrong guess or too many candidates falls back to a full exchanged pass per byte.  All CTAs of the
// cluster call this with identical (K, visible), so the cluster barriers inside match up.
template <int NT>
__device__ void cluster_select(const uint32_t* keys, const uint32_t* hist0, uint32_t* allh, uint32_t* sbuf, int n,
                               int K, int64_t visible, int32_t* out_row, int range_start, uint32_t rank, uint32_t C,
                               SelectSmem& S, const int32_t* pages, int32_t* rows_row, float* score_row,
                               int pos_begin) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // physical cache row of local key i (its page from this CTA's page list), -1 for a missing page
    auto row_of = [&](int i) -> int32_t {
        const int32_t pg = pages[i >> 6];
        return pg >= 0 ? pg * kPage + (i & (kPage - 1)) : -1;
    };
    if (visible <= K) {
        // every visible position is kept: pos_begin..pos_begin+visible-1 in order (each CTA writes those of
        // its own range), then -1
        const int64_t own_hi = min((int64_t)range_start + n, (int64_t)pos_begin + visible);
        for (int64_t s = (int64_t)range_start + tid; s < own_hi; s += NT) {
            const int64_t o = s - pos_begin;
            out_row[o] = (int32_t)s;
            if (rows_row) rows_row[o] = row_of((int)(s - range_start));
            if (score_row) score_row[o] = key_score(keys[s - range_start]);
        }
        const int pad = K - (int)visible;
        const int per = (pad + (int)C - 1) / (int)C;
        const int lo = (int)visible + (int)rank * per, hi = min(K, lo + per);
        for (int s = lo + tid; s < hi; s += NT) {
            out_row[s] = -1;
            if (rows_row) rows_row[s] = -1;
            if (score_row) score_row[s] = -INFINITY;
        }
        return;
    }
    uint32_t remaining = (uint32_t)K, prefix = 0, bstar = 0;
    if (tid < kMaxCluster) S.gt[tid] = 0;
    uint32_t* ahA = allh;             // round A: [C][512] = top-byte | guessed second-byte histograms
    uint32_t* cand = allh + C * 512;  // round B: [C][kCandCap] candidate keys
    static_assert(kCandCap <= 256, "round-B candidates share the 768-word slot");

    // ---- round A: the top-byte histogram, and the second-byte histogram of the guessed bin ----
    if (tid < 32) {
        uint32_t g, gr;
        boundary_bin(hist0, (uint32_t)((K + (int)C - 1) / (int)C), g, gr);
        if (tid == 0) S.res[7] = g;
    }
    if (tid < 256) S.hist[1][tid] = 0;
    __syncthreads();
    const uint32_t guess = S.res[7];
    for (int i0 = 4 * tid; i0 < n; i0 += 4 * NT * 8) {
        uint4 k8[8];  // eight 16-byte loads in flight (n is a multiple of 128)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u * 4 * NT;
            k8[u] = i < n ? *reinterpret_cast<const uint4*>(keys + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const uint32_t kv[4] = {k8[u].x, k8[u].y, k8[u].z, k8[u].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (i0 + u * 4 * NT < n && (kv[e] >> 24) == guess) atomicAdd(&S.hist[1][(kv[e] >> 16) & 255u], 1u);
        }
    }
    __syncthreads();
    if (tid < 256) {
        const uint32_t slot = smem_u32(ahA + rank * 512 + tid);
        const uint32_t h0 = hist0[tid], h1 = S.hist[1][tid];
        for (uint32_t r = 0; r < C; ++r) {
            const uint32_t a = mapa_shared(slot, r);
            st_dsmem_u32(a, h0);
            st_dsmem_u32(a + 256 * 4, h1);
        }
    }
    if (tid < (int)C) st_dsmem_u32(mapa_shared(smem_u32(&S.guess_in[rank]), (uint32_t)tid), guess);
    cluster_sync();  // also: every CTA of the cluster has finished scoring, so sbuf may now be written
    if (tid < 256) {
        uint32_t t0 = 0, t1 = 0;
        for (uint32_t r = 0; r < C; ++r) {
            t0 += ahA[r * 512 + tid];
            t1 += ahA[r * 512 + 256 + tid];
        }
        S.totals[tid] = t0;
        S.hist[0][tid] = t1;
    }
    __syncthreads();
    if (tid < 32) {
        uint32_t b0, r0, b1 = 0, r1 = 0;
        boundary_bin(S.totals, remaining, b0, r0);
        // the guessed second-byte histograms count the right keys when every CTA guessed this bin
        const bool agree = __all_sync(0xFFFFFFFFu, lane >= (int)C || S.guess_in[lane] == b0);
        if (agree) boundary_bin(S.hist[0], r0, b1, r1);
        if (tid == 0) {
            S.res[0] = b0;
            S.res[1] = r0;
            S.res[2] = agree ? 1u : 0u;
            S.res[3] = b1;
            S.res[4] = r1;
        }
    }
    __syncthreads();
    bstar = S.res[0];
    remaining = S.res[1];
    const bool spec = S.res[2] != 0;
    prefix = bstar << 24;
    if (spec) {
        bstar = S.res[3];
        remaining = S.res[4];
        __syncthreads();  // S.res is reused
    } else {
        __syncthreads();
        exchange_pass<NT>(keys, n, prefix, 16, sbuf, rank, C, remaining, bstar, S);
    }
    prefix |= bstar << 16;

    // ---- round B: the keys that still match the 16-bit prefix, sent to every CTA ----
    // Warp w scans the contiguous segment [w*seg, (w+1)*seg) of the local keys (the segments of the ordered
    // compaction below), four keys per lane.  It counts the keys whose top 16 bits exceed the prefix (they
    // are selected whatever the K-th key turns out to be) and sends every key that matches the prefix to
    // every CTA, noting which warp's segment it came from.
    const int nw = NT / 32;
    const int seg = ((n + nw - 1) / nw + 127) / 128 * 128;
    const int lo = min(n, warp * seg), hi = min(n, lo + seg);
    const uint32_t p16 = prefix >> 16;
    if (tid == 0) S.ncand = 0;
    if (tid < kMaxWarps) S.scan_e[tid] = 0;
    __syncthreads();
    {
        uint32_t sure = 0;
        for (int b0 = lo; b0 < hi; b0 += 4 * 128) {
            uint4 k4[4];  // four 16-byte loads in flight (segments are multiples of 128 keys)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = b0 + u * 128 + 4 * lane;
                k4[u] = i < hi ? *reinterpret_cast<const uint4*>(keys + i) : make_uint4(0, 0, 0, 0);
            }
            // matches are rare: mark them in a mask here, send them from a small rolled loop below
            uint32_t mask = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t kv[4] = {k4[u].x, k4[u].y, k4[u].z, k4[u].w};
                const bool in = b0 + u * 128 + 4 * lane < hi;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sure += (in && (kv[e] >> 16) > p16) ? 1u : 0u;
                    if (in && (kv[e] >> 16) == p16) mask |= 1u << (4 * u + e);
                }
            }
#pragma unroll 1
            while (mask != 0) {
                const int bit = __ffs(mask) - 1;
                mask &= mask - 1;
                const uint32_t key = keys[b0 + (bit >> 2) * 128 + 4 * lane + (bit & 3)];
                const uint32_t j = atomicAdd(&S.ncand, 1u);
                if (j < (uint32_t)kCandCap) {
                    S.cwarp[j] = (uint8_t)warp;
                    const uint32_t slot = smem_u32(cand + rank * kCandCap + j);
                    for (uint32_t r = 0; r < C; ++r) st_dsmem_u32(mapa_shared(slot, r), key);
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sure += __shfl_xor_sync(0xFFFFFFFFu, sure, off);
        if (lane == 0) S.scan_s[warp] = sure;
    }
    __syncthreads();
    if (tid < (int)C) {
        uint32_t sure_cta = 0;
        for (int w = 0; w < nw; ++w) sure_cta += S.scan_s[w];
        st_dsmem_u32(mapa_shared(smem_u32(&S.ncand_in[rank]), (uint32_t)tid), S.ncand);
        st_dsmem_u32(mapa_shared(smem_u32(&S.sure_in[rank]), (uint32_t)tid), sure_cta);
    }
    cluster_sync();
    const bool fits = __syncthreads_and(tid >= (int)C || S.ncand_in[tid] <= (uint32_t)kCandCap) != 0;
    // keys above the K-th key per CTA: the sure ones, plus the candidates (or exchanged bins) above it
    if (tid < kMaxCluster) {
        S.gt[tid] = tid < (int)C ? S.sure_in[tid] : 0u;
        S.ecnt[tid] = 0;
    }
    uint32_t n_c = 0;  // candidates of the whole cluster
    for (uint32_t r = 0; r < C; ++r) n_c += S.ncand_in[r];
    uint32_t T;
    if (fits && n_c <= (uint32_t)kRankPick) {
        // Every CTA holds the same few candidates: the remaining-th largest of them is the K-th key.  They
        // are flattened into the idle stage ring first; then a group of `subs` lanes per candidate splits
        // the count of the candidates above and equal to its own, and sums it with shuffles.
        __syncthreads();
        for (uint32_t c = (uint32_t)tid; c < n_c; c += NT) {
            uint32_t r = 0, j = c;
            while (j >= S.ncand_in[r]) j -= S.ncand_in[r++];
            sbuf[c] = cand[r * kCandCap + j];
        }
        __syncthreads();
        const uint32_t subs = n_c * 8 <= (uint32_t)NT ? 8u : n_c * 4 <= (uint32_t)NT ? 4u : n_c * 2 <= (uint32_t)NT ? 2u : 1u;
        for (uint32_t base = 0; base < n_c * subs; base += NT) {  // the same trip count in every thread
            const uint32_t idx = base + (uint32_t)tid, c = idx / subs, sb = idx % subs;
            const bool valid = c < n_c;
            const uint32_t key = valid ? sbuf[c] : 0u;
            uint32_t above = 0, equal = 0;
            if (valid) {
#pragma unroll 4
                for (uint32_t j = sb; j < n_c; j += subs) {
                    const uint32_t k2 = sbuf[j];
                    above += k2 > key ? 1u : 0u;
                    equal += k2 == key ? 1u : 0u;
                }
            }
            for (uint32_t off = 1; off < subs; off <<= 1) {  // the group's lanes are consecutive within a warp
                above += __shfl_xor_sync(0xFFFFFFFFu, above, off);
                equal += __shfl_xor_sync(0xFFFFFFFFu, equal, off);
            }
            if (valid && sb == 0 && above < remaining && remaining <= above + equal) {  // all equal keys agree
                S.res[0] = key;
                S.res[1] = remaining - above;
            }
        }
        __syncthreads();
        T = S.res[0];
        remaining = S.res[1];  // keys equal to T still to take
    } else if (fits) {
        // many candidates: their two low bytes, a histogram at a time
        if (tid < 256) {
            S.hist[0][tid] = 0;
            S.hist[1][tid] = 0;
        }
        __syncthreads();
        for (int idx = tid; idx < (int)C * kCandCap; idx += NT) {
            const uint32_t r = (uint32_t)idx / kCandCap, j = (uint32_t)idx % kCandCap;
            if (j < S.ncand_in[r]) atomicAdd(&S.hist[0][(cand[idx] >> 8) & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            uint32_t b2, r2;
            boundary_bin(S.hist[0], remaining, b2, r2);
            if (tid == 0) {
                S.res[0] = b2;
                S.res[1] = r2;
            }
        }
        __syncthreads();
        const uint32_t b2 = S.res[0];
        remaining = S.res[1];
        for (int idx = tid; idx < (int)C * kCandCap; idx += NT) {
            const uint32_t r = (uint32_t)idx / kCandCap, j = (uint32_t)idx % kCandCap;
            if (j < S.ncand_in[r] && ((cand[idx] >> 8) & 255u) == b2) atomicAdd(&S.hist[1][cand[idx] & 255u], 1u);
        }
        __syncthreads();
        if (tid < 32) {
            uint32_t b3, r3;
            boundary_bin(S.hist[1], remaining, b3, r3);
            if (tid == 0) {
                S.res[2] = b3;
                S.res[3] = r3;
            }
        }
        __syncthreads();
        remaining = S.res[3];
        T = prefix | (b2 << 8) | S.res[2];
    }
    if (fits) {
        // the candidates above T and equal to it: per CTA (one warp per CTA of the cluster, counted with
        // ballots), and per warp segment for this CTA's own
        for (uint32_t r = (uint32_t)warp; r < C; r += (uint32_t)nw) {
            const uint32_t nr = S.ncand_in[r];
            uint32_t above = 0, equal = 0;
            for (uint32_t j = (uint32_t)lane; j < ((nr + 31u) & ~31u); j += 32) {
                const uint32_t key = j < nr ? cand[r * kCandCap + j] : 0u;
                const bool a = j < nr && key > T, e = j < nr && key == T;
                above += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, a));
                equal += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, e));
                if (r == rank) {
                    if (a) atomicAdd(&S.scan_s[S.cwarp[j]], 1u);
                    if (e) atomicAdd(&S.scan_e[S.cwarp[j]], 1u);
                }
            }
            if (lane == 0) {
                S.gt[r] += above;
                S.ecnt[r] += equal;
            }
        }
    } else {
        // too many candidates: a full exchanged pass for each of the two low bytes, then this CTA's
        // per-warp counts by a pass over its keys
        exchange_pass<NT>(keys, n, prefix, 8, sbuf + C * 256, rank, C, remaining, bstar, S);
        prefix |= bstar << 8;
        exchange_pass<NT>(keys, n, prefix, 0, sbuf, rank, C, remaining, bstar, S);
        T = prefix | bstar;
        if (tid < (int)C) S.ecnt[tid] = sbuf[tid * 256 + bstar];
        uint32_t cg = 0, ce = 0;
        for (int b0 = lo; b0 < hi; b0 += 128) {
            const uint4 k4 = *reinterpret_cast<const uint4*>(keys + b0 + 4 * lane);
            const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                cg += kv[e] > T ? 1u : 0u;
                ce += kv[e] == T ? 1u : 0u;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            cg += __shfl_xor_sync(0xFFFFFFFFu, cg, off);
            ce += __shfl_xor_sync(0xFFFFFFFFu, ce, off);
        }
        if (lane == 0) {
            S.scan_s[warp] = cg;
            S.scan_e[warp] = ce;
        }
    }
    __syncthreads();  // the per-CTA counts (gt, ecnt) and the per-warp counts are complete
    if (tid == 0) {
        // this CTA's share of the ties (they go to the lowest positions, so to the lowest ranks first) and
        // its output offset
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
    // Ordered compaction: warp w writes the selected positions of its segment after those of the warps
    // before it (the same prefix sums over the warps, one lane per warp).  Per 128 keys (four per lane),
    // ballots give each key the number of selected keys in earlier lanes; only a chunk that holds a key
    // equal to the K-th key ranks its ties the same way.
    uint32_t tie_base, out_base;
    {
        const uint32_t e = lane < nw ? S.scan_e[lane] : 0u, g = lane < nw ? S.scan_s[lane] : 0u;
        uint32_t ties_incl = e;
#pragma unroll
        for (int off = 1; off < kMaxWarps; off <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, ties_incl, off);
            if (lane >= off) ties_incl += v;
        }
        const uint32_t tb = ties_incl - e;
        const uint32_t take_k = take_me > tb ? min(e, take_me - tb) : 0u;
        uint32_t run_incl = g + take_k;
#pragma unroll
        for (int off = 1; off < kMaxWarps; off <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, run_incl, off);
            if (lane >= off) run_incl += v;
        }
        tie_base = __shfl_sync(0xFFFFFFFFu, tb, warp);
        out_base = off_me + __shfl_sync(0xFFFFFFFFu, run_incl - (g + take_k), warp);
    }
    if (S.scan_s[warp] == 0 && (S.scan_e[warp] == 0 || tie_base >= take_me)) return;  // nothing selected here
    const uint32_t lt = lanemask_lt();
    uint32_t run_tie = tie_base, run_sel = out_base;
    for (int b0 = lo; b0 < hi; b0 += 128) {
        const int i = b0 + 4 * lane;
        const uint4 k4 = *reinterpret_cast<const uint4*>(keys + i);
        const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
        uint32_t tm = 0, sm = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            tm |= (kv[e] == T ? 1u : 0u) << e;
            sm |= (kv[e] > T ? 1u : 0u) << e;
        }
        if (__any_sync(0xFFFFFFFFu, tm != 0u)) {
            // ties in this chunk: rank them among the CTA's ties at earlier positions
            uint32_t bt[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) bt[e] = __ballot_sync(0xFFFFFFFFu, (tm >> e) & 1u);
            uint32_t tie_rank = run_tie;
#pragma unroll
            for (int e = 0; e < 4; ++e) tie_rank += (uint32_t)__popc(bt[e] & lt);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if ((tm >> e) & 1u) {
                    if (tie_rank < take_me) sm |= 1u << e;
                    ++tie_rank;
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) run_tie += (uint32_t)__popc(bt[e]);
        }
        uint32_t bs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) bs[e] = __ballot_sync(0xFFFFFFFFu, (sm >> e) & 1u);
        uint32_t pos = run_sel;
#pragma unroll
        for (int e = 0; e < 4; ++e) pos += (uint32_t)__popc(bs[e] & lt);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if ((sm >> e) & 1u) {
                if (pos < (uint32_t)K) {
                    out_row[pos] = range_start + i + e;
                    if (rows_row) rows_row[pos] = row_of(i + e);
                    if (score_row) score_row[pos] = key_score(kv[e]);
                }
                ++pos;
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) run_sel += (uint32_t)__popc(bs[e]);
    }
}

// One CTA of the indexer: scoring of this CTA's position range, then the cluster Top-K.  NT threads (the
// scoring roles use warps 0-9: producer, MMA issuer, two epilogue groups or, for MX keys, one epilogue
// group and four converters; all NT threads take part in the select).  smem_raw: the dynamic shared memory.
// LAST_TMEM: no later phase of the kernel allocates tensor memory, so the allocation permit is given up
// after this CTA's allocation.
template <int HI, int DI, int QB, bool FP8, int NT, bool LAST_TMEM, bool MX = false>
__device__ __forceinline__ void indexer_cta(const CUtensorMap& kmap, const CUtensorMap& qmap, const IndexerParams& p,
                                            uint8_t* smem_raw) {
    using Cfg = IdxCfg<HI, DI, QB, FP8, MX>;
    // four queries of 64 heads per block (two accumulator buffers): both epilogue groups read every tile,
    // two queries each
    constexpr bool kSplitQueries = !MX && QB == 4 && Cfg::kAccBufs == 2;
    // Several queries per block (scoring bound by the MMA thread's loop rather than by the K-cache
    // stream): the producer also waits until the tile's accumulator buffer is free before loading it, so
    // the MMA thread waits only for the landed stage.  With one query the stream sets the pace, and the
    // producer runs ahead by the full ring instead.
    constexpr bool kProducerWaitsAcc = !MX && QB >= 2;
    static_assert(!kSplitQueries || HI % 32 == 0, "split epilogue: the 32-column head loop");
    static_assert(NT % 32 == 0 && NT >= 256 && NT / 32 <= kMaxWarps, "thread count of the indexer body");
    // 1024-byte alignment for the swizzled operand tiles, by pointer arithmetic on the shared array (an
    // integer round trip would hide from the compiler that the derived pointers are shared, turning every
    // access into a slower generic one)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages;
    uint8_t* a_tiles = smem;                                   // S * kStageBytes
    uint8_t* q_tile = a_tiles + (size_t)S * Cfg::kStageBytes;  // kQBytes
    uint8_t* kexp_ring = q_tile + Cfg::kQBytes;                // MX: S * kScaleStageBytes, beside the stages
    uint32_t* keys = reinterpret_cast<uint32_t*>(kexp_ring + (size_t)S * Cfg::kScaleStageBytes);  // QB * chunk
    float* w_s = reinterpret_cast<float*>(keys + (size_t)QB * p.chunk);   // kN
    int32_t* pages_s = reinterpret_cast<int32_t*>(w_s + Cfg::kN);         // chunk / 64, padded to 16 bytes
    // everything after the page list is read with 16-byte vector loads: keep it 16-byte aligned
    uint32_t* hist0 = reinterpret_cast<uint32_t*>(pages_s + page_words(p.chunk));  // QB x 256
    uint32_t* allh = hist0 + QB * 256;                                      // C x 768 (select exchange)
    SelectSmem* sel = reinterpret_cast<SelectSmem*>(allh + 3 * cluster_nctarank() * 256);
    uint8_t* ctl_raw = reinterpret_cast<uint8_t*>(sel + 1);
    CtrlSmem* ctl = reinterpret_cast<CtrlSmem*>(ctl_raw + ((16u - (smem_u32(ctl_raw) & 15u)) & 15u));

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
    // this CTA's positions: its chunk of the candidate range [pos_begin, pos_end), up to the block's last query
    const int range_start = p.pos_begin + (int)rank * p.chunk;
    const int64_t range_end = (int64_t)range_start + p.chunk;
    const int64_t hi = min(min(range_end, p_last + 1), (int64_t)p.pos_end);
    const int n_pos = hi > range_start ? (int)(hi - range_start) : 0;
    const int ntiles = (n_pos + kTileM - 1) / kTileM;
    const int n_keys = ntiles * kTileM;

    // ---- set-up: page list, head weights, barriers, tensor memory --------------------------------------
    const int32_t* pt_row = p.page_table + (int64_t)b * p.max_pages;
    for (int i = tid; i < ntiles * 2; i += NT) {
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
    for (int i = tid; i < QB * 256; i += NT) hist0[i] = 0;
    for (int c = tid; c < Cfg::kN; c += NT) {
        float wv = 0.f;
        if (c < nq * HI) {
            const int64_t idx = (int64_t)(t0 + c / HI) * HI + (c % HI);
            wv = p.w[idx];
            if (FP8 && !MX) wv *= p.q_scale[idx];
        }
        w_s[c] = wv;
    }
    if constexpr (MX) {
        // the query tile dequantised to bf16 (exact: a code times a power of two) in the MMA's swizzled
        // K-major layout: head row h, 16-byte chunk j (dims 8j..8j+7) of atom j / 8
        const uint8_t* qc = reinterpret_cast<const uint8_t*>(p.q_idx_codes);
        const uint8_t* qe = reinterpret_cast<const uint8_t*>(p.q_scale);
        const uint32_t qb = smem_u32(q_tile);
        for (int i = tid; i < Cfg::kN * (DI / 8); i += NT) {
            const int h = i / (DI / 8), j = i % (DI / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < nq * HI) {
                const int64_t qrow = (int64_t)t0 * HI + h;
                const uint2 codes = __ldg(reinterpret_cast<const uint2*>(qc + qrow * DI + 8 * j));
                v = e4m3x8_to_bf16x8(codes, e8m0_factor(__ldg(qe + qrow * (DI / 32) + j / 4)));
            }
            st_shared_v4(qb + (j / 8) * (Cfg::kN * 128) + h * 128 + (((j % 8) ^ (h & 7)) << 4), v);
        }
        fence_proxy_async_smem();  // read by the MMAs through the async proxy
    }
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&ctl->full[s], 1);
            mbar_init(&ctl->empty[s], MX ? 4 : 1);  // MX: the four converter warps free the stage; else the MMA commit
        }
        for (int i = 0; i < 4; ++i) {
            mbar_init(&ctl->tfull[i], 1);
            // one arrival per epilogue warp that reads it: one group, or both groups with split queries
            mbar_init(&ctl->tempty[i], kSplitQueries ? 8 : 4);
        }
        mbar_init(&ctl->qbar, 1);
        mbar_init(&ctl->mma_done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->bfull[i], 4);  // MX: one arrival per converter warp
            mbar_init(&ctl->bempty[i], 1);
        }
        ctl->consumed = 0;
        ctl->issued = 0;
        ctl->qwaited = 0;
        fence_mbar_init();
    }
    if (warp == 1 && ntiles > 0) {
        tmem_alloc(&ctl->tmem_base, Cfg::kTmemCols);
        if (LAST_TMEM) tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (MX && tid == 0) mbar_arrive(&ctl->qbar);  // the dequantised query tile is in place

    // ---- scoring pipeline -----------------------------------------------------------------------------
    if (ntiles > 0) {
        // The producer and MMA warps run their loops with all 32 lanes (every lane waits on the barriers,
        // one lane issues), so no lane of these warps sits at the block barrier while the loop runs.
        if (warp == 0) {
            if (lane == 0) {
                prefetch_tensormap(&kmap);
                if (!MX) {
                    prefetch_tensormap(&qmap);
                    mbar_arrive_expect_tx(&ctl->qbar, Cfg::kQBytes);
#pragma unroll
                    for (int a = 0; a < Cfg::kAtoms; ++a)
                        tma_load_2d(q_tile + a * Cfg::kN * 128, &qmap, &ctl->qbar, a * (128 / Cfg::kElem), t0 * HI);
                }
            }
            int issued = 0;
            // the K cache is read once per step: evict-first, so its stream does not push the kernel's code
            // and later inputs out of L2
            const uint64_t kpol = l2_policy_evict_first();
            int s = 0;  // ring slot and its phase, advanced without a division by the runtime depth
            uint32_t ph = 0;
            for (int i = 0; i < ntiles; ++i, s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->empty[s], ph ^ 1u, p.err, p.wait_ns))) break;
                if constexpr (kProducerWaitsAcc) {
                    const uint32_t aph = (uint32_t)(i / Cfg::kAccBufs) & 1u;
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->tempty[i % Cfg::kAccBufs], aph ^ 1u, p.err, p.wait_ns)))
                        break;
                }
                if (elect_one_sync()) {  // one lane issues, with the warp converged (uniform issue path)
                    const int32_t pg0 = pages_s[2 * i], pg1 = pages_s[2 * i + 1];
                    const uint32_t bytes = (uint32_t)((pg0 >= 0) + (pg1 >= 0)) *
                                           (kPage * Cfg::kRowBytes + Cfg::kScaleStageBytes / 2);
                    if (bytes == 0) {
                        mbar_arrive(&ctl->full[s]);
                    } else {
                        mbar_arrive_expect_tx(&ctl->full[s], bytes);
                        uint8_t* dst = a_tiles + (size_t)s * Cfg::kStageBytes;
#pragma unroll
                        for (int a = 0; a < Cfg::kAtoms; ++a) {
                            if (pg0 >= 0)
                                tma_load_3d_hint(dst + a * (kTileM * 128), &kmap, &ctl->full[s],
                                                 a * (128 / Cfg::kElem), 0, pg0, kpol);
                            if (pg1 >= 0)
                                tma_load_3d_hint(dst + a * (kTileM * 128) + kPage * 128, &kmap, &ctl->full[s],
                                                 a * (128 / Cfg::kElem), 0, pg1, kpol);
                        }
                        if (MX) {  // each page's 64 x 4 scale bytes, contiguous in the cache
                            constexpr uint32_t kPageScaleBytes = Cfg::kScaleStageBytes / 2;
                            uint8_t* sdst = kexp_ring + (size_t)s * Cfg::kScaleStageBytes;
                            const uint8_t* ssrc = reinterpret_cast<const uint8_t*>(p.k_scale);
                            if (pg0 >= 0)
                                bulk_copy_g2s(sdst, ssrc + (int64_t)pg0 * kPageScaleBytes, kPageScaleBytes, &ctl->full[s]);
                            if (pg1 >= 0)
                                bulk_copy_g2s(sdst + kPageScaleBytes, ssrc + (int64_t)pg1 * kPageScaleBytes,
                                              kPageScaleBytes, &ctl->full[s]);
                        }
                    }
                }
                // (no warp barrier here: the next iteration's vote and elect.sync reconverge the warp)
                issued = i + 1;
            }
            if (lane == 0) ctl->issued = issued;
        } else if (warp == 1) {
            // The whole warp runs the issue loop and one elected lane issues each tile's MMAs and commit: the
            // issue path then stays warp-uniform (about 30 cycles per tcgen05.mma, against about 90 from a
            // single-lane branch, measured on this GPU).  elect.sync picks the lowest lane every time, so the
            // same thread issues every MMA and the commits that track them.
            const uint32_t tmem = ctl->tmem_base;
            int consumed = 0;
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&ctl->qbar, 0, p.err, p.wait_ns));
            if (lane == 0) ctl->qwaited = ok ? 1 : 0;
            // Precomputed descriptors: each is a base plus a compile-time offset (the start address field holds
            // address / 16 and no address here reaches 2^18, so adding to the descriptor adds to the address).
            const uint64_t ad0 = smem_desc(smem_u32(a_tiles), 16, 1024, kSwizzle128B);  // stage s: + s * kStageBytes / 16
            const uint64_t bd0 = smem_desc(smem_u32(q_tile), 16, 1024, kSwizzle128B);
            int s = 0;
            uint32_t ph = 0;
            for (int i = 0; ok && i < ntiles; ++i, s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                const int ab = i % Cfg::kAccBufs;
                const uint32_t aph = (uint32_t)(i / Cfg::kAccBufs) & 1u;
                // the accumulator buffer is free (seen here, or by the producer before it loaded the stage)
                if (!kProducerWaitsAcc && !__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->tempty[ab], aph ^ 1u, p.err, p.wait_ns)))
                    break;
                // the tile to score: the loaded stage, or (MX) its dequantised copy in TMEM
                uint64_t* ready = MX ? &ctl->bfull[i & 1] : &ctl->full[s];
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(ready, MX ? (((uint32_t)i >> 1) & 1u) : ph, p.err, p.wait_ns)))
                    break;
                consumed = i + 1;
                tc_fence_after();
                if (elect_one_sync()) {
                    const uint64_t ads = ad0 + (uint64_t)((uint32_t)s * (uint32_t)(Cfg::kStageBytes / 16));
#pragma unroll
                    for (int k = 0; k < Cfg::kKSteps; ++k) {
                        constexpr int kStep = Cfg::kMmaK * Cfg::kMmaElem;  // bytes along K per MMA
                        const int kb = k * kStep;
                        const int atom = kb / 128, off = kb % 128;
                        const uint64_t ad = ads + (uint64_t)((atom * (kTileM * 128) + off) / 16);
                        const uint64_t bd = bd0 + (uint64_t)((atom * (Cfg::kN * 128) + off) / 16);
                        if (MX)
                            umma_f16_ts(tmem + ab * Cfg::kN, tmem + Cfg::kACol + (i & 1) * Cfg::kACols + k * 8, bd,
                                        Cfg::kIdesc, k > 0);
                        else if (Cfg::kMmaBf16)
                            umma_f16_ss(tmem + ab * Cfg::kN, ad, bd, Cfg::kIdesc, k > 0);
                        else
                            umma_f8_ss(tmem + ab * Cfg::kN, ad, bd, Cfg::kIdesc, k > 0);
                    }
                    // the stage is free once these MMAs complete (MX: the converters free the FP8 stage, and
                    // this commit frees their TMEM tile); then the accumulator is ready for the epilogue
                    umma_commit(MX ? &ctl->bempty[i & 1] : &ctl->empty[s]);
                    umma_commit(&ctl->tfull[ab]);
                }
                // (no warp barrier here: the next iteration's votes and elect.sync reconverge the warp)
            }
            if (lane == 0 && !MX) ctl->consumed = consumed;
            // Drain: tensor memory is released below only once every MMA issued here has completed (the
            // epilogue has waited for all of them unless a pipeline wait gave up)
            if (consumed > 0 && elect_one_sync()) {
                umma_commit(&ctl->mma_done);
                mbar_wait(&ctl->mma_done, 0, p.err);
            }
            __syncwarp();
        } else if (MX && warp >= 6 && warp < 10) {
            // MX converters: each landed FP8 tile, dequantised to bf16 with the key's group scales, goes to
            // one of two TMEM tiles the MMA reads as its A operand; the FP8 stage is then free again
            static_assert(NT >= 320, "the MX converters are warps 6-9");
            const int row = (warp & 3) * 32 + lane;  // position within the tile = the TMEM lane this warp may write
            const uint32_t trow = ctl->tmem_base + (((uint32_t)(warp & 3) * 32u) << 16) + Cfg::kACol;
            int consumed = 0, s = 0;
            uint32_t ph = 0;
            // half a row: chunks h*4 .. h*4+3 of 16 codes (chunk c: dims 16c..16c+15, scale group c / 2)
            // times their group factors, stored as TMEM columns 32h .. 32h+31 of the row; BIG: factors
            // beyond 2^127 take a second product
            auto convert = [&](auto big_tag, int h, uint32_t kexp, uint32_t src, uint32_t dst) {
                constexpr bool BIG = decltype(big_tag)::value;
                uint4 in[4];
                uint32_t o[32];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                 : "=r"(in[j].x), "=r"(in[j].y), "=r"(in[j].z), "=r"(in[j].w)
                                 : "r"(src + (((4 * h + j) ^ (row & 7)) << 4)));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = 4 * h + j;
                    const uint32_t e = (kexp >> (8 * (c / 2))) & 255u;
                    const uint32_t flo = mx_factor_lo(e);
                    const uint32_t fhi = BIG ? mx_factor_hi(e) : 0u;
                    const uint32_t wd[4] = {in[j].x, in[j].y, in[j].z, in[j].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t& lo = o[8 * j + 2 * k];
                        uint32_t& hi = o[8 * j + 2 * k + 1];
                        lo = bf16x2_mul(e4m3x2_to_bf16x2_unscaled(wd[k], 0x1804u), flo);
                        hi = bf16x2_mul(e4m3x2_to_bf16x2_unscaled(wd[k], 0x3A24u), flo);
                        if (BIG) {
                            lo = bf16x2_mul(lo, fhi);
                            hi = bf16x2_mul(hi, fhi);
                        }
                    }
                }
                tmem_st16_u32(dst + 32 * h, o);
                tmem_st16_u32(dst + 32 * h + 16, o + 16);
            };
            for (int i = 0; i < ntiles; ++i, s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0) ? 1u : 0u) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->full[s], ph, p.err, p.wait_ns))) break;
                consumed = i + 1;
                if (!__all_sync(0xFFFFFFFFu,
                                mbar_wait(&ctl->bempty[i & 1], (((uint32_t)i >> 1) & 1u) ^ 1u, p.err, p.wait_ns)))
                    break;
                tc_fence_after();  // the MMAs that read this TMEM tile have completed
                const uint32_t src = smem_u32(a_tiles + (size_t)s * Cfg::kStageBytes) + row * 128;
                const uint32_t dst = trow + (uint32_t)((i & 1) * Cfg::kACols);
                uint32_t kexp;  // the row's four scale bytes (group g in byte g)
                asm volatile("ld.shared.b32 %0, [%1];"
                             : "=r"(kexp)
                             : "r"(smem_u32(kexp_ring + (size_t)s * Cfg::kScaleStageBytes) + row * 4));
                if (__any_sync(0xFFFFFFFFu, __vcmpgtu4(kexp, 0x86868686u) != 0u)) {
                    convert(std::true_type{}, 0, kexp, src, dst);
                    convert(std::true_type{}, 1, kexp, src, dst);
                } else {
                    convert(std::false_type{}, 0, kexp, src, dst);
                    convert(std::false_type{}, 1, kexp, src, dst);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ctl->empty[s]);
                    mbar_arrive(&ctl->bfull[i & 1]);
                }
            }
            if (lane == 0 && warp == 6) ctl->consumed = consumed;
        } else if (warp >= 2 && warp < (MX ? 6 : 10)) {
            // Two epilogue groups (warps 2-5 and 6-9; MX keeps warps 6-9 for its converters), each covering
            // the four TMEM lane quadrants.  With up to two queries per block they take alternate tiles (an
            // accumulator buffer is read by one group).  With four queries a tile's accumulator is 256
            // columns, only two buffers fit in tensor memory, and the MMA of tile i + 2 waits for the
            // epilogue of tile i: both groups then read every tile, each for two of the queries, which
            // halves the epilogue's chain of tensor-memory loads per tile.
            static_assert(MX || NT >= 320, "the second epilogue group is warps 6-9");
            const int group = (warp - 2) >> 2;
            const uint32_t quad = (uint32_t)(warp & 3);  // TMEM lanes this warp may access
            const int row = (int)quad * 32 + lane;       // position within the tile
            const uint32_t tmem = ctl->tmem_base + ((quad * 32u) << 16);
            int64_t pq[QB];
#pragma unroll
            for (int q = 0; q < QB; ++q) pq[q] = (int64_t)L - n_b + j0 + q;
            for (int i = kSplitQueries ? 0 : group; i < ntiles; i += (MX || kSplitQueries) ? 1 : 2) {
                const int ab = i % Cfg::kAccBufs;
                const uint32_t aph = (uint32_t)(i / Cfg::kAccBufs) & 1u;
                const int local = i * kTileM + row;
                const int pos = range_start + local;
                const int32_t pg = pages_s[2 * i + (row >> 6)];
                float ksc = 1.f;
                if (FP8 && !MX && pg >= 0) ksc = __ldg(p.k_scale + (int64_t)pg * kPage + (row & 63));
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->tfull[ab], aph, p.err, p.wait_ns))) break;
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
                        if (kSplitQueries && (q >> 1) != group) continue;  // the other group's queries
                        // partial sums in pairs (2k, 2k+1), advanced by the packed fp32x2 FMA: one instruction
                        // per two heads, each lane of it the same rounding as a scalar FMA
                        float2 part[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                          make_float2(0.f, 0.f)};
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
                                float2& pk = part[j4 & 3];
                                pk = __ffma2_rn(make_float2(wv.x, wv.y), make_float2(fmaxf(v[0], 0.f), fmaxf(v[1], 0.f)), pk);
                                pk = __ffma2_rn(make_float2(wv.z, wv.w), make_float2(fmaxf(v[2], 0.f), fmaxf(v[3], 0.f)), pk);
                            }
                        }
                        acc[q] = ((part[0].x + part[0].y) + (part[1].x + part[1].y)) +
                                 ((part[2].x + part[2].y) + (part[3].x + part[3].y));
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
                    if (kSplitQueries && (q >> 1) != group) continue;
                    uint32_t key = 0;
                    if (q < nq && pg >= 0 && (int64_t)pos <= pq[q] && pos < p.pos_end)
                        key = score_key((FP8 && !MX) ? acc[q] * ksc : acc[q]);
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
        // candidate positions of this query: [pos_begin, min(p + 1, pos_end))
        const int64_t visible = max((int64_t)0, min((int64_t)L - n_b + j0 + q + 1, (int64_t)p.pos_end) - p.pos_begin);
        // the smem stage ring is idle once every CTA has scored: it holds the select's fallback exchange space
        cluster_select<NT>(keys + (size_t)q * p.chunk, hist0 + q * 256, allh, reinterpret_cast<uint32_t*>(a_tiles),
                       n_keys, p.top_k, visible,
                       p.topk + (int64_t)(t0 + q) * p.top_k, range_start, rank, C, *sel, pages_s,
                       p.rows_out ? p.rows_out + (int64_t)(t0 + q) * p.top_k : nullptr,
                       p.topk_score ? p.topk_score + (int64_t)(t0 + q) * p.top_k : nullptr, p.pos_begin);
    }
    // No cluster barrier here: every remote access is a histogram push, and the pushes of a pass complete
    // before that pass's barrier, so after the last pass no CTA touches another's shared memory.
    __syncthreads();
    if (tid == 0) {  // the barriers' memory may be reused by whatever runs next in this CTA
        for (int s = 0; s < S; ++s) {
            mbar_inval(&ctl->full[s]);
            mbar_inval(&ctl->empty[s]);
        }
        for (int i = 0; i < 4; ++i) {
            mbar_inval(&ctl->tfull[i]);
            mbar_inval(&ctl->tempty[i]);
        }
        mbar_inval(&ctl->qbar);
        mbar_inval(&ctl->mma_done);
        for (int i = 0; i < 2; ++i) {
            mbar_inval(&ctl->bfull[i]);
            mbar_inval(&ctl->bempty[i]);
        }
    }
}

template <int HI, int DI, int QB, bool FP8, bool MX = false>
size_t indexer_smem_bytes(int stages, int chunk, int cluster) {
    using Cfg = IdxCfg<HI, DI, QB, FP8, MX>;
    return 1024 + (size_t)stages * Cfg::kStageBytes + Cfg::kQBytes + (size_t)QB * chunk * 4 + Cfg::kN * 4 +
           (size_t)stages * Cfg::kScaleStageBytes +
           (size_t)page_words(chunk) * 4 + (size_t)(QB + 3 * cluster) * 256 * 4 + sizeof(SelectSmem) + sizeof(CtrlSmem) +
           64;
}

}  // namespace
}  // namespace dsa
