// Device code of the sparse flash attention over the Top-K selected rows of a paged MLA latent-KV cache
// (shared by the standalone attention kernel and the single-launch decode kernel), for sm_103a.
//
// For each query token t and head h: z_s = scale * q[t,h,:] . kv[s,:] over the selected positions s,
// out[t,h,:] = softmax(z) . kv[:, :Dv], lse = logsumexp(z) ("Optimizing Inference for Hybrid Attention
// Architectures: From Operator Fusion to Sequence Sharding", section "Breaking Down the Computational
// Path of Hybrid Attention", step 2; "Day0 Inference Support and Performance Optimization for New LLM
// Architectures", section 3.2: only the selected positions' KV rows are read; "Optimizing Inference for
// Hybrid Attention LLMs: Practices for Fast Adaptation", section 3.2: gather of the next rows overlaps
// the computation on the current ones).
//
// One CTA pair per (query token, position split):
//   * the 128 query heads are the UMMA M dimension.  Q[t] (128 x 576 bf16) is split by 64-dim atoms:
//     atoms 0-3 stay in shared memory (SMEM A operand), atoms 4-8 live in tensor memory (TMEM A
//     operand), which leaves shared memory for double-buffered row tiles;
//   * at start every thread helps translate the split's selected positions (Top-K entry -> page table
//     -> physical row) into a row list in smem, in two dependent rounds of independent loads (the
//     entries together with a parallel search for the token's sequence, then the pages together with
//     the sequence length), so no global lookup sits on the per-tile path;
//   * the selected rows are processed 64 at a time (UMMA N = 64: below that a tcgen05.mma costs about
//     as much as at N = 64).  Each tile is kept as the 256 value dims this CTA owns (the "V part") and
//     the other 320 dims (the "K part"), each double-buffered and refilled by its own four gather warps
//     with cp.async pieces written straight into the 128B-swizzled operand layout (per-lane 16-byte
//     copies issue faster here than TMA tile::gather4, which moves only 4 rows per copy).  The loads of
//     a tile are issued about two tiles ahead of its use, which hides the HBM latency without an L2
//     prefetch; bf16 rows are copied under an evict-first L2 policy (read once per step, they would
//     otherwise push the kernel's own code out of L2);
//   * the MMA issuer runs S(i) = Q K(i)^T over the K part, then O += P(i-1) V(i-1), then the V-part
//     atoms of S(i).  The V buffer of a tile is busy until its P V has run, so this order gives its
//     refill a whole tile period; the K buffer is free as soon as the K-part MMAs of S(i) complete;
//   * the softmax of tile i (one thread per head row, online max raised only when it grows by more
//     than 2^8 so O rarely needs rescaling) overlaps the K-part MMAs of S(i+1);
//   * O += P V (M=128, N=256, K=64; A = P from TMEM, B = the V part read as an MN-major operand)
//     accumulates in TMEM.  The 512 value dims are split between the two CTAs of the pair (each owns 256
//     columns of O) because a full 128 x 512 fp32 O would fill all of TMEM; both CTAs compute the same S.
//   * With more than one position split, the partial (O, max, sum) of the splits are merged through L2:
//     bulk copies of the rows each split owns into the workspace, one cluster barrier, bulk copies back,
//     and a combine straight from TMEM.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kDim = 576;  // latent + rope
constexpr int kVDim = 512;
// warp 0: Q load, 1: MMA, 2-5: softmax, then the K-part and the V-part gather warps
constexpr int kKWarps = 4;
constexpr int kVWarps = 4;
constexpr int kFirstGatherWarp = 6;
constexpr int kThreadsSfa = 32 * (kFirstGatherWarp + kKWarps + kVWarps);
constexpr int kRows = 64;         // selected rows per tile
constexpr int kAtoms = kDim / 64;  // 128-byte swizzle atoms per row
constexpr int kSmemQAtoms = 4;     // Q atoms 0-3 in smem, 4-8 in TMEM
constexpr int kKAtoms = 5;         // atoms of the K part (the V part has 4)
constexpr int kAtomBytes = kRows * 128;
constexpr int kQAtomBytes = 128 * 128;
constexpr int kQBytes = kSmemQAtoms * kQAtomBytes;
constexpr int kKBufBytes = kKAtoms * kAtomBytes;
constexpr int kVBufBytes = 4 * kAtomBytes;
constexpr int kMaxEntries = kSfaMaxEntries;  // selected entries per CTA (per position split)
constexpr int kEntPerThread = (kMaxEntries + kThreadsSfa - 1) / kThreadsSfa;
constexpr int kMaxSplits = 8;
constexpr int kOCols = 256;        // TMEM columns [0, 256): O (this CTA's value half)
constexpr int kSCol = 256;         // [256, 320): S
constexpr int kPCol = 320;         // [320, 352): P, 64 bf16 per row
constexpr int kQCol = 352;         // [352, 512): Q atoms 4-8, 32 columns each
constexpr int kTmemCols = 512;
constexpr uint32_t kIdescQK = make_idesc(128, kRows, 1, 1, 0, 0);
constexpr uint32_t kIdescPV = make_idesc(128, kOCols, 1, 1, 0, 1);
constexpr float kRescaleLog2 = 8.f;  // raise the running max only when it grows by more than this

struct SfaCtrl {
    uint64_t q_full;   // Q atoms 0-3 in smem
    uint64_t qt_full;  // Q atoms 4-8 in TMEM
    uint64_t k_full[2], k_empty[2];
    uint64_t v_full[2], v_empty[2];
    uint64_t s_full, s_empty;
    uint64_t p_full, p_empty;
    uint64_t mma_done;
    uint64_t merge_full;  // split merge: the other splits' rows of this CTA have landed in smem
    uint32_t tmem_base;
    int32_t q_waited;
    int32_t tok_b, tok_cu0, tok_cu1;  // sequence of this CTA's query token and its query offsets
};

constexpr size_t kSfaSmem =
    1024 + kQBytes + 2 * kKBufBytes + 2 * kVBufBytes + kMaxEntries * 4 + sizeof(SfaCtrl);

// 2^x by the SFU approximation (relative error about 2^-22, far below the bf16 rounding of P);
// ex2(-inf) = +0.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Atom a (64 dims) of a row belongs to the V part of the CTA that owns value half dvh.
__device__ __forceinline__ bool is_v_atom(int a, int dvh) { return a >= 4 * dvh && a < 4 * dvh + 4; }
// Slot of atom a inside its part's buffer.
__device__ __forceinline__ int part_slot(int a, int dvh) {
    if (is_v_atom(a, dvh)) return a - 4 * dvh;
    return dvh == 0 ? a - 4 : (a < 4 ? a : 4);
}

// One CTA of the sparse attention (kThreadsSfa threads).  smem_raw: the dynamic shared memory.
// KVFP8: the latent-KV rows are in the FP8 row layout (dequantised to bf16 by the gather warps).
template <bool KVFP8>
__device__ __forceinline__ void sfa_cta(const CUtensorMap& qmap, const SfaParams& p, uint8_t* smem_raw) {
    // 1024-byte alignment by pointer arithmetic on the shared array (an integer round trip would hide from
    // the compiler that the derived pointers are shared, turning every access into a slower generic one)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* q_s = smem;                         // Q atoms 0-3: [atom][128 rows][128 B]
    uint8_t* kbuf = q_s + kQBytes;               // 2 x K part: [slot][64 rows][128 B]
    uint8_t* vbuf = kbuf + 2 * kKBufBytes;       // 2 x V part
    int32_t* rows_s = reinterpret_cast<int32_t*>(vbuf + 2 * kVBufBytes);  // physical row per entry, -1 = skip
    SfaCtrl* ctl = reinterpret_cast<SfaCtrl*>(rows_s + kMaxEntries);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = p.splits;
    const int dvh = blockIdx.x & 1;
    const int ps = (blockIdx.x >> 1) % P;
    const int t = blockIdx.x / (2 * P);
    if (t >= p.total_q) return;  // uniform over the cluster
    const int per = ((p.top_k + P - 1) / P + kRows - 1) / kRows * kRows;
    const int e0 = ps * per;
    const int n_ent = max(0, min(p.top_k, e0 + per) - e0);
    const int ntiles = (n_ent + kRows - 1) / kRows;

    // ---- set-up.  Launched right behind this library's indexer (early_setup), everything up to the wait
    // below overlaps the indexer's tail: only the Top-K entries come from it.  Otherwise any input may come
    // from the previous kernel in the stream, so the kernel waits first.
    if (tid == 0) prefetch_tensormap(&qmap);
    if (!p.early_setup) grid_dependency_wait();
    int32_t ent[kEntPerThread];
    // the split's Top-K entries, or (rows_in: written by the indexer phase of this launch) their physical rows
    auto load_entries = [&]() {
        const int32_t* sel = (p.rows_in ? p.rows_in : p.topk) + (int64_t)t * p.top_k + e0;
#pragma unroll
        for (int k = 0; k < kEntPerThread; ++k) {
            const int e = tid + k * kThreadsSfa;
            ent[k] = e < n_ent ? __ldcg(sel + e) : -1;  // L2: may have been written earlier in this launch
        }
    };
    if (!p.early_setup) load_entries();  // overlaps the sequence search
    // the sequence that holds token t: a parallel search over the query offsets, or (one query token per
    // sequence) sequence t, whose offsets and length are then loaded together and checked
    int b, cu0, cu1, L;
    if (p.one_query_per_seq) {
        b = t;
        cu0 = __ldg(p.cu_q_lens + t);
        cu1 = __ldg(p.cu_q_lens + t + 1);
        L = __ldg(p.seq_lens + t);
        if (cu0 != t || cu1 != t + 1) {
            if (tid == 0 && dvh == 0 && ps == 0) raise_error(p.err, DSA_DEVERR_SEQ);
            return;  // uniform over the cluster (same token)
        }
    } else {
        if (tid == 0) ctl->tok_b = -1;
        __syncthreads();
        for (int j = tid; j < p.batch; j += kThreadsSfa) {
            const int c0 = __ldg(p.cu_q_lens + j), c1 = __ldg(p.cu_q_lens + j + 1);
            if (c0 <= t && t < c1) {  // one sequence when the offsets are non-decreasing
                ctl->tok_b = j;
                ctl->tok_cu0 = c0;
                ctl->tok_cu1 = c1;
            }
        }
        __syncthreads();
        b = ctl->tok_b;
        if (b < 0) {
            if (tid == 0 && dvh == 0 && ps == 0) raise_error(p.err, DSA_DEVERR_SEQ);
            return;  // uniform over the cluster (same token)
        }
        cu0 = ctl->tok_cu0;
        cu1 = ctl->tok_cu1;
        L = __ldg(p.seq_lens + b);
    }
    const int n_b = cu1 - cu0;
    if (n_b > L || L > p.max_pages * 64) {
        if (tid == 0 && dvh == 0 && ps == 0) raise_error(p.err, DSA_DEVERR_SEQ);
        return;  // uniform over the cluster (same token)
    }
    const int64_t pos = (int64_t)L - n_b + (t - cu0);
    if (tid == 0) {
        mbar_init(&ctl->q_full, 1);
        mbar_init(&ctl->qt_full, 4);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->k_full[i], 32 * kKWarps);  // one cp.async-tracked arrival per gather lane
            mbar_init(&ctl->k_empty[i], 1);
            mbar_init(&ctl->v_full[i], 32 * kVWarps);
            mbar_init(&ctl->v_empty[i], 1);
        }
        mbar_init(&ctl->s_full, 1);
        mbar_init(&ctl->s_empty, 4);
        mbar_init(&ctl->p_full, 4);
        mbar_init(&ctl->p_empty, 1);
        mbar_init(&ctl->mma_done, 1);
        mbar_init(&ctl->merge_full, 1);
        ctl->q_waited = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    if (tid == 0) {
        // Q atoms 0-3 into shared memory (TMA)
        mbar_arrive_expect_tx(&ctl->q_full, kQBytes);
        for (int a = 0; a < kSmemQAtoms; ++a) tma_load_2d(q_s + a * kQAtomBytes, &qmap, &ctl->q_full, a * 64, t * p.heads);
    }
    if (warp >= 2 && warp < 6) {
        // Q atoms 4-8 of this head row into TMEM (the A operand of those atoms' MMAs)
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t trow = tmem + ((quad * 32u) << 16);
        const int h = (int)quad * 32 + lane;
        const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)t * p.heads + h) * kDim + 64 * kSmemQAtoms);
        constexpr int kGroups = (kAtoms - kSmemQAtoms) * 2;  // 16-column groups
        static_assert(kGroups % 2 == 0, "two batches");
#pragma unroll 1
        for (int c0 = 0; c0 < kGroups; c0 += kGroups / 2) {
            // one batch of independent 16-byte loads in flight, then the TMEM stores
            uint32_t qv[kGroups / 2][16];
#pragma unroll
            for (int c = 0; c < kGroups / 2; ++c) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 v = h < p.heads ? __ldg(src + (c0 + c) * 4 + j) : make_uint4(0, 0, 0, 0);
                    qv[c][4 * j] = v.x;
                    qv[c][4 * j + 1] = v.y;
                    qv[c][4 * j + 2] = v.z;
                    qv[c][4 * j + 3] = v.w;
                }
            }
#pragma unroll
            for (int c = 0; c < kGroups / 2; ++c) tmem_st16_u32(trow + kQCol + (c0 + c) * 16, qv[c]);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->qt_full);
    }
    // ---- this split's entries -> physical rows (the Top-K entries, then their pages) ----
    if (p.early_setup) {
        grid_dependency_wait();
        load_entries();
    }
    if (p.rows_in) {
        // physical rows already: only a bounds check (a row that no valid selection can produce is an error)
#pragma unroll
        for (int k = 0; k < kEntPerThread; ++k) {
            const int e = tid + k * kThreadsSfa;
            if (e >= ntiles * kRows) continue;
            int32_t row = ent[k];
            if (row < -1 || (int64_t)row >= (int64_t)p.num_pages * 64) {
                if (dvh == 0) raise_error(p.err, DSA_DEVERR_PAGE);
                row = -1;
            }
            rows_s[e] = row;
        }
    } else {
    int32_t pg[kEntPerThread];
    {
        const int32_t* pt_row = p.page_table + (int64_t)b * p.max_pages;
#pragma unroll
        for (int k = 0; k < kEntPerThread; ++k)
            pg[k] = (ent[k] >= p.pos_begin && ent[k] >= 0 && ent[k] < p.pos_end && (ent[k] >> 6) < p.max_pages)
                        ? __ldg(pt_row + (ent[k] >> 6))
                        : -1;
    }
#pragma unroll
    for (int k = 0; k < kEntPerThread; ++k) {
        const int e = tid + k * kThreadsSfa;
        if (e >= ntiles * kRows) continue;
        int32_t row = -1;
        const int32_t s_pos = ent[k];
        // entries of another context shard are skipped (valid, not this call's)
        if (s_pos >= 0 && s_pos >= p.pos_begin && s_pos < p.pos_end) {
            if ((int64_t)s_pos > pos) {
                if (dvh == 0) raise_error(p.err, DSA_DEVERR_INDEX);
            } else if (pg[k] < 0 || pg[k] >= p.num_pages) {
                if (dvh == 0) raise_error(p.err, DSA_DEVERR_PAGE);
            } else {
                row = pg[k] * 64 + (s_pos & 63);
            }
        }
        rows_s[e] = row;
    }
    }
    __syncthreads();

    float m_used = -INFINITY, l_sum = 0.f;  // softmax threads: running max (log2 units) and sum
    if (warp >= kFirstGatherWarp) {
        // ---------------- gather: kKWarps warps fill the K part, kVWarps warps the V part ----------------
        const int gw = warp - kFirstGatherWarp;
        const bool v_part = gw >= kKWarps;
        const int pw = v_part ? gw - kKWarps : gw;  // warp index within its part
        const int nw = v_part ? kVWarps : kKWarps;
        const int c8 = lane & 7;
        if constexpr (KVFP8) {
            // FP8 rows through registers.  The loads of a tile need no buffer, only its stores do: each lane
            // loads the next tile's data (its four rows: the codes of the part's four latent atoms, their two
            // tile scales, the K part's rotary piece) right after storing the current one, so the HBM
            // latency is spent while the buffer is still in use; once it is free, the lane dequantises into
            // the swizzled bf16 layout, fences for the async proxy and arrives.
            static_assert(kRows == 4 * 4 * kKWarps && kKWarps == kVWarps, "four rows per lane");
            const int a0 = 4 * (v_part ? dvh : 1 - dvh);  // first latent atom of this part
            const uint8_t* kvb = reinterpret_cast<const uint8_t*>(p.kv_cache);
            uint2 cd[4][4], sc[4];
            uint4 rope[4];
            auto load_tile = [&](int i) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int32_t row = rows_s[i * kRows + 4 * pw + 16 * k + (lane >> 3)];
                    const bool ok = row >= 0;
                    const uint8_t* src = kvb + (int64_t)(ok ? row : 0) * kKvFp8RowBytes;
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2)
                        cd[k][s2] = ok ? __ldg(reinterpret_cast<const uint2*>(src + (a0 + s2) * 64 + c8 * 8))
                                       : make_uint2(0, 0);
                    sc[k] = ok ? __ldg(reinterpret_cast<const uint2*>(src + kKvFp8ScaleOff + 4 * (a0 / 2)))
                               : make_uint2(0, 0);
                    rope[k] = (ok && !v_part)
                                  ? __ldg(reinterpret_cast<const uint4*>(src + kKvFp8RopeOff + c8 * 16))
                                  : make_uint4(0, 0, 0, 0);
                }
            };
            if (ntiles > 0) load_tile(0);
            for (int i = 0; i < ntiles; ++i) {
                const int bsel = i & 1;
                uint64_t* full = v_part ? &ctl->v_full[bsel] : &ctl->k_full[bsel];
                uint64_t* empty = v_part ? &ctl->v_empty[bsel] : &ctl->k_empty[bsel];
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty, (((uint32_t)i >> 1) & 1u) ^ 1u, p.err, p.wait_ns))) break;
                const uint32_t base = smem_u32(v_part ? vbuf + bsel * kVBufBytes : kbuf + bsel * kKBufBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 4 * pw + 16 * k + (lane >> 3);
                    const uint32_t row_base = base + r * 128 + ((c8 ^ (r & 7)) << 4);
#pragma unroll
                    for (int s2 = 0; s2 < 4; ++s2) {
                        const float scale = __uint_as_float(s2 < 2 ? sc[k].x : sc[k].y);
                        st_shared_v4(row_base + part_slot(a0 + s2, dvh) * kAtomBytes, e4m3x8_to_bf16x8(cd[k][s2], scale));
                    }
                    if (!v_part) st_shared_v4(row_base + part_slot(kAtoms - 1, dvh) * kAtomBytes, rope[k]);
                }
                fence_proxy_async_smem();  // the MMAs read these bytes through the async proxy
                mbar_arrive(full);
                if (i + 1 < ntiles) load_tile(i + 1);
            }
        } else {
            // The selected rows are read once per step (by both CTAs of a pair, within a tile period): an
            // evict-first L2 policy keeps their 75 MB stream from pushing the kernel's code and the step's
            // other inputs out of L2 (code fetched from HBM made the first tiles several us slower).  The
            // FP8 rows above keep plain loads: the hinted loads measured slower there.
            const uint64_t kvpol = l2_policy_evict_first();
            for (int i = 0; i < ntiles; ++i) {
                const int bsel = i & 1;
                uint64_t* full = v_part ? &ctl->v_full[bsel] : &ctl->k_full[bsel];
                uint64_t* empty = v_part ? &ctl->v_empty[bsel] : &ctl->k_empty[bsel];
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(empty, (((uint32_t)i >> 1) & 1u) ^ 1u, p.err, p.wait_ns))) break;
                const uint32_t base = smem_u32(v_part ? vbuf + bsel * kVBufBytes : kbuf + bsel * kKBufBytes);
    #pragma unroll 1
                for (int r0 = 4 * pw; r0 < kRows; r0 += 4 * nw) {
                    const int r = r0 + (lane >> 3);
                    const int32_t row = rows_s[i * kRows + r];
                    const uint16_t* src = p.kv_cache + (int64_t)row * kDim + c8 * 8;
                    const uint32_t row_base = base + r * 128 + ((c8 ^ (r & 7)) << 4);
    #pragma unroll
                    for (int a = 0; a < kAtoms; ++a) {
                        if (is_v_atom(a, dvh) != v_part) continue;
                        const uint32_t dst = row_base + part_slot(a, dvh) * kAtomBytes;
                        if (row >= 0)
                            cp_async_16_hint(dst, src + a * 64, kvpol);
                        else
                            cp_async_zero16(dst, p.kv_cache);
                    }
                }
                // every lane signals once its own copies have landed; the warp moves on to the next tile at once
                cp_async_mbar_arrive(full);
            }
            cp_async_wait_all();
        }
    }
    else if (warp == 1) {
        // ---------------- MMA issuer: S(i) = Q K(i)^T, then O += P(i-1) V(i-1) ----------------
        // The whole warp runs the loop and waits; one elected lane issues each group of MMAs and its commits.
        // The issue path then stays warp-uniform (about 30 cycles per tcgen05.mma, against about 90 from a
        // single-lane branch, measured on this GPU), and elect.sync picks the lowest lane every time, so one
        // thread issues every MMA and the commits that track them.  Each shared-memory descriptor is a
        // precomputed base plus a constant offset (the start address field holds address / 16 and no address
        // here reaches 2^18, so adding to the descriptor adds to the address), and the atom order of each
        // value half is a compile-time list.
        {
            bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&ctl->q_full, 0, p.err, p.wait_ns));
            if (lane == 0) ctl->q_waited = ok ? 1 : 0;
            ok = ok && __all_sync(0xFFFFFFFFu, mbar_wait(&ctl->qt_full, 0, p.err, p.wait_ns));
            const uint64_t qd0 = smem_desc(smem_u32(q_s), 16, 1024, kSwizzle128B);   // Q atom a: + a * (kQAtomBytes / 16)
            const uint64_t kd0 = smem_desc(smem_u32(kbuf), 16, 1024, kSwizzle128B);  // K part buffer, slot
            const uint64_t vd0 = smem_desc(smem_u32(vbuf), 16, 1024, kSwizzle128B);  // V part buffer, slot
            // the V part as an MN-major operand of P V: 64-dim atoms kAtomBytes apart, 8-row groups 1024 B apart
            const uint64_t pvd0 = smem_desc(smem_u32(vbuf), kAtomBytes, 1024, kSwizzle128B);
            constexpr uint32_t kAtomStep = kAtomBytes / 16, kKBufStep = kKBufBytes / 16, kVBufStep = kVBufBytes / 16;
            auto pv = [&](int j) -> bool {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->p_full, (uint32_t)j & 1u, p.err, p.wait_ns))) return false;
                tc_fence_after();
                if (elect_one_sync()) {
                    const uint64_t bd = pvd0 + (uint64_t)((j & 1) * kVBufStep);
#pragma unroll
                    for (int kk = 0; kk < kRows / 16; ++kk)
                        umma_f16_ts(tmem, tmem + kPCol + kk * 8, bd + (uint64_t)(kk * 128), kIdescPV,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                    umma_commit(&ctl->v_empty[j & 1]);
                    umma_commit(&ctl->p_empty);
                }
                return true;  // (the next vote or elect.sync reconverges the warp)
            };
            // S += Q atom A . (the part's slot at descriptor bd), K = 64 dims as four MMAs of K = 16 (called
            // by the elected lane)
            auto qk_atom = [&](auto a_c, uint64_t bd, bool first) {
                constexpr int A = decltype(a_c)::value;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint32_t acc = (first && kk == 0) ? 0u : 1u;
                    if constexpr (A < kSmemQAtoms)
                        umma_f16_ss(tmem + kSCol, qd0 + (uint64_t)(A * (kQAtomBytes / 16) + 2 * kk), bd + 2 * kk, kIdescQK, acc);
                    else
                        umma_f16_ts(tmem + kSCol, tmem + kQCol + (A - kSmemQAtoms) * 32 + kk * 8, bd + 2 * kk, kIdescQK, acc);
                }
            };
            auto main_loop = [&](auto dvh_c) {
                constexpr int DVH = decltype(dvh_c)::value;
                // K part (slots 0-4): the other value half's four latent atoms, then the rotary atom; V part
                // (slots 0-3): this half's four latent atoms
                using K0 = std::integral_constant<int, DVH == 0 ? 4 : 0>;
                using K1 = std::integral_constant<int, DVH == 0 ? 5 : 1>;
                using K2 = std::integral_constant<int, DVH == 0 ? 6 : 2>;
                using K3 = std::integral_constant<int, DVH == 0 ? 7 : 3>;
                using K4 = std::integral_constant<int, kAtoms - 1>;
                using V0 = std::integral_constant<int, 4 * DVH>;
                using V1 = std::integral_constant<int, 4 * DVH + 1>;
                using V2 = std::integral_constant<int, 4 * DVH + 2>;
                using V3 = std::integral_constant<int, 4 * DVH + 3>;
                for (int i = 0; ok && i < ntiles; ++i) {
                    const uint32_t ph = ((uint32_t)i >> 1) & 1u;
                    // K part of S(i): needs its rows and the softmax to have read S(i-1)
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->k_full[i & 1], ph, p.err, p.wait_ns)) ||
                        !__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->s_empty, ((uint32_t)i & 1u) ^ 1u, p.err, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    // the rows were written by cp.async (generic proxy); the MMAs read them through the async proxy
                    fence_proxy_async_smem();
                    tc_fence_after();
                    if (elect_one_sync()) {
                        const uint64_t kd = kd0 + (uint64_t)((i & 1) * kKBufStep);
                        qk_atom(K0{}, kd, true);
                        qk_atom(K1{}, kd + kAtomStep, false);
                        qk_atom(K2{}, kd + 2 * kAtomStep, false);
                        qk_atom(K3{}, kd + 3 * kAtomStep, false);
                        qk_atom(K4{}, kd + 4 * kAtomStep, false);
                        umma_commit(&ctl->k_empty[i & 1]);
                    }
                    if (i > 0 && !pv(i - 1)) {
                        ok = false;
                        break;
                    }
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->v_full[i & 1], ph, p.err, p.wait_ns))) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_smem();
                    tc_fence_after();
                    if (elect_one_sync()) {
                        const uint64_t vd = vd0 + (uint64_t)((i & 1) * kVBufStep);
                        qk_atom(V0{}, vd, false);
                        qk_atom(V1{}, vd + kAtomStep, false);
                        qk_atom(V2{}, vd + 2 * kAtomStep, false);
                        qk_atom(V3{}, vd + 3 * kAtomStep, false);
                        umma_commit(&ctl->s_full);
                    }
                }
            };
            if (dvh == 0)
                main_loop(std::integral_constant<int, 0>{});
            else
                main_loop(std::integral_constant<int, 1>{});
            if (ok && ntiles > 0) pv(ntiles - 1);
            // drain (default limit): every MMA has completed before tensor memory is read back or released
            if (elect_one_sync()) {
                umma_commit(&ctl->mma_done);
                mbar_wait(&ctl->mma_done, 0, p.err);
            }
            __syncwarp();
        }
    } else if (warp >= 2) {
        // ---------------- softmax: one thread per head row ----------------
        const uint32_t quad = (uint32_t)(warp & 3);
        const uint32_t trow = tmem + ((quad * 32u) << 16);
        // i = -1 is a dry pass over the loop body (no waits, tensor-memory accesses, state updates or
        // arrivals) run while the first tile's rows are still in flight: it fetches the body's code, which the
        // first real pass would otherwise wait for (in the single-launch kernel it follows the indexer phase's
        // code, and its first pass took several microseconds).
#pragma unroll 1
        for (int i = -1; i < ntiles; ++i) {
            const bool dry = i < 0;
            const int it = dry ? 0 : i;  // rows_s holds kMaxEntries entries: row 0..63 is always in bounds
            const uint32_t vm0 = __ballot_sync(0xFFFFFFFFu, rows_s[it * kRows + lane] >= 0);
            const uint32_t vm1 = __ballot_sync(0xFFFFFFFFu, rows_s[it * kRows + 32 + lane] >= 0);
            if (!dry && !__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->s_full, (uint32_t)i & 1u, p.err, p.wait_ns))) break;
            tc_fence_after();
            float sv[kRows];
            if (dry) {
#pragma unroll
                for (int j = 0; j < kRows; ++j) sv[j] = 0.f;
            } else {
                // all four column groups in flight before one wait
                float a0[16], a1[16], a2[16], a3[16];
                tmem_ld16(trow + kSCol, a0);
                tmem_ld16(trow + kSCol + 16, a1);
                tmem_ld16(trow + kSCol + 32, a2);
                tmem_ld16(trow + kSCol + 48, a3);
                tmem_ld_wait();
                tmem_regs_ready(a0);
                tmem_regs_ready(a1);
                tmem_regs_ready(a2);
                tmem_regs_ready(a3);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    sv[j] = a0[j];
                    sv[16 + j] = a1[j];
                    sv[32 + j] = a2[j];
                    sv[48 + j] = a3[j];
                }
            }
            if (!dry) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->s_empty);
            }
            // a row that is not selected (padding, another shard's entry) scores -inf; a tile without one
            // skips the selects
            if ((vm0 & vm1) != 0xFFFFFFFFu) {
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const uint32_t m = j < 32 ? vm0 : vm1;
                    if (!((m >> (j & 31)) & 1u)) sv[j] = -INFINITY;
                }
            }
            // row max as a tree (short dependency chains), on the unscaled scores: the scale is positive,
            // so the scaled maximum is the maximum's scaled value, and the scale joins each exponent's
            // argument in one fused multiply-add below
            float mx[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) mx[k] = fmaxf(fmaxf(sv[k], sv[k + 16]), fmaxf(sv[k + 32], sv[k + 48]));
#pragma unroll
            for (int w = 8; w > 0; w >>= 1)
#pragma unroll
                for (int k = 0; k < w; ++k) mx[k] = fmaxf(mx[k], mx[k + w]);
            const float mt = mx[0] * p.scale_log2;
            const bool raise = mt > m_used + kRescaleLog2;
            const float m_new = raise ? mt : m_used;
            const float alpha = (raise && m_used != -INFINITY) ? exp2f(m_used - m_new) : 1.f;
            // P before the wait for P(i-1) V(i-1): only the P store and an O rescale need it done.  With no
            // row seen yet every score is -inf, and exp2(-inf - 0) = 0.
            const float mu = m_new == -INFINITY ? 0.f : m_new;
            uint32_t packed[kRows / 2];
            float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < kRows; j += 2) {
                const uint32_t pk = f2_to_bf2(ex2_approx(fmaf(sv[j], p.scale_log2, -mu)),
                                              ex2_approx(fmaf(sv[j + 1], p.scale_log2, -mu)));
                packed[j / 2] = pk;
                // the row sum takes the bf16-rounded values that P V uses
                ps[(j / 2) & 7] += __uint_as_float(pk << 16) + __uint_as_float(pk & 0xFFFF0000u);
            }
            const float rs = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            // P(i-1) V(i-1) has completed: the P columns are free and O is stable
            if (dry) {
                asm volatile("" ::"f"(rs));  // the dry pass computes the row sum (so the whole body) for real
                continue;
            }
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(&ctl->p_empty, ((uint32_t)i & 1u) ^ 1u, p.err, p.wait_ns))) break;
            tc_fence_after();
            if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
#pragma unroll 1
                for (int c = 0; c < kOCols / 16; ++c) {
                    float o[16];
                    tmem_ld16(trow + c * 16, o);
                    tmem_ld_wait();
                    tmem_regs_ready(o);
#pragma unroll
                    for (int j = 0; j < 16; ++j) o[j] *= alpha;
                    tmem_st16(trow + c * 16, o);
                }
            }
            l_sum = l_sum * alpha + rs;
            m_used = m_new;
            tmem_st16_u32(trow + kPCol, packed);
            tmem_st16_u32(trow + kPCol + 16, packed + 16);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->p_full);
        }
        if (ntiles > 0) mbar_wait(&ctl->p_empty, ((uint32_t)(ntiles - 1)) & 1u, p.err, p.wait_ns);
        tc_fence_after();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0 && lane == 0 && !ctl->q_waited) mbar_wait(&ctl->q_full, 0, p.err);

    // ---------------- epilogue ----------------
    const bool softmax_thread = warp >= 2 && warp < 6;
    const int h = softmax_thread ? (warp & 3) * 32 + lane : 0;
    const uint32_t trow = tmem + (((uint32_t)(warp & 3) * 32u) << 16);
    if (P == 1) {
        if (softmax_thread) {
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
#pragma unroll 1
            for (int c = 0; c < kOCols / 16; ++c) {
                float o[16];
                tmem_ld16(trow + c * 16, o);
                tmem_ld_wait();
                tmem_regs_ready(o);
                if (h < p.heads) {
                    uint32_t pk[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) pk[j] = f2_to_bf2(o[2 * j] * inv, o[2 * j + 1] * inv);
                    uint4* dst =
                        reinterpret_cast<uint4*>(p.out + ((int64_t)t * p.heads + h) * kVDim + dvh * kOCols + c * 16);
                    dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
            }
            if (dvh == 0 && h < p.heads && p.lse)
                p.lse[(int64_t)t * p.heads + h] = l_sum > 0.f ? (m_used + log2f(l_sum)) * 0.69314718055994531f : -INFINITY;
        }
    } else {
        // Merge the P position splits of this value half through L2.  Split o owns the head rows
        // [o*slice, (o+1)*slice).  Every CTA stages the rows other splits own in its shared memory (16-byte
        // chunks swizzled by row), sends each owner its rows with one bulk copy into this CTA's region of
        // the workspace, and writes the (max, sum) of its rows there.  After one cluster barrier each owner
        // pulls its rows from every other split with one bulk copy per split and combines them with its own
        // O, read straight from TMEM.  (An exchange through distributed shared memory was measured at ~10
        // bytes/cycle per SM here, several times slower; per-row stores or copies issue too slowly.)
        const int slice = (128 + P - 1) / P;
        const int rows_here = max(0, min(slice, p.heads - ps * slice));
        float* my_region = p.merge + (size_t)blockIdx.x * kSfaMergeFloatsPerCta;  // [o*slice + r][256], then ml
        float2* my_ml = reinterpret_cast<float2*>(my_region + kSfaMergeRows * 256);
        const int cta0 = (int)blockIdx.x - 2 * ps;  // CTA of split 0 for this token and value half
        uint8_t* stage = q_s;  // row (o*slice + r) at (o*slice + r) KiB, chunk q at (q ^ (r & 7)) * 16
        if (softmax_thread) {
            my_ml[h] = make_float2(m_used, l_sum);
            const int o = h / slice, r = h - o * slice;
            const bool send = o != ps && h < p.heads;
            if (__any_sync(0xFFFFFFFFu, send)) {
                const uint32_t row = smem_u32(stage) + (uint32_t)h * 1024u;
#pragma unroll 1
                for (int c = 0; c < kOCols / 16; c += 4) {
                    float v4[4][16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) tmem_ld16(trow + (c + u) * 16, v4[u]);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 4; ++u) tmem_regs_ready(v4[u]);
                    if (send) {
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float* v = &v4[q >> 2][4 * (q & 3)];
                            const int qc = c * 4 + q;
                            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(row + ((qc ^ (r & 7)) << 4)),
                                         "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3])
                                         : "memory");
                        }
                    }
                }
            }
        }
        fence_proxy_async_smem();  // the staged rows are read by the bulk copies (async proxy)
        __syncthreads();
        if (tid == 0) {
            for (int o = 0; o < P; ++o) {
                const int n = max(0, min(slice, p.heads - o * slice));
                if (o == ps || n == 0) continue;
                bulk_copy_s2g(my_region + (size_t)o * slice * 256, stage + (size_t)o * slice * 1024, (uint32_t)n * 1024u);
            }
            bulk_commit_and_wait();  // written to global memory (and the staging may be reused)
            asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        cluster_sync();  // every split's rows and (max, sum) are visible
        // this CTA's rows from every other split, row j*slice + r, same swizzle
        uint8_t* obuf = q_s;
        if (tid == 0) {
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t bytes = (uint32_t)((P - 1) * rows_here * 1024);
            if (bytes > 0) {
                mbar_arrive_expect_tx(&ctl->merge_full, bytes);
                for (int j = 0; j < P; ++j) {
                    if (j == ps) continue;
                    bulk_copy_g2s(obuf + (size_t)j * slice * 1024,
                                  p.merge + (size_t)(cta0 + 2 * j) * kSfaMergeFloatsPerCta + (size_t)ps * slice * 256,
                                  (uint32_t)rows_here * 1024u, &ctl->merge_full);
                }
            } else {
                mbar_arrive(&ctl->merge_full);
            }
        }
        // Combine: the three warps of each TMEM lane quadrant (one softmax warp, two gather warps) share the
        // 16 column chunks of that quadrant's rows.
        if (warp >= 2) {
            const int quad = warp & 3, part = (warp - 2) >> 2;  // part 0..2 within the quadrant
            const int hh = quad * 32 + lane, r = hh - ps * slice;
            const bool own_row = r >= 0 && r < rows_here;
            if (P == 2 && __any_sync(0xFFFFFFFFu, own_row)) {
                // the common case, two splits: the same arithmetic as below with one other split, in compact
                // code (this runs once per launch)
                const uint32_t tr = tmem + (((uint32_t)quad * 32u) << 16);
                const int jo = 1 - ps;
                float2 mo = make_float2(-INFINITY, 0.f), mt = make_float2(-INFINITY, 0.f);
                if (own_row) {
                    const float* base = p.merge + kSfaMergeRows * 256;
                    mo = __ldcg(reinterpret_cast<const float2*>(base + (size_t)(cta0 + 2 * ps) * kSfaMergeFloatsPerCta) + hh);
                    mt = __ldcg(reinterpret_cast<const float2*>(base + (size_t)(cta0 + 2 * jo) * kSfaMergeFloatsPerCta) + hh);
                }
                float M = -INFINITY;
                if (mo.y > 0.f) M = fmaxf(M, mo.x);
                if (mt.y > 0.f) M = fmaxf(M, mt.x);
                float w_own = mo.y > 0.f ? exp2f(mo.x - M) : 0.f, w_oth = mt.y > 0.f ? exp2f(mt.x - M) : 0.f;
                const float Lsum = mo.y * w_own + mt.y * w_oth;
                const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
                w_own *= inv;
                w_oth *= inv;
                if (part == 0 && own_row && dvh == 0 && p.lse)
                    p.lse[(int64_t)t * p.heads + hh] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
                const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(&ctl->merge_full, 0, p.err, p.wait_ns));
                const int c_lo = part == 0 ? 0 : (part == 1 ? 6 : 11), c_hi = part == 0 ? 6 : (part == 1 ? 11 : 16);
                const uint32_t rowp = smem_u32(obuf) + (uint32_t)(jo * slice + r) * 1024u;
#pragma unroll 1
                for (int c = c_lo; c < c_hi; ++c) {
                    float o[16];
                    tmem_ld16(tr + c * 16, o);
                    tmem_ld_wait();
                    tmem_regs_ready(o);
                    if (own_row && got) {
                        // a split with no selected row has weight 0 and an O that is never read: select, not scale
                        float acc[16];
#pragma unroll
                        for (int k = 0; k < 16; ++k) acc[k] = w_own != 0.f ? o[k] * w_own : 0.f;
                        if (w_oth != 0.f) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                float4 v;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                             : "r"(rowp + (((c * 4 + k) ^ (r & 7)) << 4)));
                                acc[4 * k] += v.x * w_oth;
                                acc[4 * k + 1] += v.y * w_oth;
                                acc[4 * k + 2] += v.z * w_oth;
                                acc[4 * k + 3] += v.w * w_oth;
                            }
                        }
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) pk[k] = f2_to_bf2(acc[2 * k], acc[2 * k + 1]);
                        uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)t * p.heads + hh) * kVDim + dvh * kOCols + c * 16);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            } else if (__any_sync(0xFFFFFFFFu, own_row)) {
                const uint32_t tr = tmem + (((uint32_t)quad * 32u) << 16);
                // weights of the splits for this row: exp2(m_j - M) / sum_j l_j exp2(m_j - M)
                float2 ml[kMaxSplits];
                float M = -INFINITY;
#pragma unroll
                for (int j = 0; j < kMaxSplits; ++j) {
                    ml[j] = make_float2(-INFINITY, 0.f);
                    if (j < P && own_row)
                        ml[j] = __ldcg(reinterpret_cast<const float2*>(p.merge + (size_t)(cta0 + 2 * j) *
                                                                       kSfaMergeFloatsPerCta + kSfaMergeRows * 256) + hh);
                    if (ml[j].y > 0.f) M = fmaxf(M, ml[j].x);
                }
                float wj[kMaxSplits], Lsum = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxSplits; ++j) {
                    wj[j] = ml[j].y > 0.f ? exp2f(ml[j].x - M) : 0.f;
                    Lsum += ml[j].y * wj[j];
                }
                const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
                float w_own = 0.f;
#pragma unroll
                for (int j = 0; j < kMaxSplits; ++j) {
                    wj[j] *= inv;
                    if (j == ps) w_own = wj[j];
                }
                if (part == 0 && own_row && dvh == 0 && p.lse)
                    p.lse[(int64_t)t * p.heads + hh] = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
                const bool got = __all_sync(0xFFFFFFFFu, mbar_wait(&ctl->merge_full, 0, p.err, p.wait_ns));
                const int c_lo = part == 0 ? 0 : (part == 1 ? 6 : 11), c_hi = part == 0 ? 6 : (part == 1 ? 11 : 16);
#pragma unroll 1
                for (int c = c_lo; c < c_hi; ++c) {
                    float o[16];
                    tmem_ld16(tr + c * 16, o);
                    tmem_ld_wait();
                    tmem_regs_ready(o);
                    if (own_row && got) {
                        float acc[16];
                        // a split with no selected row has weight 0 and an O that is never read: select, not scale
#pragma unroll
                        for (int k = 0; k < 16; ++k) acc[k] = w_own != 0.f ? o[k] * w_own : 0.f;
#pragma unroll
                        for (int j = 0; j < kMaxSplits; ++j) {
                            if (j >= P || j == ps || wj[j] == 0.f) continue;
                            const uint32_t rowp = smem_u32(obuf) + (uint32_t)(j * slice + r) * 1024u;
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                float4 v;
                                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                                             : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                                             : "r"(rowp + (((c * 4 + k) ^ (r & 7)) << 4)));
                                acc[4 * k] += v.x * wj[j];
                                acc[4 * k + 1] += v.y * wj[j];
                                acc[4 * k + 2] += v.z * wj[j];
                                acc[4 * k + 3] += v.w * wj[j];
                            }
                        }
                        uint32_t pk[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) pk[k] = f2_to_bf2(acc[2 * k], acc[2 * k + 1]);
                        uint4* dst = reinterpret_cast<uint4*>(p.out + ((int64_t)t * p.heads + hh) * kVDim + dvh * kOCols + c * 16);
                        dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                        dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                    }
                }
            }
        }
        // drain (default limit): every bulk copy into this CTA has landed before it exits (the combining
        // warps saw the barrier unless their wait gave up; a CTA without owned rows waits here)
        if (tid == 0) mbar_wait(&ctl->merge_full, 0, p.err);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace
}  // namespace dsa
