// Context-parallel decode building blocks ("Day0 Inference Support and Performance Optimization for New
// LLM Architectures", section 5 "Context Parallelism (CP)", 5.1): when one long sequence is sharded by
// position across devices, each shard scores its own positions and keeps a local Top-K of (score,
// position) pairs; the shards' lists are exchanged and merged into the global Top-K with the same
// ordering key (score descending, then position ascending); each shard then runs the sparse attention
// over the selected rows it holds, and the partial (out, lse) pairs are combined with log-sum-exp
// weights.  This file holds the two device steps that are not the indexer or the attention themselves:
//   merge_kernel    the S shards' candidate lists of one query token -> its global Top-K;
//   combine_kernel  the S shards' partial attention outputs of one (token, head) -> the final output.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kMergeThreads = 512;

// 64-bit ordering key of a candidate: the score's order-preserving key above the complement of the
// position, so that a larger key means a higher score or, at equal scores, a lower position.  0 marks an
// empty slot (a real score never maps to key 0).
__device__ __forceinline__ uint64_t cand_key(int32_t idx, float score) {
    if (idx < 0) return 0ull;
    return ((uint64_t)score_key(score) << 32) | (uint64_t)(~(uint32_t)idx);
}

// One CTA per query token.  Candidates of shard s are idx[s][t][0..K) (ascending positions, -1 padded);
// shards are taken in order, so the output is ascending when shard s holds positions below shard s+1's.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeParams p) {
    extern __shared__ __align__(16) uint64_t mkeys[];  // S * K candidate keys
    __shared__ uint32_t hist[256];
    __shared__ uint32_t warp_cnt[kMergeThreads / 32];
    __shared__ uint32_t res[2];
    const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.top_k, n = p.shards * K;
    for (int i = tid; i < n; i += kMergeThreads) {
        const int s = i / K, k = i - s * K;
        const int64_t off = ((int64_t)s * p.total_q + t) * K + k;
        mkeys[i] = cand_key(__ldg(p.idx + off), __ldg(p.score + off));
    }
    // count the valid candidates (each thread its own strided share, then the block)
    uint32_t nv = 0;
    {
        uint32_t c = 0;
        for (int i = tid; i < n; i += kMergeThreads) c += mkeys[i] != 0ull ? 1u : 0u;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, off);
        if (lane == 0) warp_cnt[warp] = c;
        __syncthreads();
        for (int w = 0; w < kMergeThreads / 32; ++w) nv += warp_cnt[w];
        __syncthreads();
    }
    // the K-th largest key, a byte at a time (every key is distinct when the shards' positions are)
    uint64_t thr = 1ull;  // with no more valid candidates than K every valid one is kept
    if (nv > (uint32_t)K) {
        uint64_t prefix = 0, mask = 0;
        uint32_t remaining = (uint32_t)K;
        for (int shift = 56; shift >= 0; shift -= 8) {
            if (tid < 256) hist[tid] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kMergeThreads) {
                const uint64_t key = mkeys[i];
                if (key != 0ull && (key & mask) == prefix) atomicAdd(&hist[(uint32_t)(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds bins 8l..8l+7; count from the top bin down
                uint32_t v[8], lsum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    v[j] = hist[8 * lane + j];
                    lsum += v[j];
                }
                uint32_t incl = lsum;  // keys in bins >= 8*lane
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t o = __shfl_down_sync(0xFFFFFFFFu, incl, off);
                    if (lane + off < 32) incl += o;
                }
                uint32_t above = incl - lsum;
                for (int j = 7; j >= 0; --j) {
                    if (above < remaining && remaining <= above + v[j]) {
                        res[0] = (uint32_t)(8 * lane + j);
                        res[1] = remaining - above;
                    }
                    above += v[j];
                }
            }
            __syncthreads();
            prefix |= (uint64_t)res[0] << shift;
            mask |= 0xFFull << shift;
            remaining = res[1];
            __syncthreads();
        }
        thr = prefix;
    }
    // ordered compaction of the keys >= thr, in candidate order
    int32_t* out_idx = p.out_idx + (int64_t)t * K;
    float* out_score = p.out_score ? p.out_score + (int64_t)t * K : nullptr;
    uint32_t base = 0;
    for (int i0 = 0; i0 < n; i0 += kMergeThreads) {
        const int i = i0 + tid;
        const uint64_t key = i < n ? mkeys[i] : 0ull;
        const bool sel = key != 0ull && key >= thr;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, sel);
        if (lane == 0) warp_cnt[warp] = __popc(bal);
        __syncthreads();
        uint32_t before = base;
        for (int w = 0; w < warp; ++w) before += warp_cnt[w];
        uint32_t total = 0;
        for (int w = 0; w < kMergeThreads / 32; ++w) total += warp_cnt[w];
        if (sel) {
            const uint32_t o = before + __popc(bal & ((1u << lane) - 1u));
            if (o < (uint32_t)K) {
                out_idx[o] = (int32_t)~(uint32_t)key;
                if (out_score) out_score[o] = key_score((uint32_t)(key >> 32));
            }
        }
        base += total;
        __syncthreads();
    }
    for (int o = (int)min(base, (uint32_t)K) + tid; o < K; o += kMergeThreads) {
        out_idx[o] = -1;
        if (out_score) out_score[o] = -INFINITY;
    }
}

constexpr int kCombineWarps = 8;

// One warp per (token, head): out = sum_s exp(lse_s - LSE) out_s, LSE = log sum_s exp(lse_s).
__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(const CombineParams p) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * kCombineWarps + warp;  // t * heads + h
    if (row >= (int64_t)p.total_q * p.heads) return;
    const int64_t plane = (int64_t)p.total_q * p.heads;
    float m = -INFINITY;
    for (int s = 0; s < p.shards; ++s) m = fmaxf(m, __ldg(p.lse_in + s * plane + row));
    uint16_t* out = p.out + row * p.v_dim;
    if (m == -INFINITY) {  // no shard selected any row
        for (int d = lane; d < p.v_dim; d += 32) out[d] = 0;
        if (lane == 0 && p.lse) p.lse[row] = -INFINITY;
        return;
    }
    float lsum = 0.f;
    for (int s = 0; s < p.shards; ++s) {
        const float l = __ldg(p.lse_in + s * plane + row);
        lsum += l == -INFINITY ? 0.f : expf(l - m);
    }
    const float inv = 1.f / lsum;
    for (int d = 2 * lane; d < p.v_dim; d += 64) {
        float a0 = 0.f, a1 = 0.f;
        for (int s = 0; s < p.shards; ++s) {
            const float l = __ldg(p.lse_in + s * plane + row);
            if (l == -INFINITY) continue;
            const float wgt = expf(l - m) * inv;
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(p.out_in + (s * plane + row) * p.v_dim + d));
            a0 += wgt * __uint_as_float(v << 16);
            a1 += wgt * __uint_as_float(v & 0xFFFF0000u);
        }
        *reinterpret_cast<uint32_t*>(out + d) = f2_to_bf2(a0, a1);
    }
    if (lane == 0 && p.lse) p.lse[row] = m + logf(lsum);
}

}  // namespace

size_t merge_smem_bytes(int shards, int top_k) { return (size_t)shards * (size_t)top_k * sizeof(uint64_t); }

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    const size_t smem = merge_smem_bytes(p.shards, p.top_k);
    cudaError_t e = cudaFuncSetAttribute(merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    merge_kernel<<<p.total_q, kMergeThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.total_q * p.heads;
    const unsigned blocks = (unsigned)((rows + kCombineWarps - 1) / kCombineWarps);
    combine_kernel<<<blocks, 32 * kCombineWarps, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
