// Sparse flash attention over the Top-K selected rows of a paged MLA latent-KV cache, for sm_103a.
//
// For each query token t and head h: z_s = scale * q[t,h,:] . kv[s,:] over the selected positions s,
// out[t,h,:] = softmax(z) . kv[:, :Dv], lse = logsumexp(z) ("Optimizing Inference for Hybrid Attention
// Architectures: From Operator Fusion to Sequence Sharding", section "Breaking Down the Computational
// Path of Hybrid Attention", step 2; "Day0 Inference Support and Performance Optimization for New LLM
// Architectures", section 3.2: only the selected positions' KV rows are read).
//
// This translation unit holds the warp-per-head kernel: one warp per (token, head); every warp of a
// CTA walks the same selected rows, so each gathered row is read from L2 once per CTA and served to
// the other warps from L1.  Online softmax in fp32 (base-2 exponent), fp32 accumulation.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kHeadsPerCta = 8;
constexpr int kDim = 576;  // latent + rope
constexpr int kVDim = 512;
constexpr int kPairs = kDim / 64;   // bf16 pairs per lane: lane owns dims 2*lane + 64*j (+1)
constexpr int kVPairs = kVDim / 64;

__device__ __forceinline__ float2 bf2_to_f2(uint32_t u) {
    return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t f2_to_bf2(float a, float b) {
    // round to nearest even (finite inputs)
    uint32_t ua = __float_as_uint(a), ub = __float_as_uint(b);
    ua += 0x7FFFu + ((ua >> 16) & 1u);
    ub += 0x7FFFu + ((ub >> 16) & 1u);
    return (ua >> 16) | (ub & 0xFFFF0000u);
}

__global__ void __launch_bounds__(kHeadsPerCta * 32) sfa_warp_kernel(const SfaParams p) {
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * kHeadsPerCta + warp;
    if (t >= p.total_q || h >= p.heads) return;
    // sequence of this token
    int b = 0;
    {
        int lo = 0, hi = p.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (p.cu_q_lens[mid] <= t) lo = mid; else hi = mid - 1;
        }
        b = lo;
    }
    const int n_b = p.cu_q_lens[b + 1] - p.cu_q_lens[b];
    const int L = p.seq_lens[b];
    if (t < p.cu_q_lens[b] || t >= p.cu_q_lens[b + 1] || n_b > L || L > p.max_pages * 64) {
        if (lane == 0) raise_error(p.err, DSA_DEVERR_SEQ);
        return;
    }
    const int64_t pos = (int64_t)L - n_b + (t - p.cu_q_lens[b]);
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + ((int64_t)t * p.heads + h) * kDim);
    float2 q[kPairs];
#pragma unroll
    for (int j = 0; j < kPairs; ++j) q[j] = bf2_to_f2(__ldg(qrow + lane + 32 * j));
    float m = -INFINITY, l = 0.f;
    float2 o[kVPairs];
#pragma unroll
    for (int j = 0; j < kVPairs; ++j) o[j] = make_float2(0.f, 0.f);
    const int32_t* sel = p.topk + (int64_t)t * p.top_k;
    const int32_t* pt_row = p.page_table + (int64_t)b * p.max_pages;
    for (int k = 0; k < p.top_k; ++k) {
        const int32_t s = __ldg(sel + k);
        if (s < 0) continue;
        if ((int64_t)s > pos) {
            if (lane == 0 && h == 0) raise_error(p.err, DSA_DEVERR_INDEX);
            continue;
        }
        const int32_t pg = __ldg(pt_row + (s >> 6));
        if (pg < 0 || pg >= p.num_pages) {
            if (lane == 0 && h == 0) raise_error(p.err, DSA_DEVERR_PAGE);
            continue;
        }
        const uint32_t* row = reinterpret_cast<const uint32_t*>(p.kv_cache + ((int64_t)pg * 64 + (s & 63)) * kDim);
        float2 kv[kPairs];
#pragma unroll
        for (int j = 0; j < kPairs; ++j) kv[j] = bf2_to_f2(__ldg(row + lane + 32 * j));
        float dot = 0.f;
#pragma unroll
        for (int j = 0; j < kPairs; ++j) dot = fmaf(q[j].x, kv[j].x, fmaf(q[j].y, kv[j].y, dot));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xFFFFFFFFu, dot, off);
        const float z = dot * p.scale_log2;  // base-2 logit
        const float m_new = fmaxf(m, z);
        const float corr = exp2f(m - m_new);
        const float e = exp2f(z - m_new);
        l = l * corr + e;
#pragma unroll
        for (int j = 0; j < kVPairs; ++j) {
            o[j].x = fmaf(o[j].x, corr, e * kv[j].x);
            o[j].y = fmaf(o[j].y, corr, e * kv[j].y);
        }
        m = m_new;
    }
    uint32_t* orow = reinterpret_cast<uint32_t*>(p.out + ((int64_t)t * p.heads + h) * kVDim);
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int j = 0; j < kVPairs; ++j) orow[lane + 32 * j] = f2_to_bf2(o[j].x * inv, o[j].y * inv);
    if (p.lse && lane == 0) p.lse[(int64_t)t * p.heads + h] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

cudaError_t launch_sfa(const SfaLaunch& L, cudaStream_t stream) {
    const SfaParams& p = L.params;
    dim3 grid((unsigned)p.total_q, (unsigned)((p.heads + kHeadsPerCta - 1) / kHeadsPerCta));
    sfa_warp_kernel<<<grid, kHeadsPerCta * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
