// Appending one step's new rows to the paged caches: every query token's new indexer key and latent-KV
// row go to the cache rows of its own position ("Day0 Inference Support and Performance Optimization
// for New LLM Architectures", section 3.3: the indexer's K input is prepared ahead of the indexer).
// FP8 caches are quantised dynamically per group ("Optimizing Inference for Hybrid Attention LLMs:
// Practices for Fast Adaptation", section 1, layered quantization; "Day0 Inference Support ...",
// section 4, hierarchical quantization): scale = absmax / 448 (1 for an all-zero group) and
// code = E4M3(x / scale), nearest with ties to even, saturated at 448, in fp32 with correctly rounded
// divisions.  Groups: the whole indexer key row (one scale per row), and each 128-element tile of the
// latent part of a latent-KV row (the 64 rotary dims stay bf16).
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {
namespace {

constexpr int kAppendThreads = 128;  // one token per CTA; thread i owns key element i and latent dims 4i..4i+3

// Two E4M3 codes (a in the low byte), nearest-even, saturating at +-448.
__device__ __forceinline__ uint16_t f2_to_e4m3x2(float a, float b) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits) { return __uint_as_float(bits << 16); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    return v;
}

// absmax / 448 in fp32 (1 for an all-zero group)
__device__ __forceinline__ float group_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f; }

__global__ void __launch_bounds__(kAppendThreads) append_kernel(const AppendParams p) {
    __shared__ int s_b, s_cu0, s_cu1;
    __shared__ float s_amax[kAppendThreads / 32];
    const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the sequence that holds token t: a parallel search over the query offsets
    if (tid == 0) s_b = -1;
    __syncthreads();
    for (int j = tid; j < p.batch; j += kAppendThreads) {
        const int c0 = __ldg(p.cu_q_lens + j), c1 = __ldg(p.cu_q_lens + j + 1);
        if (c0 <= t && t < c1) {
            s_b = j;
            s_cu0 = c0;
            s_cu1 = c1;
        }
    }
    __syncthreads();
    const int b = s_b;
    if (b < 0) {
        if (tid == 0) raise_error(p.err, DSA_DEVERR_SEQ);
        return;
    }
    const int n_b = s_cu1 - s_cu0;
    const int L = __ldg(p.seq_lens + b);
    if (n_b > L || L < 0 || (int64_t)L > (int64_t)p.max_pages * 64) {
        if (tid == 0) raise_error(p.err, DSA_DEVERR_SEQ);
        return;
    }
    const int pos = L - n_b + (t - s_cu0);
    const int32_t pg = __ldg(p.page_table + (int64_t)b * p.max_pages + pos / 64);
    if (pg < 0 || pg >= p.num_pages) {
        if (tid == 0) raise_error(p.err, DSA_DEVERR_PAGE);
        return;
    }
    const int64_t row = (int64_t)pg * 64 + (pos & 63);

    // ---- indexer key row ----
    if (p.k_new != nullptr) {
        const int Di = p.idx_dim;
        const uint16_t* src = p.k_new + (int64_t)t * Di;
        if (!p.idx_fp8) {
            // bf16 copy, 4 bytes per thread (Di is even)
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.k_cache + row * Di * 2);
            for (int i = tid; i < Di / 2; i += kAppendThreads) dst[i] = __ldg(reinterpret_cast<const uint32_t*>(src) + i);
        } else {
            const float x = tid < Di ? bf16_bits_to_f32(__ldg(src + tid)) : 0.f;
            const float wmax = warp_max(fabsf(x));
            if (lane == 0) s_amax[warp] = wmax;
            __syncthreads();
            float amax = 0.f;
#pragma unroll
            for (int w = 0; w < kAppendThreads / 32; ++w) amax = fmaxf(amax, s_amax[w]);
            const float scale = group_scale(amax);
            const float y = __fdiv_rn(x, scale);
            const float y_next = __shfl_down_sync(0xFFFFFFFFu, y, 1);
            if ((tid & 1) == 0 && tid < Di)
                *reinterpret_cast<uint16_t*>(p.k_cache + row * Di + tid) = f2_to_e4m3x2(y, y_next);
            if (tid == 0) p.k_scale[row] = scale;
        }
    }

    // ---- latent-KV row ----
    if (p.kv_new != nullptr) {
        const uint16_t* src = p.kv_new + (int64_t)t * 576;
        if (!p.kv_fp8) {
            // bf16 copy: 72 pieces of 16 bytes
            const uint4* s4 = reinterpret_cast<const uint4*>(src);
            uint4* d4 = reinterpret_cast<uint4*>(p.kv_cache + row * 1152);
            for (int i = tid; i < 72; i += kAppendThreads) d4[i] = __ldg(s4 + i);
        } else {
            uint8_t* dst = p.kv_cache + row * kKvFp8RowBytes;
            // latent dims 4*tid .. 4*tid+3: warp w holds tile w (128 dims)
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + tid);
            const float x0 = bf16_bits_to_f32(v.x & 0xFFFFu), x1 = bf16_bits_to_f32(v.x >> 16);
            const float x2 = bf16_bits_to_f32(v.y & 0xFFFFu), x3 = bf16_bits_to_f32(v.y >> 16);
            const float amax = warp_max(fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(x2), fabsf(x3))));
            const float scale = group_scale(amax);
            const uint32_t lo = f2_to_e4m3x2(__fdiv_rn(x0, scale), __fdiv_rn(x1, scale));
            const uint32_t hi = f2_to_e4m3x2(__fdiv_rn(x2, scale), __fdiv_rn(x3, scale));
            *reinterpret_cast<uint32_t*>(dst + 4 * tid) = lo | (hi << 16);
            if (lane == 0) *reinterpret_cast<float*>(dst + kKvFp8ScaleOff + 4 * warp) = scale;
            // rotary dims 512..575 unquantised: 8 pieces of 16 bytes
            if (tid < 8)
                *reinterpret_cast<uint4*>(dst + kKvFp8RopeOff + 16 * tid) =
                    __ldg(reinterpret_cast<const uint4*>(src + 512) + tid);
        }
    }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
    if (p.total_q <= 0) return cudaSuccess;
    append_kernel<<<dim3((unsigned)p.total_q), dim3(kAppendThreads), 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
