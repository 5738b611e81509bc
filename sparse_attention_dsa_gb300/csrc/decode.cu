// Single-launch fused decode: for every query token, the lightning indexer + Top-K and then the sparse
// flash attention over the selected rows run back to back in one thread-block cluster, in one kernel
// launch ("Optimizing Inference for Hybrid Attention Architectures: From Operator Fusion to Sequence
// Sharding", section "Breaking Down the Computational Path of Hybrid Attention": steps 1 and 2 of one
// decode step; "Day0 Inference Support and Performance Optimization for New LLM Architectures", section
// 3.1: launch overhead dominates decode).  The two phases are the device code of the standalone kernels
// (indexer_impl.cuh, sfa_impl.cuh).  A cluster of 2P CTAs serves one token: in the first phase its CTAs
// score 1/(2P) of the context each and select the token's Top-K together; after a cluster barrier the
// same CTAs run the attention as P position splits x 2 value halves.  Shared memory and tensor memory
// are reused from one phase to the next; the Top-K goes through L2.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "indexer_impl.cuh"
#include "sfa_impl.cuh"

namespace dsa {
namespace {

template <int HI, int DI, bool FP8, bool MX, bool KVFP8>
__global__ void __launch_bounds__(kThreadsSfa, 1)
    decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap_idx,
                  const IndexerParams ip, const __grid_constant__ CUtensorMap qmap_q, const SfaParams sp) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // (the attention phase allocates tensor memory again, so the indexer phase keeps the allocation permit)
    indexer_cta<HI, DI, 1, FP8, kThreadsSfa, false, MX>(kmap, qmap_idx, ip, smem_raw);
    // shared memory this thread wrote is next written by the attention phase's copies (async proxy)
    fence_proxy_async_smem();
    // the cluster's Top-K is written and visible to every CTA of the cluster; nothing of the indexer
    // phase is still in use in shared or tensor memory
    cluster_sync();
    sfa_cta<KVFP8>(qmap_q, sp, smem_raw);
}

struct DecodePlan {
    int P, C, stages;
    int chunk;
    size_t smem;
};

// Chooses the split count P (a cluster of C = 2P CTAs per token) as the attention launcher would, then
// smaller until the indexer's slice of the scores fits next to at least two pipeline stages and every
// cluster of the grid can be resident at once.  False when no P works.
template <int HI, int DI, bool FP8, bool MX, bool KVFP8>
bool plan_decode_variant(const IndexerLaunch& IL, const SfaLaunch& SL, DecodePlan* out) {
    auto kern = decode_kernel<HI, DI, FP8, MX, KVFP8>;
    const int64_t T = SL.params.total_q;
    const int64_t max_ctx = (int64_t)IL.params.max_pages * 64;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    for (int P = sfa_splits(T, SL.params.top_k, SL.num_sms); P >= 1; --P) {
        if ((SL.params.top_k + P - 1) / P > kSfaMaxEntries) break;
        const int C = 2 * P;
        const int64_t per = (max_ctx + C - 1) / C;
        const int64_t chunk = (per + 127) / 128 * 128;
        if (chunk > INT32_MAX) continue;
        int stages = kMaxStages;
        while (stages > 2 && indexer_smem_bytes<HI, DI, 1, FP8, MX>(stages, (int)chunk, C) > (size_t)SL.smem_limit) --stages;
        const size_t idx_smem = indexer_smem_bytes<HI, DI, 1, FP8, MX>(stages, (int)chunk, C);
        const size_t smem = idx_smem > kSfaSmem ? idx_smem : kSfaSmem;
        if (smem > (size_t)SL.smem_limit) continue;
        if (P > 1 && (size_t)T * 2 * P > sfa_merge_ctas(T, SL.params.top_k)) continue;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(T * C));
        cfg.blockDim = dim3(kThreadsSfa);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int nclusters = 0;
        if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            continue;
        }
        if (nclusters < T) continue;  // a second wave of clusters would double the time: fewer splits
        *out = DecodePlan{P, C, stages, (int)chunk, smem};
        return true;
    }
    return false;
}

template <int HI, int DI, bool FP8, bool MX, bool KVFP8>
cudaError_t launch_decode_variant(const IndexerLaunch& IL, const SfaLaunch& SL, cudaStream_t stream) {
    DecodePlan d;
    if (!plan_decode_variant<HI, DI, FP8, MX, KVFP8>(IL, SL, &d)) return cudaErrorNotSupported;
    auto kern = decode_kernel<HI, DI, FP8, MX, KVFP8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)d.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)d.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(SL.params.total_q * d.C));
    cfg.blockDim = dim3(kThreadsSfa);
    cfg.dynamicSmemBytes = d.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    IndexerParams ip = IL.params;
    ip.chunk = d.chunk;
    ip.stages = d.stages;
    SfaParams sp = SL.params;
    sp.splits = d.P;
    sp.one_query_per_seq = 1;  // decode_shape_ok: every sequence has exactly one query token
    sp.early_setup = 0;
    return cudaLaunchKernelEx(&cfg, kern, IL.kmap, IL.qmap, ip, SL.qmap, sp);
}

bool decode_shape_ok(const IndexerLaunch& IL, const SfaLaunch& SL) {
    // one query token per sequence (so one indexer work item per token) and a query-block-1 variant
    return IL.params.qb == 1 && IL.params.blocks_per_seq == 1 && (int64_t)IL.items == (int64_t)SL.params.total_q &&
           IL.idx_heads == 64 && IL.idx_dim == 128;
}

}  // namespace

cudaError_t launch_decode(const IndexerLaunch& IL, const SfaLaunch& SL, cudaStream_t stream) {
    if (!decode_shape_ok(IL, SL)) return cudaErrorNotSupported;
    const bool kv8 = SL.params.kv_fp8 != 0;
    if (IL.mx) return kv8 ? launch_decode_variant<64, 128, true, true, true>(IL, SL, stream)
                          : launch_decode_variant<64, 128, true, true, false>(IL, SL, stream);
    if (IL.fp8) return kv8 ? launch_decode_variant<64, 128, true, false, true>(IL, SL, stream)
                           : launch_decode_variant<64, 128, true, false, false>(IL, SL, stream);
    return kv8 ? launch_decode_variant<64, 128, false, false, true>(IL, SL, stream)
               : launch_decode_variant<64, 128, false, false, false>(IL, SL, stream);
}

bool decode_single_launch(const IndexerLaunch& IL, const SfaLaunch& SL) {
    if (!decode_shape_ok(IL, SL)) return false;
    DecodePlan d;
    const bool kv8 = SL.params.kv_fp8 != 0;
    if (IL.mx) return kv8 ? plan_decode_variant<64, 128, true, true, true>(IL, SL, &d)
                          : plan_decode_variant<64, 128, true, true, false>(IL, SL, &d);
    if (IL.fp8) return kv8 ? plan_decode_variant<64, 128, true, false, true>(IL, SL, &d)
                           : plan_decode_variant<64, 128, true, false, false>(IL, SL, &d);
    return kv8 ? plan_decode_variant<64, 128, false, false, true>(IL, SL, &d)
               : plan_decode_variant<64, 128, false, false, false>(IL, SL, &d);
}

}  // namespace dsa
