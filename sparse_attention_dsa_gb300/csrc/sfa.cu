// The standalone sparse-attention kernel (one launch per dsa_sparse_attn call), its launch planning and
// launcher.  The device code lives in sfa_impl.cuh.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "sfa_impl.cuh"

namespace dsa {
namespace {

template <bool KVFP8>
__global__ void __launch_bounds__(kThreadsSfa, 1) sfa_kernel(const __grid_constant__ CUtensorMap qmap, const SfaParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    sfa_cta<KVFP8>(qmap, p, smem_raw);
}

}  // namespace

// Position splits P (a cluster of 2P CTAs per query token): the fewest that keep a split within
// kMaxEntries entries, grown while the grid still fits on `sms` SMs.
static int splits_for(int64_t total_q, int top_k, int sms) {
    int P = 1;
    while (P < kMaxSplits && (top_k + P - 1) / P > kMaxEntries) ++P;
    const int max_splits = (top_k + kRows - 1) / kRows;
    while (P < kMaxSplits && P + 1 <= max_splits && total_q * 2 * (P + 1) <= sms) ++P;
    return P;
}

int sfa_splits(int64_t total_q, int32_t top_k, int num_sms) {
    return splits_for(total_q, top_k, num_sms < 256 ? num_sms : 256);
}

size_t sfa_merge_ctas(int64_t total_q, int32_t top_k) {
    // the launcher never counts more than 256 SMs, so this grid bounds the one it picks
    const int P = splits_for(total_q, top_k, 256);
    return P > 1 ? (size_t)total_q * 2 * P : 0;
}

// Clusters of `size` CTAs of this kernel that can be resident at once (cached per device, variant, size).
template <bool KVFP8>
static int max_active_clusters(int size) {
    static int cache[64][2 * kMaxSplits + 1];  // 0 = not queried yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int& c = cache[dev][size];
    if (c == 0) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)size;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)size);
        cfg.blockDim = dim3(kThreadsSfa);
        cfg.dynamicSmemBytes = kSfaSmem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, sfa_kernel<KVFP8>, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        c = n > 0 ? n : -1;
    }
    return c;
}

template <bool KVFP8>
static cudaError_t launch_sfa_variant(const SfaLaunch& L, cudaStream_t stream) {
    auto kern = sfa_kernel<KVFP8>;
    SfaParams p = L.params;
    static_assert(kQBytes + 2 * kKBufBytes >= kSfaMergeRows * 1024, "split merge rows must fit in the Q and K-part buffers");
    static_assert(kSfaMergeRows >= 128 + kMaxSplits - 1, "P * ceil(128 / P) rows at most");
    if (kSfaSmem > (size_t)L.smem_limit) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSfaSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    // Position splits: grown while the CTAs still fit on the SMs, then shrunk until every cluster of the
    // grid can be resident at once (a second wave of clusters would double the time).
    int P = splits_for(p.total_q, p.top_k, L.num_sms < 256 ? L.num_sms : 256);
    if ((p.top_k + P - 1) / P > kMaxEntries) return cudaErrorInvalidValue;
    const int min_p = splits_for(p.total_q, p.top_k, 0);
    while (P > min_p && P > 1 && p.total_q > max_active_clusters<KVFP8>(2 * P)) --P;
    if (P > 1 && (size_t)p.total_q * 2 * P > sfa_merge_ctas(p.total_q, p.top_k)) return cudaErrorInvalidValue;
    p.splits = P;
    p.early_setup = L.after_indexer ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)(P == 1 ? 1 : 2 * P);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // right behind the indexer: start early, wait on the device before reading the Top-K
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)(p.total_q * 2 * P));
    cfg.blockDim = dim3(kThreadsSfa);
    cfg.dynamicSmemBytes = kSfaSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = L.after_indexer ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, L.qmap, p);
}

cudaError_t launch_sfa(const SfaLaunch& L, cudaStream_t stream) {
    return L.params.kv_fp8 ? launch_sfa_variant<true>(L, stream) : launch_sfa_variant<false>(L, stream);
}

}  // namespace dsa
