// The standalone indexer kernel (one launch per dsa_indexer_topk call) and its launcher.  The device
// code lives in indexer_impl.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "indexer_impl.cuh"

namespace dsa {
namespace {

template <int HI, int DI, int QB, bool FP8, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_topk_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                        const IndexerParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    indexer_cta<HI, DI, QB, FP8, kThreads, true, MX>(kmap, qmap, p, smem_raw);
}

template <int HI, int DI, int QB, bool FP8, bool MX = false>
cudaError_t launch_variant(const IndexerLaunch& L, cudaStream_t stream) {
    auto kern = indexer_topk_kernel<HI, DI, QB, FP8, MX>;
    const int chunk = L.params.chunk;
    // choose the number of pipeline stages from the shared-memory budget
    int stages = kMaxStages;
    while (stages > 2 && indexer_smem_bytes<HI, DI, QB, FP8, MX>(stages, chunk, L.cluster) > (size_t)L.smem_limit) --stages;
    size_t smem = indexer_smem_bytes<HI, DI, QB, FP8, MX>(stages, chunk, L.cluster);
    if (smem > (size_t)L.smem_limit) return cudaErrorInvalidConfiguration;
    // a CTA that takes all of TMEM must be alone on its SM (a second one would wait in its allocation
    // for a cluster peer that waits for it): more than half the shared memory keeps it alone
    if (IdxCfg<HI, DI, QB, FP8, MX>::kTmemCols == 512 && 2 * smem <= (size_t)L.smem_limit) smem = L.smem_limit / 2 + 1024;
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
    if (fp8 == 2) return (idx_heads == 64 && idx_dim == 128 && qb == 1) ? 64 : 0;
    if (!fp8 && idx_heads == 4 && idx_dim == 64 && qb >= 1 && qb <= 4) return 16;
    if (idx_heads == 64 && idx_dim == 128 && (qb == 1 || qb == 2 || (qb == 4 && !fp8))) return 64 * qb;
    return 0;
}

size_t indexer_smem_estimate(int idx_heads, int idx_dim, int fp8, int qb, int stages, int chunk, int cluster) {
    if (fp8 == 2)
        return (idx_heads == 64 && idx_dim == 128 && qb == 1) ? indexer_smem_bytes<64, 128, 1, true, true>(stages, chunk, cluster)
                                                               : ~size_t(0);
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
    if (L.mx) {
        if (L.idx_heads == 64 && L.idx_dim == 128 && qb == 1) return launch_variant<64, 128, 1, true, true>(L, stream);
        return cudaErrorInvalidValue;
    }
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
