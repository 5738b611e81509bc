// dsa_indexer_topk_static: the fused indexer + Top-K without a caller-allocated workspace.
//
// Some callers cannot allocate device memory when they run the indexer: code that lives inside another
// runtime which owns all device memory (a pooled allocator or an inference server that forbids raw
// cudaMalloc), real-time decode loops that must not allocate after start-up, and hosts that expose no
// allocator to plugins at all.  dsa_indexer_topk needs a workspace for its scratch (the device error
// word), so those callers would have to obtain one.  This entry point instead keeps the scratch in a
// file-scope device array that exists on every GPU that loads the library, for the life of the process.
//
// The kernels are exactly those of dsa_indexer_topk; only the scratch location differs.  Every argument
// is checked (with the same checks as dsa_indexer_topk) before anything is put on the stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"
#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 4096;  // maximum scratch this entry point can provide

// Scratch shared by every call of dsa_indexer_topk_static on this device.  In host code this name is a
// host-side stand-in; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch in the current device's context.  Looked up on every call (the
// lookup allocates nothing and is cheap): a cached address would go stale if the context were destroyed
// and recreated (cudaDeviceReset), since the module is then loaded again, possibly elsewhere.
dsa_status_t scratch_address(void** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p) {
        dsa::set_last_error("dsa_indexer_topk_static: cudaGetSymbolAddress of the static scratch failed");
        return DSA_ERR_CUDA;
    }
    *out = p;
    return DSA_OK;
}

}  // namespace

extern "C" dsa_status_t dsa_indexer_topk_static(const dsa_dims_t* dims, const void* q_idx, const void* q_scale,
                                                const float* w, const void* k_cache, const void* k_scale,
                                                const int32_t* page_table, const int32_t* seq_lens,
                                                const int32_t* cu_q_lens, int32_t* topk_idx, float* topk_score,
                                                int32_t* device_error, void* stream) {
    dsa::set_last_error("");
    if (!dims) {
        dsa::set_last_error("dims is NULL");
        return DSA_ERR_INVALID_ARG;
    }
    if (device_error && (reinterpret_cast<uintptr_t>(device_error) & 3u) != 0) {
        dsa::set_last_error("device_error is not 4-byte aligned");
        return DSA_ERR_INVALID_ARG;
    }
    // the indexer uses only the error word area of a workspace (the rest is the attention kernel's)
    const size_t need = dsa::kErrorWordArea;
    static_assert(dsa::kErrorWordArea <= kStaticScratchBytes, "the static array holds the indexer's scratch");
    void* scratch = nullptr;
    dsa_status_t st = scratch_address(&scratch);
    if (st != DSA_OK) return st;
    // every check and the launch plan first: a rejected call puts nothing on the stream and leaves
    // *device_error as it was
    dsa::IndexerLaunch L;
    bool launch = false;
    st = dsa::prepare_indexer_call(dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens,
                                   topk_idx, topk_score, scratch, &L, &launch);
    if (st != DSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the scratch keeps the previous call's contents; the error word must start at zero
    cudaError_t e = cudaMemsetAsync(scratch, 0, need, s);
    if (e != cudaSuccess) {
        dsa::set_last_error("dsa_indexer_topk_static: clearing the static scratch failed");
        return DSA_ERR_CUDA;
    }
    if (launch && (st = dsa::launch_indexer_call(L, stream)) != DSA_OK) return st;
    if (device_error) {
        e = cudaMemcpyAsync(device_error, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) {
            dsa::set_last_error("dsa_indexer_topk_static: copying the device error word failed");
            return DSA_ERR_CUDA;
        }
    }
    return DSA_OK;
}
