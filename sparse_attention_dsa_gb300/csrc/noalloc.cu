// dsa_indexer_topk_static: the fused indexer + Top-K without a caller-allocated workspace.
//
// Some callers cannot allocate device memory when they run the indexer: code that lives inside another
// runtime which owns all device memory (a pooled allocator or an inference server that forbids raw
// cudaMalloc), real-time decode loops that must not allocate after start-up, and hosts that expose no
// allocator to plugins at all.  dsa_indexer_topk needs a workspace for its scratch (the device error
// word), so those callers would have to obtain one.  This entry point instead keeps the scratch in a
// file-scope device array that exists on every GPU that loads the library, for the life of the process.
//
// The kernels are exactly those of dsa_indexer_topk; only the scratch location differs.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "dsa.h"
#include "internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 4096;  // maximum scratch this entry point can provide

// Scratch shared by every call of dsa_indexer_topk_static on this device.  In host code this name is a
// host-side stand-in; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (looked up once per device).
dsa_status_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        dsa::set_last_error("dsa_indexer_topk_static: cudaGetDevice failed");
        return DSA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        dsa::set_last_error("dsa_indexer_topk_static: device ordinal out of range");
        return DSA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) {
            dsa::set_last_error("dsa_indexer_topk_static: cudaGetSymbolAddress of the static scratch failed");
            return DSA_ERR_CUDA;
        }
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return DSA_OK;
}

}  // namespace

extern "C" dsa_status_t dsa_indexer_topk_static(const dsa_dims_t* dims, const void* q_idx, const void* q_scale,
                                                const float* w, const void* k_cache, const void* k_scale,
                                                const int32_t* page_table, const int32_t* seq_lens,
                                                const int32_t* cu_q_lens, int32_t* topk_idx, int32_t* device_error,
                                                void* stream) {
    if (!dims) {
        dsa::set_last_error("dims is NULL");
        return DSA_ERR_INVALID_ARG;
    }
    // the indexer uses only the error word area of a workspace (the rest is the attention kernel's)
    const size_t need = dsa::kErrorWordArea;
    static_assert(dsa::kErrorWordArea <= kStaticScratchBytes, "the static array holds the indexer's scratch");
    void* scratch = nullptr;
    dsa_status_t st = scratch_address(&scratch);
    if (st != DSA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the scratch keeps the previous call's contents; the error word must start at zero
    cudaError_t e = cudaMemsetAsync(scratch, 0, need, s);
    if (e != cudaSuccess) {
        dsa::set_last_error("dsa_indexer_topk_static: clearing the static scratch failed");
        return DSA_ERR_CUDA;
    }
    st = dsa_indexer_topk(dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens, topk_idx,
                          scratch, stream);
    if (st != DSA_OK) return st;
    if (device_error) {
        e = cudaMemcpyAsync(device_error, scratch, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) {
            dsa::set_last_error("dsa_indexer_topk_static: copying the device error word failed");
            return DSA_ERR_CUDA;
        }
    }
    return DSA_OK;
}
