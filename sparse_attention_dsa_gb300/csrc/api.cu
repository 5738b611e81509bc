// C ABI (include/dsa.h): argument validation, work planning, tensor-map encoding and kernel launches.
// No device memory is allocated here and nothing synchronises with the host except
// dsa_get_device_error().
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>

#include "dsa.h"
#include "internal.h"

namespace {

thread_local std::string g_last_error;
std::atomic<uint64_t> g_wait_limit_ns{1000000000ull};  // limit of the kernels' pipeline waits

dsa_status_t fail(dsa_status_t st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

dsa_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(DSA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceInfo {
    int num_sms = 0;
    int smem_optin = 0;
};

dsa_status_t device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lk(mu);
    if (!have[dev]) {
        DeviceInfo d;
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(DSA_ERR_UNSUPPORTED, "this library is built for sm_103a; device %d is sm_%d%d", dev, major, minor);
        cache[dev] = d;
        have[dev] = true;
    }
    *out = cache[dev];
    return DSA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Workspace layout: the error word area, the attention kernel's split-merge scratch for the largest grid
// it may use, then (decode shapes: one query token per sequence) the physical rows of the Top-K that the
// single-launch decode kernel hands from its indexer phase to its attention phase.
size_t merge_bytes(int64_t T, int32_t K) { return dsa::sfa_merge_ctas(T, K) * dsa::kSfaMergeFloatsPerCta * sizeof(float); }
size_t decode_rows_bytes(const dsa_dims_t* d) {
    if (d->max_q_len != 1 || d->total_q <= 0 || d->top_k <= 0) return 0;
    return ((size_t)d->total_q * (size_t)d->top_k * sizeof(int32_t) + 15) / 16 * 16;
}

dsa_status_t check_ptr(const void* p, const char* name, bool required = true) {
    if (!p) return required ? fail(DSA_ERR_INVALID_ARG, "%s is NULL", name) : DSA_OK;
    if (!aligned16(p)) return fail(DSA_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
    return DSA_OK;
}

dsa_status_t check_common(const dsa_dims_t* d) {
    if (!d) return fail(DSA_ERR_INVALID_ARG, "dims is NULL");
    if (d->batch < 1) return fail(DSA_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", d->batch);
    if (d->total_q < 0) return fail(DSA_ERR_INVALID_ARG, "total_q must be >= 0 (got %d)", d->total_q);
    if (d->max_q_len < 1) return fail(DSA_ERR_INVALID_ARG, "max_q_len must be >= 1 (got %d)", d->max_q_len);
    if (d->num_pages < 1) return fail(DSA_ERR_INVALID_ARG, "num_pages must be >= 1 (got %d)", d->num_pages);
    if (d->page_size < 1) return fail(DSA_ERR_INVALID_ARG, "page_size must be >= 1 (got %d)", d->page_size);
    if (d->page_size != 64) return fail(DSA_ERR_UNSUPPORTED, "page_size must be 64 (got %d)", d->page_size);
    if (d->max_pages_per_seq < 1)
        return fail(DSA_ERR_INVALID_ARG, "max_pages_per_seq must be >= 1 (got %d)", d->max_pages_per_seq);
    if ((int64_t)d->max_pages_per_seq * 64 > (int64_t)INT32_MAX)
        return fail(DSA_ERR_UNSUPPORTED, "max_pages_per_seq * 64 exceeds int32");
    if (d->top_k < 1) return fail(DSA_ERR_INVALID_ARG, "top_k must be >= 1 (got %d)", d->top_k);
    if (d->top_k > 16384) return fail(DSA_ERR_UNSUPPORTED, "top_k must be <= 16384 (got %d)", d->top_k);
    return DSA_OK;
}

constexpr int kMaxClusterSize = 16;

// Candidate positions of an indexer call: [pos_begin, pos_end) (the whole context by default).
struct PosRange {
    int32_t begin = 0;
    int32_t end = INT32_MAX;
};

dsa_status_t plan_indexer(const dsa_dims_t* d, const DeviceInfo& dev, dsa::IndexerLaunch* L, PosRange r = PosRange()) {
    if (d->idx_heads < 1 || d->idx_dim < 1)
        return fail(DSA_ERR_INVALID_ARG, "idx_heads and idx_dim must be >= 1 (got %d, %d)", d->idx_heads, d->idx_dim);
    if (d->idx_dtype != DSA_BF16 && d->idx_dtype != DSA_FP8_E4M3 && d->idx_dtype != DSA_MXFP8_E4M3)
        return fail(DSA_ERR_INVALID_ARG, "idx_dtype %d is not a dsa_dtype_t", d->idx_dtype);
    const bool mx = d->idx_dtype == DSA_MXFP8_E4M3;
    const bool fp8 = d->idx_dtype == DSA_FP8_E4M3 || mx;  // one-byte codes
    const int quant = mx ? 2 : fp8 ? 1 : 0;
    // the positions one work item scores: the candidate range within the longest context
    const int64_t max_ctx = std::max<int64_t>(0, std::min<int64_t>((int64_t)d->max_pages_per_seq * 64, r.end) - r.begin);
    int qb_max;
    if (mx) {
        if (d->idx_heads != 64 || d->idx_dim != 128)
            return fail(DSA_ERR_UNSUPPORTED, "MXFP8 indexer supports 64 heads of 128 dims (got %d, %d)", d->idx_heads,
                        d->idx_dim);
        qb_max = 1;
    } else if (!fp8 && d->idx_heads == 4 && d->idx_dim == 64)
        qb_max = 4;
    else if (d->idx_heads == 64 && d->idx_dim == 128)
        qb_max = (!fp8 && max_ctx <= 65536) ? 4 : 2;
    else
        return fail(DSA_ERR_UNSUPPORTED, "indexer shape (heads %d, dim %d, %s) has no kernel variant", d->idx_heads,
                    d->idx_dim, fp8 ? "fp8" : "bf16");
    int qb_want = d->max_q_len < qb_max ? d->max_q_len : qb_max;
    if (qb_want == 3) qb_want = 4;
    auto chunk_for = [&](int C) -> int64_t {
        const int64_t per = (max_ctx + C - 1) / C;
        return (per + 127) / 128 * 128;
    };
    // Largest query block (up to qb_want) and smallest cluster for which a CTA's slice of the scores fits
    // in shared memory next to a pipeline of at least 3 stages (2 accepted as a last resort).
    int qb = 0, c_min = 0;
    for (int min_stages = 3; min_stages >= 2 && c_min == 0; --min_stages)
        for (int q = qb_want; q >= 1 && c_min == 0; q /= 2) {
            if (dsa::indexer_variant_n(d->idx_heads, d->idx_dim, quant, q) == 0) continue;
            for (int C = 1; C <= kMaxClusterSize; C *= 2)
                if (chunk_for(C) <= INT32_MAX &&
                    dsa::indexer_smem_estimate(d->idx_heads, d->idx_dim, quant, q, min_stages, (int)chunk_for(C),
                                               C) <= (size_t)dev.smem_optin) {
                    qb = q;
                    c_min = C;
                    break;
                }
        }
    if (c_min == 0)
        return fail(DSA_ERR_UNSUPPORTED, "context of %lld positions exceeds the on-chip score capacity of a %d-CTA "
                    "cluster", (long long)max_ctx, kMaxClusterSize);
    const int blocks_per_seq = (d->max_q_len + qb - 1) / qb;
    const int64_t items = (int64_t)d->batch * blocks_per_seq;
    if (items > (1 << 26)) return fail(DSA_ERR_UNSUPPORTED, "too many work items (%lld)", (long long)items);
    // Otherwise as many CTAs per work item as keep every CTA resident (portable cluster sizes up to 8).
    int c_target = 1;
    while (c_target < 8 && items * (c_target * 2) <= dev.num_sms) c_target *= 2;
    const int C = c_min > c_target ? c_min : c_target;
    L->cluster = C;
    L->items = (int)items;
    L->idx_heads = d->idx_heads;
    L->idx_dim = d->idx_dim;
    L->fp8 = fp8;
    L->mx = mx;
    L->smem_limit = dev.smem_optin;
    L->check_occupancy = true;
    dsa::IndexerParams& p = L->params;
    memset(&p, 0, sizeof p);
    p.batch = d->batch;
    p.total_q = d->total_q;
    p.num_pages = d->num_pages;
    p.max_pages = d->max_pages_per_seq;
    p.top_k = d->top_k;
    p.qb = qb;
    p.blocks_per_seq = blocks_per_seq;
    p.chunk = (int)chunk_for(C) > 0 ? (int)chunk_for(C) : 128;
    p.pos_begin = r.begin;
    p.pos_end = r.end;
    p.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    return DSA_OK;
}

dsa_status_t encode_indexer_maps(const dsa_dims_t* d, const void* q_idx, const void* k_cache, int n_cols,
                                 dsa::IndexerLaunch* L) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const bool fp8 = L->fp8;
    const int elem = fp8 ? 1 : 2;
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint32_t inner_box = (cuuint32_t)(128 / elem);
    {
        const cuuint64_t gdim[3] = {(cuuint64_t)d->idx_dim, 64, (cuuint64_t)d->num_pages};
        const cuuint64_t gstride[2] = {(cuuint64_t)d->idx_dim * elem, (cuuint64_t)64 * d->idx_dim * elem};
        const cuuint32_t box[3] = {inner_box, 64, 1};
        const cuuint32_t es[3] = {1, 1, 1};
        CUresult r = enc(&L->kmap, dt, 3, const_cast<void*>(k_cache), gdim, gstride, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "tensor map for k_cache: CUresult %d", (int)r);
    }
    {
        const cuuint64_t gdim[2] = {(cuuint64_t)d->idx_dim, (cuuint64_t)d->total_q * d->idx_heads};
        const cuuint64_t gstride[1] = {(cuuint64_t)d->idx_dim * elem};
        const cuuint32_t box[2] = {inner_box, (cuuint32_t)n_cols};
        const cuuint32_t es[2] = {1, 1};
        CUresult r = enc(&L->qmap, dt, 2, const_cast<void*>(q_idx), gdim, gstride, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "tensor map for q_idx: CUresult %d", (int)r);
    }
    return DSA_OK;
}

// Everything of an indexer call but the launch.  *launch is false when there is nothing to launch.
dsa_status_t prepare_indexer(const dsa_dims_t* d, const void* q_idx, const float* q_scale, const float* w,
                             const void* k_cache, const float* k_scale, const int32_t* page_table,
                             const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t* topk_idx, float* topk_score,
                             void* workspace, dsa::IndexerLaunch* Lout, bool* launch, PosRange range = PosRange()) {
    *launch = false;
    dsa_status_t st = check_common(d);
    if (st) return st;
    if (range.begin < 0 || range.begin % 64 != 0 || range.end <= range.begin)
        return fail(DSA_ERR_INVALID_ARG, "position range [%d, %d) must be non-empty with a start that is a multiple of 64",
                    range.begin, range.end);
    const bool fp8 = d->idx_dtype == DSA_FP8_E4M3 || d->idx_dtype == DSA_MXFP8_E4M3;
    if ((st = check_ptr(q_idx, "q_idx")) || (st = check_ptr(w, "w")) || (st = check_ptr(k_cache, "k_cache")) ||
        (st = check_ptr(page_table, "page_table")) || (st = check_ptr(seq_lens, "seq_lens")) ||
        (st = check_ptr(cu_q_lens, "cu_q_lens")) || (st = check_ptr(topk_idx, "topk_idx")) ||
        (st = check_ptr(topk_score, "topk_score", false)) || (st = check_ptr(workspace, "workspace")))
        return st;
    if (fp8 && ((st = check_ptr(q_scale, "q_scale")) || (st = check_ptr(k_scale, "k_scale")))) return st;
    // argument checks that need no device come before the device query
    if (d->idx_dtype != DSA_BF16 && d->idx_dtype != DSA_FP8_E4M3 && d->idx_dtype != DSA_MXFP8_E4M3)
        return fail(DSA_ERR_INVALID_ARG, "idx_dtype %d is not a dsa_dtype_t", d->idx_dtype);
    if (d->idx_dtype == DSA_MXFP8_E4M3 && (d->idx_heads != 64 || d->idx_dim != 128))
        return fail(DSA_ERR_UNSUPPORTED, "MXFP8 indexer supports 64 heads of 128 dims (got %d, %d)", d->idx_heads,
                    d->idx_dim);
    DeviceInfo dev;
    if ((st = device_info(&dev))) return st;
    dsa::IndexerLaunch& L = *Lout;
    memset(&L, 0, sizeof L);
    if ((st = plan_indexer(d, dev, &L, range))) return st;
    if (d->total_q == 0) return DSA_OK;
    const int n_cols = dsa::indexer_variant_n(d->idx_heads, d->idx_dim, L.mx ? 2 : fp8 ? 1 : 0, L.params.qb);
    if ((st = encode_indexer_maps(d, q_idx, k_cache, n_cols, &L))) return st;
    dsa::IndexerParams& p = L.params;
    p.q_scale = fp8 ? q_scale : nullptr;
    p.q_idx_codes = L.mx ? q_idx : nullptr;
    p.w = w;
    p.k_scale = fp8 ? k_scale : nullptr;
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.topk = topk_idx;
    p.topk_score = topk_score;
    p.err = static_cast<int32_t*>(workspace);
    *launch = true;
    return DSA_OK;
}

dsa_status_t launch_indexer_checked(const dsa::IndexerLaunch& L, void* stream) {
    cudaError_t e = dsa::launch_indexer(L, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorInvalidClusterSize)
        return fail(DSA_ERR_UNSUPPORTED, "a cluster of %d CTAs does not fit on this device", L.cluster);
    if (e != cudaSuccess) return cuda_fail(e, "indexer launch");
    return DSA_OK;
}

dsa_status_t run_indexer(const dsa_dims_t* d, const void* q_idx, const float* q_scale, const float* w,
                         const void* k_cache, const float* k_scale, const int32_t* page_table, const int32_t* seq_lens,
                         const int32_t* cu_q_lens, int32_t* topk_idx, float* topk_score, void* workspace, void* stream,
                         PosRange range = PosRange()) {
    dsa::IndexerLaunch L;
    bool launch = false;
    dsa_status_t st = prepare_indexer(d, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens,
                                      topk_idx, topk_score, workspace, &L, &launch, range);
    if (st || !launch) return st;
    return launch_indexer_checked(L, stream);
}

// Everything of an attention call but the launch.  *launch is false when there is nothing to launch.
dsa_status_t prepare_sfa(const dsa_dims_t* d, const void* q, const void* kv_cache, const int32_t* page_table,
                         const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* topk_idx, void* out,
                         float* lse, void* workspace, dsa::SfaLaunch* Lout, bool* launch, PosRange range = PosRange()) {
    *launch = false;
    dsa_status_t st = check_common(d);
    if (st) return st;
    if (d->attn_heads < 1) return fail(DSA_ERR_INVALID_ARG, "attn_heads must be >= 1 (got %d)", d->attn_heads);
    if (d->kv_dim < 1 || d->v_dim < 1 || d->v_dim > d->kv_dim)
        return fail(DSA_ERR_INVALID_ARG, "need 1 <= v_dim <= kv_dim (got %d, %d)", d->v_dim, d->kv_dim);
    if (d->kv_dim != 576 || d->v_dim != 512)
        return fail(DSA_ERR_UNSUPPORTED, "sparse attention supports kv_dim 576 / v_dim 512 (got %d / %d)", d->kv_dim,
                    d->v_dim);
    if (d->attn_heads > 128) return fail(DSA_ERR_UNSUPPORTED, "attn_heads must be <= 128 (got %d)", d->attn_heads);
    if (d->kv_dtype != DSA_BF16 && d->kv_dtype != DSA_FP8_E4M3)
        return fail(DSA_ERR_INVALID_ARG, "kv_dtype %d is not a dsa_dtype_t", d->kv_dtype);
    if ((int64_t)d->num_pages * 64 > (int64_t)INT32_MAX)
        return fail(DSA_ERR_UNSUPPORTED, "num_pages * 64 must fit in int32 (got %d pages)", d->num_pages);
    if (!(d->softmax_scale > 0.f) || d->softmax_scale > 1e30f)
        return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be a positive finite number");
    if ((st = check_ptr(q, "q")) || (st = check_ptr(kv_cache, "kv_cache")) ||
        (st = check_ptr(page_table, "page_table")) || (st = check_ptr(seq_lens, "seq_lens")) ||
        (st = check_ptr(cu_q_lens, "cu_q_lens")) || (st = check_ptr(topk_idx, "topk_idx")) ||
        (st = check_ptr(out, "out")) || (st = check_ptr(lse, "lse", false)) ||
        (st = check_ptr(workspace, "workspace")))
        return st;
    DeviceInfo dev;
    if ((st = device_info(&dev))) return st;
    if (d->total_q == 0) return DSA_OK;
    dsa::SfaLaunch& L = *Lout;
    memset(&L, 0, sizeof L);
    dsa::SfaParams& p = L.params;
    p.q = static_cast<const uint16_t*>(q);
    p.kv_cache = static_cast<const uint16_t*>(kv_cache);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.topk = topk_idx;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.err = static_cast<int32_t*>(workspace);
    p.batch = d->batch;
    p.total_q = d->total_q;
    p.num_pages = d->num_pages;
    p.max_pages = d->max_pages_per_seq;
    p.top_k = d->top_k;
    p.heads = d->attn_heads;
    p.kv_dim = d->kv_dim;
    p.v_dim = d->v_dim;
    p.scale_log2 = d->softmax_scale * 1.4426950408889634f;
    p.merge = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + dsa::kErrorWordArea);
    p.kv_fp8 = d->kv_dtype == DSA_FP8_E4M3 ? 1 : 0;
    p.pos_begin = range.begin;
    p.pos_end = range.end;
    p.wait_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    L.smem_limit = dev.smem_optin;
    L.num_sms = dev.num_sms;
    {
        EncodeTiledFn enc = encode_fn();
        if (!enc) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
        const cuuint64_t gdim[2] = {(cuuint64_t)d->kv_dim, (cuuint64_t)d->total_q * d->attn_heads};
        const cuuint64_t gstride[1] = {(cuuint64_t)d->kv_dim * 2};
        const cuuint32_t box[2] = {64, 128};
        const cuuint32_t es[2] = {1, 1};
        CUresult r = enc(&L.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), gdim, gstride, box, es,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "tensor map for q: CUresult %d", (int)r);
    }
    *launch = true;
    return DSA_OK;
}

// after_indexer: the previous launch on this stream is this library's indexer, made in the same call on the
// same inputs, so the attention kernel may start before it ends (it waits on the device for the Top-K).
dsa_status_t launch_sfa_checked(dsa::SfaLaunch L, void* stream, bool after_indexer) {
    L.after_indexer = after_indexer;
    cudaError_t e = dsa::launch_sfa(L, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "sparse attention launch");
    return DSA_OK;
}

dsa_status_t run_sfa(const dsa_dims_t* d, const void* q, const void* kv_cache, const int32_t* page_table,
                     const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* topk_idx, void* out, float* lse,
                     void* workspace, void* stream, PosRange range = PosRange()) {
    dsa::SfaLaunch L;
    bool launch = false;
    dsa_status_t st = prepare_sfa(d, q, kv_cache, page_table, seq_lens, cu_q_lens, topk_idx, out, lse, workspace, &L,
                                  &launch, range);
    if (st || !launch) return st;
    return launch_sfa_checked(L, stream, false);
}

}  // namespace

void dsa::set_last_error(const char* message) { g_last_error = message ? message : ""; }

uint64_t dsa::wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

dsa_status_t dsa::prepare_indexer_call(const dsa_dims_t* d, const void* q_idx, const void* q_scale, const float* w,
                                       const void* k_cache, const void* k_scale, const int32_t* page_table,
                                       const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t* topk_idx,
                                       float* topk_score, void* workspace, IndexerLaunch* L, bool* launch) {
    g_last_error.clear();
    return prepare_indexer(d, q_idx, static_cast<const float*>(q_scale), w, k_cache, static_cast<const float*>(k_scale),
                           page_table, seq_lens, cu_q_lens, topk_idx, topk_score, workspace, L, launch);
}

dsa_status_t dsa::launch_indexer_call(const IndexerLaunch& L, void* stream) { return launch_indexer_checked(L, stream); }

extern "C" {

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

const char* dsa_status_string(dsa_status_t s) {
    switch (s) {
        case DSA_OK: return "DSA_OK";
        case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: invalid argument";
        case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: valid arguments this build does not implement";
        case DSA_ERR_CUDA: return "DSA_ERR_CUDA: a CUDA call failed";
        case DSA_ERR_DEVICE: return "DSA_ERR_DEVICE: the device error word is set";
        case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: a bounded device wait gave up";
    }
    return "unknown dsa_status_t";
}

const char* dsa_last_error_message(void) { return g_last_error.c_str(); }

size_t dsa_workspace_size(const dsa_dims_t* dims) {
    if (!dims) return 0;
    const int64_t T = dims->total_q > 0 ? dims->total_q : 0;
    const int32_t K = dims->top_k > 0 ? dims->top_k : 0;
    return dsa::kErrorWordArea + merge_bytes(T, K) + decode_rows_bytes(dims);
}

dsa_status_t dsa_indexer_topk(const dsa_dims_t* dims, const void* q_idx, const void* q_scale, const float* w,
                              const void* k_cache, const void* k_scale, const int32_t* page_table,
                              const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t* topk_idx, float* topk_score,
                              void* workspace, void* stream) {
    g_last_error.clear();
    // the scale arrays are fp32 (DSA_FP8_E4M3) or E8M0 bytes (DSA_MXFP8_E4M3); the kernels read them by type
    return run_indexer(dims, q_idx, static_cast<const float*>(q_scale), w, k_cache, static_cast<const float*>(k_scale),
                       page_table, seq_lens, cu_q_lens, topk_idx, topk_score, workspace, stream);
}

dsa_status_t dsa_indexer_topk_shard(const dsa_dims_t* dims, const void* q_idx, const void* q_scale, const float* w,
                                    const void* k_cache, const void* k_scale, const int32_t* page_table,
                                    const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t pos_begin,
                                    int32_t pos_end, int32_t* topk_idx, float* topk_score, void* workspace,
                                    void* stream) {
    g_last_error.clear();
    PosRange r;
    r.begin = pos_begin;
    r.end = pos_end;
    return run_indexer(dims, q_idx, static_cast<const float*>(q_scale), w, k_cache, static_cast<const float*>(k_scale),
                       page_table, seq_lens, cu_q_lens, topk_idx, topk_score, workspace, stream, r);
}

dsa_status_t dsa_sparse_attn(const dsa_dims_t* dims, const void* q, const void* kv_cache, const int32_t* page_table,
                             const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* topk_idx, void* out,
                             float* lse, void* workspace, void* stream) {
    g_last_error.clear();
    return run_sfa(dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk_idx, out, lse, workspace, stream);
}

dsa_status_t dsa_sparse_attn_shard(const dsa_dims_t* dims, const void* q, const void* kv_cache,
                                   const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q_lens,
                                   const int32_t* topk_idx, int32_t pos_begin, int32_t pos_end, void* out, float* lse,
                                   void* workspace, void* stream) {
    g_last_error.clear();
    if (pos_begin < 0 || pos_end <= pos_begin)
        return fail(DSA_ERR_INVALID_ARG, "position range [%d, %d) must be non-empty and non-negative", pos_begin, pos_end);
    PosRange r;
    r.begin = pos_begin;
    r.end = pos_end;
    return run_sfa(dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk_idx, out, lse, workspace, stream, r);
}

dsa_status_t dsa_topk_merge(int32_t shards, int32_t total_q, int32_t top_k, const int32_t* topk_idx,
                            const float* topk_score, int32_t* out_idx, float* out_score, void* stream) {
    g_last_error.clear();
    if (shards < 1 || total_q < 0 || top_k < 1)
        return fail(DSA_ERR_INVALID_ARG, "need shards >= 1, total_q >= 0, top_k >= 1 (got %d, %d, %d)", shards, total_q,
                    top_k);
    dsa_status_t st;
    if ((st = check_ptr(topk_idx, "topk_idx")) || (st = check_ptr(topk_score, "topk_score")) ||
        (st = check_ptr(out_idx, "out_idx")) || (st = check_ptr(out_score, "out_score", false)))
        return st;
    if ((int64_t)shards * top_k > dsa::kMaxMergeCandidates)
        return fail(DSA_ERR_UNSUPPORTED, "shards * top_k must be <= %d (got %lld)", dsa::kMaxMergeCandidates,
                    (long long)shards * top_k);
    DeviceInfo dev;
    if ((st = device_info(&dev))) return st;
    if (total_q == 0) return DSA_OK;
    dsa::MergeParams p;
    memset(&p, 0, sizeof p);
    p.idx = topk_idx;
    p.score = topk_score;
    p.out_idx = out_idx;
    p.out_score = out_score;
    p.shards = shards;
    p.total_q = total_q;
    p.top_k = top_k;
    cudaError_t e = dsa::launch_merge(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return DSA_OK;
}

dsa_status_t dsa_attn_combine(int32_t shards, int32_t total_q, int32_t heads, int32_t v_dim, const void* out_parts,
                              const float* lse_parts, void* out, float* lse, void* stream) {
    g_last_error.clear();
    if (shards < 1 || total_q < 0 || heads < 1 || v_dim < 2 || (v_dim & 1))
        return fail(DSA_ERR_INVALID_ARG, "need shards >= 1, total_q >= 0, heads >= 1 and an even v_dim >= 2 "
                    "(got %d, %d, %d, %d)", shards, total_q, heads, v_dim);
    dsa_status_t st;
    if ((st = check_ptr(out_parts, "out_parts")) || (st = check_ptr(lse_parts, "lse_parts")) ||
        (st = check_ptr(out, "out")) || (st = check_ptr(lse, "lse", false)))
        return st;
    DeviceInfo dev;
    if ((st = device_info(&dev))) return st;
    if (total_q == 0) return DSA_OK;
    dsa::CombineParams p;
    memset(&p, 0, sizeof p);
    p.out_in = static_cast<const uint16_t*>(out_parts);
    p.lse_in = lse_parts;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.shards = shards;
    p.total_q = total_q;
    p.heads = heads;
    p.v_dim = v_dim;
    cudaError_t e = dsa::launch_combine(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    return DSA_OK;
}

uint64_t dsa_set_wait_limit_ns(uint64_t limit_ns) {
    return g_wait_limit_ns.exchange(limit_ns == 0 ? 1000000000ull : limit_ns);
}

dsa_status_t dsa_append_rows(const dsa_dims_t* d, const void* k_new, const void* kv_new, const int32_t* page_table,
                             const int32_t* seq_lens, const int32_t* cu_q_lens, void* k_cache, void* k_scale,
                             void* kv_cache, void* workspace, void* stream) {
    g_last_error.clear();
    dsa_status_t st = check_common(d);
    if (st) return st;
    if ((st = check_ptr(k_new, "k_new", false)) || (st = check_ptr(kv_new, "kv_new", false)) ||
        (st = check_ptr(page_table, "page_table")) || (st = check_ptr(seq_lens, "seq_lens")) ||
        (st = check_ptr(cu_q_lens, "cu_q_lens")) || (st = check_ptr(workspace, "workspace")))
        return st;
    const bool idx_fp8 = d->idx_dtype == DSA_FP8_E4M3, kv_fp8 = d->kv_dtype == DSA_FP8_E4M3;
    if (k_new) {
        if (d->idx_dtype == DSA_MXFP8_E4M3)
            return fail(DSA_ERR_UNSUPPORTED, "appending MXFP8 indexer keys is not supported");
        if (d->idx_dtype != DSA_BF16 && !idx_fp8)
            return fail(DSA_ERR_INVALID_ARG, "idx_dtype %d is not a dsa_dtype_t", d->idx_dtype);
        if (d->idx_dim < 2 || d->idx_dim > 128 || (d->idx_dim & 1))
            return fail(DSA_ERR_UNSUPPORTED, "appending supports an even idx_dim in [2, 128] (got %d)", d->idx_dim);
        if ((st = check_ptr(k_cache, "k_cache")) || (st = check_ptr(k_scale, "k_scale", idx_fp8))) return st;
    }
    if (kv_new) {
        if (d->kv_dtype != DSA_BF16 && !kv_fp8)
            return fail(DSA_ERR_INVALID_ARG, "kv_dtype %d is not a dsa_dtype_t", d->kv_dtype);
        if (d->kv_dim != 576 || d->v_dim != 512)
            return fail(DSA_ERR_UNSUPPORTED, "appending supports kv_dim 576 / v_dim 512 (got %d / %d)", d->kv_dim,
                        d->v_dim);
        if ((st = check_ptr(kv_cache, "kv_cache"))) return st;
    }
    if ((int64_t)d->num_pages * 64 > (int64_t)INT32_MAX)
        return fail(DSA_ERR_UNSUPPORTED, "num_pages * 64 must fit in int32 (got %d pages)", d->num_pages);
    if (d->total_q == 0 || (!k_new && !kv_new)) return DSA_OK;
    dsa::AppendParams p;
    memset(&p, 0, sizeof p);
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.kv_new = static_cast<const uint16_t*>(kv_new);
    p.page_table = page_table;
    p.seq_lens = seq_lens;
    p.cu_q_lens = cu_q_lens;
    p.k_cache = static_cast<uint8_t*>(k_cache);
    p.k_scale = static_cast<float*>(k_scale);
    p.kv_cache = static_cast<uint8_t*>(kv_cache);
    p.err = static_cast<int32_t*>(workspace);
    p.batch = d->batch;
    p.total_q = d->total_q;
    p.num_pages = d->num_pages;
    p.max_pages = d->max_pages_per_seq;
    p.idx_dim = d->idx_dim;
    p.idx_fp8 = idx_fp8 ? 1 : 0;
    p.kv_fp8 = kv_fp8 ? 1 : 0;
    cudaError_t e = dsa::launch_append(p, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return DSA_OK;
}

dsa_status_t dsa_fused_decode(const dsa_dims_t* dims, const void* q_idx, const void* q_scale_v, const float* w,
                              const void* k_cache, const void* k_scale_v, const void* q, const void* kv_cache,
                              const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q_lens,
                              int32_t* topk_idx, void* out, float* lse, void* workspace, void* stream) {
    g_last_error.clear();
    const float* q_scale = static_cast<const float*>(q_scale_v);  // fp32, or E8M0 bytes (MXFP8)
    const float* k_scale = static_cast<const float*>(k_scale_v);
    dsa::IndexerLaunch IL;
    dsa::SfaLaunch SL;
    bool li = false, ls = false;
    dsa_status_t st = prepare_indexer(dims, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens,
                                      topk_idx, nullptr, workspace, &IL, &li);
    if (st) return st;
    st = prepare_sfa(dims, q, kv_cache, page_table, seq_lens, cu_q_lens, topk_idx, out, lse, workspace, &SL, &ls);
    if (st) return st;
    if (!li || !ls) return DSA_OK;  // no query token
    // one launch when every query token can have a cluster of its own for both phases; its indexer phase
    // hands the Top-K's physical rows to its attention phase through the workspace
    if (decode_rows_bytes(dims) > 0) {
        int32_t* rows = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + dsa::kErrorWordArea +
                                                   merge_bytes(dims->total_q, dims->top_k));
        IL.params.rows_out = rows;
        SL.params.rows_in = rows;
    }
    cudaError_t e = dsa::launch_decode(IL, SL, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) return DSA_OK;
    if (e != cudaErrorNotSupported) return cuda_fail(e, "fused decode launch");
    // otherwise the indexer, then the attention kernel as its programmatic dependent
    IL.params.rows_out = nullptr;
    SL.params.rows_in = nullptr;
    if ((st = launch_indexer_checked(IL, stream))) return st;
    return launch_sfa_checked(SL, stream, true);
}

int32_t dsa_fused_decode_launches(const dsa_dims_t* dims) {
    g_last_error.clear();
    if (!dims) {
        dsa::set_last_error("dims is NULL");
        return -1;
    }
    if (check_common(dims) != DSA_OK) return -1;
    if (dims->total_q == 0) return 0;
    DeviceInfo dev;
    if (device_info(&dev) != DSA_OK) return -1;
    dsa::IndexerLaunch IL;
    memset(&IL, 0, sizeof IL);
    if (plan_indexer(dims, dev, &IL) != DSA_OK) return -1;
    dsa::SfaLaunch SL;
    memset(&SL, 0, sizeof SL);
    SL.params.total_q = dims->total_q;
    SL.params.top_k = dims->top_k;
    SL.num_sms = dev.num_sms;
    SL.smem_limit = dev.smem_optin;
    return dsa::decode_single_launch(IL, SL) ? 1 : 2;
}

dsa_status_t dsa_get_device_error(const void* workspace, void* stream, int32_t* code) {
    g_last_error.clear();
    if (!workspace || !code) return fail(DSA_ERR_INVALID_ARG, "workspace and code must be non-NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    *code = v;
    if (v == 0) return DSA_OK;
    if (v & DSA_DEVERR_TIMEOUT) return fail(DSA_ERR_TIMEOUT, "device error word 0x%x", v);
    return fail(DSA_ERR_DEVICE, "device error word 0x%x", v);
}

dsa_status_t dsa_clear_device_error(void* workspace, void* stream) {
    g_last_error.clear();
    if (!workspace) return fail(DSA_ERR_INVALID_ARG, "workspace is NULL");
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
    return DSA_OK;
}

}  // extern "C"
