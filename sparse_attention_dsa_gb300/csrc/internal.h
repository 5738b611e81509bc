// Launch descriptions shared between the C-ABI layer (api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

constexpr int kMaxStages = 8;

// ---- lightning indexer + Top-K -----------------------------------------------------------------------
struct IndexerParams {
    const float* q_scale;  // [T, Hi] (FP8 only)
    const float* w;        // [T, Hi]
    const float* k_scale;  // [num_pages, 64] (FP8 only)
    const int32_t* page_table;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    int32_t* topk;  // [T, K]
    int32_t* err;   // device error word
    int32_t batch;
    int32_t total_q;
    int32_t num_pages;
    int32_t max_pages;
    int32_t top_k;
    int32_t qb;              // query tokens per cluster work item
    int32_t blocks_per_seq;  // ceil(max_q_len / qb)
    int32_t chunk;           // positions per CTA (multiple of 128)
    int32_t stages;          // filled in by the launcher
    int32_t* rows_out;       // [T, K] physical cache row of every selected position (-1 for padding), or null
    const void* q_idx_codes;  // MXFP8: the q_idx codes [T, Hi, Di] (dequantised at set-up instead of loaded by TMA)
    float* topk_score;        // [T, K] fp32 score of every selected position (-inf for padding), or null
    int32_t pos_begin;        // only positions in [pos_begin, pos_end) are candidates (pos_begin % 64 == 0)
    int32_t pos_end;
    uint64_t wait_ns;         // limit of every pipeline wait (drains keep the default limit)
};

struct IndexerLaunch {
    CUtensorMap kmap;  // 3-D view [num_pages][64][Di] of the indexer K cache
    CUtensorMap qmap;  // 2-D view [T*Hi][Di] of q_idx
    IndexerParams params;
    int items;    // work items (clusters)
    int cluster;  // CTAs per cluster
    int idx_heads;
    int idx_dim;
    bool fp8;
    bool mx;         // FP8 with one E8M0 scale per 32 elements (q_scale / k_scale hold scale bytes)
    int smem_limit;  // opt-in dynamic shared memory per block
    bool check_occupancy;
};

// UMMA N of the kernel variant serving (Hi, Di, dtype, qb), 0 when no variant exists.
int indexer_variant_n(int idx_heads, int idx_dim, int fp8, int qb);  // fp8: 0 bf16, 1 row scales, 2 MXFP8
// Dynamic shared memory of that variant for the given pipeline depth, positions per CTA and cluster size.
size_t indexer_smem_estimate(int idx_heads, int idx_dim, int fp8, int qb, int stages, int chunk, int cluster);  // fp8 as above
cudaError_t launch_indexer(const IndexerLaunch& launch, cudaStream_t stream);

// ---- sparse flash attention --------------------------------------------------------------------------
struct SfaParams {
    const uint16_t* q;         // [T, Hq, D] bf16 bits
    const uint16_t* kv_cache;  // [num_pages, 64, D] bf16 bits, or FP8 rows of kKvFp8RowBytes (kv_fp8)
    const int32_t* page_table;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    const int32_t* topk;  // [T, K]
    uint16_t* out;        // [T, Hq, Dv] bf16 bits
    float* lse;           // [T, Hq] or null
    int32_t* err;
    int32_t batch;
    int32_t total_q;
    int32_t num_pages;
    int32_t max_pages;
    int32_t top_k;
    int32_t heads;
    int32_t kv_dim;
    int32_t v_dim;
    float scale_log2;  // softmax_scale * log2(e)
    int32_t splits;    // position splits per query (filled in by the launcher)
    int32_t early_setup;  // launched right behind this library's indexer: only topk comes from it
    float* merge;         // split-merge scratch: sfa_merge_floats_per_cta() floats per CTA of the grid
    int32_t kv_fp8;       // kv_cache rows are in the FP8 row layout
    const int32_t* rows_in;  // [T, K] physical rows of topk written by the indexer phase in the same launch, or null
    int32_t one_query_per_seq;  // every sequence has exactly one query token: token t belongs to sequence t
    int32_t pos_begin;          // Top-K entries outside [pos_begin, pos_end) are skipped (a context shard)
    int32_t pos_end;
    uint64_t wait_ns;           // limit of every pipeline wait (drains keep the default limit)
};

struct SfaLaunch {
    CUtensorMap qmap;  // 2-D view [T*Hq][576] of q, 128-row boxes
    SfaParams params;
    int smem_limit;
    int num_sms;
    bool after_indexer;  // the previous kernel in the stream is this library's indexer (programmatic launch)
};

cudaError_t launch_sfa(const SfaLaunch& launch, cudaStream_t stream);

// Position splits the attention launcher starts from for these sizes on `num_sms` SMs (before its
// co-residency check), and the most entries one split may hold.
int sfa_splits(int64_t total_q, int32_t top_k, int num_sms);
constexpr int kSfaMaxEntries = 2048;
// FP8 latent-KV row: 512 E4M3 codes (4 tiles of 128), 4 fp32 tile scales, 64 bf16 rotary values
constexpr int kKvFp8RowBytes = 656;
constexpr int kKvFp8ScaleOff = 512;
constexpr int kKvFp8RopeOff = 528;

// ---- appending a step's rows to the paged caches ------------------------------------------------------
struct AppendParams {
    const uint16_t* k_new;   // [T, Di] bf16 bits or null
    const uint16_t* kv_new;  // [T, 576] bf16 bits or null
    const int32_t* page_table;
    const int32_t* seq_lens;
    const int32_t* cu_q_lens;
    uint8_t* k_cache;   // bf16 rows of Di, or E4M3 rows of Di bytes (idx_fp8)
    float* k_scale;     // [num_pages * 64] (idx_fp8)
    uint8_t* kv_cache;  // bf16 rows of 576, or FP8 rows of kKvFp8RowBytes (kv_fp8)
    int32_t* err;
    int32_t batch;
    int32_t total_q;
    int32_t num_pages;
    int32_t max_pages;
    int32_t idx_dim;
    int32_t idx_fp8;
    int32_t kv_fp8;
};
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);

// Single-launch decode (indexer + Top-K + attention of each token in one cluster, one kernel).  Returns
// cudaErrorNotSupported, without launching anything, when the sizes do not map one query token to one
// cluster (the caller then launches the two kernels).
cudaError_t launch_decode(const IndexerLaunch& indexer, const SfaLaunch& attention, cudaStream_t stream);
// Whether launch_decode would launch for these plans (no launch).
bool decode_single_launch(const IndexerLaunch& indexer, const SfaLaunch& attention);

// Split-merge scratch of the attention kernel: each CTA of a grid with position splits owns one region
// of kSfaMergeRows partial O rows (256 fp32 each; P * ceil(128 / P) of them are used) and 128
// (max, sum) pairs.
constexpr int kSfaMergeRows = 136;
constexpr size_t kSfaMergeFloatsPerCta = (size_t)kSfaMergeRows * 256 + 2 * 128;
// The largest grid (in CTAs) the attention launcher can choose with position splits for these sizes
// (0 when it never splits): at most 256 SMs' worth, or more when top_k forces splits.
size_t sfa_merge_ctas(int64_t total_q, int32_t top_k);
// Bytes of workspace the library uses: the 256-byte error word area, plus the attention merge scratch.
constexpr size_t kErrorWordArea = 256;

// ---- context-parallel decode: merge of shard Top-K lists, combine of shard attention outputs -----------
struct MergeParams {
    const int32_t* idx;   // [shards, T, K] shard-local selections (positions, -1 padded)
    const float* score;   // [shards, T, K] their scores
    int32_t* out_idx;     // [T, K]
    float* out_score;     // [T, K] or null
    int32_t shards;
    int32_t total_q;
    int32_t top_k;
};
size_t merge_smem_bytes(int shards, int top_k);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

struct CombineParams {
    const uint16_t* out_in;  // [shards, T, Hq, Dv] bf16 bits
    const float* lse_in;     // [shards, T, Hq]
    uint16_t* out;           // [T, Hq, Dv] bf16 bits
    float* lse;              // [T, Hq] or null
    int32_t shards;
    int32_t total_q;
    int32_t heads;
    int32_t v_dim;
};
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);

// Sets the message returned by dsa_last_error_message() on this host thread.
void set_last_error(const char* message);

// Limit of the kernels' pipeline waits for launches made from now on (dsa_set_wait_limit_ns).
uint64_t wait_limit_ns();

// The host half of dsa_indexer_topk: every argument check and the launch plan, nothing enqueued (*launch
// is false when there is nothing to launch); then the launch itself.
dsa_status_t prepare_indexer_call(const dsa_dims_t* dims, const void* q_idx, const void* q_scale, const float* w,
                                  const void* k_cache, const void* k_scale, const int32_t* page_table,
                                  const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t* topk_idx,
                                  float* topk_score, void* workspace, IndexerLaunch* launch_out, bool* launch);
dsa_status_t launch_indexer_call(const IndexerLaunch& launch, void* stream);

// Candidates one dsa_topk_merge call may hold per query token (shards * top_k): its shared-memory keys.
constexpr int kMaxMergeCandidates = 16384;

}  // namespace dsa
