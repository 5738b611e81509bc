/*
 * dsa.h - C ABI of the GB300 (sm_103a) library for the DSA decode/prefill hot path:
 * a fused lightning indexer with on-chip Top-K selection, followed by sparse flash attention (SFA)
 * over the selected rows of a paged MLA latent-KV cache.
 *
 * The operations follow these published articles (cited by title and section):
 *  [A1] "Optimizing Inference for Hybrid Attention LLMs: Practices for Fast Adaptation", sections 1 and
 *       3.2 (index-gather-compute integration; paged KV management; gather/compute overlap; layered
 *       quantization: FP8 KV cache with one scale per 128 elements of each token).
 *  [A2] "Optimizing Inference for Hybrid Attention Architectures: From Operator Fusion to Sequence
 *       Sharding", section "Breaking Down the Computational Path of Hybrid Attention" (steps 1 and 2) and
 *       section "Fusing Index Screening with Multi-Stream Orchestration".
 *  [A3] "Day0 Inference Optimization for Next-Generation Hybrid-Architecture LLMs Based on CANN",
 *       sections 2.1 (deep operator fusion) and 3.1 (FP8 indexer inputs).
 *  [A4] "Day0 Inference Support and Performance Optimization for New LLM Architectures", sections 3.1
 *       (integrated indexer fusion), 3.2 (sparse attention kernel), 3.3 (input preparation ahead of the
 *       indexer), 4 (hierarchical quantization: "Token-Head-Tile" FP8 KV cache, tiles of 128) and 5
 *       (context parallelism: 5.1 decode by context shards, 5.2 the Zigzag layout of prefill).
 *
 * Conventions shared by every entry point
 *  - Ownership: the caller owns every buffer.  All array arguments are DEVICE pointers (memory of the
 *    current CUDA device) unless stated otherwise; `dims` is a host pointer read during the call only.
 *    The library keeps no state between calls and allocates no device memory.
 *  - Execution: compute calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and never synchronise with the host, so they can be captured in a CUDA graph.
 *  - Errors: argument problems are detected on the host and returned synchronously before any launch
 *    (DSA_ERR_INVALID_ARG / DSA_ERR_UNSUPPORTED; dsa_last_error_message() explains).  Problems found on
 *    the device (an out-of-range page id, inconsistent lengths, a bounded wait that gave up) set bits in
 *    the workspace error word; the kernels skip the affected work and return normally.  Read the word
 *    with dsa_get_device_error().  A failed launch returns DSA_ERR_CUDA.
 *  - Layout: tensors are dense and row-major in the shapes given below; every array pointer must be
 *    16-byte aligned.
 *  - Paging ([A1] 3.2): logical position s of sequence b lives in row s % page_size of physical page
 *    page_table[b * max_pages_per_seq + s / page_size].  The indexer K cache and the latent-KV cache
 *    share one page table.  page_size must be 64.
 *  - Queries: sequence b owns query tokens cu_q_lens[b] .. cu_q_lens[b+1]-1 (n_b of them).
 *    seq_lens[b] = L_b counts the cached tokens INCLUDING those n_b new ones, so query j of sequence b
 *    sits at position p = L_b - n_b + j and sees positions 0..p (causal, itself included).
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 4

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* a null/misaligned pointer, a negative or inconsistent size */
    DSA_ERR_UNSUPPORTED = 2, /* valid arguments outside what this build implements (see each call) */
    DSA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    DSA_ERR_DEVICE = 4,      /* dsa_get_device_error(): the device error word is non-zero */
    DSA_ERR_TIMEOUT = 5      /* dsa_get_device_error(): a bounded device wait gave up */
} dsa_status_t;

typedef enum {
    DSA_BF16 = 0,       /* bfloat16 */
    DSA_FP8_E4M3 = 1,   /* OCP OFP8 E4M3 codes times fp32 scales: indexer rows with one scale per row
                           ([A3] 3.1); latent-KV rows in the FP8 row layout below */
    DSA_MXFP8_E4M3 = 2  /* indexer only: E4M3 codes with one E8M0 scale byte per 32 consecutive elements
                           of a row (OCP MX: the byte e means 2^(e - 127); [A1] 1, [A4] 4.1 "MXFP8,
                           per-group 32").  The NaN codes 0x7F and 0xFF, which a saturating encoder
                           never writes, are not propagated from k_cache (the kernel reads them as
                           +-480 times the scale); a scale byte of 255 (NaN) is. */
} dsa_dtype_t;

/*
 * FP8 latent-KV row layout ([A1] 1 and [A4] 4: FP8 with one scale per 128 elements of each token), used
 * when dims->kv_dtype == DSA_FP8_E4M3 (D = 576, Dv = 512).  One row is DSA_KV_FP8_ROW_BYTES bytes:
 *   bytes   0..511  E4M3 codes of dims 0..511 (the latent part, also V), in 4 tiles of 128;
 *   bytes 512..527  4 fp32 scales, tile i covering dims 128*i .. 128*i+127;
 *   bytes 528..655  dims 512..575 (the rotary part) as bf16, unquantised (576 is not a multiple of 128).
 * Element d < 512 of the row is e4m3(code[d]) * scale[d / 128]; the kernels dequantise to bf16.
 */
#define DSA_KV_FP8_ROW_BYTES 656

/* Bits of the device error word (the first int32 of the workspace). */
#define DSA_DEVERR_PAGE 0x1    /* a page-table entry outside [0, num_pages) was needed */
#define DSA_DEVERR_SEQ 0x2     /* n_b > L_b, or L_b > max_pages_per_seq * page_size */
#define DSA_DEVERR_INDEX 0x4   /* a Top-K entry outside [-1, p] reached the attention kernel */
#define DSA_DEVERR_TIMEOUT 0x8 /* a pipeline wait exceeded its limit (one second unless
                                  dsa_set_wait_limit_ns() says otherwise) */

typedef struct {
    int32_t batch;             /* B >= 1 sequences */
    int32_t total_q;           /* T = cu_q_lens[B] query tokens (0 allowed: nothing to do) */
    int32_t max_q_len;         /* >= max_b n_b, >= 1 */
    int32_t num_pages;         /* physical pages in each cache */
    int32_t page_size;         /* tokens per page; must be 64 */
    int32_t max_pages_per_seq; /* row length of page_table */
    int32_t idx_heads;         /* Hi, indexer heads */
    int32_t idx_dim;           /* Di, indexer head dim */
    int32_t idx_dtype;         /* dsa_dtype_t of q_idx and the indexer K cache */
    int32_t top_k;             /* K, positions kept per query */
    int32_t attn_heads;        /* Hq, attention heads sharing the latent KV rows */
    int32_t kv_dim;            /* D, latent KV row width (512 latent + 64 RoPE = 576) */
    int32_t v_dim;             /* Dv, leading dims of each row used as V (512) */
    float softmax_scale;       /* multiplies q . kv before the softmax (1/sqrt(576)) */
    int32_t kv_dtype;          /* dsa_dtype_t of the latent-KV cache: DSA_BF16 rows of D values, or
                                  DSA_FP8_E4M3 rows in the FP8 row layout above */
} dsa_dims_t;

/* ABI version of the loaded library (DSA_ABI_VERSION). */
int32_t dsa_abi_version(void);

/* Static description of a status code. */
const char* dsa_status_string(dsa_status_t status);

/* Human-readable reason for the last non-OK status returned on this host thread ("" if none). */
const char* dsa_last_error_message(void);

/*
 * Bytes of device workspace the compute calls need for `dims`: 256 bytes whose first int32 is the
 * device error word, then (when the attention kernel may split one query's positions across several
 * CTAs: few query tokens) scratch for merging those splits, 137 KiB per CTA of the largest grid it may
 * use (at most about 33 MiB), then (when max_q_len == 1) T x K int32 through which the single-launch
 * dsa_fused_decode hands the physical cache rows of the Top-K from its indexer phase to its attention
 * phase.  The caller allocates it once (16-byte aligned, as from cudaMalloc),
 * zero-fills at least the first 256 bytes before first use, and passes the same buffer to later calls;
 * the error word latches until dsa_clear_device_error().  Returns 0 when dims is NULL.  Calls that may
 * overlap on the GPU need separate workspaces.
 */
size_t dsa_workspace_size(const dsa_dims_t* dims);

/*
 * Lightning indexer + Top-K ([A2] step 1; [A3] 2.1; [A4] 3.1): for every query token t,
 *     I[t,s] = sum_h w[t,h] * max(0, q_idx[t,h,:] . k[s,:])      for s = 0..p_t,
 * and keep the K positions with the largest I (ties: the lower position wins).  The scores stay on
 * chip; only the selected positions (and, on request, their scores) are written.  With FP8 inputs,
 * q_idx[t,h,:] and k[s,:] are the codes times their row scales.
 *   q_idx        [T, Hi, Di]  bf16, or E4M3 codes (uint8) when dims->idx_dtype is DSA_FP8_E4M3 or
 *                DSA_MXFP8_E4M3
 *   q_scale      [T, Hi] fp32 row scales of q_idx (DSA_FP8_E4M3), [T, Hi, Di/32] E8M0 bytes
 *                (DSA_MXFP8_E4M3), NULL for bf16
 *   w            [T, Hi]      fp32 head weights
 *   k_cache      [num_pages, 64, Di]  paged indexer keys, same dtype as q_idx
 *   k_scale      [num_pages, 64] fp32 row scales of k_cache (DSA_FP8_E4M3), [num_pages, 64, Di/32] E8M0
 *                bytes (DSA_MXFP8_E4M3), NULL for bf16
 *   page_table   [B, max_pages_per_seq] int32;  seq_lens [B] int32;  cu_q_lens [B+1] int32
 *   topk_idx     [T, K] int32 output: the selected positions of each query in ascending order; when
 *                fewer than K positions are visible all of them are kept and the rest is -1.
 *   topk_score   [T, K] fp32 output or NULL: I[t, topk_idx[t,k]] as the kernel computed it (fp32
 *                accumulation; -0 is written as +0), -inf where topk_idx is -1.  These are the keys
 *                dsa_topk_merge orders by.
 *   workspace    dsa_workspace_size(dims) bytes (see above)
 * Supported: (Hi, Di) = (4, 64) or (64, 128) in bf16, (64, 128) in FP8 and MXFP8; K <= 4096 (MXFP8 runs
 * one query token per thread-block cluster, any number per sequence).
 */
dsa_status_t dsa_indexer_topk(const dsa_dims_t* dims, const void* q_idx, const void* q_scale, const float* w,
                              const void* k_cache, const void* k_scale, const int32_t* page_table,
                              const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t* topk_idx,
                              float* topk_score, void* workspace, void* stream);

/*
 * dsa_indexer_topk restricted to the positions of one context shard ([A4] 5.1: under context
 * parallelism each device scores the positions it holds and keeps a local Top-K of (score, position)):
 * only positions s with pos_begin <= s < pos_end (and s <= p_t) are candidates; the result holds the K
 * best of them (all of them, -1 padded, if there are fewer), in ascending order, with their scores.
 * Positions are the sequence's logical positions; page_table entries of pages outside the range are
 * never read (a shard's table may hold anything there).  pos_begin must be a multiple of 64 (page
 * aligned); pos_end > pos_begin (INT32_MAX: to the end).  Other arguments and limits as for
 * dsa_indexer_topk.  Selecting each shard's Top-K and merging them with dsa_topk_merge gives exactly the
 * selection of dsa_indexer_topk over the whole context (the scores of a position do not depend on the
 * range it is scored in).
 */
dsa_status_t dsa_indexer_topk_shard(const dsa_dims_t* dims, const void* q_idx, const void* q_scale, const float* w,
                                    const void* k_cache, const void* k_scale, const int32_t* page_table,
                                    const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t pos_begin,
                                    int32_t pos_end, int32_t* topk_idx, float* topk_score, void* workspace,
                                    void* stream);

/*
 * Merge of context-shard selections ([A4] 5.1: the shards' local Top-K lists are gathered and merged
 * into the global Top-K with the same key).  For every query token t, from the candidates
 * (topk_idx[s,t,k], topk_score[s,t,k]) of all shards s (entries with topk_idx < 0 are empty), keep the K
 * with the largest score, ties to the lower position; write them in candidate order (shard 0 first),
 * which is ascending when shard s holds positions below those of shard s+1 and each list is ascending
 * (as dsa_indexer_topk_shard writes them), then -1 / -inf padding.
 *   topk_idx    [shards, T, K] int32;  topk_score [shards, T, K] fp32 (from dsa_indexer_topk_shard)
 *   out_idx     [T, K] int32 output;   out_score  [T, K] fp32 output or NULL
 * Positions must be distinct across shards.  No workspace.  Supported: shards * K <= 16384.
 */
dsa_status_t dsa_topk_merge(int32_t shards, int32_t total_q, int32_t top_k, const int32_t* topk_idx,
                            const float* topk_score, int32_t* out_idx, float* out_score, void* stream);

/*
 * Sparse flash attention over the selected rows ([A2] step 2; [A4] 3.2; [A1] 3.2): for every query
 * token t and head h, with S_t = { topk_idx[t,k] : topk_idx[t,k] >= 0 } (any order; -1 entries are
 * skipped),
 *     z_s = softmax_scale * q[t,h,:] . kv[s,:]           (all kv_dim dims)
 *     out[t,h,:] = sum_{s in S_t} softmax(z)_s * kv[s, 0:v_dim]
 *     lse[t,h]   = log sum_{s in S_t} exp(z_s)           (natural log; -inf and out = 0 if S_t is empty)
 *   q          [T, Hq, D] bf16
 *   kv_cache   [num_pages, 64, D] bf16, or [num_pages, 64, DSA_KV_FP8_ROW_BYTES] bytes in the FP8 row
 *              layout when dims->kv_dtype == DSA_FP8_E4M3 (V = the first Dv dims of each row)
 *   topk_idx   [T, K] int32 logical positions (entries outside [-1, p_t] set DSA_DEVERR_INDEX and are
 *              skipped)
 *   out        [T, Hq, Dv] bf16 output;  lse [T, Hq] fp32 output (may be NULL)
 * Supported: D = 576, Dv = 512, Hq <= 128, K <= 4096.
 */
dsa_status_t dsa_sparse_attn(const dsa_dims_t* dims, const void* q, const void* kv_cache, const int32_t* page_table,
                             const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* topk_idx, void* out,
                             float* lse, void* workspace, void* stream);

/*
 * dsa_sparse_attn over the selected rows one context shard holds ([A4] 5.1: each device attends to the
 * selected rows in its own cache, giving a partial (out, lse)): entries of topk_idx outside
 * [pos_begin, pos_end) are skipped like -1 (they are not an error).  out and lse are the attention over
 * the shard's rows alone (out = 0 and lse = -inf when it holds none); dsa_attn_combine joins the
 * shards' partials.  Other arguments and limits as for dsa_sparse_attn.
 */
dsa_status_t dsa_sparse_attn_shard(const dsa_dims_t* dims, const void* q, const void* kv_cache,
                                   const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q_lens,
                                   const int32_t* topk_idx, int32_t pos_begin, int32_t pos_end, void* out, float* lse,
                                   void* workspace, void* stream);

/*
 * Combine of partial attention results ([A4] 5.1: the shards' partial outputs are merged with their
 * log-sum-exp values): for every token t and head h,
 *     LSE = log sum_s exp(lse_parts[s,t,h]),   out[t,h,:] = sum_s exp(lse_parts[s,t,h] - LSE) * out_parts[s,t,h,:]
 * (shards with lse = -inf have weight 0; with none left, out = 0 and lse = -inf).
 *   out_parts [shards, T, heads, v_dim] bf16;  lse_parts [shards, T, heads] fp32
 *   out       [T, heads, v_dim] bf16 output;   lse [T, heads] fp32 output or NULL
 * Arithmetic in fp32.  No workspace.  v_dim must be even.
 */
dsa_status_t dsa_attn_combine(int32_t shards, int32_t total_q, int32_t heads, int32_t v_dim, const void* out_parts,
                              const float* lse_parts, void* out, float* lse, void* stream);

/*
 * The whole decode/prefill step: the work of dsa_indexer_topk followed by that of dsa_sparse_attn on
 * the same stream ([A2] "Fusing Index Screening with Multi-Stream Orchestration"; [A4] 3.1-3.2).
 * topk_idx is an output (the selection used by the attention).  Arguments and limits are those of the
 * two calls.  When every sequence has exactly one query token and both stages fit one thread-block
 * cluster per token (64 indexer heads of 128 dims), this is ONE kernel launch: each cluster scores its
 * token's context, selects the Top-K and runs the attention.  Otherwise it is the two kernels, the
 * attention launched as a programmatic dependent of the indexer.  dsa_fused_decode_launches() tells
 * which.
 */
dsa_status_t dsa_fused_decode(const dsa_dims_t* dims, const void* q_idx, const void* q_scale, const float* w,
                              const void* k_cache, const void* k_scale, const void* q, const void* kv_cache,
                              const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q_lens,
                              int32_t* topk_idx, void* out, float* lse, void* workspace, void* stream);

/*
 * Kernel launches dsa_fused_decode makes for `dims` on the current device: 1 (the single-launch
 * kernel), 2 (indexer, then attention), 0 (no query token), or -1 when dims are invalid or unsupported
 * (the reason is in dsa_last_error_message()).  Host-only: launches nothing.  The articles have no
 * counterpart to this call.
 */
int32_t dsa_fused_decode_launches(const dsa_dims_t* dims);

/*
 * dsa_indexer_topk without a workspace argument.  The articles have no counterpart to this call; it
 * exists for callers that cannot allocate device memory when they run the indexer: code living inside
 * another runtime that owns all device memory (a pooled allocator or a server that forbids raw
 * cudaMalloc), decode loops that must not allocate after start-up, and plug-in hosts that offer no
 * allocator.  The kernels are those of dsa_indexer_topk and so are the arguments, except:
 *   - the scratch (the device error word: the indexer uses only the first 256 bytes of a workspace)
 *     lives in a static device array of 4096 bytes inside the library; every GPU that loads the
 *     library holds it until the process exits;
 *   - device_error (optional DEVICE pointer to one int32, 4-byte aligned) receives this call's device
 *     error word (see dsa_get_device_error) on `stream` after the kernel.  With NULL the word is
 *     discarded: device-side problems (bad pages, lengths, a wait that gave up) are then not reported.
 * Every call looks up the array's device address in the current device's context
 * (cudaGetSymbolAddress, with that device current; this allocates nothing).  Every argument is checked
 * first: a call that returns an error has put nothing on `stream` and left *device_error unchanged.
 * Otherwise the call clears the error word on `stream`, launches, and copies the word out.  All calls
 * share the one array, so calls that may overlap on the GPU (different streams, or different host
 * threads) race on it.  Nothing is allocated: no cudaMalloc, cudaFree or allocating library routine is
 * called.
 */
dsa_status_t dsa_indexer_topk_static(const dsa_dims_t* dims, const void* q_idx, const void* q_scale,
                                     const float* w, const void* k_cache, const void* k_scale,
                                     const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q_lens,
                                     int32_t* topk_idx, float* topk_score, int32_t* device_error, void* stream);

/*
 * Synchronises `stream`, then reads the device error word of `workspace` into *code (host pointer).
 * Returns DSA_OK if it is zero, DSA_ERR_TIMEOUT if DSA_DEVERR_TIMEOUT is set, DSA_ERR_DEVICE for any
 * other bit, DSA_ERR_CUDA if the synchronisation or the copy fails.
 */
dsa_status_t dsa_get_device_error(const void* workspace, void* stream, int32_t* code);

/*
 * Appends one step's new rows to the paged caches ([A4] 3.3: the indexer's K input is prepared ahead of
 * the indexer; quantisation per [A1] 1 and [A4] 4): for every query token t (at position p_t, see the
 * conventions), its indexer key goes to the indexer cache row of p_t and its latent-KV row to the
 * latent-KV cache row of p_t.  FP8 caches are quantised dynamically per group (the whole indexer key
 * row; each 128-element latent tile): scale = absmax / 448 (1 for an all-zero group), code =
 * E4M3(x / scale) rounded to nearest with ties to even and saturated at 448, all in fp32.
 *   k_new      [T, Di] bf16 new indexer keys, or NULL to leave the indexer cache alone
 *   kv_new     [T, D] bf16 new latent-KV rows, or NULL to leave the latent-KV cache alone
 *   k_cache, k_scale   as for dsa_indexer_topk (k_scale: FP8 only, receives the fp32 row scales;
 *                      MXFP8 keys are not appended: DSA_ERR_UNSUPPORTED)
 *   kv_cache   as for dsa_sparse_attn (bf16 rows, or the FP8 row layout)
 *   workspace  dsa_workspace_size(dims) bytes (only its error word is used)
 * A token whose page is out of range (DSA_DEVERR_PAGE) or whose position is inconsistent
 * (DSA_DEVERR_SEQ) writes nothing.  Supported: Di <= 128 and even; D = 576, Dv = 512.
 */
dsa_status_t dsa_append_rows(const dsa_dims_t* dims, const void* k_new, const void* kv_new,
                             const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q_lens,
                             void* k_cache, void* k_scale, void* kv_cache, void* workspace, void* stream);

/* Zeroes the device error word (asynchronously on `stream`). */
dsa_status_t dsa_clear_device_error(void* workspace, void* stream);

/*
 * Failure detection: sets the limit, in nanoseconds, after which a pipeline wait inside the kernels gives
 * up (sets DSA_DEVERR_TIMEOUT, abandons its work, and the kernel still drains its copies in flight and
 * frees its tensor memory under the default limit before it returns).  Applies to launches made after
 * the call, from any host thread; 0 restores the default of one second.  Returns the previous limit.  A
 * wait's clock starts when it first finds its phase incomplete; with a limit below the default, waits
 * poll instead of suspending, so that the limit is looked at within its own span.  A short limit makes
 * correct launches report DSA_DEVERR_TIMEOUT (with unspecified outputs): it exists to test that path.
 * The articles have no counterpart to this call.
 */
uint64_t dsa_set_wait_limit_ns(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */
