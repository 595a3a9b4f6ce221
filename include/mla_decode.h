/*
 * mla_decode.h -- C ABI of libmla: split-KV absorbed-MLA decode over a paged
 * fp8 e4m3fn KV cache on GB300 (sm_103a).
 *
 * The operation (moonmath-ai/amd-kernels README, "MLA absorbed decode",
 * "Use / MLA decode" and "Constraints / MLA decode"):
 *   one fused fp8 row per cached token is both K (all d_v + d_rope columns) and
 *   V (the first d_v columns), dequantized by ONE per-tensor kv_scale; queries
 *   come split into a latent part q_lat and a RoPE part q_pe; the pool is paged
 *   with page_size 1, so kv_indices is a flat per-token slot list in which any
 *   permutation or subset of the pool is legal; a call serves plain decode
 *   (q_len 1) and speculative verify (q_len > 1: draft position t of a request of
 *   S keys attends KV positions [0, S - q_len + t], inclusive); the output is
 *   written in place and an optional base-2 log-sum-exp is returned.
 *
 * For query row r = b*q_len + t and head h, with k_j the dequantized rows of
 * request b's visible positions:
 *   s_j  = scale * (q_lat[r,h,:] . k_j[0:d_v] + q_pe[r,h,:] . k_j[d_v:d_v+d_rope])
 *   o    = sum_j softmax(s)_j k_j[0:d_v]                    (bf16, round to nearest)
 *   lse  = log2 sum_j 2^(s_j * log2 e)                        (fp32, base 2)
 * A row that sees no key gets o = 0 and lse = -inf.
 *
 * Split-KV ("flash-decoding"): the planner splits each request's positions into
 * num_splits contiguous ranges (hip_mha_decoding_num_partitions: wave-aligned
 * split-K target, MLA-style branch); each (request, head block, split) CTA
 * writes a normalized fp32 partial and its base-2 LSE to the workspace and a
 * split-K reduce merges them in increasing split order, a fixed association
 * (README, "Numerics": the merge sums in a fixed association, so results are
 * deterministic run to run).
 *
 * Conventions shared by every entry point:
 *   - Pointers named q_*, pool, *indices, *indptr, seq_lens, o*, lse*, workspace
 *     are DEVICE pointers owned by the caller; the library never allocates,
 *     frees or keeps them past the call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work on it: no host synchronisation, no allocation, so a call
 *     can be captured into a CUDA graph (the plan depends on shapes alone).
 *   - Return value: MLA_OK (0) or a negative MLA_ERR_* status; nothing is
 *     enqueued when a status other than MLA_OK or MLA_ERR_LAUNCH_FAILED is
 *     returned.  mla_status_string() names each status.
 *   - Faults found on the device (a slot outside [0, pool_rows), a bounded wait
 *     that ran out) are never raised as GPU faults: the kernel skips the bad
 *     access, ORs an MLA_DEVERR_* bit into the workspace's error word and
 *     finishes; outputs of the affected rows are then unspecified.  The word
 *     is sticky: clear it with mla_workspace_reset() and read it with
 *     mla_read_device_error().
 */
#ifndef MLA_DECODE_H
#define MLA_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------- */
#define MLA_OK 0
#define MLA_ERR_INVALID_ARG (-1)         /* null pointer, negative size, plan/shape mismatch */
#define MLA_ERR_UNSUPPORTED_SHAPE (-2)   /* d_v/d_rope not (512,64) dense or (448,64) sparse,
                                            heads outside [1,128], too many splits,
                                            more than 65535 requests or tokens */
#define MLA_ERR_MISALIGNED (-3)          /* a buffer is not 16-byte aligned */
#define MLA_ERR_WORKSPACE_TOO_SMALL (-4) /* workspace_bytes < plan->workspace_bytes */
#define MLA_ERR_UNSUPPORTED_DEVICE (-5)  /* current device is not compute capability 10.3 */
#define MLA_ERR_LAUNCH_FAILED (-6)       /* a kernel launch returned a CUDA error */
#define MLA_ERR_CUDA (-7)                /* another CUDA runtime/driver call failed */

/* ---- device error bits (workspace error word) ------------------------------- */
#define MLA_DEVERR_BAD_SLOT 1u       /* a dense slot outside [0, pool_rows): key skipped */
#define MLA_DEVERR_TIMEOUT 2u        /* a bounded pipeline wait ran out: CTA gave up */
#define MLA_DEVERR_BAD_LENGTH 4u     /* seq_lens[b] outside [0, kv_indptr[b+1]-kv_indptr[b]] */

/* Element types of the DCP share buffers (mla_decode_dcp, mla_dcp_lse_merge_ranks). */
#define MLA_DTYPE_BF16 0
#define MLA_DTYPE_F32 1

/* Largest split count the reducer accepts (hip_mha_decoding_num_partitions: the
 * reducer's 256-partition specialization caps the MLA-style split count). */
#define MLA_MAX_SPLITS 256
/* Bytes at the start of every workspace that hold the device error word and
 * the fused merge's arrival tickets; zero them before a workspace's first use
 * (mla_workspace_reset does). */
#define MLA_WORKSPACE_HEADER_BYTES 65536

/*
 * A launch plan: a pure function of shapes and the SM count (README, "MLA
 * absorbed decode": the op plans from tensor shapes alone, so it is CUDA-graph
 * capturable with no host synchronisation).  Plain data: copy it, store it,
 * recompute it; it holds no pointer.  Fields after `variant` echo the shape the
 * plan was made for; the decode entry points reject a plan whose echo differs
 * from their arguments.
 */
typedef struct {
    int32_t num_splits;      /* KV ranges per request (1..MLA_MAX_SPLITS) */
    int32_t rows_per_cta;    /* query rows (draft position x head) per CTA: 16, or 32
                                when a request has more than 16 rows; above 16 the
                                planners take 16 where a CTA's work is short (a
                                32-row CTA starts later), else 32; results agree
                                with the oracle either way */
    int32_t block_n;         /* keys per pipeline block */
    int32_t head_blocks;     /* CTAs sharing one (request, split) */
    int32_t grid_x, grid_y, grid_z;  /* head_blocks, num_splits, batch (or tokens) */
    int32_t variant;         /* kernel variant: 2 = tcgen05 split kernel, then the
                                split-K reduce kernel when num_splits > 1;
                                other values are rejected (MLA_ERR_INVALID_ARG) */
    int64_t workspace_bytes; /* bytes of device workspace the call needs */
    int32_t batch, q_len, num_heads, d_v, d_rope, sm_count;
    int64_t total_keys;      /* dense: kv_indices length; sparse: tokens * (topk + extra_topk) */
    int32_t kv_share;        /* 1: every CTA gathers its own KV rows (a request's
                                head blocks read the same rows, the repeats
                                served from L2); other values are rejected */
    int32_t extra_topk;      /* sparse: candidates per token in the second
                                (compressed) cache, 0 without one; dense: 0 */
    int32_t long_first;      /* dense, 1: grid slice z serves the z-th longest
                                request (ties by index), so the longest work is
                                scheduled first; set when the grid outlasts one
                                wave and batch <= 256; results do not depend on it */
    int32_t merge_cluster;   /* 1: the split-K merge is a second kernel (the split-K
                                reduce); 2 or 4: it is fused into the split kernel,
                                whose CTAs form clusters of that many consecutive
                                splits (num_splits a multiple of it) that merge
                                their partials through each other's shared memory,
                                the last cluster of a tile to finish merging the
                                clusters' results; results do not depend on the
                                timing.  The planner sets 1 (measured on GB300
                                the fused merge never beat the reduce kernel);
                                a caller may opt in by setting a size that fits */
} mla_plan_t;

/*
 * Dense plan.  total_keys = number of entries of kv_indices (a shape, not a
 * value); sm_count = the device's multiProcessorCount.  d_v must be 512 and
 * d_rope 64 (README, "Constraints / MLA decode": kv_lora_rank 512,
 * qk_rope_head_dim 64); num_heads in [1, 128] (same passage: H 1..128); any
 * q_len >= 1 with q_len * num_heads <= 2^20; batch <= 65535 (the requests are
 * the split grid's third dimension).  Writes *out and returns MLA_OK, or a
 * status.
 */
int mla_decode_plan(int32_t batch, int32_t q_len, int32_t num_heads, int64_t total_keys,
                    int32_t d_v, int32_t d_rope, int32_t sm_count, mla_plan_t* out);

/*
 * Sparse top-k plan (flashinfer.mla.cake_sparse_mla_sm120_dsv4_nvfp4_plan_splits:
 * one decode call's (num_splits, chunks per CTA) from tokens, heads, top-k, the
 * second cache's extra_topk and the SM count; "[Perf] pa_decode_sparse ..."
 * issue: 64 heads, 448 NoPE + 64 RoPE columns, top-k 2048).  d_v must be 448
 * and d_rope 64.  extra_topk = candidates per token in a second (compressed)
 * cache, 0 without one (mla_sparse_decode_extra).  max_splits caps num_splits
 * (0 = MLA_MAX_SPLITS).  Every split count from 1 up is valid for this kernel
 * (a split may even be empty), so a small cap costs speed only and is never an
 * error.  num_tokens <= 65535 (the tokens are the split grid's third dimension).
 */
int mla_sparse_decode_plan(int32_t num_tokens, int32_t num_heads, int32_t topk,
                           int32_t extra_topk, int32_t d_v, int32_t d_rope, int32_t sm_count,
                           int32_t max_splits, mla_plan_t* out);

/*
 * Dense decode: enqueues the split kernel and, when plan->num_splits > 1, the
 * split-K reduce (launched as a programmatic dependent of the split kernel, so
 * it is scheduled while the split kernel drains).  Layouts (row-major,
 * contiguous):
 *   q_lat    bf16 [batch*q_len, num_heads, 512]   row r = b*q_len + t
 *   q_pe     bf16 [batch*q_len, num_heads, 64]
 *   pool     e4m3fn bytes [pool_rows, 576] (a [pool_rows, 1, 576] tensor), 16-byte aligned
 *   seq_lens int32 [batch]; kv_indptr int32 [batch+1]; kv_indices int32 [kv_indptr[batch]]
 *            request b's position j lives in slot kv_indices[kv_indptr[b] + j],
 *            j < seq_lens[b] <= kv_indptr[b+1] - kv_indptr[b]
 *   o_lat    bf16 [batch*q_len, num_heads, 512], written
 *   lse      fp32 [batch*q_len, num_heads] base 2, written when non-NULL
 *   workspace >= plan->workspace_bytes bytes, 256-byte aligned; its first
 *            MLA_WORKSPACE_HEADER_BYTES hold the error word, the rest is
 *            scratch for the fp32 partials.  Calls that share a workspace must
 *            not overlap on the GPU.
 * scale multiplies the raw q.k dot product of dequantized rows (typically
 * (512+64)^-0.5); kv_scale dequantizes the pool.  Rows are copied in 128-key
 * blocks: the keys of a block that a call masks (past a request's length, or
 * invalid sparse entries) become zero rows without reading the pool, so only
 * the rows the page table names need finite e4m3fn bytes.
 */
int mla_decode(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
               const void* pool, int64_t pool_rows, const int32_t* seq_lens,
               const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
               int32_t q_len, int32_t num_heads, float scale, float kv_scale,
               void* o_lat, float* lse, void* workspace, int64_t workspace_bytes,
               void* stream);

/*
 * Sparse top-k decode: token t attends the pool rows indices[t, 0:topk]
 * (a negative entry is invalid and skipped, the has_invalid case of the
 * pa_decode_sparse issue; a token with no valid entry gets o = 0, lse = -inf).
 *   q_nope bf16 [num_tokens, num_heads, 448]; q_pe bf16 [num_tokens, num_heads, 64]
 *   pool   e4m3fn bytes [pool_rows, 512]; indices int32 [num_tokens, topk]
 *   o      bf16 [num_tokens, num_heads, 448]; lse fp32 [num_tokens, num_heads] or NULL
 * Other arguments as for mla_decode.
 */
int mla_sparse_decode(const mla_plan_t* plan, const void* q_nope, const void* q_pe,
                      const void* pool, int64_t pool_rows, const int32_t* indices,
                      int32_t num_tokens, int32_t num_heads, int32_t topk, float scale,
                      float kv_scale, void* o, float* lse, void* workspace,
                      int64_t workspace_bytes, void* stream);

/*
 * Dense decode of one rank's share under decode context parallelism (DCP;
 * moonmath-ai/amd-kernels README, "MLA absorbed decode" and "Use / MLA decode":
 * one op serves plain decode, speculative verify and DCP; under DCP seq_lens
 * counts this rank's positions, glen gives the global lengths, and the op
 * returns a base-2 LSE for the cross-rank merge; "Constraints / MLA decode":
 * DCP needs glen whenever cp_world > 1).
 *   Rank cp_rank of cp_world holds the positions p of every request with
 *   p % cp_world == cp_rank, in increasing order: its kv_indices/kv_indptr/
 *   seq_lens list those positions' slots, so local key j is the global
 *   position j * cp_world + cp_rank.
 *   glen  int32 [batch] device: global lengths.  Draft row t of request b sees
 *         the local keys j < seq_lens[b] with j * cp_world + cp_rank <=
 *         glen[b] - q_len + t (the draft window of mla_decode in global
 *         positions); a row that sees none gets o = 0, lse = -inf.
 *   o     [batch*q_len, num_heads, 512]: the share's normalised output
 *         (softmax over the rank's visible keys, times kv_scale), bf16 when
 *         o_dtype is MLA_DTYPE_BF16 (the op's own output type, as in the
 *         pages) or fp32 when MLA_DTYPE_F32 (no rounding before the merge, at
 *         twice the exchange bytes); 16-byte aligned;
 *   lse   fp32 [batch*q_len, num_heads] base 2 of the share, required when
 *         cp_world > 1.
 * cp_world in [1, MLA_MAX_SPLITS], cp_rank in [0, cp_world); glen and lse are
 * required when cp_world > 1 (else MLA_ERR_INVALID_ARG), as is a known
 * o_dtype.  With cp_world == 1, glen == NULL and MLA_DTYPE_BF16 the call is
 * mla_decode.  The plan is mla_decode_plan's for the rank's own kv_indices
 * length.  Other arguments as for mla_decode.
 */
int mla_decode_dcp(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                   const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                   const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                   int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                   const int32_t* glen, int32_t cp_rank, int32_t cp_world, int32_t o_dtype,
                   void* o, float* lse, void* workspace, int64_t workspace_bytes,
                   void* stream);

/*
 * The split kernel of mla_decode_dcp alone (as mla_decode_splits is to
 * mla_decode): with plan->num_splits == 1 it writes the share o / lse; with
 * more it leaves the fp32 partials in the workspace for mla_splitk_reduce.
 * Arguments as for mla_decode_dcp.
 */
int mla_decode_dcp_splits(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                          const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                          const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                          int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                          const int32_t* glen, int32_t cp_rank, int32_t cp_world,
                          int32_t o_dtype, void* o, float* lse, void* workspace,
                          int64_t workspace_bytes, void* stream);

/*
 * Cross-rank merge of DCP shares (README, "Use / MLA decode":
 * mla_dcp_lse_merge_ranks combines the ranks' outputs and base-2 LSEs after
 * the all-to-all).  For each of `rows` rows, with k over the cp_world ranks:
 *   M = max_k lse_in[k, row];  w_k = 2^(lse_in[k, row] - M)
 *   out[row, :] = bf16(sum_k w_k parts_in[k, row, :] / sum_k w_k)
 *   lse_out[row] = M + log2 sum_k w_k           (when lse_out is non-NULL)
 * in a fixed association (each column sums its terms in increasing k).  A row whose
 * shares are all -inf gets out = 0 and lse_out = -inf.
 *   parts_in [cp_world, rows, d_v] (rank-major, as an all-gather leaves it),
 *            bf16 or fp32 as parts_dtype (MLA_DTYPE_BF16 / MLA_DTYPE_F32) says
 *   lse_in   fp32 [cp_world, rows] base 2
 *   out      bf16 [rows, d_v], written; lse_out fp32 [rows] or NULL
 * d_v a multiple of 8 up to 512; cp_world in [1, MLA_MAX_SPLITS]; parts_in and
 * out 16-byte aligned.  Device pointers; enqueued on `stream`.
 */
int mla_dcp_lse_merge_ranks(const void* parts_in, int32_t parts_dtype, const float* lse_in,
                            int32_t cp_world, int64_t rows, int32_t d_v, void* out,
                            float* lse_out, void* stream);

/*
 * Sparse top-k decode over two caches in one call (flashinfer
 * cake_sparse_mla_sm120_dsv4_nvfp4_plan_splits: extra_topk candidate slots per
 * token in the second (compressed) cache).  Token t attends, in one softmax,
 * the valid entries of indices[t, 0:topk] (rows of pool) together with the
 * valid entries of extra_indices[t, 0:extra_topk] (rows of extra_pool); a
 * negative entry in either table is invalid and skipped, and a token with no
 * valid entry gets o = 0, lse = -inf.
 *   extra_pool    e4m3fn bytes [extra_rows, 512], the main pool's row format
 *                 (448 NoPE + 64 RoPE columns) and kv_scale; 16-byte aligned
 *   extra_indices int32 [num_tokens, extra_topk]
 * The plan is mla_sparse_decode_plan's with the same topk and extra_topk.
 * With extra_topk == 0 the call is mla_sparse_decode (extra_pool and
 * extra_indices may be NULL).  Other arguments as for mla_sparse_decode.
 */
int mla_sparse_decode_extra(const mla_plan_t* plan, const void* q_nope, const void* q_pe,
                            const void* pool, int64_t pool_rows, const int32_t* indices,
                            const void* extra_pool, int64_t extra_rows,
                            const int32_t* extra_indices, int32_t num_tokens, int32_t num_heads,
                            int32_t topk, int32_t extra_topk, float scale, float kv_scale,
                            void* o, float* lse, void* workspace, int64_t workspace_bytes,
                            void* stream);
/* The split kernel of mla_sparse_decode_extra alone (see mla_decode_splits). */
int mla_sparse_decode_extra_splits(const mla_plan_t* plan, const void* q_nope,
                                   const void* q_pe, const void* pool, int64_t pool_rows,
                                   const int32_t* indices, const void* extra_pool,
                                   int64_t extra_rows, const int32_t* extra_indices,
                                   int32_t num_tokens, int32_t num_heads, int32_t topk,
                                   int32_t extra_topk, float scale, float kv_scale, void* o,
                                   float* lse, void* workspace, int64_t workspace_bytes,
                                   void* stream);

/*
 * The two halves of mla_decode / mla_sparse_decode, for callers that keep the
 * per-split partials (for example to merge them with another rank's) or time
 * the kernels one by one.  mla_decode_splits enqueues only the split kernel:
 * with plan->num_splits == 1 it writes o_lat / lse exactly as mla_decode does;
 * otherwise it leaves the normalized fp32 partials and their base-2 LSEs in the
 * workspace, where mla_workspace_partials() finds them, and
 * mla_splitk_reduce(o_part, lse_part, rows, num_splits, d_v, kv_scale, ...)
 * finishes the call.  Arguments as for mla_decode / mla_sparse_decode.
 */
int mla_decode_splits(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                      const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                      const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                      int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                      void* o_lat, float* lse, void* workspace, int64_t workspace_bytes,
                      void* stream);
int mla_sparse_decode_splits(const mla_plan_t* plan, const void* q_nope, const void* q_pe,
                             const void* pool, int64_t pool_rows, const int32_t* indices,
                             int32_t num_tokens, int32_t num_heads, int32_t topk, float scale,
                             float kv_scale, void* o, float* lse, void* workspace,
                             int64_t workspace_bytes, void* stream);

/*
 * Device addresses, inside `workspace`, of the partials a plan's split kernel
 * writes: o_part fp32 [rows, num_splits, d_v] and lse_part fp32
 * [rows, num_splits], rows = batch * q_len * num_heads.  Host arithmetic only;
 * both are NULL when plan->num_splits == 1.
 */
int mla_workspace_partials(const mla_plan_t* plan, void* workspace, float** o_part,
                           float** lse_part);

/*
 * Split-K reduce on its own (hip_mha_decoding_num_partitions: the split-K
 * reducer that merges up to 256 partitions).  For each of `rows` rows:
 *   M = max_s lse_part[row, s];  w_s = 2^(lse_part[row, s] - M)
 *   o[row, :]  = bf16(out_scale * sum_s w_s o_part[row, s, :] / sum_s w_s)
 *   lse[row]   = M + log2 sum_s w_s            (when lse is non-NULL)
 * in a fixed association (sum_s w_s is 32 lane-strided partial sums joined by a
 * butterfly; each column sums its terms in increasing s, or, above 16 splits
 * and above 8 splits when rows <= 128, as four interleaved sums, s = g, g + 4,
 * ... for g = 0..3, each in increasing s, added in increasing g), so the result
 * does not vary from call to call; a row whose partials are all -inf gets o = 0 and
 * lse = -inf.  o_part fp32 [rows, num_splits, d_v] (normalized partials),
 * lse_part fp32 [rows, num_splits] base 2, o bf16 [rows, d_v]; d_v a multiple
 * of 8, num_splits in [1, MLA_MAX_SPLITS]; all 16-byte aligned.
 */
int mla_splitk_reduce(const float* o_part, const float* lse_part, int64_t rows,
                      int32_t num_splits, int32_t d_v, float out_scale, void* o,
                      float* lse, void* stream);

/*
 * Re-target a plan to a forced split count (1..MLA_MAX_SPLITS), updating its
 * grid, its merge cluster size (1, as the planner sets it) and its workspace
 * size.  For split sweeps
 * (moonmath-ai/amd-kernels README, "Results -- MLA decode": num_kv_splits swept
 * per shape) and tests; the planner's own choice needs no call to it.  A
 * caller may set merge_cluster to 1 afterwards (the separate reduce) or to
 * another size that fits; the decode calls reject one that does not.
 */
int mla_plan_force_splits(mla_plan_t* plan, int32_t num_splits);

/* Zero the workspace header, which holds the error word (enqueued on `stream`). */
int mla_workspace_reset(void* workspace, void* stream);

/*
 * Read the error word (MLA_DEVERR_* bits) into *code.  Synchronises `stream`;
 * not for the hot path.
 */
int mla_read_device_error(const void* workspace, int32_t* code, void* stream);

/*
 * Dense decode for callers that cannot allocate device memory: code running
 * where cudaMalloc is unavailable or not allowed (a no-allocation region of a
 * serving loop with a fixed memory budget, or a host framework that hands over
 * only its input and output buffers).  It is mla_decode with the workspace
 * replaced by a static scratch array inside the library, so the caller passes
 * inputs and outputs only and the call itself allocates nothing.  The pages
 * have no counterpart of this entry point.
 *   - Scratch: a file-scope __device__ array of MLA_NOALLOC_SCRATCH_BYTES; every
 *     GPU that loads the library holds it until the process exits.  A plan with
 *     plan->workspace_bytes above that size is rejected with
 *     MLA_ERR_WORKSPACE_TOO_SMALL and nothing is enqueued.
 *   - Set-up: the first call on a device (with that device current) looks up
 *     the array's device address once; make that first call before any stream
 *     capture on the device.  The address is kept for the life of the process,
 *     so do not use this entry point on a device after cudaDeviceReset.
 *   - Every call shares the one array and it keeps the last call's contents, so
 *     calls that overlap on the GPU (on different streams, or from different
 *     threads) race and must be serialised by the caller.
 *   - Device-side error bits (MLA_DEVERR_*) are not reported by this entry
 *     point: bad slots are still skipped safely, but there is no workspace to
 *     read them from.
 * Other arguments, layouts and status codes as for mla_decode.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (32 * 1024 * 1024)
int mla_decode_noalloc(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                       const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                       const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                       int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                       void* o_lat, float* lse, void* stream);

/* Static text for a status code. */
const char* mla_status_string(int status);

/*
 * Gather probe, for tests of the page-table gather (step a2): copies
 * out[i, :] = pool[indices[i], :] for i < n, byte for byte, through the split
 * kernel's own gather path (TMA tile::gather4 into the swizzled shared-memory
 * stage layout, then read back de-swizzled).  row_bytes is 576 (dense rows:
 * four 128-byte chunks and a 64-byte RoPE chunk) or 512 (sparse rows).  An
 * index outside [0, pool_rows) is not read; its output row is zero.  pool and
 * out 16-byte aligned; workspace (>= MLA_WORKSPACE_HEADER_BYTES, 256-byte
 * aligned) receives MLA_DEVERR_TIMEOUT if a bounded wait ran out.  Not on the
 * decode path.
 */
int mla_debug_gather(const void* pool, int64_t pool_rows, int32_t row_bytes,
                     const int32_t* indices, int64_t n, void* out, void* workspace,
                     void* stream);

/*
 * Sets the bound, in SM clock cycles, of the split kernel's pipeline waits
 * for launches enqueued after the call (process-wide; every device), and
 * returns the previous bound; cycles <= 0 restores the default, about one
 * second at GB300 clocks.  A wait that runs out ends its CTA's work: the CTA
 * stops issuing copies and MMAs, waits (with the full bound) for those it
 * already issued, writes what it has (its output rows are then unspecified),
 * sets MLA_DEVERR_TIMEOUT in the workspace error word and exits; the call
 * completes normally and the device stays usable.  For tests of that path:
 * while a bound other than the default is set, every CTA also starts with a
 * wait on a barrier that nothing completes, so at least that wait runs out
 * while the CTA's first copies are in flight.  Not on the decode path; not
 * thread-safe against concurrent decode calls that expect the default.
 */
int64_t mla_debug_wait_limit(int64_t cycles);

/*
 * The split count that the wave-fill rule of hip_mha_decoding_num_partitions
 * (MLA-style branch) gives for the given constants: ctas = ceil(heads/bm) *
 * batch; one_wave = sm/ctas; two_wave = 2*sm/ctas; pages = ceil(keys/page);
 * work_floor = ceil(pages/max_pages_per_split); np = clamp(work_floor,
 * one_wave, two_wave) rounded up to a power of two, capped by two_wave, by
 * max_splits and by pages; heads <= small_heads uses min(two_wave, pages).
 * The dense planner calls it with GB300 constants; it is exported so the
 * constants of the page it comes from can be checked against that page's
 * printed sweep.
 */
int32_t mla_wave_fill_splits(int32_t batch, int64_t keys_per_request, int32_t heads,
                             int32_t sm_count, int32_t bm, int32_t page,
                             int32_t max_pages_per_split, int32_t max_splits,
                             int32_t small_heads);

#ifdef __cplusplus
}
#endif
#endif /* MLA_DECODE_H */
