// mla_internal.h -- host-side declarations shared by the libmla translation units.
#pragma once
#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/mla_decode.h"

namespace mla {

// Runs a set-up step (a kernel attribute, a symbol lookup: state the runtime
// keeps per device) once for each device that is current when run() is called.
// Thread-safe; a step that fails is tried again on the next call.
class DeviceOnce {
public:
    template <class F>
    cudaError_t run(F&& step)
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        if (done_[dev].load(std::memory_order_acquire)) return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev].load(std::memory_order_relaxed)) return cudaSuccess;
        e = step();
        if (e == cudaSuccess) done_[dev].store(true, std::memory_order_release);
        return e;
    }

private:
    static constexpr int kMaxDevices = 64;
    std::atomic<bool> done_[kMaxDevices]{};
    std::mutex mu_;
};

// Parameters of one split-kernel launch (dense or sparse).
// Largest batch for which the split kernel orders requests longest first.
constexpr int kLongFirstMaxBatch = 256;

struct SplitArgs {
    const uint16_t* q_lat;      // bf16 [rows, H, d_v]  (dense q_lat / sparse q_nope)
    const uint16_t* q_pe;       // bf16 [rows, H, d_rope]
    const uint8_t* pool;        // e4m3fn [pool_rows, d_v + d_rope]
    int64_t pool_rows;
    const int32_t* seq_lens;    // dense: [batch]; sparse: NULL (every token has topk entries)
    const int32_t* kv_indices;  // dense: flat slot list; sparse: [tokens, topk]
    const int32_t* kv_indptr;   // dense: [batch+1]; sparse: NULL (token t starts at t*topk)
    int32_t topk;               // sparse only
    int32_t batch;              // requests (dense) or tokens (sparse)
    int32_t q_len;              // 1 for sparse
    int32_t num_heads;
    int32_t d_v, d_rope;
    int32_t num_splits, rows_per_cta, head_blocks;
    float logit_scale;          // scale * kv_scale * log2(e): raw fp8 dot -> base-2 logit
    float out_scale;            // kv_scale: raw fp8 V units -> output units
    uint16_t* o;                // bf16 [rows, H, d_v]   (written when num_splits == 1)
    float* o_f32;               // fp32 [rows, H, d_v] instead of o, or NULL
    float* lse;                 // fp32 [rows, H] or NULL
    float* o_part;              // fp32 [rows*H, ns, d_v] (num_splits > 1)
    float* lse_part;            // fp32 [rows*H, ns]
    uint32_t* err;              // workspace error word
    int sparse;
    // sparse only: a second (compressed) cache, extra_indices [tokens, extra_topk]
    // into extra_pool [extra_rows, d_v + d_rope]; extra_topk 0 without one
    const uint8_t* extra_pool = nullptr;
    int64_t extra_rows = 0;
    const int32_t* extra_indices = nullptr;
    int32_t extra_topk = 0;
    // dense only: grid slice z takes the z-th longest request (batch at most
    // kLongFirstMaxBatch)
    int32_t long_first = 0;
    // decode context parallelism (dense only): local key i is global position
    // i * cp_world + cp_rank; glen [batch] global lengths, or NULL to use seq_lens
    const int32_t* glen = nullptr;
    int32_t cp_rank = 0;
    int32_t cp_world = 1;
    // fused merge (plan.merge_cluster > 1): per (request x head block, cluster
    // rank) arrival tickets in the workspace header, zero between calls
    uint32_t* tickets = nullptr;
    // phase time stamps (builds with MLA_TRACE only): kTraceSlots per CTA
    unsigned long long* trace = nullptr;
    // cycle bound of the pipeline's waits (mla_debug_wait_limit; the waits that
    // drain copies and MMAs before the CTA exits keep the full bound)
    long long wait_limit = 2000000000ll;
    // tests of the timeout path: the softmax warps first wait on a barrier that
    // nothing completes, so that wait runs out while copies are in flight
    int32_t stall_probe = 0;
};

// The pipeline wait bound that launches use (mla_debug_wait_limit sets it),
// and whether that call armed the unsatisfiable wait of the timeout tests.
long long pipeline_wait_limit();
bool stall_probe_armed();

// Phase stamps of a traced build (compiled with -DMLA_TRACE): per CTA of the
// split kernel, globaltimer nanoseconds at kTraceSlots points, for at most
// kTraceCtas CTAs (linear CTA index x + grid_x (y + grid_y z)).
constexpr int kTraceSlots = 12;
constexpr int kTraceCtas = 8192;
// ... followed by per-block events of the first kTraceBlockCtas CTAs.
constexpr int kTraceBlockCtas = 4;
constexpr int kTraceBlocks = 64;
constexpr int kTraceBlockEvents = 8;
constexpr int kTraceWords =
    kTraceCtas * kTraceSlots + kTraceBlockCtas * kTraceBlocks * kTraceBlockEvents;

// Merge-ticket counters in the workspace header: after the 256-byte error-word
// area, one uint32 per (tile, cluster rank) of a fused-merge launch.
constexpr int64_t kErrorAreaBytes = 256;
constexpr int64_t kMaxTickets = (MLA_WORKSPACE_HEADER_BYTES - kErrorAreaBytes) / 4;
// Largest number of (row, cluster) partials one CTA of the last cluster merges
// from the workspace in a fused merge (its slice rows x the tile's clusters).
constexpr int kMaxMergeTerms = 32;

// Kernel variants (mla_plan_t::variant).  Value 1 belonged to a CUDA-core
// bring-up kernel that the tcgen05 kernel replaced; it is rejected.
enum Variant : int32_t {
    kVariantTc = 2,   // tcgen05 + TMA split kernel, then the split-K reduce kernel
};

// The split kernel; mc > 1 fuses the split-K merge (clusters of mc splits).
cudaError_t launch_split_tc(const SplitArgs& a, const mla_plan_t& plan, int mc,
                            cudaStream_t stream);

// Workspace bytes that a plan needs, recomputed from its shape and split count.
int64_t needed_workspace(const mla_plan_t* plan);

// 2-D uint8 tensor map of the pool (row_bytes columns x rows) with one-row
// boxes of `box` columns (the shape tile::gather4 reads); false on failure.
bool make_row_map(CUtensorMap* m, const void* pool, int64_t rows, int row_bytes, int box,
                  CUtensorMapSwizzle sw);

// Merge of decode-context-parallel ranks' bf16 shares (mla_dcp_lse_merge_ranks).
cudaError_t launch_dcp_merge(const void* parts, bool parts_f32, const float* lse_in,
                             int32_t world, int64_t rows, int32_t d_v, uint16_t* o, float* lse,
                             cudaStream_t stream);

// Gather probe (mla_debug_gather).
cudaError_t launch_gather_probe(const void* pool, int64_t pool_rows, int32_t row_bytes,
                                const int32_t* indices, int64_t n, uint8_t* out, uint32_t* err,
                                cudaStream_t stream);
// Split-K reduce; writes o as bf16, or as fp32 when out_f32.
cudaError_t launch_splitk_reduce(const float* o_part, const float* lse_part, int64_t rows,
                                 int32_t num_splits, int32_t d_v, float out_scale, void* o,
                                 bool out_f32, float* lse, cudaStream_t stream);

}  // namespace mla
