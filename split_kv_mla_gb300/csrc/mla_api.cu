// mla_api.cu -- the extern "C" boundary of libmla: planning, argument checks,
// kernel dispatch and the workspace error word.  See include/mla_decode.h for
// the contract of every entry point.
#include <cmath>
#include <cstring>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kDenseDv = 512, kDenseDr = 64;
constexpr int kSparseDv = 448, kSparseDr = 64;
constexpr int kMaxHeads = 128;
constexpr int32_t kMaxBatch = 65535;   // requests (tokens) are the split grid's z dimension
constexpr float kLog2e = 1.4426950408889634f;

// Split-kernel geometry: 128 keys per block; 16 query rows per CTA when a
// request has at most 16 (heads x draft positions); above that 32, or 16 where
// the planners find the smaller tile faster (short work per CTA, below).
constexpr int kBlockN = 128;

inline int32_t rows_per_cta_for(int64_t rows) { return rows <= 16 ? 16 : 32; }

// A plan's rows per CTA: 16 for any row count, 32 only above 16 rows.
inline bool rows_per_cta_ok(int64_t rows, int32_t rpc)
{
    return rpc == 16 || (rpc == 32 && rows > 16);
}

// GB300 split rule (the wave-fill idea of hip_mha_decoding_num_partitions,
// re-derived for this kernel: one resident CTA per SM, 128-key blocks).  A
// small cost model in microseconds picks the split count.  Each wave of CTAs
// costs its blocks per CTA times the slower of the block's latency-bound time
// and the wave's share of the GPU-wide gather rate, plus a fixed time per CTA;
// several splits add the reduce (a launch and the fp32 partial traffic).  The
// constants come from phase traces and split sweeps of this kernel on GB300.
constexpr double kBlockUs16 = 2.1;     // a 128-key block, 16 query rows per CTA (latency-bound)
constexpr double kBlockUs32 = 2.2;     // ... 32 query rows per CTA
constexpr double kGather32 = 5.0e6;    // bytes/us gathered GPU-wide by 32-row CTAs (a
                                       // request's head blocks gather the same rows); 16-row
                                       // CTAs measured no GPU-wide cap up to a full wave
constexpr double kCtaUs = 6.0;         // start-up to the first QK, and the epilogue
constexpr double kFirstBlockUs32 = 5.0;  // a 32-row CTA's extra start-up over a 16-row one
                                         // (its query tile and first softmax): CTAs of one
                                         // block took 4.9-5.2 us longer at 32 rows than at
                                         // 16 (H=64, S=256..4096)
constexpr double kReduceUs = 3.0;      // reduce launch and its latency chain
constexpr double kBytesPerUs = 6.8e6;  // HBM bytes per microsecond

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t align_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// CTAs resident at once, one per SM, in clusters of `mc` (GB300, measured with
// cudaOccupancyMaxActiveClusters at this kernel's shared memory: clusters of 2
// fill all 152 SMs, clusters of 4 leave 8 idle).
int64_t wave_ctas(int32_t sm_count, int32_t mc = 1)
{
    return mc >= 4 ? (int64_t)sm_count - sm_count / 19 : sm_count;
}

// Whether clusters of `mc` splits can fuse the merge of a plan: the split count
// divides into clusters, every (tile, rank) has a ticket, and a CTA of the last
// cluster merges at most kMaxMergeTerms (row, cluster) partials.
bool fused_merge_ok(int64_t tiles, int32_t ns, int32_t rows_per_cta, int32_t mc)
{
    if (mc != 2 && mc != 4) return false;
    if (ns < mc || ns % mc != 0 || rows_per_cta % mc != 0) return false;
    if (tiles * mc > kMaxTickets) return false;
    const int64_t nclus = ns / mc;
    return nclus == 1 || nclus * (rows_per_cta / mc) <= kMaxMergeTerms;
}

int device_ok()
{
    static int cached[64];  // 0 unknown, 1 ok, 2 not ok
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return MLA_ERR_UNSUPPORTED_DEVICE;
    if (cached[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return MLA_ERR_CUDA;
        cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    return cached[dev] == 1 ? MLA_OK : MLA_ERR_UNSUPPORTED_DEVICE;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t workspace_for(int64_t items, int ns, int d_v)
{
    int64_t bytes = MLA_WORKSPACE_HEADER_BYTES;
    if (ns > 1) {
        bytes += align_up(items * ns * (int64_t)d_v * 4, 256);
        bytes += align_up(items * ns * 4, 256);
    }
    return bytes;
}

// The merge cluster size the planner uses: 1, the separate reduce (see
// gb300_splits); callers may opt into the fused merge by setting the plan's
// merge_cluster to a size that fits.
int32_t planned_merge_cluster(int64_t, int32_t, int32_t) { return 1; }

struct SplitChoice {
    int32_t ns, mc;
    double us;   // the cost model's time of the call
};

// Split count and merge cluster size for `tiles` (request, head block) tiles
// of `rows_per_cta` rows, `keys` keys per request of `row_bytes`-byte rows and
// `items` output rows (row x head) in the call: the cheapest by the cost
// model, over every split count with the separate reduce and the fused merge
// where one cluster holds a tile's splits.
SplitChoice gb300_splits(int64_t tiles, int64_t keys, int64_t items, int32_t d_v,
                         int32_t row_bytes, int32_t sm_count, int32_t rows_per_cta)
{
    const int64_t blocks = ceil_div(keys > 0 ? keys : 1, kBlockN);
    const int64_t ctas1 = tiles > 0 ? tiles : 1;
    const int64_t max_ns = blocks < MLA_MAX_SPLITS ? blocks : MLA_MAX_SPLITS;
    const double block_us = rows_per_cta == 16 ? kBlockUs16 : kBlockUs32;
    const double us_per_cta_block =
        rows_per_cta == 16 ? 0.0 : (double)kBlockN * row_bytes / kGather32;
    const double cta_us = kCtaUs + (rows_per_cta == 16 ? 0.0 : kFirstBlockUs32);
    double best = 0.0;
    SplitChoice pick{1, 1, 0.0};
    auto consider = [&](int64_t ns, int32_t mc) {
        const int64_t ctas = ctas1 * ns;
        const int64_t wave = wave_ctas(sm_count, mc);
        const double bpc = (double)ceil_div(blocks, ns);
        auto wave_us = [&](int64_t active) {
            const double b = (double)active * us_per_cta_block;
            return bpc * (b > block_us ? b : block_us) + cta_us;
        };
        double t = (double)(ctas / wave) * wave_us(wave);
        if (ctas % wave != 0) t += wave_us(ctas % wave);
        if (ns > 1 && mc == 1) t += kReduceUs + (double)items * ns * d_v * 4.0 * 2.0 / kBytesPerUs;
        if ((pick.ns == 1 && pick.mc == 1 && ns == 1) || t < best - 1e-9) {
            best = t;
            pick = SplitChoice{(int32_t)ns, mc, t};
        }
    };
    // The fused merge is not a candidate: measured on GB300 it never beat the
    // reduce kernel (tiles of several clusters: c1 21.3 vs 19.5 us; one
    // cluster per tile: B=1 S=256 11.4 vs 10.2 us, sparse 24 tokens equal).
    for (int64_t ns = 1; ns <= max_ns; ++ns) consider(ns, 1);
    return pick;
}

// Sparse split rule, after flashinfer.mla.cake_sparse_mla_sm120_dsv4_nvfp4_plan_splits
// ("Measured split rules") with this kernel's geometry: a chunk is 64
// candidates and a CTA should keep at least one 128-key block (two chunks).
// The page splits only grids that cover at most 40 % of the SMs, and by powers
// of two up to 80 % of them.  Re-derived on GB300: while the unsplit grid is
// below one wave, take the largest split that keeps the grid within the SM
// count and two chunks per CTA (64 heads, top-k 2048: 24 tokens 27.7 us at 3
// splits against 31.4 at 2; 32 tokens 32.3 us at 2 against 42.8 unsplit; 12
// tokens 20.0 at 6 against 21.2 at 4); on a full grid, split 16-chunk work in
// two when the doubled grid ends in a wave at least half full; otherwise run
// unsplit.
int32_t sparse_splits(int64_t ctas, int64_t topk, int32_t sm_count)
{
    const int64_t chunks = ceil_div(topk > 0 ? topk : 1, 64);
    if (chunks <= 2) return 1;
    if (ctas < sm_count) {
        int64_t ns = (int64_t)sm_count / (ctas > 0 ? ctas : 1);
        if (ns > chunks / 2) ns = chunks / 2;
        if (ns < 1) ns = 1;
        return (int32_t)(ns < MLA_MAX_SPLITS ? ns : MLA_MAX_SPLITS);
    }
    if (chunks == 16) {
        const int64_t tail = (2 * ctas) % sm_count;
        if (tail == 0 || tail * 2 >= sm_count) return 2;
    }
    return 1;
}

void fill_plan(mla_plan_t* p, int32_t batch, int32_t q_len, int32_t heads, int32_t d_v,
               int32_t d_rope, int32_t sm_count, int64_t total_keys, int32_t ns, int32_t mc,
               int32_t rpc)
{
    const int32_t rows = q_len * heads;
    std::memset(p, 0, sizeof *p);
    p->num_splits = ns;
    p->rows_per_cta = rpc;
    p->block_n = kBlockN;
    p->head_blocks = (int32_t)ceil_div(rows, p->rows_per_cta);
    p->grid_x = p->head_blocks;
    p->grid_y = ns;
    p->grid_z = batch;
    p->variant = kVariantTc;
    p->workspace_bytes = workspace_for((int64_t)batch * rows, ns, d_v);
    p->batch = batch;
    p->q_len = q_len;
    p->num_heads = heads;
    p->d_v = d_v;
    p->d_rope = d_rope;
    p->sm_count = sm_count;
    p->total_keys = total_keys;
    p->kv_share = 1;
    p->merge_cluster = mc;
}

}  // namespace

// The bound of the split kernel's pipeline waits, in SM cycles (about a second
// by default; mla_debug_wait_limit lowers it for tests of the timeout path).
constexpr long long kDefaultWaitLimit = 2000000000ll;
static std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
long long pipeline_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }
bool stall_probe_armed() { return pipeline_wait_limit() != kDefaultWaitLimit; }

// The workspace bytes a plan needs, from its shape and split count (the plan's
// own workspace_bytes field is only a copy of this, and is checked against it).
int64_t needed_workspace(const mla_plan_t* plan)
{
    return workspace_for((int64_t)plan->batch * plan->q_len * plan->num_heads,
                         plan->num_splits, plan->d_v);
}

namespace {

int check_workspace(const mla_plan_t* plan, const void* ws, int64_t bytes)
{
    if (!ws) return MLA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MLA_ERR_MISALIGNED;
    if (plan->workspace_bytes != needed_workspace(plan)) return MLA_ERR_INVALID_ARG;
    if (bytes < plan->workspace_bytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
    return MLA_OK;
}

void carve(const mla_plan_t* plan, void* ws, int64_t items, SplitArgs* a)
{
    char* base = static_cast<char*>(ws);
    a->err = reinterpret_cast<uint32_t*>(base);
    if (plan->num_splits > 1) {
        const int64_t obytes = align_up(items * plan->num_splits * (int64_t)plan->d_v * 4, 256);
        a->o_part = reinterpret_cast<float*>(base + MLA_WORKSPACE_HEADER_BYTES);
        a->lse_part = reinterpret_cast<float*>(base + MLA_WORKSPACE_HEADER_BYTES + obytes);
    } else {
        a->o_part = nullptr;
        a->lse_part = nullptr;
    }
}

// A plan's launch geometry must follow from its shape, its tile (16 rows per
// CTA, or 32 above 16 rows) and its split count: the kernels index the
// workspace and the outputs by it.
bool variant_ok(const mla_plan_t* plan)
{
    if (plan->variant != kVariantTc) return false;
    if (plan->q_len < 1 || plan->num_heads < 1 || plan->batch < 0) return false;
    if (plan->batch > kMaxBatch) return false;
    const int64_t rows = (int64_t)plan->q_len * plan->num_heads;
    if (rows > (1 << 20)) return false;
    if (!rows_per_cta_ok(rows, plan->rows_per_cta) || plan->block_n != kBlockN ||
        plan->head_blocks != ceil_div(rows, plan->rows_per_cta) ||
        plan->grid_x != plan->head_blocks || plan->grid_y != plan->num_splits ||
        plan->grid_z != plan->batch)
        return false;
    if (plan->merge_cluster != 1 &&
        !fused_merge_ok((int64_t)plan->batch * plan->head_blocks, plan->num_splits,
                        plan->rows_per_cta, plan->merge_cluster))
        return false;
    if (plan->long_first != 0 && (plan->long_first != 1 || plan->batch > kLongFirstMaxBatch))
        return false;
    return plan->kv_share == 1;
}

// The split kernel, then the split-K reduce when the plan has several splits
// and does not fuse the merge.  Without the reduce (the *_splits entry points)
// the kernel leaves every split's partial in the workspace.
int run(const mla_plan_t* plan, SplitArgs& a, int64_t items, cudaStream_t stream,
        bool with_reduce)
{
    a.wait_limit = pipeline_wait_limit();
    a.stall_probe = stall_probe_armed() ? 1 : 0;
    const int mc = with_reduce ? plan->merge_cluster : 1;
    a.tickets = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(a.err) + kErrorAreaBytes);
    cudaError_t e = launch_split_tc(a, *plan, mc, stream);
    if (e != cudaSuccess) return MLA_ERR_LAUNCH_FAILED;
    if (with_reduce && mc == 1 && plan->num_splits > 1) {
        void* out = a.o_f32 ? static_cast<void*>(a.o_f32) : static_cast<void*>(a.o);
        e = launch_splitk_reduce(a.o_part, a.lse_part, items, plan->num_splits, plan->d_v,
                                 a.out_scale, out, a.o_f32 != nullptr, a.lse, stream);
        if (e != cudaSuccess) return MLA_ERR_LAUNCH_FAILED;
    }
    return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int32_t mla_wave_fill_splits(int32_t batch, int64_t keys_per_request, int32_t heads,
                             int32_t sm_count, int32_t bm, int32_t page,
                             int32_t max_pages_per_split, int32_t max_splits,
                             int32_t small_heads)
{
    if (batch <= 0 || heads <= 0 || sm_count <= 0 || bm <= 0 || page <= 0 ||
        max_pages_per_split <= 0 || max_splits <= 0)
        return 1;
    const int64_t ctas = ceil_div(heads, bm) * batch;
    const int64_t one_wave = sm_count / ctas;
    const int64_t two_wave = 2LL * sm_count / ctas;
    const int64_t pages = ceil_div(keys_per_request > 0 ? keys_per_request : 1, page);
    int64_t np;
    if (heads <= small_heads) {
        np = two_wave < pages ? two_wave : pages;
    } else {
        const int64_t work_floor = ceil_div(pages, max_pages_per_split);
        np = work_floor < one_wave ? one_wave : work_floor;
        if (np > two_wave) np = two_wave;
        int64_t p2 = 1;
        while (p2 < np) p2 <<= 1;
        np = p2 < two_wave ? p2 : two_wave;
    }
    if (np > max_splits) np = max_splits;
    if (np > pages) np = pages;
    if (np < 1) np = 1;
    return (int32_t)np;
}

int mla_decode_plan(int32_t batch, int32_t q_len, int32_t num_heads, int64_t total_keys,
                    int32_t d_v, int32_t d_rope, int32_t sm_count, mla_plan_t* out)
{
    if (!out || batch < 0 || q_len < 1 || total_keys < 0 || sm_count < 1)
        return MLA_ERR_INVALID_ARG;
    if (d_v != kDenseDv || d_rope != kDenseDr || num_heads < 1 || num_heads > kMaxHeads ||
        batch > kMaxBatch)
        return MLA_ERR_UNSUPPORTED_SHAPE;
    const int64_t rows = (int64_t)q_len * num_heads;
    if (rows > (1 << 20)) return MLA_ERR_UNSUPPORTED_SHAPE;
    const int64_t keys = batch > 0 ? ceil_div(total_keys, batch) : 0;
    auto choose = [&](int32_t rpc) {
        return gb300_splits(ceil_div(rows, rpc) * (batch > 0 ? batch : 1), keys,
                            (int64_t)batch * rows, d_v, d_v + d_rope, sm_count, rpc);
    };
    // Above 16 rows, the 32-row tile against the 16-row one (twice the head
    // blocks, each gathering the same rows): the smaller tile wins where a
    // CTA's work is short, since a 32-row CTA starts about 5 us later (a cost
    // the model charges each wave of 32-row CTAs).
    int32_t rpc = rows_per_cta_for(rows);
    SplitChoice ch = choose(rpc);
    if (rpc == 32) {
        const SplitChoice ch16 = choose(16);
        if (ch16.us < ch.us) {
            rpc = 16;
            ch = ch16;
        }
    }
    fill_plan(out, batch, q_len, num_heads, d_v, d_rope, sm_count, total_keys, ch.ns, ch.mc,
              rpc);
    // Longest requests first once the grid outlasts one wave (variable lengths
    // then leave the short requests for the last wave).
    const int64_t ctas = (int64_t)out->grid_x * out->grid_y * out->grid_z;
    out->long_first = (batch >= 2 && batch <= kLongFirstMaxBatch &&
                       ctas > wave_ctas(sm_count, ch.mc)) ? 1 : 0;
    return MLA_OK;
}

int mla_sparse_decode_plan(int32_t num_tokens, int32_t num_heads, int32_t topk,
                           int32_t extra_topk, int32_t d_v, int32_t d_rope, int32_t sm_count,
                           int32_t max_splits, mla_plan_t* out)
{
    if (!out || num_tokens < 0 || topk < 0 || extra_topk < 0 || sm_count < 1 || max_splits < 0)
        return MLA_ERR_INVALID_ARG;
    if ((int64_t)topk + extra_topk + 3 > (1LL << 30)) return MLA_ERR_UNSUPPORTED_SHAPE;
    if (d_v != kSparseDv || d_rope != kSparseDr || num_heads < 1 || num_heads > kMaxHeads ||
        num_tokens > kMaxBatch)
        return MLA_ERR_UNSUPPORTED_SHAPE;
    const int32_t cap = max_splits == 0 ? MLA_MAX_SPLITS
                                        : (max_splits < MLA_MAX_SPLITS ? max_splits : MLA_MAX_SPLITS);
    const int64_t keys = (int64_t)topk + extra_topk;
    auto splits_for = [&](int32_t rpc) {
        const int32_t ns = sparse_splits(ceil_div(num_heads, rpc) * (num_tokens > 0 ? num_tokens : 1),
                                         keys, sm_count);
        return ns > cap ? cap : ns;
    };
    // Above 16 heads, 16-row CTAs (twice the head blocks) where the 32-row
    // split would leave each CTA at most two 128-key blocks: a 32-row CTA
    // starts about 5 us later, which short work cannot amortise.  Measured on
    // GB300 (64 heads, top-k 2048): T=1 14.1 -> 10.5 us, T=4 16.4 -> 11.6, T=8
    // 16.4 -> 15.5; at T=16 (four blocks per 32-row CTA) 32 rows stay faster.
    int32_t rpc = rows_per_cta_for(num_heads);
    int32_t ns = splits_for(rpc);
    if (rpc == 32 && ceil_div(ceil_div(keys > 0 ? keys : 1, ns), kBlockN) <= 2) {
        rpc = 16;
        ns = splits_for(16);
    }
    const int64_t head_blocks = ceil_div(num_heads, rpc);
    fill_plan(out, num_tokens, 1, num_heads, d_v, d_rope, sm_count,
              (int64_t)num_tokens * keys, ns,
              planned_merge_cluster(head_blocks * num_tokens, ns, rpc), rpc);
    out->extra_topk = extra_topk;
    return MLA_OK;
}

static int dense_call(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                      const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                      const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                      int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                      void* o_lat, float* lse, void* workspace, int64_t workspace_bytes,
                      void* stream, bool with_reduce, const int32_t* glen = nullptr,
                      int32_t cp_rank = 0, int32_t cp_world = 1, bool o_f32 = false)
{
    if (!plan) return MLA_ERR_INVALID_ARG;
    if (cp_world < 1 || cp_world > MLA_MAX_SPLITS || cp_rank < 0 || cp_rank >= cp_world)
        return MLA_ERR_INVALID_ARG;
    if (plan->batch != batch || plan->q_len != q_len || plan->num_heads != num_heads ||
        plan->d_v != kDenseDv || plan->d_rope != kDenseDr ||
        !variant_ok(plan) ||
        plan->num_splits < 1 || plan->num_splits > MLA_MAX_SPLITS)
        return MLA_ERR_INVALID_ARG;
    if (batch == 0) return MLA_OK;
    if (!q_lat || !q_pe || !pool || !seq_lens || !kv_indptr || !o_lat || pool_rows < 1)
        return MLA_ERR_INVALID_ARG;
    if (cp_world > 1 && (!glen || !lse)) return MLA_ERR_INVALID_ARG;
    if (plan->total_keys > 0 && !kv_indices) return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned16(pool) || !aligned16(o_lat))
        return MLA_ERR_MISALIGNED;
    if (!std::isfinite(scale) || !std::isfinite(kv_scale)) return MLA_ERR_INVALID_ARG;
    int rc = check_workspace(plan, workspace, workspace_bytes);
    if (rc != MLA_OK) return rc;
    rc = device_ok();
    if (rc != MLA_OK) return rc;

    SplitArgs a{};
    a.q_lat = static_cast<const uint16_t*>(q_lat);
    a.q_pe = static_cast<const uint16_t*>(q_pe);
    a.pool = static_cast<const uint8_t*>(pool);
    a.pool_rows = pool_rows;
    a.seq_lens = seq_lens;
    a.kv_indices = kv_indices;
    a.kv_indptr = kv_indptr;
    a.topk = 0;
    a.batch = batch;
    a.q_len = q_len;
    a.num_heads = num_heads;
    a.d_v = kDenseDv;
    a.d_rope = kDenseDr;
    a.num_splits = plan->num_splits;
    a.rows_per_cta = plan->rows_per_cta;
    a.head_blocks = plan->head_blocks;
    a.logit_scale = scale * kv_scale * kLog2e;
    a.out_scale = kv_scale;
    a.o = o_f32 ? nullptr : static_cast<uint16_t*>(o_lat);
    a.o_f32 = o_f32 ? static_cast<float*>(o_lat) : nullptr;
    a.lse = lse;
    a.sparse = 0;
    a.glen = glen;
    a.cp_rank = cp_rank;
    a.cp_world = cp_world;
    a.long_first = plan->long_first;
    const int64_t items = (int64_t)batch * q_len * num_heads;
    carve(plan, workspace, items, &a);
    return run(plan, a, items, static_cast<cudaStream_t>(stream), with_reduce);
}

static int sparse_call(const mla_plan_t* plan, const void* q_nope, const void* q_pe,
                       const void* pool, int64_t pool_rows, const int32_t* indices,
                       int32_t num_tokens, int32_t num_heads, int32_t topk, float scale,
                       float kv_scale, void* o, float* lse, void* workspace,
                       int64_t workspace_bytes, void* stream, bool with_reduce,
                       const void* extra_pool = nullptr, int64_t extra_rows = 0,
                       const int32_t* extra_indices = nullptr, int32_t extra_topk = 0)
{
    if (!plan) return MLA_ERR_INVALID_ARG;
    if (topk < 0 || extra_topk < 0) return MLA_ERR_INVALID_ARG;
    if (plan->batch != num_tokens || plan->q_len != 1 || plan->num_heads != num_heads ||
        plan->d_v != kSparseDv || plan->d_rope != kSparseDr ||
        !variant_ok(plan) || plan->extra_topk != extra_topk || plan->long_first != 0 ||
        plan->total_keys != (int64_t)num_tokens * ((int64_t)topk + extra_topk) ||
        plan->num_splits < 1 || plan->num_splits > MLA_MAX_SPLITS)
        return MLA_ERR_INVALID_ARG;
    if (num_tokens == 0) return MLA_OK;
    if (!q_nope || !q_pe || !pool || !o || pool_rows < 1) return MLA_ERR_INVALID_ARG;
    if (topk > 0 && !indices) return MLA_ERR_INVALID_ARG;
    if (extra_topk > 0 && (!extra_pool || !extra_indices || extra_rows < 1))
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(pool) || !aligned16(o) ||
        (extra_topk > 0 && !aligned16(extra_pool)))
        return MLA_ERR_MISALIGNED;
    if (!std::isfinite(scale) || !std::isfinite(kv_scale)) return MLA_ERR_INVALID_ARG;
    int rc = check_workspace(plan, workspace, workspace_bytes);
    if (rc != MLA_OK) return rc;
    rc = device_ok();
    if (rc != MLA_OK) return rc;

    SplitArgs a{};
    a.q_lat = static_cast<const uint16_t*>(q_nope);
    a.q_pe = static_cast<const uint16_t*>(q_pe);
    a.pool = static_cast<const uint8_t*>(pool);
    a.pool_rows = pool_rows;
    a.seq_lens = nullptr;
    a.kv_indices = indices;
    a.kv_indptr = nullptr;
    a.topk = topk;
    a.batch = num_tokens;
    a.q_len = 1;
    a.num_heads = num_heads;
    a.d_v = kSparseDv;
    a.d_rope = kSparseDr;
    a.num_splits = plan->num_splits;
    a.rows_per_cta = plan->rows_per_cta;
    a.head_blocks = plan->head_blocks;
    a.logit_scale = scale * kv_scale * kLog2e;
    a.out_scale = kv_scale;
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.sparse = 1;
    if (extra_topk > 0) {
        a.extra_pool = static_cast<const uint8_t*>(extra_pool);
        a.extra_rows = extra_rows;
        a.extra_indices = extra_indices;
        a.extra_topk = extra_topk;
    }
    const int64_t items = (int64_t)num_tokens * num_heads;
    carve(plan, workspace, items, &a);
    return run(plan, a, items, static_cast<cudaStream_t>(stream), with_reduce);
}

int mla_decode(const mla_plan_t* plan, const void* q_lat, const void* q_pe, const void* pool,
               int64_t pool_rows, const int32_t* seq_lens, const int32_t* kv_indices,
               const int32_t* kv_indptr, int32_t batch, int32_t q_len, int32_t num_heads,
               float scale, float kv_scale, void* o_lat, float* lse, void* workspace,
               int64_t workspace_bytes, void* stream)
{
    return dense_call(plan, q_lat, q_pe, pool, pool_rows, seq_lens, kv_indices, kv_indptr,
                      batch, q_len, num_heads, scale, kv_scale, o_lat, lse, workspace,
                      workspace_bytes, stream, true);
}

int mla_decode_splits(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                      const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                      const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                      int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                      void* o_lat, float* lse, void* workspace, int64_t workspace_bytes,
                      void* stream)
{
    return dense_call(plan, q_lat, q_pe, pool, pool_rows, seq_lens, kv_indices, kv_indptr,
                      batch, q_len, num_heads, scale, kv_scale, o_lat, lse, workspace,
                      workspace_bytes, stream, false);
}

int mla_decode_dcp(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                   const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                   const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                   int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                   const int32_t* glen, int32_t cp_rank, int32_t cp_world, int32_t o_dtype,
                   void* o, float* lse, void* workspace, int64_t workspace_bytes, void* stream)
{
    if (o_dtype != MLA_DTYPE_BF16 && o_dtype != MLA_DTYPE_F32) return MLA_ERR_INVALID_ARG;
    return dense_call(plan, q_lat, q_pe, pool, pool_rows, seq_lens, kv_indices, kv_indptr,
                      batch, q_len, num_heads, scale, kv_scale, o, lse, workspace,
                      workspace_bytes, stream, true, glen, cp_rank, cp_world,
                      o_dtype == MLA_DTYPE_F32);
}

int mla_decode_dcp_splits(const mla_plan_t* plan, const void* q_lat, const void* q_pe,
                          const void* pool, int64_t pool_rows, const int32_t* seq_lens,
                          const int32_t* kv_indices, const int32_t* kv_indptr, int32_t batch,
                          int32_t q_len, int32_t num_heads, float scale, float kv_scale,
                          const int32_t* glen, int32_t cp_rank, int32_t cp_world,
                          int32_t o_dtype, void* o, float* lse, void* workspace,
                          int64_t workspace_bytes, void* stream)
{
    if (o_dtype != MLA_DTYPE_BF16 && o_dtype != MLA_DTYPE_F32) return MLA_ERR_INVALID_ARG;
    return dense_call(plan, q_lat, q_pe, pool, pool_rows, seq_lens, kv_indices, kv_indptr,
                      batch, q_len, num_heads, scale, kv_scale, o, lse, workspace,
                      workspace_bytes, stream, false, glen, cp_rank, cp_world,
                      o_dtype == MLA_DTYPE_F32);
}

int mla_dcp_lse_merge_ranks(const void* parts_in, int32_t parts_dtype, const float* lse_in,
                            int32_t cp_world, int64_t rows, int32_t d_v, void* out,
                            float* lse_out, void* stream)
{
    if (rows < 0 || cp_world < 1 || cp_world > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
    if (parts_dtype != MLA_DTYPE_BF16 && parts_dtype != MLA_DTYPE_F32) return MLA_ERR_INVALID_ARG;
    if (d_v < 8 || (d_v % 8) != 0 || d_v > 4 * 128) return MLA_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MLA_OK;
    if (!parts_in || !lse_in || !out) return MLA_ERR_INVALID_ARG;
    if (!aligned16(parts_in) || !aligned16(out)) return MLA_ERR_MISALIGNED;
    int rc = device_ok();
    if (rc != MLA_OK) return rc;
    cudaError_t e = launch_dcp_merge(parts_in, parts_dtype == MLA_DTYPE_F32, lse_in, cp_world,
                                     rows, d_v, static_cast<uint16_t*>(out), lse_out,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH_FAILED;
}

int mla_sparse_decode(const mla_plan_t* plan, const void* q_nope, const void* q_pe,
                      const void* pool, int64_t pool_rows, const int32_t* indices,
                      int32_t num_tokens, int32_t num_heads, int32_t topk, float scale,
                      float kv_scale, void* o, float* lse, void* workspace,
                      int64_t workspace_bytes, void* stream)
{
    return sparse_call(plan, q_nope, q_pe, pool, pool_rows, indices, num_tokens, num_heads,
                       topk, scale, kv_scale, o, lse, workspace, workspace_bytes, stream, true);
}

int mla_sparse_decode_extra(const mla_plan_t* plan, const void* q_nope, const void* q_pe,
                            const void* pool, int64_t pool_rows, const int32_t* indices,
                            const void* extra_pool, int64_t extra_rows,
                            const int32_t* extra_indices, int32_t num_tokens, int32_t num_heads,
                            int32_t topk, int32_t extra_topk, float scale, float kv_scale,
                            void* o, float* lse, void* workspace, int64_t workspace_bytes,
                            void* stream)
{
    return sparse_call(plan, q_nope, q_pe, pool, pool_rows, indices, num_tokens, num_heads,
                       topk, scale, kv_scale, o, lse, workspace, workspace_bytes, stream, true,
                       extra_pool, extra_rows, extra_indices, extra_topk);
}

int mla_sparse_decode_extra_splits(const mla_plan_t* plan, const void* q_nope,
                                   const void* q_pe, const void* pool, int64_t pool_rows,
                                   const int32_t* indices, const void* extra_pool,
                                   int64_t extra_rows, const int32_t* extra_indices,
                                   int32_t num_tokens, int32_t num_heads, int32_t topk,
                                   int32_t extra_topk, float scale, float kv_scale, void* o,
                                   float* lse, void* workspace, int64_t workspace_bytes,
                                   void* stream)
{
    return sparse_call(plan, q_nope, q_pe, pool, pool_rows, indices, num_tokens, num_heads,
                       topk, scale, kv_scale, o, lse, workspace, workspace_bytes, stream, false,
                       extra_pool, extra_rows, extra_indices, extra_topk);
}

int mla_sparse_decode_splits(const mla_plan_t* plan, const void* q_nope, const void* q_pe,
                             const void* pool, int64_t pool_rows, const int32_t* indices,
                             int32_t num_tokens, int32_t num_heads, int32_t topk, float scale,
                             float kv_scale, void* o, float* lse, void* workspace,
                             int64_t workspace_bytes, void* stream)
{
    return sparse_call(plan, q_nope, q_pe, pool, pool_rows, indices, num_tokens, num_heads,
                       topk, scale, kv_scale, o, lse, workspace, workspace_bytes, stream, false);
}

int mla_workspace_partials(const mla_plan_t* plan, void* workspace, float** o_part,
                           float** lse_part)
{
    if (!plan || !workspace || !o_part || !lse_part) return MLA_ERR_INVALID_ARG;
    SplitArgs a{};
    carve(plan, workspace, (int64_t)plan->batch * plan->q_len * plan->num_heads, &a);
    *o_part = a.o_part;
    *lse_part = a.lse_part;
    return MLA_OK;
}

int mla_splitk_reduce(const float* o_part, const float* lse_part, int64_t rows,
                      int32_t num_splits, int32_t d_v, float out_scale, void* o, float* lse,
                      void* stream)
{
    if (rows < 0 || num_splits < 1 || num_splits > MLA_MAX_SPLITS || d_v < 8 || (d_v % 8) != 0 ||
        d_v > 4 * 128)
        return rows < 0 || num_splits < 1 ? MLA_ERR_INVALID_ARG : MLA_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return MLA_OK;
    if (!o_part || !lse_part || !o) return MLA_ERR_INVALID_ARG;
    if (!aligned16(o_part) || !aligned16(o)) return MLA_ERR_MISALIGNED;
    if (!std::isfinite(out_scale)) return MLA_ERR_INVALID_ARG;
    int rc = device_ok();
    if (rc != MLA_OK) return rc;
    cudaError_t e = launch_splitk_reduce(o_part, lse_part, rows, num_splits, d_v, out_scale, o,
                                         false, lse, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH_FAILED;
}

int mla_plan_force_splits(mla_plan_t* plan, int32_t num_splits)
{
    if (!plan || num_splits < 1 || num_splits > MLA_MAX_SPLITS) return MLA_ERR_INVALID_ARG;
    if (plan->q_len < 1 || plan->num_heads < 1 || plan->batch < 0) return MLA_ERR_INVALID_ARG;
    plan->num_splits = num_splits;
    plan->grid_y = num_splits;
    plan->merge_cluster = planned_merge_cluster((int64_t)plan->batch * plan->head_blocks,
                                                num_splits, plan->rows_per_cta);
    plan->workspace_bytes = workspace_for((int64_t)plan->batch * plan->q_len * plan->num_heads,
                                          num_splits, plan->d_v);
    return MLA_OK;
}

int mla_workspace_reset(void* workspace, void* stream)
{
    if (!workspace) return MLA_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(workspace, 0, MLA_WORKSPACE_HEADER_BYTES,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_read_device_error(const void* workspace, int32_t* code, void* stream)
{
    if (!workspace || !code) return MLA_ERR_INVALID_ARG;
    uint32_t v = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
    *code = (int32_t)v;
    return MLA_OK;
}

int mla_debug_gather(const void* pool, int64_t pool_rows, int32_t row_bytes,
                     const int32_t* indices, int64_t n, void* out, void* workspace, void* stream)
{
    if (n < 0 || pool_rows < 1 || (row_bytes != 576 && row_bytes != 512))
        return row_bytes != 576 && row_bytes != 512 ? MLA_ERR_UNSUPPORTED_SHAPE : MLA_ERR_INVALID_ARG;
    if (n == 0) return MLA_OK;
    if (!pool || !indices || !out || !workspace) return MLA_ERR_INVALID_ARG;
    if (!aligned16(pool) || !aligned16(out)) return MLA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MLA_ERR_MISALIGNED;
    int rc = device_ok();
    if (rc != MLA_OK) return rc;
    cudaError_t e = launch_gather_probe(pool, pool_rows, row_bytes, indices, n,
                                        static_cast<uint8_t*>(out),
                                        static_cast<uint32_t*>(workspace),
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH_FAILED;
}

int64_t mla_debug_wait_limit(int64_t cycles)
{
    const long long v = cycles > 0 ? (long long)cycles : kDefaultWaitLimit;
    return (int64_t)g_wait_limit.exchange(v);
}

const char* mla_status_string(int status)
{
    switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MLA_ERR_MISALIGNED: return "buffer not 16-byte aligned (workspace: 256-byte)";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_UNSUPPORTED_DEVICE: return "unsupported device (need compute capability 10.3)";
    case MLA_ERR_LAUNCH_FAILED: return "kernel launch failed";
    case MLA_ERR_CUDA: return "CUDA runtime call failed";
    default: return "unknown status";
    }
}

}  // extern "C"
