// mla_split_kernel.cuh -- tcgen05 split kernel for absorbed-MLA decode (sm_103a).
//
// Included by the translation units that instantiate it (mla_split_dense.cu,
// mla_split_sparse.cu); mla_split_tc.cu holds the host-side dispatch.
//
// One CTA computes one (request, head block, split) of the split-KV decode
// (moonmath-ai/amd-kernels README, "MLA absorbed decode": one fused fp8 row per
// token is both K and V, page_size 1, base-2 LSE; hip_mha_decoding_num_partitions:
// per-split partials merged by a split-K reducer).  Output of a CTA: for each of
// its query rows the normalized fp32 partial o_s = O / l and lse_s, or the final
// bf16 row when the plan has a single split.
//
// GB300 design (the pages' MFMA/LDS designs are prior art, not followed):
//
// * Swapped operands.  Keys are the MMA's M (128 per block, one per TMEM lane)
//   and query rows (heads x draft positions) are N, so 16 heads need no padding:
//   S^T[128 x N] = K[128 x 576] . Q^T and O^T[512 x N] += V^T[512 x 128] . P^T.
// * fp8-native operands.  K and V stay e4m3 exactly as gathered from the pool
//   (the latent part of the same rows is V, read as an MN-major operand), so no
//   dequantised copy is ever written.  The small operands are split into two
//   e4m3 terms, the second one a residual stored scaled up by a power of two:
//   each query row q is scaled by a power of two and written as
//   q_hi + 2^-5 q_lo (exact for every element within 2^-14 of the row maximum,
//   bf16 having 8 significant bits), and each probability p as
//   p_hi + 2^-4 p_lo (about as precise as rounding p to bf16 down to 2^-10 of
//   the row's reference, weights below about 2^-19 of it dropped).  hi and lo
//   are stacked along N (2N MMA columns), so the big operand is read from
//   shared memory once per MMA.  kv_scale and the powers of two are folded into
//   the logit and output scales.
// * Warp roles (16 warps).  Warps 0-6 gather the block's 128 rows with TMA
//   tile::gather4 (four slots per instruction; 128-byte latent boxes land
//   128B-swizzled, the 64-byte RoPE box 64B-swizzled: exactly the K-major operand
//   layout) into a two-stage ring, the block's 160 copies dealt out over the
//   seven warps; warp 7 issues the tcgen05.mma (kind::f8f6f4, fp32 accumulators
//   in TMEM) and commits to mbarriers; warps 8-11 and 12-15 are two softmax sets,
//   each owning half the query rows, and warp w % 4 of a set owns TMEM lanes
//   32 (w % 4)..+31 (one key per thread).  Measured on GB300, a block's 160
//   gather4 copies take ~3,800 SM cycles to issue from seven warps (~3,200 from
//   sixteen), and an SM streams random 576-byte rows at ~30-35 GB/s: the copy
//   engine, not the number of issuing warps, sets the rate.  One softmax warp per
//   SM sub-partition left its dependent chains exposed, so every key has two.
//   Registers move with setmaxnreg from warpgroups 0-1 (64 per thread) to the
//   softmax warpgroups (192).
// * Lazy rescaling.  Each row keeps a reference m that bounds its logits; p is
//   2^(s - m).  A block only moves the reference of a row whose logits exceed it
//   by more than kTau (then to the block maximum plus kHeadroom, so the next
//   move needs a jump of kTau + kHeadroom); otherwise p stays below 2^kTau.  The
//   decision is one hardware barrier-reduction (bar.red.or) of the four softmax
//   warps; O in TMEM is rescaled, column by column, only for the rows that moved.
// * Sums.  Each block's exact fp32 p (for the LSE) is summed over the warp's
//   32 keys with a transposing shuffle reduction, so each lane carries one row's
//   running sum.  The sums of p_hi + p_lo (what the tensor core consumed, used
//   to normalise O) are kept per thread and row across blocks (the split into
//   e4m3 terms yields them) and reduced once, at the end.
// * Memory in flight.  Two stages hold gathered blocks; right after issuing
//   block j, the gather warps prefetch the rows of block j+1 into L2 so its
//   gather finds them there.
// * Work order.  When the grid outlasts one wave, grid slice z serves the z-th
//   longest request, so variable-length batches start their longest work first.
// * Safety.  Every mbarrier wait is time-bounded and warp-uniform; the softmax
//   warps meet at bar.sync only at points every one of them reaches, and agree
//   on giving up through the same barrier-reduction, so a stuck pipeline ends
//   with an error bit instead of a hang.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <climits>

#include "mla_internal.h"
#include "mla_layout.cuh"
#include "mla_sm100.cuh"

namespace mla {
namespace {

// Phase stamps of a traced build: slot i of this CTA gets the global timer.
#ifdef MLA_TRACE
__device__ __forceinline__ void trace_stamp(const SplitArgs& a, int i)
{
    const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (a.trace == nullptr || cta >= (unsigned)kTraceCtas) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    a.trace[(size_t)cta * kTraceSlots + i] = t;
}
#define MLA_STAMP(i) trace_stamp(a, (i))
// Per-block events of the first kTraceBlockCtas CTAs: block j, event e.
__device__ __forceinline__ void trace_block(const SplitArgs& a, int j, int e)
{
    const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (a.trace == nullptr || cta >= (unsigned)kTraceBlockCtas || j >= kTraceBlocks) return;
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    a.trace[(size_t)kTraceCtas * kTraceSlots +
            ((size_t)cta * kTraceBlocks + j) * kTraceBlockEvents + e] = t;
}
#define MLA_BLOCK_STAMP(j, e) trace_block(a, (j), (e))
#else
#define MLA_STAMP(i) ((void)0)
#define MLA_BLOCK_STAMP(j, e) ((void)0)
#endif
// Block events: 0 gather warp 0 starts issuing the block, 1 it has issued its
// copies, 2 QK issued, 3 S loaded by the first softmax set's first warp, 4 its
// P published, 5 P.V issued, 6 and 7 as 3 and 4 for the second softmax set.
// Stamp slots: 0 CTA start, 1 after the wait for the preceding kernel,
// 2 first gather issued, 3 first QK issued, 4 last P.V issued, 5 epilogue has
// O, 6 rows staged, 7 rows stored, 8 end, 9 query tile written (first query
// warp), 10 the MMA warp past the query tile's barrier, 11 the first query warp
// starts converting its rows.


using namespace sm100;

constexpr int kBlockN = 128;          // keys per block (MMA M)
constexpr int kThreads = 512;         // warps 0-6 gather, 7 MMA, 8-11 and 12-15 softmax
constexpr int kWarps = kThreads / 32;
constexpr int kGatherWarps = 7;
constexpr int kMmaWarp = 7;
constexpr int kSoftmaxWarp0 = 8;      // two sets of four warps, each set owns half the rows
constexpr int kSets = 2;
constexpr uint32_t kRegsLow = 64;     // registers per thread of warpgroups 0-1 after set-up
constexpr uint32_t kRegsHigh = 192;   // ... of the softmax warpgroups 2-3
static_assert(2 * 128 * kRegsLow + 2 * 128 * kRegsHigh == 65536, "register split = the file");
constexpr float kTau = 2.75f;        // lazy-rescale threshold, base-2 logit units
constexpr float kShift = 6.f;         // p is fed as p * 2^kShift: at most 2^(kTau + kShift) < 448
constexpr float kHeadroom = 1.f;      // a new reference sits this far above the block maximum
static_assert(kTau + kShift < 8.807f, "p * 2^kShift stays below e4m3's largest finite 448");
// Every residual term is stored scaled up by a power of two, which moves its
// representable range down by as many bits.  A query row scaled to max |q| < 256
// leaves residuals |q - q_hi| <= 8 (half an e4m3 step at 2^7), so 2^5 keeps them
// at or below 256, and the same holds for the residual of that residual; a
// probability p * 2^kShift <= 2^8.75 leaves residuals <= 16, so 2^4 does.  The
// MMA results of the residual terms land in their own TMEM columns and are
// scaled back when the terms are added.
constexpr int kQLoBits = 5;
constexpr int kPLoBits = 4;
constexpr float kQLoBack = 1.f / (1 << kQLoBits);
constexpr float kPLoBack = 1.f / (1 << kPLoBits);
constexpr int kQWarps = kWarps - kSoftmaxWarp0;   // warps 8-15 split the query tile
constexpr uint32_t kQBar = 2;                     // Q tile + MMA warp (1 and 3: softmax sets)
constexpr uint32_t kGatherSleepNs = 32;
constexpr int kPrefetchMaxBlocks = 8;             // unshared CTAs of more blocks prefetch by line
constexpr uint32_t kMmaSleepNs = 32;

template <int N, bool SPARSE>
struct Cfg {
    static constexpr int NQ = 3 * N;                       // QK MMA columns: q_hi, q_mid, q_lo rows
    static constexpr int NC = 2 * N;                       // P.V MMA columns: p_hi rows, then p_lo rows
    static constexpr int kRowBytes = SPARSE ? 512 : 576;   // pool row width
    static constexpr bool kRope = !SPARSE;                 // separate 64-byte RoPE chunk
    static constexpr int kLatChunkBytes = kBlockN * 128;   // 16 KB per 128-column chunk
    static constexpr int kStageBytes = kBlockN * kRowBytes;
    static constexpr int kQChunkBytes = NQ * 128;
    static constexpr int kQBytes = 4 * kQChunkBytes + (kRope ? NQ * 64 : 0);
    static constexpr int kPBytes = kBlockN * NC;
    static constexpr int kDv = SPARSE ? 448 : 512;
    static constexpr int kOffStage = 0;
    static constexpr int kOffQ = 2 * kStageBytes;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffMisc = (kOffP + 2 * kPBytes + 127) / 128 * 128;
    static constexpr uint32_t kTmemCols = (2 * NQ + 4 * NC <= 256) ? 256u : 512u;
    static constexpr uint32_t kColS = 0;                   // S^T buffers: [0, 2 NQ)
    static constexpr uint32_t kColO = 2 * NQ;              // O^T chunks:  [2 NQ, 2 NQ + 4 NC)
    static constexpr int kGroups = kRowBytes / 8;          // 8-column query groups per row
    static constexpr int kVec = (kGroups + 31) / 32;       // query groups per lane
    static constexpr int kQRowsPerWarp = (N + kQWarps - 1) / kQWarps;
    static_assert(kOffQ % 1024 == 0 && kQChunkBytes % 1024 == 0, "128B-swizzle atoms");
    static_assert(kOffP % 16 == 0, "P tile alignment");
    static_assert(2 * NQ + 4 * NC <= 512, "TMEM columns");
    static_assert(NQ % 16 == 0 && NQ <= 256, "QK MMA N: a multiple of 16 up to 256");
    static_assert(N * 512 * 4 <= 2 * kStageBytes, "epilogue staging fits in the stages");
};

struct Misc {
    uint64_t kv_full[2], kv_empty[2], pv_done[2], s_full[2], s_free[2], p_full[2], o_done;
    uint64_t mma_drain;   // after an abort: every MMA the CTA issued has completed
    uint64_t never;       // tests of the timeout path: a barrier nothing completes
    uint32_t tmem_base;
    int abort;
    int q3;   // some query row of the tile needs its third (q_lo) term
    int kvalid[2][kBlockN];
    alignas(16) float cq[32];   // per query row: raw dot -> base-2 logit
    alignas(16) int win[32];   // per query row: keys at positions < win are visible
    float red[8][32];   // cross-warp reduction scratch, [set * 4 + warp of the set][row]
    alignas(16) float redt[8][32];   // epilogue: the same for the consumed sums (p_hi + p_lo)
    alignas(16) float fin[2][32];   // epilogue: the base-2 LSE per row (fin[1])
    float mlse[32];                 // fused merge: the cluster peers' LSEs of this CTA's slice rows
    float xw[kMaxMergeTerms];       // fused merge: the cluster partials' weights per slice row
    float xs[32];                   // fused merge: output scale per slice row
    uint32_t ticket;                // fused merge: this cluster's arrival rank at its slice
    long long row_item[32];   // epilogue: output row (request row x head) per query row, -1 if none
    int lens[kLongFirstMaxBatch];   // longest-first ordering: the requests' lengths
    int req;                        // longest-first ordering: this CTA's request
};

template <int N, bool SPARSE>
constexpr int smem_bytes()
{
    return Cfg<N, SPARSE>::kOffMisc + (int)sizeof(Misc);
}


// 2^x by the hardware's approximation (relative error about 2^-22; results
// below the smallest normal fp32 flush to 0).
__device__ __forceinline__ float ex2_approx(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// x * 2^k, exact whenever the result is a normal fp32 number.
__device__ __forceinline__ float mul_pow2(float x, int k)
{
    if (k > 127) {
        x *= __uint_as_float(254u << 23);
        k -= 127;
    } else if (k < -126) {
        x *= __uint_as_float(1u << 23);
        k += 126;
    }
    return x * __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

// Power-of-two shift that brings max |q| into [128, 256).
__device__ __forceinline__ int q_shift(float amax)
{
    if (!(amax > 0.f)) return 0;
    const uint32_t bits = __float_as_uint(amax);
    int e;  // amax = f * 2^e with f in [0.5, 1)
    if ((bits >> 23) != 0) e = (int)(bits >> 23) - 126;
    else frexpf(amax, &e);
    return 8 - e;
}

// Packed e4m3x2 -> two fp32 through the conversion unit (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2_cvt(uint16_t v)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
    float lo, hi;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi) : "r"(h2));
    return make_float2(lo, hi);
}

// Split two fp32 values into e4m3 hi bytes and e4m3 bytes of the residual
// times 2^kLoBits (pairs packed lo-byte first); returns the values the pairs
// represent, hi + lo * 2^-kLoBits (exact in fp32: the subtraction and the
// power-of-two scalings are exact).
template <int kLoBits>
__device__ __forceinline__ float2 split_pair(float a, float b, uint16_t& hi, uint16_t& lo)
{
    constexpr float up = (float)(1 << kLoBits);
    constexpr float back = 1.f / up;
    hi = f32x2_to_e4m3x2(a, b);
    const float2 h = e4m3x2_to_f32x2_cvt(hi);
    lo = f32x2_to_e4m3x2((a - h.x) * up, (b - h.y) * up);
    const float2 l = e4m3x2_to_f32x2_cvt(lo);
    return make_float2(fmaf(l.x, back, h.x), fmaf(l.y, back, h.y));
}

// Split two fp32 values of a scaled query row (max |x| < 256) into three e4m3
// terms, x = hi + 2^-5 (mid + 2^-5 lo), bytes packed lo-byte first.  Exact for
// every element of at least 2^-12 (the residuals are formed exactly in fp32).
// Returns |lo| of the two values (before lo is rounded to e4m3).
__device__ __forceinline__ float split_q3(float a, float b, uint16_t& hi, uint16_t& mid,
                                          uint16_t& lo)
{
    constexpr float up = (float)(1 << kQLoBits);
    hi = f32x2_to_e4m3x2(a, b);
    const float2 h = e4m3x2_to_f32x2_cvt(hi);
    const float ra = (a - h.x) * up, rb = (b - h.y) * up;
    mid = f32x2_to_e4m3x2(ra, rb);
    const float2 m = e4m3x2_to_f32x2_cvt(mid);
    const float la = (ra - m.x) * up, lb = (rb - m.y) * up;
    lo = f32x2_to_e4m3x2(la, lb);
    return fabsf(la) + fabsf(lb);   // the two lo terms' size, before their rounding
}

// Reduce N values held by every lane of a warp (max or sum); afterwards lane l
// holds the result for value index (l * N) / 32.
template <int N, bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[N], int lane)
{
    int count = N;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        if (count > 1) {
            const int half = count >> 1;
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int k = 0; k < N / 2; ++k) {
                if (k < half) {
                    const float send = upper ? v[k] : v[k + half];
                    const float keep = upper ? v[k + half] : v[k];
                    const float recv = __shfl_xor_sync(0xffffffffu, send, off);
                    v[k] = MAX ? fmaxf(keep, recv) : keep + recv;
                }
            }
            count = half;
        } else {
            const float recv = __shfl_xor_sync(0xffffffffu, v[0], off);
            v[0] = MAX ? fmaxf(v[0], recv) : v[0] + recv;
        }
    }
    return v[0];
}

// Barrier of the four warps of one softmax set (id 1 or 3, 128 threads).  Only
// used at points that all four warps of the set always reach.
__device__ __forceinline__ void softmax_bar(uint32_t id)
{
    asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// The same barrier, returning the OR of `v` over the set's four warps.
__device__ __forceinline__ bool softmax_bar_or(uint32_t id, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %2, 0;\n\t"
        "bar.red.or.pred po, %1, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(id), "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

// Bounded wait whose outcome is the same on every lane of the warp (all lanes
// must call it), so no warp-collective instruction is reached divergently.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t sleep_ns = 0,
                                          long long limit = kWaitLimitCycles)
{
    const bool ok = mbar_wait_or_abort(bar, parity, abort, sleep_ns, limit);
    return __all_sync(0xffffffffu, ok);
}

// One TMEM row of R query-row columns: hi columns at taddr_hi plus lo columns
// at taddr_lo (the two halves of the stacked MMA output), summed.
// The hi and lo columns of R rows, loads issued without waiting.
template <int R>
__device__ __forceinline__ void issue_rows(uint32_t taddr_hi, uint32_t taddr_lo,
                                           uint32_t (&h)[R], uint32_t (&l)[R])
{
    static_assert(R == 8 || R == 16, "a softmax set holds 8 or 16 rows");
    if constexpr (R == 16) {
        tmem_ld16(taddr_hi, h);
        tmem_ld16(taddr_lo, l);
    } else {
        tmem_ld8(taddr_hi, h);
        tmem_ld8(taddr_lo, l);
    }
}

// One TMEM row of R query-row columns of S^T from the q_hi and q_mid column
// groups only (a tile whose q_lo terms are all negligible).
template <int R>
__device__ __forceinline__ void load_rows(uint32_t taddr_hi, uint32_t taddr_mid, float (&s)[R])
{
    static_assert(R == 8 || R == 16, "a softmax set holds 8 or 16 rows");
    uint32_t h[R], m[R];
    if constexpr (R == 16) {
        tmem_ld16(taddr_hi, h);
        tmem_ld16(taddr_mid, m);
    } else {
        tmem_ld8(taddr_hi, h);
        tmem_ld8(taddr_mid, m);
    }
    tmem_wait_ld();
    reg_fence(h);
    reg_fence(m);
#pragma unroll
    for (int n = 0; n < R; ++n) s[n] = fmaf(__uint_as_float(m[n]), kQLoBack, __uint_as_float(h[n]));
}

// One TMEM row of R query-row columns of S^T: the q_hi, q_mid and q_lo column
// groups (the three parts of the stacked MMA output), combined.
template <int R>
__device__ __forceinline__ void load_rows(uint32_t taddr_hi, uint32_t taddr_mid,
                                          uint32_t taddr_lo, float (&s)[R])
{
    static_assert(R == 8 || R == 16, "a softmax set holds 8 or 16 rows");
    uint32_t h[R], m[R], l[R];
    if constexpr (R == 16) {
        tmem_ld16(taddr_hi, h);
        tmem_ld16(taddr_mid, m);
        tmem_ld16(taddr_lo, l);
    } else {
        tmem_ld8(taddr_hi, h);
        tmem_ld8(taddr_mid, m);
        tmem_ld8(taddr_lo, l);
    }
    tmem_wait_ld();
    reg_fence(h);
    reg_fence(m);
    reg_fence(l);
#pragma unroll
    for (int n = 0; n < R; ++n)
        s[n] = fmaf(fmaf(__uint_as_float(l[n]), kQLoBack, __uint_as_float(m[n])), kQLoBack,
                    __uint_as_float(h[n]));
}

// ---- fused split-K merge -------------------------------------------------------------------
// The MC splits of a cluster (consecutive split indices, cluster rank = split
// % MC) each hold their normalised fp32 partial rows o_s (staged in the idle KV
// stages) and base-2 LSEs lse_s in shared memory.  Cluster rank r merges rows
// [r RS, (r + 1) RS) of the tile, RS = N / MC, over the MC peers' shared memory
// (the merge of mla_splitk_reduce: M = max lse_s, w_s = 2^(lse_s - M),
// o = sum w_s o_s / sum w_s in increasing split order, lse = M + log2 sum w_s).
// With one cluster per tile that is the final row.  Otherwise each cluster
// writes its merged slice (normalised, with its LSE) to the workspace and takes
// a ticket per (tile, rank); the rank-r CTA of the last cluster to arrive merges
// the tile's cluster partials of its slice in increasing cluster order and
// writes the final rows, so the association is fixed: splits within a cluster,
// then clusters.  It resets the ticket to zero for the next call.
//
// Every thread of the CTA calls it (the cluster barriers count all threads);
// warps 8-15 do the work.
template <int N, bool SPARSE, int MC>
__device__ __forceinline__ void fused_merge(uint8_t* smem, Misc& ms, const SplitArgs& a, int b,
                                            int hb, int split)
{
    using C = Cfg<N, SPARSE>;
    constexpr int RS = N / MC;                      // slice rows of one CTA
    constexpr int kQuads = C::kDv / 4;              // float4 per output row
    constexpr int kWork = RS * kQuads;              // float4 of the slice
    constexpr int kThr = kThreads - kSoftmaxWarp0 * 32;
    constexpr int kPer = (kWork + kThr - 1) / kThr; // float4 per thread
    static_assert(N % MC == 0 && RS * MC <= 32, "slices of the tile's rows");
    const int tid = threadIdx.x;
    const bool worker = tid >= kSoftmaxWarp0 * 32;
    const int t = tid - kSoftmaxWarp0 * 32;
    const float* ostage = reinterpret_cast<const float*>(smem + C::kOffStage);  // [N][512]
    const uint32_t rank = cluster_ctarank();
    const int r0 = (int)rank * RS;

    cluster_sync();   // every peer's partial rows and LSEs are staged
    float4 acc[kPer];
    float wsum[kPer];
    int rr_of[kPer];
    if (worker) {
        if (t < RS * MC) {
            const int rr = t / MC, p = t % MC;
            ms.mlse[t] = ld_dsmem_f32(dsmem_addr(&ms.fin[1][r0 + rr], (uint32_t)p));
        }
        asm volatile("bar.sync 4, %0;" ::"n"(kThr) : "memory");
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int w = t + k * kThr;
            acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            wsum[k] = 0.f;
            rr_of[k] = -1;
            if (w >= kWork) continue;
            const int rr = w / kQuads, q = w % kQuads;
            rr_of[k] = rr;
            float m = -CUDART_INF_F;
#pragma unroll
            for (int p = 0; p < MC; ++p) m = fmaxf(m, ms.mlse[rr * MC + p]);
            const float* src = ostage + (r0 + rr) * 512 + q * 4;
#pragma unroll
            for (int p = 0; p < MC; ++p) {
                const float l = ms.mlse[rr * MC + p];
                const float wp = (m == -CUDART_INF_F || l == -CUDART_INF_F) ? 0.f : exp2f(l - m);
                wsum[k] += wp;
                const float4 v = ld_dsmem_f32x4(dsmem_addr(src, (uint32_t)p));
                acc[k].x += wp * v.x;
                acc[k].y += wp * v.y;
                acc[k].z += wp * v.z;
                acc[k].w += wp * v.w;
            }
        }
    }
    cluster_sync();   // peers have read this CTA's shared memory
    if (!worker) return;

    const int ns = a.num_splits;
    const int nclus = ns / MC;
    const int clus = split / MC;
    // the merged slice's LSE per row, from its first thread
    auto slice_lse = [&](int rr) {
        float m = -CUDART_INF_F, ws = 0.f;
#pragma unroll
        for (int p = 0; p < MC; ++p) m = fmaxf(m, ms.mlse[rr * MC + p]);
#pragma unroll
        for (int p = 0; p < MC; ++p) {
            const float l = ms.mlse[rr * MC + p];
            ws += (m == -CUDART_INF_F || l == -CUDART_INF_F) ? 0.f : exp2f(l - m);
        }
        return ws > 0.f ? m + log2f(ws) : -CUDART_INF_F;
    };
    auto store_final = [&](long long item, int q, float4 v) {
        if (a.o_f32 != nullptr) {
            *reinterpret_cast<float4*>(a.o_f32 + item * C::kDv + q * 4) = v;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(a.o + item * C::kDv + q * 4) = pk;
        }
    };
    if (nclus == 1) {
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            if (rr_of[k] < 0) continue;
            const int w = t + k * kThr;
            const int rr = rr_of[k], q = w % kQuads;
            const long long item = ms.row_item[r0 + rr];
            if (item < 0) continue;
            const float f = wsum[k] > 0.f ? a.out_scale / wsum[k] : 0.f;
            store_final(item, q, make_float4(acc[k].x * f, acc[k].y * f, acc[k].z * f, acc[k].w * f));
            if (q == 0 && a.lse != nullptr) a.lse[item] = slice_lse(rr);
        }
        return;
    }
    // several clusters: publish this cluster's slice, then take the ticket
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        if (rr_of[k] < 0) continue;
        const int w = t + k * kThr;
        const int rr = rr_of[k], q = w % kQuads;
        const long long item = ms.row_item[r0 + rr];
        if (item < 0) continue;
        const float f = wsum[k] > 0.f ? 1.f / wsum[k] : 0.f;
        *reinterpret_cast<float4*>(a.o_part + (item * nclus + clus) * C::kDv + q * 4) =
            make_float4(acc[k].x * f, acc[k].y * f, acc[k].z * f, acc[k].w * f);
        if (q == 0) a.lse_part[item * nclus + clus] = slice_lse(rr);
    }
    // The barrier orders the slice's stores before thread 0's acq_rel ticket
    // (a release at GPU scope covering them); the last arriver's acquire then
    // orders every other cluster's slice before the loads below.
    asm volatile("bar.sync 4, %0;" ::"n"(kThr) : "memory");
    uint32_t* ticket = a.tickets + ((int64_t)b * a.head_blocks + hb) * MC + rank;
    if (t == 0) ms.ticket = atom_add_acq_rel_gpu(ticket, 1u);
    asm volatile("bar.sync 4, %0;" ::"n"(kThr) : "memory");
    if (ms.ticket != (uint32_t)(nclus - 1)) return;
    if (t == 0) *ticket = 0u;   // no CTA of this launch touches it again
    // Every (row, cluster) LSE loaded at once, then the weights per row.
    constexpr int kMaxClus = kMaxMergeTerms / RS;   // nclus * RS <= kMaxMergeTerms
    if (t < RS * nclus) {
        const int rr = t / nclus, c = t % nclus;
        const long long item = ms.row_item[r0 + rr];
        ms.xw[t] = item >= 0 ? __ldcg(a.lse_part + item * nclus + c) : -CUDART_INF_F;
    }
    asm volatile("bar.sync 4, %0;" ::"n"(kThr) : "memory");
    if (t < RS) {
        const long long item = ms.row_item[r0 + t];
        float* w = ms.xw + t * nclus;
        float m = -CUDART_INF_F, ws = 0.f;
        for (int c = 0; c < nclus; ++c) m = fmaxf(m, w[c]);
        for (int c = 0; c < nclus; ++c) {
            const float wc = (m == -CUDART_INF_F || w[c] == -CUDART_INF_F) ? 0.f : exp2f(w[c] - m);
            w[c] = wc;
            ws += wc;
        }
        if (item >= 0 && a.lse != nullptr) a.lse[item] = ws > 0.f ? m + log2f(ws) : -CUDART_INF_F;
        ms.xs[t] = ws > 0.f ? a.out_scale / ws : 0.f;
    }
    asm volatile("bar.sync 4, %0;" ::"n"(kThr) : "memory");
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        if (rr_of[k] < 0) continue;
        const int w = t + k * kThr;
        const int rr = rr_of[k], q = w % kQuads;
        const long long item = ms.row_item[r0 + rr];
        if (item < 0) continue;
        const float* op = a.o_part + item * nclus * C::kDv + q * 4;
        float4 v[kMaxClus];
#pragma unroll
        for (int c = 0; c < kMaxClus; ++c)   // all loads in flight together
            if (c < nclus) v[c] = __ldcg(reinterpret_cast<const float4*>(op + (int64_t)c * C::kDv));
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kMaxClus; ++c) {
            if (c < nclus) {
                const float wc = ms.xw[rr * nclus + c];
                o.x += wc * v[c].x;
                o.y += wc * v[c].y;
                o.z += wc * v[c].z;
                o.w += wc * v[c].w;
            }
        }
        const float f = ms.xs[rr];
        store_final(item, q, make_float4(o.x * f, o.y * f, o.z * f, o.w * f));
    }
}

template <int N, bool SPARSE, bool EXTRA, int MC>
__global__ void __launch_bounds__(kThreads, 1)
split_tc_kernel(const __grid_constant__ CUtensorMap tm_lat,
                const __grid_constant__ CUtensorMap tm_rope, const SplitArgs a)
{
    using C = Cfg<N, SPARSE>;
    constexpr int NQ = C::NQ;
    constexpr int NC = C::NC;
    constexpr int kWidth = C::kRowBytes;
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc& ms = *reinterpret_cast<Misc*>(smem + C::kOffMisc);
    volatile int* abort_flag = &ms.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hb = blockIdx.x, split = blockIdx.y;
    int b = blockIdx.z;   // the request (token); remapped below when long_first is set
    // Let a programmatic dependent (the split-K reduce) be scheduled as soon as
    // every CTA of this grid has started; it waits for this grid's completion
    // before reading anything.
    asm volatile("griddepcontrol.launch_dependents;");
    if (tid == 0) MLA_STAMP(0);
    const int rows_in_req = a.q_len * a.num_heads;

    // kv_empty: the stage's P.V has finished and it may be refilled; pv_done:
    // the same completion, waited for by the softmax warps.
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.kv_full[i], kGatherWarps);   // one arrival per gather warp
            mbar_init(&ms.kv_empty[i], 1);
            mbar_init(&ms.pv_done[i], 1);
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.s_free[i], 4 * kSets);   // every softmax warp
            mbar_init(&ms.p_full[i], 4 * kSets);
        }
        mbar_init(&ms.o_done, 1);
        mbar_init(&ms.mma_drain, 1);
        mbar_init(&ms.never, 1);
        ms.abort = 0;
        ms.q3 = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ms.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    // Everything above touches only this CTA's shared memory and TMEM.  This
    // launch is a programmatic dependent of the preceding kernel, which may
    // still be writing the inputs (queries, page table, cache rows): wait for it
    // before the first global read.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) MLA_STAMP(1);

    // Longest requests first.  With more CTAs than one wave, grid slice z takes
    // the z-th request in decreasing length order (ties in index order): the
    // block scheduler hands out CTAs in index order, so the longest work starts
    // first and the last wave holds the shortest (longest-processing-time
    // ordering).  Every CTA derives the same permutation from seq_lens.
    if (!SPARSE && a.long_first && a.batch <= kLongFirstMaxBatch) {
        for (int t = tid; t < a.batch; t += kThreads) ms.lens[t] = a.seq_lens[t];
        __syncthreads();
        if (tid < a.batch) {
            const int lt = ms.lens[tid];
            int rank = 0;
            for (int r = 0; r < a.batch; ++r) {
                const int lr = ms.lens[r];
                rank += (lr > lt || (lr == lt && r < tid)) ? 1 : 0;
            }
            if (rank == (int)blockIdx.z) ms.req = tid;
        }
        __syncthreads();
        b = ms.req;
    }

    // The query rows' loads go out first, ahead of the index loads and the
    // gathers that would otherwise queue in front of them (warps 8-15).
    uint4 qv[C::kQRowsPerWarp][C::kVec];
    if (warp >= kSoftmaxWarp0) {
        const int qw = warp - kSoftmaxWarp0;
#pragma unroll
        for (int rr = 0; rr < C::kQRowsPerWarp; ++rr) {
            const int n = qw + rr * kQWarps;
            const int idx = hb * N + n;
            const bool valid = n < N && idx < rows_in_req;
            int64_t item = 0;
            if (valid)
                item = ((int64_t)b * a.q_len + idx / a.num_heads) * a.num_heads + idx % a.num_heads;
#pragma unroll
            for (int v = 0; v < C::kVec; ++v) {
                const int c = (lane + 32 * v) * 8;
                qv[rr][v] = make_uint4(0u, 0u, 0u, 0u);
                if (valid && c < kWidth)
                    qv[rr][v] = c < a.d_v
                        ? __ldg(reinterpret_cast<const uint4*>(a.q_lat + item * a.d_v + c))
                        : __ldg(reinterpret_cast<const uint4*>(a.q_pe + item * a.d_rope + (c - a.d_v)));
            }
        }
    }

    // ---- the request's key list and this split's range --------------------------------
    // Sparse with a second (compressed) cache: token b's keys are its topk main
    // candidates, up to three invalid padding keys (so the second cache's keys
    // start on a four-row group), then its extra_topk candidates in the second
    // cache.  Splits then start on multiples of four keys, so every gather4
    // group reads one cache.
    int64_t base;
    int L;
    int topk4 = 0;
    const int32_t* xlist = nullptr;
    if (SPARSE) {
        base = (int64_t)b * a.topk;
        L = a.topk;
        if constexpr (EXTRA) {
            topk4 = (a.topk + 3) & ~3;
            L = topk4 + a.extra_topk;
            xlist = a.extra_indices + (int64_t)b * a.extra_topk;
        }
    } else {
        base = a.kv_indptr[b];
        const int cap = a.kv_indptr[b + 1] - a.kv_indptr[b];
        L = a.seq_lens[b];
        if (L < 0 || L > cap) {
            if (tid == 0) atomicOr(a.err, MLA_DEVERR_BAD_LENGTH);
            L = L < 0 ? 0 : cap;
        }
    }
    // The draft window.  Local key i is the request's global position
    // i * cp_world + cp_rank (decode context parallelism: this rank holds the
    // positions p with p % cp_world == cp_rank; cp_world 1 otherwise), and draft
    // row t sees the global positions up to G - q_len + t, G the request's global
    // length (glen, or L itself).  win(t) is the number of local keys row t sees.
    int G = L;
    if (!SPARSE && a.glen != nullptr) G = a.glen[b];
    auto window = [&](int t) {
        const int x = G - a.q_len + t - a.cp_rank;
        return x >= 0 ? x / a.cp_world + 1 : 0;
    };
    const int win_min = window(0);
    int chunk = (L + a.num_splits - 1) / a.num_splits;
    if constexpr (EXTRA) chunk = (chunk + 3) & ~3;
    const int k0 = min(L, split * chunk);
    const int k1 = min(L, k0 + chunk);
    const int nblk = (k1 - k0 + kBlockN - 1) / kBlockN;

    // ---- gather helpers (warps 0-6) ---------------------------------------------------------
    // A block is 32 four-row groups x kBoxes boxes (the four 128-byte latent
    // chunks, then the 64-byte RoPE chunk): kItems tile::gather4 copies, dealt
    // out kItemsPerWarp per warp and one per lane.  TMA issue is serial within a
    // warp, so spreading the copies over seven warps shortens a block's issue.
    // The key-validity bits of the 128 rows come from lanes of warps 0-3, one
    // row each.
    constexpr int kBoxes = C::kRope ? 5 : 4;
    constexpr int kItems = 32 * kBoxes;
    constexpr int kItemsPerWarp = (kItems + kGatherWarps - 1) / kGatherWarps;
    static_assert(kItemsPerWarp <= 32, "one copy per lane");
    const int32_t* list = a.kv_indices + base;
    constexpr bool has_extra = EXTRA;   // only sparse launches have a second cache
    // The index of key k of this request or token, and whether it lives in the
    // second cache (-1: a padding key, invalid).
    auto key_slot = [&](int k) -> int32_t {
        if (!has_extra) return __ldg(list + k);
        if (k < a.topk) return __ldg(list + k);
        return k < topk4 ? -1 : __ldg(xlist + (k - topk4));
    };
    auto key_extra = [&](int k) { return has_extra && k >= topk4; };
    const int my_item = warp * kItemsPerWarp + lane;
    const bool item_on = warp < kGatherWarps && lane < kItemsPerWarp && my_item < kItems;
    const int my_group = item_on ? my_item / kBoxes : 0;   // rows 4 g .. 4 g + 3
    const int my_box = item_on ? my_item % kBoxes : 0;
    const bool row_lane = tid < kBlockN;                   // warps 0-3: row tid's validity
    struct Slots {
        int32_t v[4];
        bool ex;   // the group's rows are in the second cache
    };
    // The four indices of this lane's group in block j (-1 past the split),
    // and row tid's index.
    auto raw_slots = [&](int j) -> Slots {
        Slots r;
        const int kb = k0 + j * kBlockN;
        const int nk = min(kBlockN, k1 - kb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 4 * my_group + i;
            r.v[i] = (item_on && row < nk) ? key_slot(kb + row) : -1;
        }
        r.ex = key_extra(kb + 4 * my_group);
        return r;
    };
    auto raw_row = [&](int j) -> int32_t {
        const int kb = k0 + j * kBlockN;
        const int nk = min(kBlockN, k1 - kb);
        return (row_lane && tid < nk) ? key_slot(kb + tid) : -1;
    };
    auto slot_ok = [&](int32_t v, bool ex) {
        return v >= 0 && (int64_t)v < (ex ? a.extra_rows : a.pool_rows);
    };
    // Slots to gather: masked or invalid keys take row coordinate -1, outside
    // the tensor, where the copy fills the row with zeros (p = 0 for them, and
    // no pool row is read).
    auto fix_slots = [&](Slots r) -> Slots {
#pragma unroll
        for (int i = 0; i < 4; ++i) r.v[i] = slot_ok(r.v[i], r.ex) ? r.v[i] : -1;
        return r;
    };
    // Validity of row tid (a dense slot out of range is reported, not read).
    auto row_valid = [&](int j, int32_t v) -> int {
        const int kb = k0 + j * kBlockN;
        const int nk = min(kBlockN, k1 - kb);
        if (!row_lane || tid >= nk) return 0;
        if (slot_ok(v, key_extra(kb + tid))) return 1;
        if (!(SPARSE && v < 0)) atomicOr(a.err, MLA_DEVERR_BAD_SLOT);
        return 0;
    };
    // Block j into stage j & 1.  Warp 0 announces the stage's bytes, which
    // arrive from the seven warps' copies.  The four-row groups past the split's
    // end are not fetched from block 2 on: their rows are masked, and the stage
    // still holds block j-2's rows there (finite bytes; the copy engine's issue
    // rate, not DRAM, bounds a block, so a short last block costs less).  The
    // stages' first fills copy every group (zero rows for masked keys), so no
    // row of a stage is ever read uninitialised.
    auto issue = [&](int j, const Slots& sl, int rowok) {
        const int st = j & 1;
        const int nk = min(kBlockN, k1 - (k0 + j * kBlockN));
        const int ngrp = j >= 2 ? (nk + 3) >> 2 : kBlockN / 4;
        if (row_lane) ms.kvalid[st][tid] = rowok;
        __syncwarp();
        if (lane == 0) {
            if (warp == 0)
                mbar_arrive_expect_tx(&ms.kv_full[st],
                                      (uint32_t)(ngrp * (C::kStageBytes / (kBlockN / 4))));
            else
                mbar_arrive(&ms.kv_full[st]);
        }
        __syncwarp();
        if (item_on && my_group < ngrp) {
            uint8_t* stage = smem + C::kOffStage + st * C::kStageBytes;
            uint8_t* dst = my_box < 4 ? stage + my_box * C::kLatChunkBytes + my_group * 512
                                      : stage + 4 * C::kLatChunkBytes + my_group * 256;
            // sparse: tm_rope is the second cache's map (512-byte rows, no RoPE box)
            const CUtensorMap* map = (my_box < 4 && !sl.ex) ? &tm_lat : &tm_rope;
            const int x = my_box < 4 ? my_box * 128 : 512;
            tma_gather4(dst, map, x, sl.v[0], sl.v[1], sl.v[2], sl.v[3], &ms.kv_full[st]);
        }
    };
    // L2 prefetch of the rows of block j+1 right after issuing block j, one
    // prefetch per 128-byte line, from indices loaded a block earlier so it
    // never waits on a load; the next gather then finds its rows in L2.  Two
    // ways to deal the lines out, each where it measured best on GB300:
    //  * by row: warps 0-3, thread tid prefetching row tid -- in CTAs of a few
    //    blocks (B=8 H=16 S=8192: 19.1 -> 18.7 us);
    //  * by line, over all seven gather warps -- in long unshared streams,
    //    where prefetching by row held up warps 0-3, which also issue gathers
    //    (B=8 H=16 S=131072: 139 us without a prefetch, 178 by row, 135 by line).
    const bool pf_rows = nblk <= kPrefetchMaxBlocks;
    auto prefetch_block = [&](int j, int32_t v) {
        const int kb = k0 + j * kBlockN;
        const int nk = min(kBlockN, k1 - kb);
        if (!pf_rows || !row_lane || tid >= nk) return;
        const bool ex = key_extra(kb + tid);
        if (!slot_ok(v, ex)) return;
        const uint8_t* row = (ex ? a.extra_pool : a.pool) + (int64_t)v * kWidth;
#pragma unroll
        for (int c = 0; c < kWidth; c += 128) prefetch_l2(row + c);
    };
    constexpr int kLines = (kWidth + 127) / 128;                 // 128-byte lines per row
    constexpr int kPfPer = (kBlockN * kLines + kGatherWarps * 32 - 1) / (kGatherWarps * 32);
    struct PfLines { int32_t v[kPfPer]; };   // slots of this thread's lines (-1: none)
    auto pf_lines_load = [&](int j) -> PfLines {
        PfLines r;
        const int kb = k0 + j * kBlockN;
        const int nk = min(kBlockN, k1 - kb);
#pragma unroll
        for (int i = 0; i < kPfPer; ++i) {
            const int item = tid + kGatherWarps * 32 * i;
            const int row = item / kLines;
            r.v[i] = (!pf_rows && item < kBlockN * kLines && row < nk) ? key_slot(kb + row) : -1;
        }
        return r;
    };
    auto pf_lines_issue = [&](int j, const PfLines& r) {
        const int kb = k0 + j * kBlockN;
#pragma unroll
        for (int i = 0; i < kPfPer; ++i) {
            const int item = tid + kGatherWarps * 32 * i;
            const int row = item / kLines;
            if (r.v[i] < 0) continue;
            const bool ex = key_extra(kb + row);
            if (!slot_ok(r.v[i], ex)) continue;
            prefetch_l2((ex ? a.extra_pool : a.pool) + (int64_t)r.v[i] * kWidth +
                        (item % kLines) * 128);
        }
    };
    int32_t rpf = -1;   // by row: row tid's index in the block after the next
    PfLines lpf2, lpf;   // by line: block 2's lines, then the block after the next
#pragma unroll
    for (int i = 0; i < kPfPer; ++i) lpf2.v[i] = lpf.v[i] = -1;
    Slots gnext{};
    int32_t rnext = -1;
    Slots s0{{-1, -1, -1, -1}, false}, s1{{-1, -1, -1, -1}, false};
    int32_t w0 = -1, w1 = -1;
    if (warp < kGatherWarps && nblk > 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_lat);
            if (C::kRope || has_extra) tma_prefetch_desc(&tm_rope);
        }
        // the index loads of blocks 0-2 are in flight together, during the set-up
        s0 = raw_slots(0);
        w0 = raw_row(0);
        if (nblk > 1) {
            s1 = raw_slots(1);
            w1 = raw_row(1);
        }
        if (nblk > 2) {
            gnext = raw_slots(2);
            rnext = raw_row(2);
        }
        if (pf_rows && nblk > 3) rpf = raw_row(3);
        if (!pf_rows && nblk > 2) lpf2 = pf_lines_load(2);
        if (!pf_rows && nblk > 3) lpf = pf_lines_load(3);
    }

    // ---- barriers and TMEM ----------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t smem_base = smem_u32(smem);

    if (warp < kGatherWarps && nblk > 0) {
        // start the first two blocks before anything else
        if (tid == 0) MLA_BLOCK_STAMP(0, 0);
        issue(0, fix_slots(s0), row_valid(0, w0));
        if (tid == 0) {
            MLA_STAMP(2);
            MLA_BLOCK_STAMP(0, 1);
        }
        if (nblk > 1) {
            if (tid == 0) MLA_BLOCK_STAMP(1, 0);
            issue(1, fix_slots(s1), row_valid(1, w1));
            if (tid == 0) MLA_BLOCK_STAMP(1, 1);
        }
        if (nblk > 2) {
            prefetch_block(2, rnext);
            pf_lines_issue(2, lpf2);
        }
    }

    // ---- the query tile: one warp per row, warps 8-15 --------------------------------------------
    // q is scaled by 2^sh so that max |q| is in [128, 256), then split into e4m3
    // hi (tile rows 0..N-1), mid (rows N..2N-1) and lo (rows 2N..3N-1).  The
    // gather warps go on loading meanwhile; the MMA warp waits for the tile at
    // the warps' barrier.
    if (warp >= kSoftmaxWarp0) {
        const int qw = warp - kSoftmaxWarp0;
        uint8_t* qtile = smem + C::kOffQ;
        if (warp == kSoftmaxWarp0 && lane == 0) MLA_STAMP(11);
        // With four rows per warp the loop is not unrolled, so the warp runs the
        // same (by then cached) instructions for every row (measured: B=1 H=64
        // S=131072 54.3 -> 50.8 us per call); two rows stay unrolled (one pass
        // each measured slower).  The rows' values move down the register array
        // instead of being indexed by rr.
#pragma unroll(C::kQRowsPerWarp > 2 ? 1 : C::kQRowsPerWarp)
        for (int rr = 0; rr < C::kQRowsPerWarp; ++rr) {
            const int n = qw + rr * kQWarps;
            if (n >= N) break;
            float amax = 0.f;
#pragma unroll
            for (int v = 0; v < C::kVec; ++v) {
                const uint32_t w[4] = {qv[0][v].x, qv[0][v].y, qv[0][v].z, qv[0][v].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[k] << 16)),
                                             fabsf(__uint_as_float(w[k] & 0xFFFF0000u))));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const int sh = q_shift(amax);
            float lsum = 0.f;   // sum of |q_lo| over the row (this lane's columns)
#pragma unroll
            for (int v = 0; v < C::kVec; ++v) {
                const int c = (lane + 32 * v) * 8;
                if (c >= kWidth) continue;
                const uint32_t w[4] = {qv[0][v].x, qv[0][v].y, qv[0][v].z, qv[0][v].w};
                uint32_t hw[2], mw[2], lw[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    uint16_t h0, m0, l0, h1, m1, l1;
                    lsum += split_q3(mul_pow2(__uint_as_float(w[2 * k] << 16), sh),
                                     mul_pow2(__uint_as_float(w[2 * k] & 0xFFFF0000u), sh), h0, m0, l0);
                    lsum += split_q3(mul_pow2(__uint_as_float(w[2 * k + 1] << 16), sh),
                                     mul_pow2(__uint_as_float(w[2 * k + 1] & 0xFFFF0000u), sh), h1, m1, l1);
                    hw[k] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                    mw[k] = (uint32_t)m0 | ((uint32_t)m1 << 16);
                    lw[k] = (uint32_t)l0 | ((uint32_t)l1 << 16);
                }
                *reinterpret_cast<uint2*>(qtile + tile_offset(n, c, NQ)) = make_uint2(hw[0], hw[1]);
                *reinterpret_cast<uint2*>(qtile + tile_offset(N + n, c, NQ)) = make_uint2(mw[0], mw[1]);
                *reinterpret_cast<uint2*>(qtile + tile_offset(2 * N + n, c, NQ)) = make_uint2(lw[0], lw[1]);
            }
            // The q_lo terms move a logit of this row by at most
            // sum |q_lo| 2^-10 x 448 (the largest e4m3 key) x |cq|; the tile
            // feeds them to the MMA only when that bound reaches 2^-16 (base-2
            // units) for some row.
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
            if (lane == 0) {
                const int idx = hb * N + n;
                const bool valid = idx < rows_in_req;
                const float cq = valid ? mul_pow2(a.logit_scale, -sh) : 0.f;
                ms.cq[n] = cq;
                ms.win[n] = valid ? window(idx / a.num_heads) : -1;
                if (lsum * (448.f / 1024.f) * fabsf(cq) > 1.f / 65536.f) ms.q3 = 1;
            }
#pragma unroll
            for (int k = 0; k + 1 < C::kQRowsPerWarp; ++k)
#pragma unroll
                for (int v = 0; v < C::kVec; ++v) qv[k][v] = qv[k + 1][v];
        }
        if (warp == kSoftmaxWarp0 && lane == 0) MLA_STAMP(9);
    }
    if (warp >= kMmaWarp) {   // the query warps and the MMA warp, which waits for the tile
        fence_proxy_async_smem();
        asm volatile("bar.sync %0, %1;" ::"n"(kQBar), "n"((kQWarps + 1) * 32) : "memory");
        if (warp == kMmaWarp && lane == 0) MLA_STAMP(10);
    }
    // QK runs over 3N columns (hi, mid, lo) when some row needs its q_lo term,
    // else over the first 2N; the MMA warp and the softmax warps read the
    // choice after the query barrier above.

    // Registers move from the gather and MMA warpgroups (0-1) to the softmax
    // warpgroups (2-3); the shares add up to the block's 512 x 128 registers.
    // Each branch below holds all of its warpgroups' remaining code.
    if (warp < kSoftmaxWarp0) {
    regs_lower<kRegsLow>();
    if (warp < kGatherWarps) {
        // ================= gather ============================================================
        // block j reuses the stage of block j-2: wait for its P.V, then load
        int issued = nblk < 2 ? nblk : 2;
        for (int j = 2; j < nblk; ++j) {
            if (!warp_wait(&ms.kv_empty[j & 1], ((j - 2) >> 1) & 1, abort_flag, kGatherSleepNs,
                           a.wait_limit))
                break;
            if (tid == 0) MLA_BLOCK_STAMP(j, 0);
            issue(j, fix_slots(gnext), row_valid(j, rnext));
            if (tid == 0) MLA_BLOCK_STAMP(j, 1);
            issued = j + 1;
            if (j + 1 < nblk) {
                gnext = raw_slots(j + 1);
                rnext = raw_row(j + 1);
                prefetch_block(j + 1, rpf);   // block j + 1's rows into L2
                pf_lines_issue(j + 1, lpf);
                if (pf_rows && j + 2 < nblk) rpf = raw_row(j + 2);
                if (!pf_rows && j + 2 < nblk) lpf = pf_lines_load(j + 2);
            }
        }
        // Never leave the CTA with loads in flight: the last two blocks this
        // warp issued (earlier ones were consumed before their stage was
        // reused) must land.  A fresh wait flag and the full bound keep this
        // drain going after an abort.  (After an abort another gather warp
        // may have stopped one block earlier, leaving a phase that never
        // completes; the wait then runs its full bound, about a second, long
        // after this warp's own copies have landed.)
        volatile int drain_abort = 0;
        for (int j = issued - 2; j < issued; ++j)
            if (j >= 0) warp_wait(&ms.kv_full[j & 1], (j >> 1) & 1, &drain_abort, kGatherSleepNs);
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer =====================================================
        // The whole warp runs this code converged and lane 0 issues each MMA and
        // commit (predicated, not branched to), so the descriptors stay in
        // uniform registers; a lone-lane branch cost ~80 cycles per MMA in
        // register moves.  Descriptors are built once per stage and advanced by
        // adding the byte offset / 16 to their address field (shared memory <
        // 256 KB, so the 14-bit field never carries).
        if (nblk > 0) {
            const uint32_t id_qk = idesc_e4m3(128, ms.q3 ? NQ : 2 * N, false, false);
            const uint32_t id_pv = idesc_e4m3(128, NC, true, true);
            const uint32_t stage0 = smem_base + C::kOffStage;
            const uint32_t qb = smem_base + C::kOffQ;
            const uint64_t qk_a_lat = smem_desc(stage0, 16, 1024, kSw128);
            const uint64_t qk_a_rope = smem_desc(stage0 + 4 * C::kLatChunkBytes, 16, 512, kSw64);
            const uint64_t qk_b_lat = smem_desc(qb, 16, 1024, kSw128);
            const uint64_t qk_b_rope = smem_desc(qb + 4 * C::kQChunkBytes, 16, 512, kSw64);
            const uint64_t pv_a = smem_desc(stage0, C::kLatChunkBytes, 1024, kSw128);
            const uint64_t pv_b = smem_desc(smem_base + C::kOffP, 128, 2048, kSwNone);
            auto issue_pv = [&](int blk) {
                const int st = blk & 1;
                const uint64_t a0 = pv_a + (uint64_t)((st * C::kStageBytes) >> 4);
                const uint64_t b0 = pv_b + (uint64_t)((st * C::kPBytes) >> 4);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f8_warp(tmem + C::kColO + c * NC,
                                a0 + (uint64_t)((c * C::kLatChunkBytes + kk * 4096) >> 4),
                                b0 + (uint64_t)((kk * 512) >> 4), id_pv,
                                (blk > 0 || kk > 0) ? 1u : 0u);
                umma_commit_warp(&ms.pv_done[st]);
                umma_commit_warp(&ms.kv_empty[st]);   // the stage may be refilled
            };
            auto issue_qk = [&](int blk) {
                const int st = blk & 1;
                const uint64_t soff = (uint64_t)((st * C::kStageBytes) >> 4);
                const uint32_t d = tmem + C::kColS + st * NQ;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_f8_warp(d, qk_a_lat + soff + (uint64_t)((c * C::kLatChunkBytes + kk * 32) >> 4),
                                qk_b_lat + (uint64_t)((c * C::kQChunkBytes + kk * 32) >> 4), id_qk,
                                (c > 0 || kk > 0) ? 1u : 0u);
                if (C::kRope) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        umma_f8_warp(d, qk_a_rope + soff + (uint64_t)((kk * 32) >> 4),
                                qk_b_rope + (uint64_t)((kk * 32) >> 4), id_qk, 1u);
                }
                umma_commit_warp(&ms.s_full[st]);
            };
            // Event loop: QK of the next block as soon as its rows have landed
            // and its S buffer is free (so QK of block j+1 runs while the
            // softmax works on block j), P.V of the oldest block as soon as its
            // P is published (which frees the block's stage).  Both conditions
            // are polled without blocking; P.V goes first when both are ready.
            // No progress for a.wait_limit cycles ends the loop with the abort flag.
            int next_qk = 0, next_pv = 0;
            long long t_last = clock64();
            // a poll's outcome comes from lane 0, so every lane takes the same path
            auto ready = [&](uint64_t* bar, uint32_t parity) -> bool {
                return __shfl_sync(0xffffffffu, mbar_try_wait(bar, parity) ? 1 : 0, 0) != 0;
            };
            for (uint32_t idle = 0; next_pv < nblk;) {
                bool did = false;
                if (next_pv < next_qk && ready(&ms.p_full[next_pv & 1], (next_pv >> 1) & 1)) {
                    tc_fence_after();
                    issue_pv(next_pv);
                    if (lane == 0) MLA_BLOCK_STAMP(next_pv, 5);
                    if (next_pv == nblk - 1) {
                        umma_commit_warp(&ms.o_done);
                        if (lane == 0) MLA_STAMP(4);
                    }
                    ++next_pv;
                    did = true;
                }
                if (next_qk < nblk && ready(&ms.kv_full[next_qk & 1], (next_qk >> 1) & 1) &&
                    (next_qk < 2 || ready(&ms.s_free[next_qk & 1], ((next_qk - 2) >> 1) & 1))) {
                    tc_fence_after();
                    issue_qk(next_qk);
                    if (lane == 0) MLA_BLOCK_STAMP(next_qk, 2);
                    if (next_qk == 0 && lane == 0) MLA_STAMP(3);
                    ++next_qk;
                    did = true;
                }
                if (did) {
                    idle = 0;
                    continue;
                }
                if (++idle > 4) __nanosleep(kMmaSleepNs);
                if ((idle & 63u) == 0) {
                    const long long now = clock64();
                    if (*abort_flag) break;
                    if (idle == 64) t_last = now;   // first check of this idle stretch
                    else if (now - t_last > a.wait_limit) {
                        *abort_flag = 1;
                        break;
                    }
                }
            }
            // After an abort, MMAs already issued may still be running: wait
            // for them (with the full bound) before the CTA releases TMEM and
            // its stages.  Without one, o_done has already covered them.
            if (__shfl_sync(0xffffffffu, *abort_flag != 0 ? 1 : 0, 0) != 0) {
                umma_commit_warp(&ms.mma_drain);
                volatile int drain_abort = 0;
                warp_wait(&ms.mma_drain, 0, &drain_abort);
            }
        }
        __syncwarp();
    }
    } else {
        regs_raise<kRegsHigh>();
        // ================= softmax + epilogue (warps 8..15) ====================================
        // Two sets of four warps; set s owns query rows [s R, s R + R) (R = N / 2)
        // and warp w % 4 of a set owns TMEM lanes 32 (w % 4) .. +31 (one key per
        // thread), so two warps work on every key.
        constexpr int R = N / kSets;
        const int set = (warp - kSoftmaxWarp0) / 4;       // 0 or 1
        const int sw = (warp - kSoftmaxWarp0) % 4;        // warp within the set
        const uint32_t bar_id = 1u + 2u * (uint32_t)set;  // the set's named barrier
        const int r0 = set * R;                           // the set's first row
        const int quad = warp & 3;                        // TMEM lane quadrant of this warp
        const int ti = quad * 32 + lane;                  // key within a block == TMEM lane
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        constexpr int kLanesPerRow = 32 / R;              // lanes holding one row after a reduction
        const int my_row = lane / kLanesPerRow;           // set row whose sum this lane carries
        float* red = &ms.red[set * 4][0];                 // [4][32] of this set
        const bool q3 = ms.q3 != 0;                       // S^T has a q_lo column group
        float m_ref[R];
#pragma unroll
        for (int n = 0; n < R; ++n) m_ref[n] = -CUDART_INF_F;
        float l_thr[R];                                   // this thread's key: exact sums of p per row
#pragma unroll
        for (int n = 0; n < R; ++n) l_thr[n] = 0.f;
        float lt_acc[R];                                  // this thread's key: sums of p_hi + p_lo per row
#pragma unroll
        for (int n = 0; n < R; ++n) lt_acc[n] = 0.f;
        bool alive = true;
        // tests of the timeout path: a wait that nothing ends runs out (and
        // sets the abort flag) while the CTA's first copies are in flight
        if (a.stall_probe && nblk > 0) warp_wait(&ms.never, 0, abort_flag, 0, a.wait_limit);
        for (int blk = 0; blk < nblk; ++blk) {
            const int st = blk & 1;
            const uint32_t ph = (blk >> 1) & 1;
            bool ok = warp_wait(&ms.kv_full[st], ph, abort_flag, 0, a.wait_limit) &&
                      warp_wait(&ms.s_full[st], ph, abort_flag, 0, a.wait_limit);
            float s[R];
            if (ok) {
                tc_fence_after();
                const uint32_t sa = tmem + lane_addr + C::kColS + st * NQ + r0;
                if (q3) load_rows<R>(sa, sa + N, sa + 2 * N, s);
                else load_rows<R>(sa, sa + N, s);
                if ((warp & 3) == 0 && lane == 0) MLA_BLOCK_STAMP(blk, warp == kSoftmaxWarp0 ? 3 : 6);
            } else {
#pragma unroll
                for (int n = 0; n < R; ++n) s[n] = -CUDART_INF_F;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.s_free[st]);
            const bool kval = ms.kvalid[st][ti] != 0;
            const int j = k0 + blk * kBlockN + ti;
            // Per-row logit scales and windows as 16-byte loads, and a
            // branch-free mask.  The draft window only bites in blocks that reach
            // past the shortest row's window (kval already drops keys beyond
            // the split).
            const bool tail = k0 + (blk + 1) * kBlockN > win_min;
            const int jt = tail ? j : INT_MIN;
            bool need = false;
#pragma unroll
            for (int g = 0; g < R / 4; ++g) {
                const float4 c4 = reinterpret_cast<const float4*>(ms.cq + r0)[g];
                const int4 w4 = reinterpret_cast<const int4*>(ms.win + r0)[g];
                const float cq[4] = {c4.x, c4.y, c4.z, c4.w};
                const int wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int n = 4 * g + u;
                    const bool vis = kval && jt < wv[u];
                    s[n] = vis ? s[n] * cq[u] : -CUDART_INF_F;
                    need |= s[n] > m_ref[n] + kTau;
                }
            }
            if (softmax_bar_or(bar_id, !ok || *abort_flag)) {
                alive = false;
                break;
            }
            if (softmax_bar_or(bar_id, need)) {
                // new references: block max over the 128 keys, the set's four warps
                float v[R];
#pragma unroll
                for (int n = 0; n < R; ++n) v[n] = s[n];
                const float r = warp_transpose_reduce<R, true>(v, lane);
                if ((lane % kLanesPerRow) == 0) red[sw * 32 + my_row] = r;
                softmax_bar(bar_id);
                float alpha[R];
                uint32_t moved = 0;   // rows whose reference moved (same bits in every thread)
#pragma unroll
                for (int n = 0; n < R; ++n) {
                    const float bm = fmaxf(fmaxf(red[n], red[32 + n]), fmaxf(red[64 + n], red[96 + n]));
                    // only a row whose logits passed its reference by more than
                    // kTau moves it (bm is -inf when the row saw no valid key)
                    const float mn = bm > m_ref[n] + kTau ? bm + kHeadroom : m_ref[n];
                    float al = 1.f;
                    if (mn != m_ref[n])
                        al = (m_ref[n] == -CUDART_INF_F) ? 0.f : exp2f(m_ref[n] - mn);
                    alpha[n] = al;
                    if (al != 1.f) moved |= 1u << n;
                    m_ref[n] = mn;
                }
#pragma unroll
                for (int n = 0; n < R; ++n) {
                    l_thr[n] *= alpha[n];
                    lt_acc[n] *= alpha[n];
                }
                if (moved != 0 && blk > 0) {
                    // O^T holds blocks < blk: wait for the last P.V, then scale the
                    // columns (hi and lo, four d_v chunks) of the rows whose
                    // reference moved; the loop over rows is uniform.
                    if (warp_wait(&ms.pv_done[(blk - 1) & 1], ((blk - 1) >> 1) & 1, abort_flag, 0,
                                  a.wait_limit)) {
                        tc_fence_after();
#pragma unroll 1
                        while (moved != 0) {
                            const int n = __ffs(moved) - 1;
                            moved &= moved - 1;
                            float an = 1.f;
#pragma unroll
                            for (int k = 0; k < R; ++k)
                                if (k == n) an = alpha[k];
                            uint32_t rr[8];
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t ta = tmem + lane_addr + C::kColO + c * NC + r0 + n;
                                rr[2 * c] = tmem_ld1(ta);
                                rr[2 * c + 1] = tmem_ld1(ta + N);
                            }
                            tmem_wait_ld();
                            reg_fence(rr);
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t ta = tmem + lane_addr + C::kColO + c * NC + r0 + n;
                                tmem_st1(ta, __float_as_uint(__uint_as_float(rr[2 * c]) * an));
                                tmem_st1(ta + N, __float_as_uint(__uint_as_float(rr[2 * c + 1]) * an));
                            }
                        }
                        tmem_wait_st();
                    }
                }
            }
            // P^T row ti: bytes [0, N) = p_hi, [N, 2N) = p_lo, of p * 2^kShift; this
            // set writes bytes [r0, r0 + R) of each half.
            if (blk >= 2) warp_wait(&ms.pv_done[st], ((blk - 2) >> 1) & 1, abort_flag, 0, a.wait_limit);
            uint32_t hiw[R / 4], low[R / 4];
            // the reference minus kShift, finite: a row whose reference is still
            // -inf has seen no valid key, so all its logits are -inf too
            float mfin[R];
#pragma unroll
            for (int n = 0; n < R; ++n)
                mfin[n] = m_ref[n] == -CUDART_INF_F ? 0.f : m_ref[n] - kShift;
#pragma unroll
            for (int n = 0; n < R; n += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u)   // 2^-inf = 0 (mfin is finite)
                    s[n + u] = ex2_approx(s[n + u] - mfin[n + u]);
                uint16_t h0, l0, h1, l1;
                const float2 t0 = split_pair<kPLoBits>(s[n], s[n + 1], h0, l0);
                const float2 t1 = split_pair<kPLoBits>(s[n + 2], s[n + 3], h1, l1);
                lt_acc[n] += t0.x;
                lt_acc[n + 1] += t0.y;
                lt_acc[n + 2] += t1.x;
                lt_acc[n + 3] += t1.y;
#pragma unroll
                for (int u = 0; u < 4; ++u) l_thr[n + u] += s[n + u];
                hiw[n / 4] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                low[n / 4] = (uint32_t)l0 | ((uint32_t)l1 << 16);
            }
            // P^T is stored as 16-column blocks of 128 keys x 16 bytes
            uint8_t* prow = smem + C::kOffP + st * C::kPBytes + ti * 16;
            if constexpr (R == 16) {
                *reinterpret_cast<uint4*>(prow + set * 2048) =
                    make_uint4(hiw[0], hiw[1], hiw[2], hiw[3]);
                *reinterpret_cast<uint4*>(prow + (N / 16 + set) * 2048) =
                    make_uint4(low[0], low[1], low[2], low[3]);
            } else {
                *reinterpret_cast<uint2*>(prow + set * 8) = make_uint2(hiw[0], hiw[1]);
                *reinterpret_cast<uint2*>(prow + (N / 16) * 2048 + set * 8) = make_uint2(low[0], low[1]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[st]);
            if ((warp & 3) == 0 && lane == 0) MLA_BLOCK_STAMP(blk, warp == kSoftmaxWarp0 ? 4 : 7);
        }

        // ---- epilogue ------------------------------------------------------------------------
        // Row sums over all 128 keys -> the base-2 LSE per row (from the exact
        // fp32 p), and each row's output index; the per-thread sums of what the
        // MMA consumed (lt) are reduced over the set's keys the same way.  O^T
        // leaves TMEM already normalised (times 1/lt, and kv_scale into bf16 for
        // a single split) into the idle KV stages, and one bulk TMA store per
        // row writes it out.  Each set handles its own rows.
        {
            const float l_acc = warp_transpose_reduce<R, false>(l_thr, lane);
            const float t = warp_transpose_reduce<R, false>(lt_acc, lane);
            if ((lane % kLanesPerRow) == 0) {
                red[sw * 32 + my_row] = l_acc;
                ms.redt[set * 4 + sw][my_row] = t;
            }
        }
        softmax_bar(bar_id);
        const int ns = a.num_splits;
        if (ti < R) {
            const int row = r0 + ti;
            const float lsum = red[ti] + red[32 + ti] + red[64 + ti] + red[96 + ti];
            float mr = 0.f;
#pragma unroll
            for (int n = 0; n < R; ++n)
                if (n == ti) mr = m_ref[n];
            ms.fin[1][row] = lsum > 0.f ? mr + log2f(lsum) - kShift : -CUDART_INF_F;
            const int idx = hb * N + row;
            ms.row_item[row] = idx < rows_in_req
                ? ((int64_t)b * a.q_len + idx / a.num_heads) * a.num_heads + idx % a.num_heads
                : -1;
        }
        const bool have_o = alive && nblk > 0 && warp_wait(&ms.o_done, 0, abort_flag, 0, a.wait_limit);
        if (warp == kSoftmaxWarp0 && lane == 0) MLA_STAMP(5);
        if (have_o) tc_fence_after();
        softmax_bar(bar_id);
        // One split writes the final rows: bf16 into o, or fp32 into o_f32 when
        // the caller asked for fp32 output; several splits write fp32 partials.
        const bool final_rows = ns == 1;
        const bool final16 = final_rows && a.o_f32 == nullptr;
        const float fscale = final_rows ? a.out_scale : 1.f;
        float* ostage = reinterpret_cast<float*>(smem + C::kOffStage);              // fp32 [N][512]
        uint16_t* ostage16 = reinterpret_cast<uint16_t*>(smem + C::kOffStage);      // bf16 [N][512]
        // Row scale: 1 / (the consumed sum over all 128 keys of every block),
        // times the output scale for final rows.  The four d_v chunks leave TMEM
        // in two batches of loads (chunks 0-1, then 2-3), one wait each.
        float scl[R];
#pragma unroll
        for (int n = 0; n < R; ++n) {
            const float lt = (ms.redt[set * 4][n] + ms.redt[set * 4 + 1][n]) +
                             (ms.redt[set * 4 + 2][n] + ms.redt[set * 4 + 3][n]);
            scl[n] = (have_o && lt > 0.f) ? rcp_approx(lt) * fscale : 0.f;
        }
        auto stage_chunk = [&](int c, const uint32_t (&h)[R], const uint32_t (&l)[R]) {
            if (final16) {
#pragma unroll
                for (int n = 0; n < R; ++n)
                    ostage16[(r0 + n) * 512 + c * 128 + ti] = __bfloat16_as_ushort(__float2bfloat16_rn(
                        fmaf(__uint_as_float(l[n]), kPLoBack, __uint_as_float(h[n])) * scl[n]));
            } else {
#pragma unroll
                for (int n = 0; n < R; ++n)
                    ostage[(r0 + n) * 512 + c * 128 + ti] =
                        fmaf(__uint_as_float(l[n]), kPLoBack, __uint_as_float(h[n])) * scl[n];
            }
        };
        {
            uint32_t h0[R], l0[R], h1[R], l1[R];
            if (have_o) {
                const uint32_t oa = tmem + lane_addr + C::kColO + r0;
                issue_rows<R>(oa, oa + N, h0, l0);
                issue_rows<R>(oa + NC, oa + NC + N, h1, l1);
                tmem_wait_ld();
                reg_fence(h0);
                reg_fence(l0);
                reg_fence(h1);
                reg_fence(l1);
            } else {
#pragma unroll
                for (int n = 0; n < R; ++n) h0[n] = l0[n] = h1[n] = l1[n] = 0u;
            }
            stage_chunk(0, h0, l0);
            stage_chunk(1, h1, l1);
        }
        {
            uint32_t h2[R], l2[R], h3[R], l3[R];
            if (have_o) {
                const uint32_t oa = tmem + lane_addr + C::kColO + r0;
                issue_rows<R>(oa + 2 * NC, oa + 2 * NC + N, h2, l2);
                issue_rows<R>(oa + 3 * NC, oa + 3 * NC + N, h3, l3);
                tmem_wait_ld();
                reg_fence(h2);
                reg_fence(l2);
                reg_fence(h3);
                reg_fence(l3);
            } else {
#pragma unroll
                for (int n = 0; n < R; ++n) h2[n] = l2[n] = h3[n] = l3[n] = 0u;
            }
            stage_chunk(2, h2, l2);
            stage_chunk(3, h3, l3);
        }
        fence_proxy_async_smem();
        softmax_bar(bar_id);
        if (warp == kSoftmaxWarp0 && lane == 0) MLA_STAMP(6);
        // (a fused merge reads the staged partials from shared memory instead)
        if (MC == 1 && ti < R) {
            const int row = r0 + ti;
            const long long item = ms.row_item[row];
            if (item >= 0) {
                if (final16) {
                    bulk_store(a.o + item * C::kDv, ostage16 + row * 512, C::kDv * 2);
                    if (a.lse) a.lse[item] = ms.fin[1][row];
                } else if (final_rows) {
                    bulk_store(a.o_f32 + item * C::kDv, ostage + row * 512, C::kDv * 4);
                    if (a.lse) a.lse[item] = ms.fin[1][row];
                } else {
                    bulk_store(a.o_part + (item * ns + split) * C::kDv, ostage + row * 512, C::kDv * 4);
                    a.lse_part[item * ns + split] = ms.fin[1][row];
                }
                bulk_commit();
                bulk_wait_read();
            }
        }
        if (warp == kSoftmaxWarp0 && lane == 0) MLA_STAMP(7);
        if ((!alive || *abort_flag) && lane == 0) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
    }

    // ---- teardown -------------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
    if constexpr (MC > 1) fused_merge<N, SPARSE, MC>(smem, ms, a, b, hb, split);
    if (tid == kSoftmaxWarp0 * 32) MLA_STAMP(8);
}

// ---- host side -------------------------------------------------------------------------------

// One launch of split_tc_kernel<N, SPARSE, EXTRA, MC>: a programmatic dependent
// of the preceding kernel on the stream, in clusters of MC consecutive splits
// when MC > 1 (the fused merge).
template <int N, bool SPARSE, bool EXTRA, int MC>
cudaError_t launch_variant(const CUtensorMap& lat, const CUtensorMap& rope, const SplitArgs& a,
                           const mla_plan_t& plan, cudaStream_t stream)
{
    constexpr int smem = smem_bytes<N, SPARSE>();
    static_assert(smem <= 227 * 1024, "one CTA's dynamic shared memory limit");
    // The shared-memory opt-in is a per-device attribute of the kernel: set it
    // once on every device this process launches on.
    static DeviceOnce once;
    cudaError_t e = once.run([] {
        return cudaFuncSetAttribute(split_tc_kernel<N, SPARSE, EXTRA, MC>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid_x, plan.grid_y, plan.grid_z);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute la[2];
    // a programmatic dependent of the preceding kernel: set-up overlaps its tail
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    if (MC > 1) {
        la[1].id = cudaLaunchAttributeClusterDimension;
        la[1].val.clusterDim.x = 1;
        la[1].val.clusterDim.y = MC;
        la[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelEx(&cfg, split_tc_kernel<N, SPARSE, EXTRA, MC>, lat, rope, a);
}

// The launch for rows per CTA and merge cluster size given at run time.
template <bool SPARSE, bool EXTRA>
cudaError_t launch_rows_mc(const CUtensorMap& lat, const CUtensorMap& rope, const SplitArgs& a,
                           const mla_plan_t& plan, int mc, cudaStream_t stream)
{
    if (plan.rows_per_cta == 16) {
        switch (mc) {
        case 2: return launch_variant<16, SPARSE, EXTRA, 2>(lat, rope, a, plan, stream);
        case 4: return launch_variant<16, SPARSE, EXTRA, 4>(lat, rope, a, plan, stream);
        default: return launch_variant<16, SPARSE, EXTRA, 1>(lat, rope, a, plan, stream);
        }
    }
    switch (mc) {
    case 2: return launch_variant<32, SPARSE, EXTRA, 2>(lat, rope, a, plan, stream);
    case 4: return launch_variant<32, SPARSE, EXTRA, 4>(lat, rope, a, plan, stream);
    default: return launch_variant<32, SPARSE, EXTRA, 1>(lat, rope, a, plan, stream);
    }
}

}  // namespace
}  // namespace mla
