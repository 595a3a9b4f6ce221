// mla_split_tc.cu -- tcgen05 / TMA split kernel for absorbed-MLA decode (sm_103a).
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
//   dequantised copy is ever written.  The small operands are split exactly into
//   two e4m3 terms: each query row q is scaled by a power of two and written as
//   q_hi + q_lo (exact for every element within 2^-9 of the row maximum, bf16
//   having 8 significant bits), and each probability p as p_hi + p_lo (about as
//   precise as rounding p to bf16).  hi and lo are stacked along N (2N MMA
//   columns), so the big operand is read from shared memory once per MMA.
//   kv_scale and the powers of two are folded into the logit and output scales.
// * Warp roles.  Warp 0 gathers rows with TMA tile::gather4 (four slots per
//   instruction, 128-byte latent boxes with 128B swizzle, a 64-byte RoPE box with
//   64B swizzle) into a two-stage ring; warp 1 issues the tcgen05.mma
//   (kind::f8f6f4, fp32 accumulators in TMEM) and commits to mbarriers; warps 2-5
//   own one TMEM lane (= one key) each and run the online base-2 softmax.
// * Lazy rescaling.  A block only recomputes the running maxima when some logit
//   exceeds them by more than kTau; otherwise p = 2^(s - m) stays below 2^kTau.
//   O in TMEM is rescaled only at those (rare) blocks.
// * Sums.  l (exact fp32 p, for the LSE) and lt (the fp8-split p actually fed to
//   the MMA, for normalising O) are kept per thread and reduced once at the end.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "mla_internal.h"
#include "mla_sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBlockN = 128;          // keys per block (MMA M)
constexpr int kThreads = 192;         // warp 0 TMA, warp 1 MMA, warps 2..5 softmax
constexpr float kTau = 2.f;           // lazy-rescale threshold, base-2 logit units
constexpr float kShift = 6.f;         // p is fed as p * 2^kShift: at most 2^(kTau + kShift) = 256

template <int N, bool SPARSE>
struct Cfg {
    static constexpr int NC = 2 * N;                       // MMA columns: hi rows, then lo rows
    static constexpr int kRowBytes = SPARSE ? 512 : 576;   // pool row width
    static constexpr bool kRope = !SPARSE;                 // separate 64-byte RoPE chunk
    static constexpr int kLatChunkBytes = kBlockN * 128;   // 16 KB per 128-column chunk
    static constexpr int kStageBytes = kBlockN * kRowBytes;
    static constexpr int kQChunkBytes = NC * 128;
    static constexpr int kQBytes = 4 * kQChunkBytes + (kRope ? NC * 64 : 0);
    static constexpr int kPBytes = kBlockN * NC;
    static constexpr int kDv = SPARSE ? 448 : 512;
    static constexpr int kOffStage = 0;
    static constexpr int kOffQ = 2 * kStageBytes;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffMisc = kOffP + 2 * kPBytes;
    static constexpr uint32_t kTmemCols = (6 * NC <= 256) ? 256u : 512u;
    static constexpr uint32_t kColS = 0;                   // S^T buffers: [0, 2 NC)
    static constexpr uint32_t kColO = 2 * NC;              // O^T chunks:  [2 NC, 6 NC)
    static_assert(kOffQ % 1024 == 0 && kQChunkBytes % 1024 == 0, "128B-swizzle atoms");
    static_assert(kOffP % 16 == 0, "P tile alignment");
    static_assert(6 * NC <= 512, "TMEM columns");
};

struct Misc {
    uint64_t kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full[2], o_done;
    uint64_t sm_bar;    // barrier of the 4 softmax warps (one arrival per warp)
    uint32_t tmem_base;
    int abort;
    int kvalid[2][kBlockN];
    float cq[32];       // per query row: raw dot -> base-2 logit
    int win[32];        // per query row: keys at positions < win are visible
    float red[4][32];   // cross-warp reduction scratch
    int vote[2][4];
};

template <int N, bool SPARSE>
constexpr int smem_bytes()
{
    return Cfg<N, SPARSE>::kOffMisc + (int)sizeof(Misc);
}

// Byte offset of column c (0 <= c < row width) of operand row `row` in a tile
// of `rows` rows laid out as four 128B-swizzled 128-column chunks followed by
// one 64B-swizzled 64-column chunk (the canonical K-major layouts; the same
// bytes read as MN-major give V^T).
__device__ __forceinline__ int tile_offset(int row, int c, int rows)
{
    if (c < 512) {
        const int chunk = c >> 7, kb = c & 127;
        return chunk * rows * 128 + (row >> 3) * 1024 + (row & 7) * 128 +
               (((kb >> 4) ^ (row & 7)) << 4) + (kb & 15);
    }
    const int kb = c - 512;
    return 4 * rows * 128 + (row >> 3) * 512 + (row & 7) * 64 +
           (((kb >> 4) ^ ((row & 7) >> 1)) << 4) + (kb & 15);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t u)
{
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// Split two fp32 values into e4m3 hi/lo bytes (pairs packed lo-byte first);
// returns the values the pair of bytes represents (hi + lo).
__device__ __forceinline__ float2 split_pair(float a, float b, uint16_t& hi, uint16_t& lo)
{
    hi = f32x2_to_e4m3x2(a, b);
    const float2 h = e4m3x2_to_f32x2(hi);
    lo = f32x2_to_e4m3x2(a - h.x, b - h.y);
    const float2 l = e4m3x2_to_f32x2(lo);
    return make_float2(h.x + l.x, h.y + l.y);
}

// Bounded wait whose outcome is the same on every lane of the warp (all lanes
// must call it), so no warp-collective instruction is reached divergently.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort)
{
    const bool ok = mbar_wait_or_abort(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Barrier of the four softmax warps, built on an mbarrier so that it is
// bounded: a warp that stopped early makes the others time out, not hang.
// `phase` counts the barrier instances this thread has passed.
__device__ __forceinline__ bool softmax_sync(uint64_t* bar, uint32_t& phase, volatile int* abort)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
    const bool ok = warp_wait(bar, phase & 1, abort);
    ++phase;
    return ok;
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

// Reduce N per-thread values over the 128 softmax threads; every softmax
// thread receives all N results in out[].  False if a barrier timed out.
template <int N, bool MAX>
__device__ __forceinline__ bool block_reduce(const float (&in)[N], float (&out)[N], Misc& ms,
                                             int sw, int lane, uint32_t& phase,
                                             volatile int* abort)
{
    float v[N];
#pragma unroll
    for (int n = 0; n < N; ++n) v[n] = in[n];
    const float r = warp_transpose_reduce<N, MAX>(v, lane);
    constexpr int kLanesPerValue = 32 / N;
    if ((lane % kLanesPerValue) == 0) ms.red[sw][lane / kLanesPerValue] = r;
    if (!softmax_sync(&ms.sm_bar, phase, abort)) return false;
#pragma unroll
    for (int n = 0; n < N; ++n) {
        float x = ms.red[0][n];
#pragma unroll
        for (int w = 1; w < 4; ++w) x = MAX ? fmaxf(x, ms.red[w][n]) : x + ms.red[w][n];
        out[n] = x;
    }
    return softmax_sync(&ms.sm_bar, phase, abort);
}

template <int N, bool SPARSE>
__global__ void __launch_bounds__(kThreads, 1)
split_tc_kernel(const __grid_constant__ CUtensorMap tm_lat,
                const __grid_constant__ CUtensorMap tm_rope, const SplitArgs a)
{
    using C = Cfg<N, SPARSE>;
    constexpr int NC = C::NC;
    extern __shared__ __align__(1024) uint8_t smem[];
    Misc& ms = *reinterpret_cast<Misc*>(smem + C::kOffMisc);
    volatile int* abort_flag = &ms.abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hb = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
    const int rows_in_req = a.q_len * a.num_heads;

    // ---- the request's key list and this split's range --------------------------------
    int64_t base;
    int L;
    if (SPARSE) {
        base = (int64_t)b * a.topk;
        L = a.topk;
    } else {
        base = a.kv_indptr[b];
        const int cap = a.kv_indptr[b + 1] - a.kv_indptr[b];
        L = a.seq_lens[b];
        if (L < 0 || L > cap) {
            if (tid == 0) atomicOr(a.err, MLA_DEVERR_BAD_LENGTH);
            L = L < 0 ? 0 : cap;
        }
    }
    const int chunk = (L + a.num_splits - 1) / a.num_splits;
    const int k0 = min(L, split * chunk);
    const int k1 = min(L, k0 + chunk);
    const int nblk = (k1 - k0 + kBlockN - 1) / kBlockN;

    // ---- set-up: barriers, TMEM, the query tile --------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.kv_full[i], 1);
            mbar_init(&ms.kv_empty[i], 1);
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.s_free[i], 4);
            mbar_init(&ms.p_full[i], 4);
        }
        mbar_init(&ms.o_done, 1);
        mbar_init(&ms.sm_bar, 4);
        ms.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ms.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_lat);
        if (C::kRope) tma_prefetch_desc(&tm_rope);
    }
    // Query rows: q scaled by 2^e so that max |q| is in [128, 256), then split
    // into e4m3 hi (rows 0..N-1) and lo (rows N..2N-1).
    constexpr int kWidth = C::kRowBytes;
    constexpr int kPerLane = kWidth / 32;
    uint8_t* qtile = smem + C::kOffQ;
    for (int n = warp; n < N; n += kThreads / 32) {
        const int idx = hb * N + n;
        const bool valid = idx < rows_in_req;
        int t = 0;
        int64_t item = 0;
        if (valid) {
            t = idx / a.num_heads;
            item = ((int64_t)b * a.q_len + t) * a.num_heads + idx % a.num_heads;
        }
        float qv[kPerLane];
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
            const int c = lane + 32 * k;
            float v = 0.f;
            if (valid)
                v = c < a.d_v ? bf16_bits_to_f32(a.q_lat[item * a.d_v + c])
                              : bf16_bits_to_f32(a.q_pe[item * a.d_rope + (c - a.d_v)]);
            qv[k] = v;
            amax = fmaxf(amax, fabsf(v));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        int e = 0;
        if (amax > 0.f) frexpf(amax, &e);
        const int sh = amax > 0.f ? 8 - e : 0;   // max |q * 2^sh| in [128, 256)
#pragma unroll
        for (int k = 0; k < kPerLane; k += 2) {
            uint16_t hi, lo;
            split_pair(ldexpf(qv[k], sh), ldexpf(qv[k + 1], sh), hi, lo);
            const int c0 = lane + 32 * k, c1 = c0 + 32;
            qtile[tile_offset(n, c0, NC)] = (uint8_t)(hi & 0xFF);
            qtile[tile_offset(n, c1, NC)] = (uint8_t)(hi >> 8);
            qtile[tile_offset(N + n, c0, NC)] = (uint8_t)(lo & 0xFF);
            qtile[tile_offset(N + n, c1, NC)] = (uint8_t)(lo >> 8);
        }
        if (lane == 0) {
            ms.cq[n] = valid ? a.logit_scale * ldexpf(1.f, -sh) : 0.f;
            ms.win[n] = valid ? (L - a.q_len + t + 1) : -1;
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ms.tmem_base;
    const uint32_t smem_base = smem_u32(smem);

    if (warp == 0) {
        // ================= TMA producer =================================================
        const int32_t* list = a.kv_indices + base;
        int32_t slot[4];
        int ok[4];
        auto load_slots = [&](int blk) {
            const int kb = k0 + blk * kBlockN;
            const int nk = min(kBlockN, k1 - kb);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 4 * lane + q;
                int32_t s = -1;
                ok[q] = 0;
                if (j < nk) {
                    s = __ldg(list + kb + j);
                    if (s >= 0 && (int64_t)s < a.pool_rows) ok[q] = 1;
                    else if (!(SPARSE && s < 0)) atomicOr(a.err, MLA_DEVERR_BAD_SLOT);
                }
                slot[q] = ok[q] ? s : 0;   // masked keys load row 0: finite bytes, p = 0
            }
        };
        if (nblk > 0) load_slots(0);
        for (int blk = 0; blk < nblk; ++blk) {
            const int st = blk & 1;
            if (blk >= 2 && !warp_wait(&ms.kv_empty[st], ((blk - 2) >> 1) & 1, abort_flag))
                break;
#pragma unroll
            for (int q = 0; q < 4; ++q) ms.kvalid[st][4 * lane + q] = ok[q];
            // Every block gathers all 128 rows (masked keys read pool row 0), so the
            // stage never holds stale or uninitialised bytes: a masked key's p is 0
            // and 0 * (a finite fp8 value) is 0 in P.V.
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&ms.kv_full[st], (uint32_t)(kBlockN * kWidth));
            __syncwarp();
            {
                uint8_t* stage = smem + C::kOffStage + st * C::kStageBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    tma_gather4(stage + c * C::kLatChunkBytes + lane * 512, &tm_lat, c * 128,
                                slot[0], slot[1], slot[2], slot[3], &ms.kv_full[st]);
                if (C::kRope)
                    tma_gather4(stage + 4 * C::kLatChunkBytes + lane * 256, &tm_rope, 512,
                                slot[0], slot[1], slot[2], slot[3], &ms.kv_full[st]);
            }
            if (blk + 1 < nblk) load_slots(blk + 1);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =====================================================
        if (lane == 0 && nblk > 0) {
            const uint32_t id_qk = idesc_e4m3(128, NC, false, false);
            const uint32_t id_pv = idesc_e4m3(128, NC, true, true);
            auto issue_pv = [&](int blk) {
                const int st = blk & 1;
                const uint32_t stage = smem_base + C::kOffStage + st * C::kStageBytes;
                const uint32_t pt = smem_base + C::kOffP + st * C::kPBytes;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = smem_desc(stage + c * C::kLatChunkBytes + kk * 4096,
                                                      C::kLatChunkBytes, 1024, kSw128);
                        const uint64_t bd = smem_desc(pt + kk * 512, 128, 2048, kSwNone);
                        umma_f8(tmem + C::kColO + c * NC, ad, bd, id_pv,
                                (blk > 0 || kk > 0) ? 1u : 0u);
                    }
                umma_commit(&ms.kv_empty[st]);
            };
            bool alive = true;
            for (int blk = 0; blk < nblk && alive; ++blk) {
                const int st = blk & 1;
                if (!mbar_wait_or_abort(&ms.kv_full[st], (blk >> 1) & 1, abort_flag)) break;
                if (blk >= 2 &&
                    !mbar_wait_or_abort(&ms.s_free[st], ((blk - 2) >> 1) & 1, abort_flag))
                    break;
                tc_fence_after();
                const uint32_t stage = smem_base + C::kOffStage + st * C::kStageBytes;
                const uint32_t qb = smem_base + C::kOffQ;
                const uint32_t d = tmem + C::kColS + st * NC;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad =
                            smem_desc(stage + c * C::kLatChunkBytes + kk * 32, 16, 1024, kSw128);
                        const uint64_t bd =
                            smem_desc(qb + c * C::kQChunkBytes + kk * 32, 16, 1024, kSw128);
                        umma_f8(d, ad, bd, id_qk, (c > 0 || kk > 0) ? 1u : 0u);
                    }
                if (C::kRope) {
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint64_t ad =
                            smem_desc(stage + 4 * C::kLatChunkBytes + kk * 32, 16, 512, kSw64);
                        const uint64_t bd =
                            smem_desc(qb + 4 * C::kQChunkBytes + kk * 32, 16, 512, kSw64);
                        umma_f8(d, ad, bd, id_qk, 1u);
                    }
                }
                umma_commit(&ms.s_full[st]);
                if (blk >= 1) {
                    if (!mbar_wait_or_abort(&ms.p_full[(blk - 1) & 1], ((blk - 1) >> 1) & 1,
                                            abort_flag)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(blk - 1);
                }
            }
            if (alive && !*abort_flag) {
                const int last = nblk - 1;
                if (mbar_wait_or_abort(&ms.p_full[last & 1], (last >> 1) & 1, abort_flag)) {
                    tc_fence_after();
                    issue_pv(last);
                    umma_commit(&ms.o_done);
                }
            }
        }
        __syncwarp();
    } else {
        // ================= softmax + epilogue (warps 2..5) =====================================
        const int sw = warp - 2;                  // 0..3
        const int quad = warp & 3;                // TMEM lane quadrant of this warp
        const int ti = quad * 32 + lane;          // key within a block == TMEM lane
        const uint32_t lane_addr = (uint32_t)(quad * 32) << 16;
        float m_ref[N], l_part[N], lt_part[N], cq[N];
        int win[N];
#pragma unroll
        for (int n = 0; n < N; ++n) {
            m_ref[n] = -CUDART_INF_F;
            l_part[n] = 0.f;
            lt_part[n] = 0.f;
            cq[n] = ms.cq[n];
            win[n] = ms.win[n];
        }
        bool alive = true;
        uint32_t sphase = 0;   // softmax barrier instances passed
        for (int blk = 0; blk < nblk; ++blk) {
            const int st = blk & 1;
            const uint32_t ph = (blk >> 1) & 1;
            if (!warp_wait(&ms.kv_full[st], ph, abort_flag) ||
                !warp_wait(&ms.s_full[st], ph, abort_flag)) {
                alive = false;
                break;
            }
            tc_fence_after();
            const bool kval = ms.kvalid[st][ti] != 0;
            const int j = k0 + blk * kBlockN + ti;
            float s[N];
            {
                uint32_t r[32];
                if (NC == 32) {
                    tmem_ld32(tmem + lane_addr + C::kColS + st * NC, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int n = 0; n < N; ++n)
                        s[n] = __uint_as_float(r[n]) + __uint_as_float(r[(n + N) & 31]);
                } else {
                    uint32_t r2[32];
                    tmem_ld32(tmem + lane_addr + C::kColS + st * NC, r);
                    tmem_ld32(tmem + lane_addr + C::kColS + st * NC + 32, r2);
                    tmem_wait_ld();
#pragma unroll
                    for (int n = 0; n < N; ++n)
                        s[n] = __uint_as_float(r[n & 31]) + __uint_as_float(r2[n & 31]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.s_free[st]);
            bool need = false;
#pragma unroll
            for (int n = 0; n < N; ++n) {
                s[n] = (kval && j < win[n]) ? s[n] * cq[n] : -CUDART_INF_F;
                need |= s[n] > m_ref[n] + kTau;
            }
            need = __any_sync(0xffffffffu, need);
            if (lane == 0) ms.vote[blk & 1][sw] = need ? 1 : 0;
            if (!softmax_sync(&ms.sm_bar, sphase, abort_flag)) {
                alive = false;
                break;
            }
            need = (ms.vote[blk & 1][0] | ms.vote[blk & 1][1] | ms.vote[blk & 1][2] |
                    ms.vote[blk & 1][3]) != 0;
            if (need) {
                float bm[N];
                if (!block_reduce<N, true>(s, bm, ms, sw, lane, sphase, abort_flag)) {
                    alive = false;
                    break;
                }
                float alpha[N];
                bool rescale = false;
#pragma unroll
                for (int n = 0; n < N; ++n) {
                    const float mn = fmaxf(m_ref[n], bm[n]);
                    float al = 1.f;
                    if (mn != -CUDART_INF_F)
                        al = (m_ref[n] == -CUDART_INF_F) ? 0.f : exp2f(m_ref[n] - mn);
                    alpha[n] = al;
                    rescale |= al != 1.f;
                    m_ref[n] = mn;
                    l_part[n] *= al;
                    lt_part[n] *= al;
                }
                if (rescale && blk > 0) {
                    // O^T holds blocks < blk: wait for the last P.V, then scale its columns.
                    if (!warp_wait(&ms.kv_empty[(blk - 1) & 1], ((blk - 1) >> 1) & 1,
                                   abort_flag)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
#pragma unroll
                        for (int h = 0; h < NC / 32; ++h) {
                            uint32_t r[32];
                            const uint32_t ta = tmem + lane_addr + C::kColO + c * NC + h * 32;
                            tmem_ld32(ta, r);
                            tmem_wait_ld();
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha[(h * 32 + k) % N]);
                            tmem_st32(ta, r);
                        }
                    }
                    tmem_wait_st();
                }
            }
            // P^T row ti: bytes [0, N) = p_hi, [N, 2N) = p_lo, of p * 2^kShift.
            if (blk >= 2 && !warp_wait(&ms.kv_empty[st], ((blk - 2) >> 1) & 1, abort_flag)) {
                alive = false;
                break;
            }
            uint32_t hiw[N / 4], low[N / 4];
#pragma unroll
            for (int n = 0; n < N; n += 4) {
                float p[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float x = s[n + u];
                    p[u] = (x == -CUDART_INF_F || m_ref[n + u] == -CUDART_INF_F)
                               ? 0.f : exp2f(x - m_ref[n + u] + kShift);
                    l_part[n + u] += p[u];
                }
                uint16_t h0, l0, h1, l1;
                const float2 v0 = split_pair(p[0], p[1], h0, l0);
                const float2 v1 = split_pair(p[2], p[3], h1, l1);
                lt_part[n] += v0.x;
                lt_part[n + 1] += v0.y;
                lt_part[n + 2] += v1.x;
                lt_part[n + 3] += v1.y;
                hiw[n / 4] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                low[n / 4] = (uint32_t)l0 | ((uint32_t)l1 << 16);
            }
            uint8_t* prow = smem + C::kOffP + st * C::kPBytes + ti * 16;
#pragma unroll
            for (int g = 0; g < N / 16; ++g) {
                *reinterpret_cast<uint4*>(prow + g * 2048) =
                    make_uint4(hiw[4 * g], hiw[4 * g + 1], hiw[4 * g + 2], hiw[4 * g + 3]);
                *reinterpret_cast<uint4*>(prow + (N / 16 + g) * 2048) =
                    make_uint4(low[4 * g], low[4 * g + 1], low[4 * g + 2], low[4 * g + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[st]);
        }

        // ---- epilogue ------------------------------------------------------------------------
        float l[N], lt[N];
        alive = alive && !*abort_flag;
        if (alive) alive = block_reduce<N, false>(l_part, l, ms, sw, lane, sphase, abort_flag);
        if (alive) alive = block_reduce<N, false>(lt_part, lt, ms, sw, lane, sphase, abort_flag);
        if (!alive) {
#pragma unroll
            for (int n = 0; n < N; ++n) l[n] = lt[n] = 0.f;
        }
        const bool have_o = alive && nblk > 0 && warp_wait(&ms.o_done, 0, abort_flag);
        if (have_o) tc_fence_after();
        const int ns = a.num_splits;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            const int d = c * 128 + ti;
            float o[N];
            if (have_o) {
                uint32_t r[32];
                if (NC == 32) {
                    tmem_ld32(tmem + lane_addr + C::kColO + c * NC, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int n = 0; n < N; ++n)
                        o[n] = __uint_as_float(r[n]) + __uint_as_float(r[(n + N) & 31]);
                } else {
                    uint32_t r2[32];
                    tmem_ld32(tmem + lane_addr + C::kColO + c * NC, r);
                    tmem_ld32(tmem + lane_addr + C::kColO + c * NC + 32, r2);
                    tmem_wait_ld();
#pragma unroll
                    for (int n = 0; n < N; ++n)
                        o[n] = __uint_as_float(r[n & 31]) + __uint_as_float(r2[n & 31]);
                }
            } else {
#pragma unroll
                for (int n = 0; n < N; ++n) o[n] = 0.f;
            }
            if (d >= C::kDv) continue;
#pragma unroll
            for (int n = 0; n < N; ++n) {
                const int idx = hb * N + n;
                if (idx >= rows_in_req) break;
                const int64_t item =
                    ((int64_t)b * a.q_len + idx / a.num_heads) * a.num_heads + idx % a.num_heads;
                const float val = lt[n] > 0.f ? o[n] / lt[n] : 0.f;
                if (ns == 1)
                    reinterpret_cast<__nv_bfloat16*>(a.o)[item * C::kDv + d] =
                        __float2bfloat16_rn(val * a.out_scale);
                else
                    a.o_part[(item * ns + split) * C::kDv + d] = val;
            }
        }
        if (ti < N) {
            const int idx = hb * N + ti;
            if (idx < rows_in_req) {
                const int64_t item =
                    ((int64_t)b * a.q_len + idx / a.num_heads) * a.num_heads + idx % a.num_heads;
                float lsum = 0.f, mr = 0.f;
#pragma unroll
                for (int n = 0; n < N; ++n)
                    if (n == ti) {
                        lsum = l[n];
                        mr = m_ref[n];
                    }
                const float lse2 = lsum > 0.f ? mr + log2f(lsum) - kShift : -CUDART_INF_F;
                if (ns == 1) {
                    if (a.lse) a.lse[item] = lse2;
                } else {
                    a.lse_part[item * ns + split] = lse2;
                }
            }
        }
        if (!alive || *abort_flag) {
            if (lane == 0) atomicOr(a.err, MLA_DEVERR_TIMEOUT);
        }
    }

    // ---- teardown -------------------------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---- host side -------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

bool make_row_map(CUtensorMap* m, const void* pool, int64_t rows, int row_bytes, int box,
                  CUtensorMapSwizzle sw)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t gstr[1] = {(cuuint64_t)row_bytes};
    cuuint32_t bdim[2] = {(cuuint32_t)box, 1};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(pool), gdim, gstr, bdim, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N, bool SPARSE>
cudaError_t launch_variant(const CUtensorMap& lat, const CUtensorMap& rope, const SplitArgs& a,
                           const mla_plan_t& plan, cudaStream_t stream)
{
    constexpr int smem = smem_bytes<N, SPARSE>();
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(split_tc_kernel<N, SPARSE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr != cudaSuccess) return attr;
    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    split_tc_kernel<N, SPARSE><<<grid, kThreads, smem, stream>>>(lat, rope, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_split_tc(const SplitArgs& a, const mla_plan_t& plan, cudaStream_t stream)
{
    if (plan.grid_x <= 0 || plan.grid_y <= 0 || plan.grid_z <= 0) return cudaSuccess;
    CUtensorMap lat, rope;
    const int row_bytes = a.d_v + a.d_rope;
    if (!make_row_map(&lat, a.pool, a.pool_rows, row_bytes, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!a.sparse) {
        if (!make_row_map(&rope, a.pool, a.pool_rows, row_bytes, 64, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else {
        rope = lat;
    }
    if (a.sparse) {
        if (plan.rows_per_cta == 16) return launch_variant<16, true>(lat, rope, a, plan, stream);
        return launch_variant<32, true>(lat, rope, a, plan, stream);
    }
    if (plan.rows_per_cta == 16) return launch_variant<16, false>(lat, rope, a, plan, stream);
    return launch_variant<32, false>(lat, rope, a, plan, stream);
}

}  // namespace mla
