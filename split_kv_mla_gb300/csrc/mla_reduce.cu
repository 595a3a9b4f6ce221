// mla_reduce.cu -- split-K reduce of normalized fp32 partials with base-2 LSEs.
//
// hip_mha_decoding_num_partitions (split-K target and the reducer that merges up
// to 256 partitions).  The arithmetic and its fixed association are those of
// mla_merge.cuh.  One CTA per row: each thread owns four consecutive columns and
// reads them with 16-byte loads, so every split's row is one coalesced sweep.
// In the narrow form 128 threads each load every split's columns; in the wide
// form (above 16 splits, or above 8 with at most 128 rows) four groups of 128
// threads each take every fourth split (the interleaved groups of the fixed
// association) and add their sums through shared memory.
// A thread's first kPrefetch loads are in flight while warp 0 loads the row's
// LSEs and forms the weights, so a row of up to 64 splits costs one round trip
// to L2 (measured: B=1 H=64 S=131072 at 69 splits, the rest of the call after
// the split kernel 8.8 us with one 128-thread group).
//
// The kernel is launched as a programmatic dependent of the split kernel: its
// CTAs can be scheduled while the split kernel drains, and griddepcontrol.wait
// holds them until the split kernel has completed and its writes are visible.
// Launched after anything else (or without the launch attribute) the wait
// returns at once.  It lets its own dependents (the next split kernel, whose
// set-up then overlaps this kernel) be scheduled once every row has started.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"
#include "mla_merge.cuh"

namespace mla {
namespace {

constexpr int kReduceThreads = 128;   // threads of one split group (four columns each)
constexpr int kPrefetch = 16;         // loads in flight per thread
constexpr int kWideGroups = 4;        // split groups of a row in the wide form
constexpr int kWideMaxRows = 128;     // ... also taken above 8 splits up to this many rows

// Four merged columns scaled by f, stored as bf16 or fp32.
__device__ __forceinline__ void store4(__nv_bfloat16* o, float4 acc, float f)
{
    *reinterpret_cast<uint2*>(o) = merge_pack_bf16(acc, f);
}
__device__ __forceinline__ void store4(float* o, float4 acc, float f)
{
    *reinterpret_cast<float4*>(o) = make_float4(acc.x * f, acc.y * f, acc.z * f, acc.w * f);
}

template <typename OutT, int G>
__global__ void __launch_bounds__(kReduceThreads * G)
splitk_reduce_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                     int64_t rows, int num_splits, int d_v, float out_scale,
                     OutT* __restrict__ o, float* __restrict__ lse)
{
    __shared__ float w_s[MLA_MAX_SPLITS];
    __shared__ float fscale;
    __shared__ float4 gsum[G > 1 ? G - 1 : 1][kReduceThreads];   // groups 1..G-1's sums

    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next call's split kernel may be scheduled as soon as all rows started
    asm volatile("griddepcontrol.launch_dependents;");
    const int64_t row = blockIdx.x;
    if (row >= rows) return;
    const int tid = threadIdx.x;
    const int g = tid / kReduceThreads;   // split group: s = g, g + G, ...
    const int c = (tid % kReduceThreads) * 4;
    const bool cols = c < d_v;
    const float* op = o_part + row * (int64_t)num_splits * d_v + c;
    float4 v[kPrefetch];
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u) {
        const int sp = g + G * u;
        if (cols && sp < num_splits)
            v[u] = __ldcg(reinterpret_cast<const float4*>(op + (int64_t)sp * d_v));
    }
    if (tid < 32) {
        float m, wsum;
        merge_weights(lse_part + row * num_splits, num_splits, w_s, m, wsum, tid);
        if (tid == 0) {
            fscale = wsum > 0.f ? out_scale / wsum : 0.f;
            if (lse != nullptr) lse[row] = wsum > 0.f ? m + log2f(wsum) : -CUDART_INF_F;
        }
    }
    __syncthreads();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (cols) {
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int sp = g + G * u;
            if (sp < num_splits) {
                const float ws = w_s[sp];
                acc.x += ws * v[u].x;
                acc.y += ws * v[u].y;
                acc.z += ws * v[u].z;
                acc.w += ws * v[u].w;
            }
        }
        if (num_splits > G * kPrefetch)
            acc = merge_columns<8>(op, d_v, g + G * kPrefetch, num_splits, w_s, acc, G);
    }
    if constexpr (G > 1) {
        if (g > 0) gsum[g - 1][tid % kReduceThreads] = acc;
        __syncthreads();
        if (g > 0) return;
#pragma unroll
        for (int k = 0; k < G - 1; ++k) {
            const float4 x = gsum[k][tid];
            acc.x += x.x;
            acc.y += x.y;
            acc.z += x.z;
            acc.w += x.w;
        }
    }
    if (cols) store4(o + row * d_v + c, acc, fscale);
}

// Four columns of a share as fp32, from bf16 (8 bytes) or fp32 (16 bytes).
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p)
{
    const uint2 x = __ldcg(reinterpret_cast<const uint2*>(p));
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float4 load4(const float* p)
{
    return __ldcg(reinterpret_cast<const float4*>(p));
}

// Decode-context-parallel merge of the ranks' shares (rank-major
// [world, rows, d_v], as an all-gather or all-to-all leaves them; bf16 or fp32)
// with their base-2 LSEs [world, rows]: the same weights and fixed association
// as the split-K reduce, the ranks taking the place of the splits.  One CTA per
// row, four columns per thread.
template <typename PartT>
__global__ void __launch_bounds__(kReduceThreads)
dcp_merge_kernel(const PartT* __restrict__ parts, const float* __restrict__ lse_in,
                 int64_t rows, int world, int d_v, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ lse)
{
    __shared__ float w_s[MLA_MAX_SPLITS];
    __shared__ float fscale;

    const int64_t row = blockIdx.x;
    if (row >= rows) return;
    const int tid = threadIdx.x;
    const int c = tid * 4;
    const bool cols = c < d_v;
    const int64_t rank_stride = rows * (int64_t)d_v;
    const PartT* op = parts + row * d_v + c;
    float4 v[kPrefetch];
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u)
        if (cols && u < world) v[u] = load4(op + u * rank_stride);
    if (tid < 32) {
        float m, wsum;
        merge_weights(lse_in + row, world, w_s, m, wsum, tid, rows);
        if (tid == 0) {
            fscale = wsum > 0.f ? 1.f / wsum : 0.f;
            if (lse != nullptr) lse[row] = wsum > 0.f ? m + log2f(wsum) : -CUDART_INF_F;
        }
    }
    __syncthreads();
    if (!cols) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    auto add = [&](float ws, float4 x) {
        acc.x += ws * x.x;
        acc.y += ws * x.y;
        acc.z += ws * x.z;
        acc.w += ws * x.w;
    };
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u)
        if (u < world) add(w_s[u], v[u]);
    for (int k = kPrefetch; k < world; ++k) add(w_s[k], load4(op + k * rank_stride));
    store4(o + row * d_v + c, acc, fscale);
}

}  // namespace

cudaError_t launch_dcp_merge(const void* parts, bool parts_f32, const float* lse_in,
                             int32_t world, int64_t rows, int32_t d_v, uint16_t* o, float* lse,
                             cudaStream_t stream)
{
    if (rows <= 0) return cudaSuccess;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(o);
    if (parts_f32)
        dcp_merge_kernel<float><<<(unsigned)rows, kReduceThreads, 0, stream>>>(
            static_cast<const float*>(parts), lse_in, rows, world, d_v, out, lse);
    else
        dcp_merge_kernel<__nv_bfloat16><<<(unsigned)rows, kReduceThreads, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(parts), lse_in, rows, world, d_v, out, lse);
    return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* o_part, const float* lse_part, int64_t rows,
                                 int32_t num_splits, int32_t d_v, float out_scale, void* o,
                                 bool out_f32, float* lse, cudaStream_t stream)
{
    if (rows <= 0) return cudaSuccess;
    // Four split groups when one group would need several round trips, and
    // above 8 splits for at most 128 rows (measured on GB300: B=8 H=16 S=8192
    // at 16 splits, 128 rows, 18.4 -> 17.8 us per call; the wide form lost
    // with 256 rows at 9 splits, sparse T=4 H=64, 11.9 -> 13.5, and with 512
    // rows at 9 splits, B=8 H=64 S=131072, 285 -> 291).
    const bool wide = num_splits > kPrefetch || (num_splits > 8 && rows <= kWideMaxRows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows, 1, 1);
    cfg.blockDim = dim3(kReduceThreads * (wide ? kWideGroups : 1), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    float* of = static_cast<float*>(o);
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
    if (wide)
        return out_f32 ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<float, kWideGroups>, o_part,
                                            lse_part, rows, num_splits, d_v, out_scale, of, lse)
                       : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<__nv_bfloat16, kWideGroups>,
                                            o_part, lse_part, rows, num_splits, d_v, out_scale, ob,
                                            lse);
    return out_f32 ? cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<float, 1>, o_part, lse_part,
                                        rows, num_splits, d_v, out_scale, of, lse)
                   : cudaLaunchKernelEx(&cfg, splitk_reduce_kernel<__nv_bfloat16, 1>, o_part,
                                        lse_part, rows, num_splits, d_v, out_scale, ob, lse);
}

}  // namespace mla
