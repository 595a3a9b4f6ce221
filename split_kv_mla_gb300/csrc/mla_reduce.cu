// mla_reduce.cu -- split-K reduce of normalized fp32 partials with base-2 LSEs.
//
// hip_mha_decoding_num_partitions (split-K target and the reducer that merges up
// to 256 partitions); moonmath-ai/amd-kernels README, "Numerics": the fp32
// partial merge sums in a fixed association, so the result is deterministic.
//
// Per row: M = max_s lse_s, w_s = 2^(lse_s - M), o = out_scale * sum_s w_s o_s /
// sum_s w_s, lse = M + log2 sum_s w_s, s in increasing order.  All -inf -> o = 0,
// lse = -inf.  One CTA per row; each thread owns four consecutive columns and
// reads them with 16-byte loads, so every split's row is one coalesced sweep.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kReduceThreads = 128;

__global__ void __launch_bounds__(kReduceThreads)
splitk_reduce_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                     int64_t rows, int num_splits, int d_v, float out_scale,
                     __nv_bfloat16* __restrict__ o, float* __restrict__ lse)
{
    __shared__ float w_s[MLA_MAX_SPLITS];
    __shared__ float red[kReduceThreads / 32];
    __shared__ float m_row, wsum_row;

    const int64_t row = blockIdx.x;
    if (row >= rows) return;
    const int tid = threadIdx.x;
    const float* lp = lse_part + row * num_splits;

    // max over splits
    float m = -CUDART_INF_F;
    for (int s = tid; s < num_splits; s += kReduceThreads) m = fmaxf(m, lp[s]);
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    if (tid == 0) {
        float mm = red[0];
        for (int w = 1; w < kReduceThreads / 32; ++w) mm = fmaxf(mm, red[w]);
        m_row = mm;
    }
    __syncthreads();
    m = m_row;

    // weights (fixed order; an all -inf row keeps every weight at zero)
    for (int s = tid; s < num_splits; s += kReduceThreads) {
        const float l = lp[s];
        w_s[s] = (m == -CUDART_INF_F || l == -CUDART_INF_F) ? 0.f : exp2f(l - m);
    }
    __syncthreads();
    if (tid == 0) {
        float ws = 0.f;
        for (int s = 0; s < num_splits; ++s) ws += w_s[s];
        wsum_row = ws;
    }
    __syncthreads();
    const float wsum = wsum_row;

    const int c = tid * 4;
    if (c < d_v) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* op = o_part + row * (int64_t)num_splits * d_v + c;
        // Loads of kUnroll splits are issued before their sums, so the memory
        // latency is paid once per group, not once per split; the sums still run
        // in increasing split order.
        constexpr int kUnroll = 8;
        int s = 0;
        for (; s + kUnroll <= num_splits; s += kUnroll) {
            float4 v[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                v[u] = __ldg(reinterpret_cast<const float4*>(op + (int64_t)(s + u) * d_v));
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const float w = w_s[s + u];
                acc.x += w * v[u].x;
                acc.y += w * v[u].y;
                acc.z += w * v[u].z;
                acc.w += w * v[u].w;
            }
        }
        for (; s < num_splits; ++s) {
            const float w = w_s[s];
            const float4 v = __ldg(reinterpret_cast<const float4*>(op + (int64_t)s * d_v));
            acc.x += w * v.x;
            acc.y += w * v.y;
            acc.z += w * v.z;
            acc.w += w * v.w;
        }
        const float f = wsum > 0.f ? out_scale / wsum : 0.f;
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * f, acc.y * f);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * f, acc.w * f);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(o + row * d_v + c) = pk;
    }
    if (lse != nullptr && tid == 0)
        lse[row] = wsum > 0.f ? m + log2f(wsum) : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_splitk_reduce(const float* o_part, const float* lse_part, int64_t rows,
                                 int32_t num_splits, int32_t d_v, float out_scale,
                                 uint16_t* o, float* lse, cudaStream_t stream)
{
    if (rows <= 0) return cudaSuccess;
    splitk_reduce_kernel<<<(unsigned)rows, kReduceThreads, 0, stream>>>(
        o_part, lse_part, rows, num_splits, d_v, out_scale,
        reinterpret_cast<__nv_bfloat16*>(o), lse);
    return cudaGetLastError();
}

}  // namespace mla
