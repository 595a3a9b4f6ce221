// mla_merge.cuh -- the split-K merge arithmetic of the reduce kernel.
//
// hip_mha_decoding_num_partitions (a split-K reducer merges per-split partials);
// moonmath-ai/amd-kernels README, "Numerics" (the fp32 partial merge uses a fixed
// association, so results are deterministic).  For one output row with split
// partials o_s (already normalised, o_s = O_s / l_s) and base-2 LSEs lse_s:
//   M    = max_s lse_s
//   w_s  = 2^(lse_s - M)            (0 when lse_s or M is -inf)
//   o    = out_scale * (sum_s w_s o_s) / (sum_s w_s)
//   lse  = M + log2(sum_s w_s)      (-inf when every lse_s is -inf)
// The fixed association: sum_s w_s is a per-lane sum over s = lane, lane + 32,
// ... in increasing order followed by a butterfly over the 32 lanes (every lane
// ends with the same bits, fp32 addition being commutative).  Each output
// column sums w_s o_s in G interleaved groups (group g: s = g, g + G, ... in
// increasing order) and adds the group sums in increasing g; the reduce kernel
// takes G = 4 above 16 splits, and above 8 splits for at most 128 rows, else
// G = 1 (one sequential sum).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "../../include/mla_decode.h"

namespace mla {

// One full warp: M, the weights w_s (written to w[0..ns)) and their sum for the
// row whose LSEs are lse[s * stride], s < ns <= MLA_MAX_SPLITS.  Each lane
// loads its LSEs once (s = lane + 32 k) and keeps them in registers.
__device__ __forceinline__ void merge_weights(const float* lse, int ns, float* w, float& m_out,
                                              float& wsum_out, int lane, int64_t stride = 1)
{
    constexpr int kPer = MLA_MAX_SPLITS / 32;
    float l[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int s = lane + 32 * k;
        l[k] = s < ns ? __ldcg(lse + s * stride) : -CUDART_INF_F;
    }
    float m = l[0];
#pragma unroll
    for (int k = 1; k < kPer; ++k) m = fmaxf(m, l[k]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int s = lane + 32 * k;
        if (s < ns) {
            const float ws = (m == -CUDART_INF_F || l[k] == -CUDART_INF_F) ? 0.f : exp2f(l[k] - m);
            w[s] = ws;
            part += ws;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    m_out = m;
    wsum_out = part;
}

// acc + sum_s w[s] * op[s * stride + 0..3] for s = s0, s0 + step, ... < ns in
// increasing order; loads of kUnroll splits are issued before their sums.
template <int kUnroll>
__device__ __forceinline__ float4 merge_columns(const float* op, int64_t stride, int s0, int ns,
                                                const float* w, float4 acc, int step = 1)
{
    int s = s0;
    for (; s + (kUnroll - 1) * step < ns; s += kUnroll * step) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            v[u] = __ldcg(reinterpret_cast<const float4*>(op + (int64_t)(s + u * step) * stride));
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const float ws = w[s + u * step];
            acc.x += ws * v[u].x;
            acc.y += ws * v[u].y;
            acc.z += ws * v[u].z;
            acc.w += ws * v[u].w;
        }
    }
    for (; s < ns; s += step) {
        const float ws = w[s];
        const float4 v = __ldcg(reinterpret_cast<const float4*>(op + (int64_t)s * stride));
        acc.x += ws * v.x;
        acc.y += ws * v.y;
        acc.z += ws * v.z;
        acc.w += ws * v.w;
    }
    return acc;
}

// Four merged columns scaled by f, as packed bf16 (two 32-bit words).
__device__ __forceinline__ uint2 merge_pack_bf16(float4 acc, float f)
{
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * f, acc.y * f);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * f, acc.w * f);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    return pk;
}

}  // namespace mla
