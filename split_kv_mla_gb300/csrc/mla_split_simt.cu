// mla_split_simt.cu -- CUDA-core split kernel for absorbed-MLA decode.
//
// The straightforward form of one (request, head block, split) CTA of the
// split-KV decode (moonmath-ai/amd-kernels README, "MLA absorbed decode"; the
// split-K partial format of hip_mha_decoding_num_partitions): gather a block of
// fp8 rows through the page table into shared memory, take scaled logits over
// all d_v + d_rope columns, update an online base-2 softmax, and accumulate
// P.V over the first d_v columns.  The tensor-core kernel computes the same
// partials; this one serves shapes and checks where simplicity matters more
// than speed.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <math_constants.h>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;        // query rows per CTA
constexpr int kKeys = 32;        // keys per block
constexpr int kMaxWidth = 576;   // d_v + d_rope
constexpr int kStride = kMaxWidth + 4;  // 145 words per row: conflict-free columns
constexpr int kMaxDv = 512;
constexpr int kDPerThread = kMaxDv / kThreads;  // 2

struct Smem {
    float q[kRows][kMaxWidth];
    uint8_t kv[kKeys][kStride];
    float s[kRows][kKeys];
    float alpha[kRows];
    int32_t slot[kKeys];
    int32_t valid[kKeys];
};

__device__ __forceinline__ float fp8_to_float(uint8_t b)
{
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(h));
}

__device__ __forceinline__ float bf16_to_float(uint16_t u)
{
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

__global__ void __launch_bounds__(kThreads)
split_simt_kernel(const SplitArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int tid = threadIdx.x;
    const int hb = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
    const int width = a.d_v + a.d_rope;
    const int rows_in_req = a.q_len * a.num_heads;

    // request b: its key list and length
    int64_t base;
    int L;
    if (a.sparse) {
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

    // query rows of this CTA: flattened (t, h) of request b, slice hb
    for (int e = tid; e < kRows * width; e += kThreads) {
        const int n = e / width, c = e % width;
        const int idx = hb * kRows + n;
        float v = 0.f;
        if (idx < rows_in_req) {
            const int t = idx / a.num_heads, h = idx % a.num_heads;
            const int64_t item = ((int64_t)b * a.q_len + t) * a.num_heads + h;
            v = c < a.d_v ? bf16_to_float(a.q_lat[item * a.d_v + c])
                          : bf16_to_float(a.q_pe[item * a.d_rope + (c - a.d_v)]);
        }
        sm.q[n][c] = v;
    }

    float m_run = -CUDART_INF_F, l_run = 0.f;  // owned by threads tid < kRows
    float acc[kRows][kDPerThread];
#pragma unroll
    for (int n = 0; n < kRows; ++n)
#pragma unroll
        for (int k = 0; k < kDPerThread; ++k) acc[n][k] = 0.f;

    for (int kb = k0; kb < k1; kb += kKeys) {
        const int nk = min(kKeys, k1 - kb);
        if (tid < kKeys) {
            int32_t slot = -1;
            int ok = 0;
            if (tid < nk) {
                slot = a.kv_indices[base + kb + tid];
                if (slot >= 0 && (int64_t)slot < a.pool_rows) {
                    ok = 1;
                } else if (!(a.sparse && slot < 0)) {
                    atomicOr(a.err, MLA_DEVERR_BAD_SLOT);
                }
            }
            sm.slot[tid] = ok ? slot : -1;
            sm.valid[tid] = ok;
        }
        __syncthreads();
        // gather rows (4-byte words; invalid rows read as zeros)
        const int words = width / 4;
        for (int e = tid; e < kKeys * words; e += kThreads) {
            const int j = e / words, w = e % words;
            uint32_t v = 0;
            if (sm.valid[j])
                v = __ldg(reinterpret_cast<const uint32_t*>(a.pool + (int64_t)sm.slot[j] * width) + w);
            *reinterpret_cast<uint32_t*>(&sm.kv[j][w * 4]) = v;
        }
        __syncthreads();
        // logits (base 2)
        for (int e = tid; e < kRows * kKeys; e += kThreads) {
            const int n = e / kKeys, j = e % kKeys;
            const int idx = hb * kRows + n;
            const int t = idx / a.num_heads;
            const int win = L - a.q_len + t + 1;  // keys j < win are visible
            float s = -CUDART_INF_F;
            if (idx < rows_in_req && sm.valid[j] && kb + j < win) {
                float dot = 0.f;
                for (int c = 0; c < width; ++c) dot += sm.q[n][c] * fp8_to_float(sm.kv[j][c]);
                s = dot * a.logit_scale;
            }
            sm.s[n][j] = s;
        }
        __syncthreads();
        // online softmax, one thread per row
        if (tid < kRows) {
            float bm = -CUDART_INF_F;
            for (int j = 0; j < kKeys; ++j) bm = fmaxf(bm, sm.s[tid][j]);
            const float m_new = fmaxf(m_run, bm);
            float alpha = 1.f;
            if (m_new != -CUDART_INF_F) alpha = (m_run == -CUDART_INF_F) ? 0.f : exp2f(m_run - m_new);
            float psum = 0.f;
            for (int j = 0; j < kKeys; ++j) {
                const float s = sm.s[tid][j];
                const float p = (s == -CUDART_INF_F) ? 0.f : exp2f(s - m_new);
                sm.s[tid][j] = p;
                psum += p;
            }
            l_run = l_run * alpha + psum;
            m_run = m_new;
            sm.alpha[tid] = alpha;
        }
        __syncthreads();
        // P.V over the first d_v columns
#pragma unroll
        for (int k = 0; k < kDPerThread; ++k) {
            const int d = tid + k * kThreads;
            if (d < a.d_v) {
#pragma unroll
                for (int n = 0; n < kRows; ++n) acc[n][k] *= sm.alpha[n];
                for (int j = 0; j < nk; ++j) {
                    const float v = fp8_to_float(sm.kv[j][d]);
#pragma unroll
                    for (int n = 0; n < kRows; ++n) acc[n][k] += sm.s[n][j] * v;
                }
            }
        }
        __syncthreads();
    }

    // epilogue: row sums and maxima to shared memory, then normalized outputs
    __shared__ float l_sh[kRows], m_sh[kRows];
    if (tid < kRows) {
        l_sh[tid] = l_run;
        m_sh[tid] = m_run;
    }
    __syncthreads();
    for (int n = 0; n < kRows; ++n) {
        const int idx = hb * kRows + n;
        if (idx >= rows_in_req) break;
        const int t = idx / a.num_heads, h = idx % a.num_heads;
        const int64_t item = ((int64_t)b * a.q_len + t) * a.num_heads + h;
        const float l = l_sh[n];
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const float lse2 = l > 0.f ? m_sh[n] + log2f(l) : -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < kDPerThread; ++k) {
            const int d = tid + k * kThreads;
            if (d < a.d_v) {
                const float o = acc[n][k] * inv;
                if (a.num_splits == 1) {
                    reinterpret_cast<__nv_bfloat16*>(a.o)[item * a.d_v + d] =
                        __float2bfloat16_rn(o * a.out_scale);
                } else {
                    a.o_part[(item * a.num_splits + split) * a.d_v + d] = o;
                }
            }
        }
        if (tid == 0) {
            if (a.num_splits == 1) {
                if (a.lse) a.lse[item] = lse2;
            } else {
                a.lse_part[item * a.num_splits + split] = lse2;
            }
        }
    }
}

}  // namespace

cudaError_t launch_split_simt(const SplitArgs& a, const mla_plan_t& plan, cudaStream_t stream)
{
    static bool configured = false;
    const int smem = (int)sizeof(Smem);
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(split_simt_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid(plan.grid_x, plan.grid_y, plan.grid_z);
    split_simt_kernel<<<grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace mla
