// mla_debug.cu -- gather probe: pool rows through the split kernel's own gather
// path (TMA tile::gather4 into the swizzled stage layout of mla_layout.cuh),
// written back de-swizzled, so tests can check the page-table gather byte for
// byte against pool[indices].  Not on the decode path.
#include <climits>

#include "mla_internal.h"
#include "mla_layout.cuh"
#include "mla_sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kProbeRows = 128;   // one stage: 32 four-row groups
constexpr int kProbeWarps = 4;    // eight groups per warp

template <bool ROPE>
__global__ void __launch_bounds__(kProbeWarps * 32, 1)
gather_probe_kernel(const __grid_constant__ CUtensorMap tm_lat,
                    const __grid_constant__ CUtensorMap tm_rope, int64_t pool_rows,
                    const int32_t* __restrict__ idx, int64_t n, uint8_t* __restrict__ out,
                    uint32_t* err)
{
    constexpr int kRowBytes = ROPE ? 576 : 512;
    constexpr int kBoxes = ROPE ? 5 : 4;
    constexpr int kStageBytes = kProbeRows * kRowBytes;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kStageBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t base = (int64_t)blockIdx.x * kProbeRows;

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // Every row of the stage is gathered (rows past n and out-of-range slots
    // at row coordinate -1, outside the tensor: the copy fills them with
    // zeros), so the byte count is the whole stage.
    if (tid == 0) mbar_arrive_expect_tx(bar, (uint32_t)kStageBytes);
    for (int item = lane; item < 8 * kBoxes; item += 32) {
        const int g = warp * 8 + item / kBoxes;   // four-row group
        const int c = item % kBoxes;
        int32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t row = base + 4 * g + i;
            const int32_t v = row < n ? __ldg(idx + row) : -1;
            r[i] = (v >= 0 && (int64_t)v < pool_rows) ? v : -1;
        }
        if (c < 4)
            tma_gather4(smem + c * kProbeRows * 128 + g * 512, &tm_lat, c * 128, r[0], r[1], r[2],
                        r[3], bar);
        else
            tma_gather4(smem + 4 * kProbeRows * 128 + g * 256, &tm_rope, 512, r[0], r[1], r[2],
                        r[3], bar);
    }
    // bounded wait; a timeout is reported and the copies are still waited for
    volatile int abort = 0;
    const bool ok = mbar_wait_or_abort(bar, 0, &abort);
    if (!ok) {
        if (tid == 0) atomicOr(err, MLA_DEVERR_TIMEOUT);
        volatile int drain = 0;
        mbar_wait_or_abort(bar, 0, &drain);
    }
    const int64_t left = n - base;
    const int nr = left < kProbeRows ? (int)left : kProbeRows;
    constexpr int kChunks = kRowBytes / 16;
    for (int e = tid; e < nr * kChunks; e += kProbeWarps * 32) {
        const int r = e / kChunks, c16 = e % kChunks;
        const int64_t row = base + r;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (ok)   // out-of-range slots: the rows the copy filled
            val = *reinterpret_cast<const uint4*>(smem + tile_offset(r, c16 * 16, kProbeRows));
        *reinterpret_cast<uint4*>(out + row * kRowBytes + c16 * 16) = val;
    }
}

}  // namespace

cudaError_t launch_gather_probe(const void* pool, int64_t pool_rows, int32_t row_bytes,
                                const int32_t* indices, int64_t n, uint8_t* out, uint32_t* err,
                                cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    CUtensorMap lat, rope;
    if (!make_row_map(&lat, pool, pool_rows, row_bytes, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const bool with_rope = row_bytes == 576;
    if (with_rope) {
        if (!make_row_map(&rope, pool, pool_rows, row_bytes, 64, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else {
        rope = lat;
    }
    const unsigned grid = (unsigned)((n + kProbeRows - 1) / kProbeRows);
    const int smem = kProbeRows * row_bytes + 64;
    cudaError_t e;
    if (with_rope) {
        e = cudaFuncSetAttribute(gather_probe_kernel<true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        gather_probe_kernel<true><<<grid, kProbeWarps * 32, smem, stream>>>(
            lat, rope, pool_rows, indices, n, out, err);
    } else {
        e = cudaFuncSetAttribute(gather_probe_kernel<false>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        gather_probe_kernel<false><<<grid, kProbeWarps * 32, smem, stream>>>(
            lat, rope, pool_rows, indices, n, out, err);
    }
    return cudaGetLastError();
}

}  // namespace mla
