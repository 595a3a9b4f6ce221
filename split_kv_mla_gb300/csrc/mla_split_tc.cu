// mla_split_tc.cu -- host side of the split kernel: the pool's TMA tensor maps
// and the dispatch to the kernel instantiations (mla_split_dense.cu,
// mla_split_sparse.cu; the kernel itself is in mla_split_kernel.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_internal.h"

namespace mla {

cudaError_t launch_split_dense(const CUtensorMap& lat, const CUtensorMap& rope,
                               const SplitArgs& a, const mla_plan_t& plan, int mc,
                               cudaStream_t stream);
cudaError_t launch_split_sparse(const CUtensorMap& lat, const CUtensorMap& rope,
                                const SplitArgs& a, const mla_plan_t& plan, int mc,
                                cudaStream_t stream);

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
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

// 2-D uint8 map of the pool (row_bytes columns x rows) with one-row boxes of
// `box` columns: the shape tile::gather4 reads.
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

#ifdef MLA_TRACE
// Phase stamps of the last split-kernel launch (traced builds only).
static __device__ unsigned long long g_trace[kTraceWords];
#endif

cudaError_t launch_split_tc(const SplitArgs& a_in, const mla_plan_t& plan, int mc,
                            cudaStream_t stream)
{
    SplitArgs a = a_in;
#ifdef MLA_TRACE
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&a.trace), g_trace) != cudaSuccess)
        a.trace = nullptr;
#endif
    if (plan.grid_x <= 0 || plan.grid_y <= 0 || plan.grid_z <= 0) return cudaSuccess;
    CUtensorMap lat, rope;
    const int row_bytes = a.d_v + a.d_rope;
    if (!make_row_map(&lat, a.pool, a.pool_rows, row_bytes, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (!a.sparse) {
        if (!make_row_map(&rope, a.pool, a.pool_rows, row_bytes, 64, CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    } else if (a.extra_topk > 0) {
        if (!make_row_map(&rope, a.extra_pool, a.extra_rows, row_bytes, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else {
        rope = lat;
    }
    if (a.sparse) return launch_split_sparse(lat, rope, a, plan, mc, stream);
    return launch_split_dense(lat, rope, a, plan, mc, stream);
}

}  // namespace mla

#ifdef MLA_TRACE
// Traced builds: copy the phase stamps of the last split-kernel launch
// (kTraceCtas x kTraceSlots globaltimer values, then the per-block events of
// the first CTAs; zero where none was written)
// to host memory; synchronises the device.
extern "C" int mla_trace_read(unsigned long long* host, int64_t count)
{
    if (!host || count < 0 || count > (int64_t)mla::kTraceWords)
        return MLA_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return MLA_ERR_CUDA;
    return cudaMemcpyFromSymbol(host, mla::g_trace, count * sizeof(unsigned long long)) ==
                   cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
}

// Traced builds: zero the stamps.
extern "C" int mla_trace_clear(void)
{
    static unsigned long long zeros[mla::kTraceWords];
    return cudaMemcpyToSymbol(mla::g_trace, zeros, sizeof zeros) == cudaSuccess ? MLA_OK
                                                                                 : MLA_ERR_CUDA;
}
#endif
