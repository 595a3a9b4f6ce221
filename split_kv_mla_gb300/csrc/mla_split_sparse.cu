// mla_split_sparse.cu -- instantiations of the split kernel for sparse top-k
// decode (512-byte rows: 448 NoPE + 64 RoPE columns), with or without a second
// (compressed) cache, 16 or 32 query rows per CTA, with or without the fused
// cluster merge.
#include "mla_split_kernel.cuh"

namespace mla {

cudaError_t launch_split_sparse(const CUtensorMap& lat, const CUtensorMap& rope,
                                const SplitArgs& a, const mla_plan_t& plan, int mc,
                                cudaStream_t stream)
{
    if (a.extra_topk > 0) return launch_rows_mc<true, true>(lat, rope, a, plan, mc, stream);
    return launch_rows_mc<true, false>(lat, rope, a, plan, mc, stream);
}

}  // namespace mla
