// mla_split_dense.cu -- instantiations of the split kernel for dense decode
// (576-byte rows: 512 latent + 64 RoPE columns), 16 or 32 query rows per CTA,
// with or without the fused cluster merge.
#include "mla_split_kernel.cuh"

namespace mla {

cudaError_t launch_split_dense(const CUtensorMap& lat, const CUtensorMap& rope,
                               const SplitArgs& a, const mla_plan_t& plan, int mc,
                               cudaStream_t stream)
{
    return launch_rows_mc<false, false>(lat, rope, a, plan, mc, stream);
}

}  // namespace mla
