// cake_gg_dgrad.cu -- data-gradient instantiations: dX = G W_e per expert.
#include "cake_gg_launch.h"

namespace cakegg {

cudaError_t launch_dgrad(bool out_f32, const CUtensorMap &a, const CUtensorMap &b, const KParams &p,
                         int grid, size_t smem, cudaStream_t stream)
{
    return out_f32 ? launch_one<kModeDgrad, false, true>(a, b, p, grid, smem, stream)
                   : launch_one<kModeDgrad, false, false>(a, b, p, grid, smem, stream);
}

}  // namespace cakegg
