// cake_gg_dgrad.cu -- data-gradient instantiations: dX = G W_e per expert.
#include "cake_gg_launch.h"

namespace cakegg {

cudaError_t launch_dgrad(bool out_f32, int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                         const KParams &p, int grid, size_t smem, cudaStream_t stream)
{
    return out_f32 ? launch_pair_or_single<kModeDgrad, false, true>(pair, a, b, o, p, grid, smem, stream)
                   : launch_pair_or_single<kModeDgrad, false, false>(pair, a, b, o, p, grid, smem, stream);
}

}  // namespace cakegg
