// cake_gg_fwd.cu -- forward pass instantiations: Y = X W_e^T per expert.
#include "cake_gg_launch.h"

namespace cakegg {

cudaError_t launch_fwd(bool out_f32, int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                       const KParams &p, int grid, size_t smem, cudaStream_t stream)
{
    return out_f32 ? launch_pair_or_single<kModeFwd, false, true>(pair, a, b, o, p, grid, smem, stream)
                   : launch_pair_or_single<kModeFwd, false, false>(pair, a, b, o, p, grid, smem, stream);
}

}  // namespace cakegg
