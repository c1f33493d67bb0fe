// cake_gg_fwd.cu -- forward pass instantiations: Y = X W_e^T per expert.
#include "cake_gg_launch.h"

namespace cakegg {

cudaError_t launch_fwd(bool out_f32, const CUtensorMap &a, const CUtensorMap &b, const KParams &p,
                       int grid, size_t smem, cudaStream_t stream)
{
    return out_f32 ? launch_one<kModeFwd, false, true>(a, b, p, grid, smem, stream)
                   : launch_one<kModeFwd, false, false>(a, b, p, grid, smem, stream);
}

}  // namespace cakegg
