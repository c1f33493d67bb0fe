// cake_gg_wgrad.cu -- weight-gradient instantiations: dW_e = G_e^T X_e, the
// ragged reduction over each expert's rows (optionally with swapped operands
// for thin N and split reductions).
#include "cake_gg_launch.h"

namespace cakegg {

cudaError_t launch_wgrad(bool out_f32, bool swap, const CUtensorMap &a, const CUtensorMap &b,
                         const KParams &p, int grid, size_t smem, cudaStream_t stream)
{
    if (swap)
        return out_f32 ? launch_one<kModeWgrad, true, true>(a, b, p, grid, smem, stream)
                       : launch_one<kModeWgrad, true, false>(a, b, p, grid, smem, stream);
    return out_f32 ? launch_one<kModeWgrad, false, true>(a, b, p, grid, smem, stream)
                   : launch_one<kModeWgrad, false, false>(a, b, p, grid, smem, stream);
}

}  // namespace cakegg
