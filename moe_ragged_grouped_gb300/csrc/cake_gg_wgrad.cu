// cake_gg_wgrad.cu -- weight-gradient instantiations: dW_e = G_e^T X_e, the
// ragged reduction over each expert's rows (optionally with swapped operands
// for thin N and split reductions).
#include "cake_gg_launch.h"

namespace cakegg {

cudaError_t launch_wgrad(bool out_f32, bool swap, int pair, const CUtensorMap &a, const CUtensorMap &b,
                         const CUtensorMap &o, const KParams &p, int grid, size_t smem, cudaStream_t stream)
{
    // the swapped (thin) weight gradient always runs unpaired
    if (swap)
        return out_f32 ? launch_one<kModeWgrad, true, true, 1>(a, b, o, p, grid, smem, stream)
                       : launch_one<kModeWgrad, true, false, 1>(a, b, o, p, grid, smem, stream);
    // N-split tail pieces (pairs of 256 x 512 tiles only): a kernel of their own
    if (p.ntq > 1 && pair == 2)
        return out_f32 ? launch_one<kModeWgradNT, false, true, 2>(a, b, o, p, grid, smem, stream)
                       : launch_one<kModeWgradNT, false, false, 2>(a, b, o, p, grid, smem, stream);
    return out_f32 ? launch_pair_or_single<kModeWgrad, false, true>(pair, a, b, o, p, grid, smem, stream)
                   : launch_pair_or_single<kModeWgrad, false, false>(pair, a, b, o, p, grid, smem, stream);
}

}  // namespace cakegg
