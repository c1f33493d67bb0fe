// cake_gg_fwd.cu -- forward pass instantiations: Y = X W_e^T per expert (and the FP32 router GEMM's
// fused BF16x3 variant of it).
#include "cake_gg_launch.h"

namespace cakegg {

cudaError_t launch_fwd(bool out_f32, int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                       const KParams &p, int grid, size_t smem, cudaStream_t stream)
{
    return out_f32 ? launch_pair_or_single<kModeFwd, false, true>(pair, a, b, o, p, grid, smem, stream)
                   : launch_pair_or_single<kModeFwd, false, false>(pair, a, b, o, p, grid, smem, stream);
}

cudaError_t launch_router(int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                          const KParams &p, int grid, size_t smem, cudaStream_t stream)
{
    return launch_pair_or_single<kModeRouter, false, true>(pair, a, b, o, p, grid, smem, stream);
}

}  // namespace cakegg
