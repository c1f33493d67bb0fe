// cake_gg_launch.h -- internal interface between the C ABI and the kernel
// translation units (one per pass, compiled in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "cake_gg_kernel.cuh"

namespace cakegg {

cudaError_t launch_fwd(bool out_f32, const CUtensorMap &a, const CUtensorMap &b, const KParams &p,
                       int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_dgrad(bool out_f32, const CUtensorMap &a, const CUtensorMap &b, const KParams &p,
                         int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_wgrad(bool out_f32, bool swap, const CUtensorMap &a, const CUtensorMap &b,
                         const KParams &p, int grid, size_t smem, cudaStream_t stream);

template <int MODE, bool SWAP, bool OUT_F32>
cudaError_t launch_one(const CUtensorMap &a, const CUtensorMap &b, const KParams &p, int grid,
                       size_t smem, cudaStream_t stream)
{
    auto kern = cake_gg_kernel<MODE, SWAP, OUT_F32>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, smem, stream>>>(a, b, p);
    return cudaGetLastError();
}

}  // namespace cakegg
