// cake_gg_launch.h -- internal interface between the C ABI and the kernel
// translation units (one per pass, compiled in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "cake_gg_kernel.cuh"

namespace cakegg {

cudaError_t launch_fwd(bool out_f32, int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                       const KParams &p, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_dgrad(bool out_f32, int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                         const KParams &p, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_wgrad(bool out_f32, bool swap, int pair, const CUtensorMap &a, const CUtensorMap &b,
                         const CUtensorMap &o, const KParams &p, int grid, size_t smem, cudaStream_t stream);
// the FP32 router GEMM (BF16x3): the forward pass with on-chip splitting, FP32 output
cudaError_t launch_router(int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                          const KParams &p, int grid, size_t smem, cudaStream_t stream);

template <int MODE, bool SWAP, bool OUT_F32, int PAIR>
cudaError_t launch_one(const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o, const KParams &p,
                       int grid, size_t smem, cudaStream_t stream)
{
    auto kern = cake_gg_kernel<MODE, SWAP, OUT_F32, PAIR>;
    // the opt-in shared-memory limit is raised once per device to the maximum,
    // so later calls (including ones under stream capture) skip the attribute call
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemOptInLimit));
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    if (smem > kSmemOptInLimit) return cudaErrorInvalidValue;
    // clusters: a CTA pair, the CTAs of a cluster split, or its pairs
    const int cluster = PAIR * (p.csplit > 0 ? p.csplit : 1);
    if (grid % cluster != 0) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (p.pdl) {
        // programmatic dependent launch: this grid may start while the previous
        // kernel in the stream finishes (the kernel waits before touching memory)
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.gridDim = dim3(grid, 1, 1);
    // (a forward / data gradient with one epilogue group runs without warps 6..9)
    const int threads = MODE == kModeRouter || MODE == kModeWgrad || MODE == kModeWgradNT
                            ? threads_for(MODE)
                            : (p.epi_groups == 2 ? kThreadsEpi2 : kThreads);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, a, b, o, p);
}

template <int MODE, bool SWAP, bool OUT_F32>
cudaError_t launch_pair_or_single(int pair, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &o,
                                  const KParams &p, int grid, size_t smem, cudaStream_t stream)
{
    return pair == 2 ? launch_one<MODE, SWAP, OUT_F32, 2>(a, b, o, p, grid, smem, stream)
                     : launch_one<MODE, SWAP, OUT_F32, 1>(a, b, o, p, grid, smem, stream);
}

}  // namespace cakegg
