// cake_gg_router.cu -- the FP32 router GEMM of the dense projection family by
// BF16x3 emulation (flashinfer PR #8438, "Summary", which names a router GEMM
// over 256 experts in FP32 emulated with three BF16 products): logits
// Y [T, R] = X [T, K] W^T with FP32 X and
// router weights W [R, K], FP32 output.
//
// Every FP32 value v is split as hi = bf16(v) and lo = bf16(v - hi) (round to
// nearest, ties to even), and the three leading products of
// (x_hi + x_lo)(w_hi + w_lo) are kept.  Two launches on the caller's stream:
//   1. a small kernel splits W into W' [R, 2K] = [w_hi | w_lo] (BF16) in the
//      caller's workspace and writes the offsets {0, T} of a one-expert problem;
//   2. the grouped GEMM's forward kernel in its router mode: it loads FP32 X
//      tiles, converter warps split them on chip into BF16 high and low tiles,
//      and the tensor cores sum x_hi w_hi + x_hi w_lo + x_lo w_hi, every product
//      exact, in one FP32 accumulator.
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/cake_gg.h"

namespace cakegg {
// (cake_gg_capi.cu) plan and launch of the router mode of the grouped GEMM kernel
int router_plan(cake_gg_plan_t *plan, int64_t T, int32_t R, int32_t K, int32_t max_sms);
int router_run(const cake_gg_plan_t *plan, const float *X, const void *Wsplit, float *Y, const int32_t *offsets,
               void *ws, cudaStream_t stream);
bool router_plan_matches(const cake_gg_plan_t *plan);
}  // namespace cakegg

namespace {

constexpr uint64_t kAlign = 256;
constexpr int kSplitThreads = 256;

uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

bool mul_ok(uint64_t a, uint64_t b, uint64_t *out)
{
    if (a != 0 && b > UINT64_MAX / a) return false;
    *out = a * b;
    return true;
}

// Workspace layout: GEMM workspace | offsets {0, T} | W' [R, 2K] (each 256-aligned).
struct RouterLayout {
    uint64_t offsets_off, ws_off, total;
};

RouterLayout router_layout(const cake_gg_router_plan_t &rp)
{
    RouterLayout L;
    L.offsets_off = align_up(rp.gemm.workspace_bytes, kAlign);
    L.ws_off = L.offsets_off + kAlign;
    L.total = align_up(L.ws_off + uint64_t(rp.R) * 2u * uint64_t(rp.K) * 2u, kAlign);
    return L;
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b)
{
    return uint32_t(__bfloat16_as_ushort(a)) | (uint32_t(__bfloat16_as_ushort(b)) << 16);
}

// One thread: 8 consecutive values of one row of W (two float4 loads), their
// BF16 high and low parts written as 16-byte vectors at k and K + k of W'.
// (Launched as a programmatic dependent of the previous kernel in the stream,
// which may still read W' or write W: every block first waits for it.  Each
// block lets the router kernel launch at once; that kernel's set-up touches
// no global memory before it waits for this grid in turn.)
__global__ void __launch_bounds__(kSplitThreads)
    router_split_w_kernel(const float *__restrict__ W, uint16_t *__restrict__ Ws, int32_t R, int32_t K, int64_t T,
                          int32_t *__restrict__ offsets)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t groups_per_row = K / 8;
    const int64_t total = int64_t(R) * groups_per_row;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        offsets[0] = 0;
        offsets[1] = int32_t(T);
    }
    for (int64_t gi = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; gi < total;
         gi += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = gi / groups_per_row;
        const int64_t k = (gi - row * groups_per_row) * 8;
        const float *src = W + row * K + k;
        const float4 v0 = __ldg(reinterpret_cast<const float4 *>(src));
        const float4 v1 = __ldg(reinterpret_cast<const float4 *>(src) + 1);
        const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * j]);
            const __nv_bfloat16 h1 = __float2bfloat16_rn(v[2 * j + 1]);
            const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * j] - __bfloat162float(h0));
            const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * j + 1] - __bfloat162float(h1));
            hi[j] = pack2(h0, h1);
            lo[j] = pack2(l0, l1);
        }
        uint16_t *dst = Ws + row * 2 * int64_t(K) + k;
        *reinterpret_cast<uint4 *>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(dst + K) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

}  // namespace

extern "C" {

int cake_gg_router_plan(cake_gg_router_plan_t *rp, int64_t T, int32_t R, int32_t K, int32_t max_sms)
{
    if (!rp) return CAKE_GG_ERR_INVALID_ARG;
    std::memset(rp, 0, sizeof(*rp));
    if (T < 0 || T > INT32_MAX || R < 1 || K < 1 || max_sms < 0) return CAKE_GG_ERR_INVALID_ARG;
    if (R % 8 != 0 || K % 8 != 0) return CAKE_GG_ERR_ALIGNMENT;
    if (int64_t(K) * 2 > INT32_MAX) return CAKE_GG_ERR_OVERFLOW;
    uint64_t t0;
    if (!mul_ok(uint64_t(T) + uint64_t(R), uint64_t(K) * 4u, &t0)) return CAKE_GG_ERR_OVERFLOW;
    const int rc = cakegg::router_plan(&rp->gemm, T, R, K, max_sms);
    if (rc != CAKE_GG_OK) return rc;
    rp->abi_version = CAKE_GG_ABI_VERSION;
    rp->T = T;
    rp->R = R;
    rp->K = K;
    rp->workspace_bytes = router_layout(*rp).total;
    return CAKE_GG_OK;
}

int cake_gg_router_fp32(const cake_gg_router_plan_t *rp, const float *X, const float *W, float *Y,
                        void *workspace, size_t workspace_bytes, void *stream)
{
    if (!rp || rp->abi_version != CAKE_GG_ABI_VERSION || !workspace || (rp->T > 0 && (!X || !Y)) || !W)
        return CAKE_GG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(Y) |
         reinterpret_cast<uintptr_t>(workspace)) % 16 != 0)
        return CAKE_GG_ERR_ALIGNMENT;
    if (rp->gemm.K != rp->K || rp->gemm.N != rp->R || rp->gemm.M_max != rp->T || rp->gemm.E != 1 ||
        !cakegg::router_plan_matches(&rp->gemm))
        return CAKE_GG_ERR_INVALID_ARG;
    const RouterLayout L = router_layout(*rp);
    if (workspace_bytes < L.total || rp->workspace_bytes != L.total) return CAKE_GG_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets_off);
    uint16_t *wsplit = reinterpret_cast<uint16_t *>(ws + L.ws_off);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return CAKE_GG_ERR_CUDA;
    const int64_t groups = int64_t(rp->R) * int64_t(rp->K / 8);
    int64_t blocks = (groups + kSplitThreads - 1) / kSplitThreads;
    const int64_t cap = int64_t(sms) * 8;   // a few resident blocks per SM, grid-stride beyond
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks), 1, 1);
    cfg.blockDim = dim3(kSplitThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    const char *pdl_env = std::getenv("CAKE_GG_PDL");
    if (!(pdl_env && std::atoi(pdl_env) == 0)) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, router_split_w_kernel, W, wsplit, rp->R, rp->K, rp->T, offsets) != cudaSuccess)
        return CAKE_GG_ERR_CUDA;
    return cakegg::router_run(&rp->gemm, X, wsplit, Y, offsets, workspace, s);
}

}  // extern "C"
