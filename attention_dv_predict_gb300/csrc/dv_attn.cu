// dv_attn.cu -- the stand-alone decode attention kernel (body in dv_attn.cuh),
// the copy probe used for the roofline denominator, and their launchers
// (sm_103a).
#include "dv_attn.cuh"

namespace dv {
namespace {

template <typename T, int LPK>
__global__ void __launch_bounds__(kThreads) k_attn(const AttnArgs a)
{
    unsigned long long *s = chain_stamps(a.stamps);
    attn_body<T, LPK>(a, blockIdx.x, gridDim.x, PdlDep{s});
    chain_stamp_end(s);
}

template <typename T, int LPK>
cudaError_t launch_attn_one(const AttnArgs &a, cudaLaunchConfig_t &cfg)
{
    cfg.dynamicSmemBytes = attn_smem_bytes(LPK * Elem<T>::EPC);
    return cudaLaunchKernelEx(&cfg, k_attn<T, LPK>, a);
}

template <typename T>
cudaError_t dispatch_lpk(int lpk, const AttnArgs &a, dim3 grid, cudaStream_t st, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    switch (lpk) {
    case 1: return launch_attn_one<T, 1>(a, cfg);
    case 2: return launch_attn_one<T, 2>(a, cfg);
    case 4: return launch_attn_one<T, 4>(a, cfg);
    case 8: return launch_attn_one<T, 8>(a, cfg);
    case 16: return launch_attn_one<T, 16>(a, cfg);
    case 32: return launch_attn_one<T, 32>(a, cfg);
    default: return cudaErrorInvalidValue;
    }
}

// Streaming copy: 16-byte vectors, four in flight per thread.
__global__ void __launch_bounds__(kThreads) k_copy(uint4 *__restrict__ dst,
                                                   const uint4 *__restrict__ src, size_t n)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 a0 = ld_stream(src + i);
        const uint4 a1 = ld_stream(src + i + stride);
        const uint4 a2 = ld_stream(src + i + 2 * stride);
        const uint4 a3 = ld_stream(src + i + 3 * stride);
        __stcs(dst + i, a0);
        __stcs(dst + i + stride, a1);
        __stcs(dst + i + 2 * stride, a2);
        __stcs(dst + i + 3 * stride, a3);
    }
    for (; i < n; i += stride)
        __stcs(dst + i, ld_stream(src + i));
}

}  // namespace

cudaError_t launch_attn(int dtype, int lanes_per_key, const AttnArgs &a, dim3 grid,
                        cudaStream_t st, bool pdl)
{
    if (dtype == DV_F16)
        return dispatch_lpk<__half>(lanes_per_key, a, grid, st, pdl);
    return dispatch_lpk<float>(lanes_per_key, a, grid, st, pdl);
}

cudaError_t launch_copy(void *dst, const void *src, size_t n16, int grid, cudaStream_t st)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, k_copy, static_cast<uint4 *>(dst),
                              static_cast<const uint4 *>(src), n16);
}

}  // namespace dv
