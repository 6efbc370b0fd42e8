// dv_colacc.cu -- stand-alone column-gather kernels of the sparse layer decode
// (body in dv_colacc.cuh) and their launchers (sm_103a).
#include "dv_colacc.cuh"

namespace dv {
namespace {

template <typename T, int NB, int KIND, int P>
__global__ void __launch_bounds__(kThreads, 1) k_colacc(const ColArgs a)
{
    unsigned long long *s = chain_stamps(a.stamps);
    colacc_body<T, NB, KIND, P>(a, blockIdx.x, gridDim.x, PdlDep{s});
    chain_stamp_end(s);
}

template <typename T, int NB, int KIND>
cudaError_t launch_one(const ColArgs &a, dim3 grid, cudaStream_t st, bool pdl)
{
    constexpr int P = colacc_chunks<NB>();
    constexpr int CB = 32 * P * Elem<T>::EPC;
    const size_t smem = colacc_smem_bytes(CB, NB);
    auto kern = k_colacc<T, NB, KIND, P>;
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int KIND>
cudaError_t dispatch_nb(int nb, const ColArgs &a, dim3 grid, cudaStream_t st, bool pdl)
{
    switch (nb) {
    case 1: return launch_one<T, 1, KIND>(a, grid, st, pdl);
    case 2: return launch_one<T, 2, KIND>(a, grid, st, pdl);
    case 4: return launch_one<T, 4, KIND>(a, grid, st, pdl);
    case 8: return launch_one<T, 8, KIND>(a, grid, st, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int colacc_nb(int B)
{
    int nb = 1;
    while (nb < B && nb < 8)
        nb <<= 1;
    return nb;
}

int colacc_block_cols(int dtype, int nb)
{
    const int epc = dtype == DV_F16 ? 8 : 4;
    const int p = nb == 1 ? colacc_chunks<1>() : nb == 2 ? colacc_chunks<2>()
                : nb == 4 ? colacc_chunks<4>() : colacc_chunks<8>();
    return 32 * p * epc;
}

cudaError_t launch_colacc(int kind, int dtype, int nb, const ColArgs &a, dim3 grid,
                          cudaStream_t st, bool pdl)
{
    if (dtype == DV_F16)
        return kind == CK_OPROJ ? dispatch_nb<__half, CK_OPROJ>(nb, a, grid, st, pdl)
                                : dispatch_nb<__half, CK_FC2>(nb, a, grid, st, pdl);
    return kind == CK_OPROJ ? dispatch_nb<float, CK_OPROJ>(nb, a, grid, st, pdl)
                            : dispatch_nb<float, CK_FC2>(nb, a, grid, st, pdl);
}

}  // namespace dv
