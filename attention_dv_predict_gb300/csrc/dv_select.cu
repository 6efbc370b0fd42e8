// dv_select.cu -- stand-alone top-k selection kernels for dv_predict_topk
// (the fused layer decode runs the same steps inside its QKV and attention
// kernels; see dv_select.cuh).
#include "dv_select.cuh"

namespace dv {
namespace {

// Head selection (CTA 0, one warp) and this CTA's share of the neuron pass.
__global__ void __launch_bounds__(kThreads) k_select_pass(const SelectArgs a)
{
    __shared__ unsigned hbits[2 * kHeadKPL];
    __shared__ int32_t hsel[kHeadTopkMax];
    __shared__ int sb1[DV_MAX_BATCH];
    __shared__ int hbuf[kTopkBins];
    __shared__ int scr[48];
    pdl_wait();  // the scores come from the previous kernels
    pdl_launch_dependents();
    if (blockIdx.x == 0 && threadIdx.x < 32)
        head_select(a.s_h, a.ns.B, a.H, a.k_h, hbits, hsel, true, a.idx_h, a.u_h, a.n_u_h,
                    threadIdx.x);
    if (a.ns.block > 1)  // the final kernel selects the blocks
        return;
    const int W = (a.ns.N + 31) >> 5;
    const int w0 = (int)((long long)W * blockIdx.x / gridDim.x);
    const int w1 = (int)((long long)W * (blockIdx.x + 1) / gridDim.x);
    neuron_pass(a.ns, w0, w1, sb1, hbuf, scr);
}

__global__ void __launch_bounds__(kThreads) k_select_final(const SelectArgs a)
{
    extern __shared__ __align__(16) int fsm[];
    __shared__ int fscr[48];
    pdl_wait();
    pdl_launch_dependents();
    if (a.ns.block > 1)
        block_select(a.ns, final_smem(fsm, a.ns.N, fscr));
    else
        neuron_final(a.ns, final_smem(fsm, a.ns.N, fscr));
}

}  // namespace

size_t select_final_smem(int N) { return neuron_final_smem_bytes(N); }

cudaError_t launch_select(const SelectArgs &a, int grid, cudaStream_t st)
{
    static DeviceOnce once;
    cudaError_t e = once.run([] {
        return cudaFuncSetAttribute(k_select_final, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemCap);
    });
    if (e != cudaSuccess)
        return e;
    const size_t smem = neuron_final_smem_bytes(a.ns.N);
    if (smem > kSmemCap)
        return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_select_pass, a);
    if (e != cudaSuccess)
        return e;
    cfg.gridDim = dim3(1);
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, k_select_final, a);
}

}  // namespace dv
