// dv_layer.cu -- the whole sparse layer decode as one persistent kernel
// (sm_103a).
//
// The seven steps of the fused decode (predictors, QKV, attention,
// out-projection, fc1, fc2; "DejaVu Guide: Contextual Sparsity for LLM
// Inference", listing DejaVuTransformerLayer.forward) run as phases of one
// cooperative grid of one 512-thread CTA per SM, with the same bodies as the
// stand-alone kernels (dv_rowdot.cuh, dv_attn.cuh, dv_colacc.cuh).  A phase
// waits for the counter of CTAs that finished the phase it reads from
// instead of a grid boundary, so a CTA that is done with one phase places
// its work in the next one, reads its gather list and issues its first
// weight loads while other CTAs still finish: the latency that separates
// two kernels (launch, parameters, the dependent loads of a prologue) is
// hidden behind the tail of the previous phase.
//
// Phases and the CTAs that take part (n = grid size):
//   PRED1   all n
//   PRED2   all n; the last CTA selects the heads and writes LayerNorm(x),
//           then raises the side flag
//   QKV     rows on CTAs 0 .. n-2, started by the side flag; CTA n-1 waits
//           for the whole of PRED2 and selects the neurons
//   ATTN    CTAs 0 .. n-2, after their QKV counter
//   OPROJ   CTAs 0 .. n-2, after the attention counter
//   FC1     all n, after the neuron selection and the out-projection
//   FC2     all n, after fc1
// so the neuron selection runs beside QKV, attention and the out-projection.
// Every wait is bounded (PhaseDep); the last CTA to finish resets the
// counters for the next launch.
//
// Served by dv_layer_decode_persistent.  On GB300 it is not faster than the
// chained kernels of dv_layer_decode: a phase hand-off through a counter
// (release add, acquire poll) takes about as long as the programmatic-
// dependent grid wait, and the chain already places the next kernel's CTAs
// on the SMs the previous kernel leaves, so its prologues overlap the tails
// in the same way.
#include "dv_attn.cuh"
#include "dv_colacc.cuh"
#include "dv_rowdot.cuh"

namespace dv {
namespace {

struct NoDep {  // the first phase reads only the call's inputs
    DV_DEV void wait() const {}
};

template <typename T, int NB, int LPK>
__global__ void __launch_bounds__(kThreads, 1) k_layer(const LayerArgs L)
{
    constexpr int U = 8;
    constexpr int P = colacc_chunks<NB>();
    const int cta = blockIdx.x, n = gridDim.x;
    int *bar = L.bar;
    auto after = [&](int c, int target) { return PhaseDep{bar + c, nullptr, target, 0, L.status}; };

    rowdot_body<T, NB, RK_PRED1, U>(L.pred1, cta, n, NoDep{});
    phase_arrive(bar + kBarPred1);
    rowdot_body<T, NB, RK_PRED2, U>(L.pred2, cta, n, after(kBarPred1, n));
    phase_arrive(bar + kBarPred2);
    rowdot_body<T, NB, RK_QKV, U>(L.qkv, cta, n, after(kBarPred2, n));
    if (cta == n - 1) {
        phase_arrive(bar + kBarSel);
    } else {
        phase_arrive(bar + kBarQkv);
        attn_body<T, LPK>(L.attn, cta, n - 1, after(kBarQkv, n - 1));
        phase_arrive(bar + kBarAttn);
        colacc_body<T, NB, CK_OPROJ, P>(L.oproj, cta, n - 1, after(kBarAttn, n - 1));
        phase_arrive(bar + kBarOproj);
    }
    // fc1 reads the neuron union before its own wait (gather list, first
    // rows), so the selection must be complete before the phase starts
    after(kBarSel, 1).wait();
    rowdot_body<T, NB, RK_FC1, U>(L.fc1, cta, n, after(kBarOproj, n - 1));
    phase_arrive(bar + kBarFc1);
    colacc_body<T, NB, CK_FC2, P>(L.fc2, cta, n, after(kBarFc1, n));

    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(bar + kBarExit, 1) == n - 1) {
            // every CTA has passed its last wait: clear the counters
            for (int i = 0; i < kBarCount; ++i)
                bar[i] = 0;
            __threadfence();
        }
    }
}

template <int NB>
cudaError_t launch_nb(const LayerArgs &a, int grid, size_t smem, cudaStream_t st)
{
    auto kern = k_layer<__half, NB, 16>;
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemCap);
    });
    if (e != cudaSuccess)
        return e;
    if (smem > kSmemCap)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int NB>
int ctas_nb(size_t smem)
{
    auto kern = k_layer<__half, NB, 16>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemCap) !=
        cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) != cudaSuccess)
        return 0;
    return n;
}

}  // namespace

cudaError_t launch_layer(int nb, const LayerArgs &a, int grid, size_t smem, cudaStream_t st)
{
    switch (nb) {
    case 1: return launch_nb<1>(a, grid, smem, st);
    case 2: return launch_nb<2>(a, grid, smem, st);
    default: return cudaErrorInvalidValue;
    }
}

int layer_ctas_per_sm(int nb, size_t smem)
{
    switch (nb) {
    case 1: return ctas_nb<1>(smem);
    case 2: return ctas_nb<2>(smem);
    default: return 0;
    }
}

}  // namespace dv
