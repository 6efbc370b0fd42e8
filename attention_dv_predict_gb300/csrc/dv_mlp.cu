// dv_mlp.cu -- the sparse MLP block as one streaming pass (sm_103a), for
// batches of 1 and 2 rows.
//
//   act[b][n] = ReLU(w1[n] . norm(h1[b]) + b1[n])          (fc1 rows, gathered)
//   y[b]      = h1[b] + b2 + sum over selected n of act[b][n] * w2T[n][:]
// ("DejaVu Guide: Contextual Sparsity for LLM Inference", listing
// DejaVuSparseMLP.forward_sparse: only the selected neurons' fc1 rows and
// fc2 columns are read; w2T keeps each fc2 column as one contiguous row.)
//
// Work: CTA c owns the selected neurons [n0, n1) of the union (a contiguous,
// balanced share).  It computes their activations (fc1: the rows cut into
// segments of 32 x U chunks, dealt to its warps; per-segment sums in shared
// memory, added in segment order), then accumulates their fc2 rows into a
// partial y of its own (thread t owns chunks t + 512 j of the row) and
// stores it.  Nothing waits between the two halves but the CTA's own
// barrier, and the fc2 loads are in flight while the activations are summed.
// A second kernel adds the CTAs' partials in a fixed order (results do not
// depend on scheduling), the residual and the bias.
#include "dv_partials.cuh"
#include "dv_rowdot.cuh"

namespace dv {
namespace {

constexpr int kMlpU = 8;  // 16-byte chunks per lane in one fc1 segment

// Dynamic shared memory: the w2T row offsets [kMlpMaxRows], staged norm(h1)
// [NB][d], then the per-segment sums of the fc1 rows [2 kMlpMaxRows]
// [kMlpMaxSeg][NB] (two rows per neuron for SwiGLU), the activations
// [kMlpMaxRows][NB] and the neuron ids [kMlpMaxRows].
__host__ __device__ constexpr size_t mlp_smem(int nb, int d)
{
    return (size_t)kMlpMaxRows * 8 + (size_t)nb * d * 4 +
           (size_t)2 * kMlpMaxRows * kMlpMaxSeg * nb * 4 + (size_t)kMlpMaxRows * nb * 4 +
           (size_t)kMlpMaxRows * 4;
}

template <typename T, int NB, int CJ>
__global__ void __launch_bounds__(kThreads, 1) k_mlp(const MlpArgs a)
{
    constexpr int EPC = Elem<T>::EPC;
    constexpr int U = kMlpU;
    unsigned long long *stamps = chain_stamps(a.stamps);
    const PdlDep dep{stamps};
    extern __shared__ __align__(16) float smem[];
    __shared__ float red[34];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, cpr = d / EPC, G = gridDim.x, cta = blockIdx.x;
    const int nsu = (cpr + 32 * U - 1) / (32 * U);
    long long *soff = reinterpret_cast<long long *>(smem);
    float *xs = smem + 2 * kMlpMaxRows;
    float *upart = xs + (size_t)NB * d;                    // [fc1 row][seg][b]
    float *act = upart + (size_t)2 * kMlpMaxRows * kMlpMaxSeg * NB;  // [neuron][b]
    int *ssel = reinterpret_cast<int *>(act + (size_t)kMlpMaxRows * NB);
    const T *W1 = static_cast<const T *>(a.w1);
    const T *W2 = static_cast<const T *>(a.w2T);

    // this CTA's neurons: the union comes from kernels at least two launches
    // back (or from the caller, ahead of the call's first kernel)
    const int ns = min(max(ld_cg(a.n_sel), 0), a.max_sel);
    const int n0 = (int)((long long)ns * cta / G), n1 = (int)((long long)ns * (cta + 1) / G);
    const int nr = min(n1 - n0, kMlpMaxRows);
    if (tid < nr) {
        const int h = ld_cg(a.sel + n0 + tid);
        const bool ok = h >= 0 && h < a.N;
        ssel[tid] = ok ? h : -1;
        soff[tid] = ok ? (long long)h * d : -1;
        if (!ok)
            set_status(a.status, DV_ERR_DEVICE_INDEX);
    }
    if (tid == 0 && n1 - n0 > kMlpMaxRows)
        set_status(a.status, DV_ERR_INVALID_ARG);
    __syncthreads();

    // fc1 units (row, segment) of this CTA, balanced over its warps; SwiGLU
    // layers have two fc1 rows per neuron (gate, up), side by side in w1
    const int sw = a.swiglu ? 1 : 0;
    const int units = (nr << sw) * nsu;
    const int ub = units * warp / kWarpsPerBlock, ue = units * (warp + 1) / kWarpsPerBlock;
    auto load1 = [&](int u, uint4 (&v)[U]) {
        const int row = u / nsu, sg = u - row * nsu;
        const int h = (u < ue) ? ssel[row >> sw] : -1;
        const T *p = W1 + ((size_t)(h < 0 ? 0 : h << sw) + (row & sw)) * d;
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int c = sg * 32 * U + lane + 32 * j;
            v[j] = (h >= 0 && c < cpr) ? ld_stream(p + (size_t)c * EPC)
                                       : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    uint4 cur[U];
    load1(ub, cur);  // weights only: in flight across the wait

    dep.wait();  // h1 comes from the previous kernel
    for (int b = 0; b < NB; ++b) {
        float *dst = xs + (size_t)b * d;
        if (b >= a.B) {
            for (int c = tid; c < d; c += kThreads)
                dst[c] = 0.f;
            continue;
        }
        norm_row<T>(a.h1 + (size_t)b * d, d, a.norm_g, a.norm_b, a.norm_kind, a.eps, red,
                    [&](int c, const float(&v)[EPC]) { stage_chunk_store<T>(dst, d, c, v); });
    }
    __syncthreads();

    for (int u = ub; u < ue; ++u) {
        uint4 nxt[U];
        load1(u + 1, nxt);
        const int row = u / nsu, sg = u - row * nsu;
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b)
            acc[b] = 0.f;
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int c = sg * 32 * U + lane + 32 * j;
            if (c < cpr)
                fma_chunk<T, NB>(cur[j], xs, d, c, acc);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const float s = warp_sum(acc[b]);
            if (lane == 0)
                upart[((size_t)row * kMlpMaxSeg + sg) * NB + b] = s;
        }
#pragma unroll
        for (int j = 0; j < U; ++j)
            cur[j] = nxt[j];
    }

    // fc2: a ring of four rows in flight per thread; the first three rows'
    // loads go out before the activations are summed
    uint4 w0[CJ], w1[CJ], w2[CJ];
    col_ring_load<T, NB, CJ>(W2, 0 < nr ? soff[0] : -1, d, w0);
    col_ring_load<T, NB, CJ>(W2, 1 < nr ? soff[1] : -1, d, w1);
    col_ring_load<T, NB, CJ>(W2, 2 < nr ? soff[2] : -1, d, w2);
    __syncthreads();  // every segment sum is in shared memory
    if (tid < nr * NB) {
        const int row = tid / NB, b = tid - row * NB;
        const int h = ssel[row];
        const T *b1 = static_cast<const T *>(a.b1);
        float s = 0.f, s2 = 0.f;
        for (int sg = 0; sg < nsu; ++sg) {
            s += upart[((size_t)(row << sw) * kMlpMaxSeg + sg) * NB + b];
            if (sw)
                s2 += upart[((size_t)((row << 1) + 1) * kMlpMaxSeg + sg) * NB + b];
        }
        float v = 0.f;
        if (h >= 0 && b < a.B) {
            if (sw) {  // silu(gate) * up
                const float g = s + Elem<T>::load(b1, (size_t)2 * h);
                const float u = s2 + Elem<T>::load(b1, (size_t)2 * h + 1);
                v = g / (1.f + expf(-g)) * u;
            } else {
                v = fmaxf(s + Elem<T>::load(b1, (size_t)h), 0.f);
            }
        }
        act[row * NB + b] = v;
    }
    __syncthreads();
    chain_stamp(stamps, 4);
    // this CTA's partial (zeros when it owns no neuron)
    col_ring<T, NB, CJ>(W2, soff, act, nr, d, w0, w1, w2, a.part + (size_t)cta * NB * d);
    chain_stamp_end(stamps);
}

template <typename T, int NB, int CJ>
cudaError_t launch_main(const MlpArgs &a, int grid, cudaStream_t st, bool pdl)
{
    auto kern = k_mlp<T, NB, CJ>;
    const size_t smem = mlp_smem(NB, a.d);
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemCap);
    });
    if (e != cudaSuccess)
        return e;
    if (smem > kSmemCap)
        return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int NB>
cudaError_t dispatch_cj(int cj, const MlpArgs &a, int grid, cudaStream_t st, bool pdl)
{
    switch (cj) {
    case 1: return launch_main<T, NB, 1>(a, grid, st, pdl);
    case 2: return launch_main<T, NB, 2>(a, grid, st, pdl);
    case 3: return launch_main<T, NB, 3>(a, grid, st, pdl);
    case 4:
        if constexpr (NB == 1)
            return launch_main<T, NB, 4>(a, grid, st, pdl);
        return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int mlp_chunk_cols(int dtype, int d)
{
    const int epc = dtype == DV_F16 ? 8 : 4;
    if (d % epc)
        return 0;
    return (d / epc + kThreads - 1) / kThreads;
}

bool mlp_fused_ok(const dv_layer_desc &D, int B, int max_u_n, int nsm)
{
    if (B < 1 || B > 2 || nsm > kPartMaxCtas || D.d_model % 4)
        return false;
    const int epc = D.dtype == DV_F16 ? 8 : 4;
    const int cpr = D.d_model / epc;
    const int cj = mlp_chunk_cols(D.dtype, D.d_model);
    // (at two batch rows four chunk columns would spill the accumulators)
    if (cj < 1 || cj > (B == 1 ? 4 : 3) || (cpr + 32 * kMlpU - 1) / (32 * kMlpU) > kMlpMaxSeg)
        return false;
    if ((max_u_n + nsm - 1) / nsm > kMlpMaxRows)
        return false;
    return mlp_smem(B, D.d_model) <= kSmemCap;
}

cudaError_t launch_mlp(int dtype, const MlpArgs &a, int grid, cudaStream_t st, bool pdl)
{
    const int cj = mlp_chunk_cols(dtype, a.d);
    if (dtype == DV_F16)
        return a.B == 1 ? dispatch_cj<__half, 1>(cj, a, grid, st, pdl)
                        : dispatch_cj<__half, 2>(cj, a, grid, st, pdl);
    return a.B == 1 ? dispatch_cj<float, 1>(cj, a, grid, st, pdl)
                    : dispatch_cj<float, 2>(cj, a, grid, st, pdl);
}

cudaError_t launch_part_sum(int dtype, const PartSumArgs &a, cudaStream_t st)
{
    if (a.nparts > kPartMaxCtas || a.B < 1 || a.B > 2)
        return cudaErrorInvalidValue;
    if (dtype == DV_F16)
        return a.B == 1 ? launch_part_sum_t<__half, 1>(a, st) : launch_part_sum_t<__half, 2>(a, st);
    return a.B == 1 ? launch_part_sum_t<float, 1>(a, st) : launch_part_sum_t<float, 2>(a, st);
}

}  // namespace dv
