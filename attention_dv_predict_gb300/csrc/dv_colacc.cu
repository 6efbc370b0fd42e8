// dv_colacc.cu -- column-gather GEMV kernels of the sparse layer decode (sm_103a).
//
//   OPROJ  h1[b] = x[b] + b_o + sum over selected heads h and e < dh of
//          o[b][h][e] * w_oT[h][e][:]       ("DejaVu Guide: Contextual Sparsity
//          for LLM Inference", "2. Head-Pruned Attention Dispatch": inactive
//          heads' output-projection weights are never read);
//   FC2    y[b] = h1[b] + b2 + sum over selected neurons j of a[b][j] * w2T[j][:]
//          (listing, DejaVuSparseMLP.forward_sparse, steps 3-4: the selected
//          fc2 columns, kept transposed so each is one contiguous row).
//
// The gathered rows are contiguous, so every warp reads whole 512-byte
// (binary16) slices of them with 16-byte loads.  Work is split two ways:
// column slices of 32 x 16 bytes (one per warp) and G groups of rows
// (split-K).  Each (group, slice) unit accumulates in registers and writes a
// partial; the last unit of a slice to arrive sums the G partials in group
// order and adds bias and residual, so the result does not depend on
// scheduling.
#include "dv_common.cuh"

namespace dv {
namespace {

template <typename T, int NB, int KIND>
__global__ void __launch_bounds__(kThreads, 1) k_colacc(const ColArgs a)
{
    constexpr int EPC = Elem<T>::EPC;
    constexpr int CW = 32 * EPC;  // columns per warp slice
    constexpr int U = 8;          // rows in flight per lane
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile = blockIdx.y, b0 = tile * NB;
    const int ns = min(max(*a.n_sel, 0), a.max_sel);
    const int rows = (KIND == CK_OPROJ) ? ns * a.dh : ns;
    const int S = (a.d + CW - 1) / CW;
    const int G = a.G;
    const int rg = (rows + G - 1) / G;
    const int units = G * S;
    const T *W = static_cast<const T *>(a.w);
    const int nw = gridDim.x * kWarpsPerBlock;

    for (int u = blockIdx.x * kWarpsPerBlock + warp; u < units; u += nw) {
        const int g = u / S, s = u - g * S;
        const int r0 = min(rows, g * rg), r1 = min(rows, r0 + rg);
        const int col = s * CW + lane * EPC;
        const bool colok = col < a.d;
        float acc[NB][EPC];
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int e = 0; e < EPC; ++e)
                acc[b][e] = 0.f;

        for (int i0 = r0; i0 < r1; i0 += 32) {
            const int nr = min(32, r1 - i0);
            // lane l fetches the metadata of row i0 + l: weight row offset and
            // the row's coefficient for every batch row of the tile
            long long off = -1;
            float cf[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                cf[b] = 0.f;
            if (lane < nr) {
                const int i = i0 + lane;
                int wrow;
                if constexpr (KIND == CK_OPROJ) {
                    const int j = i / a.dh, e = i - j * a.dh;
                    const int h = a.sel[j];
                    wrow = (h >= 0 && h < a.sel_range) ? h * a.dh + e : -1;
                } else {
                    const int j = a.sel[i];
                    wrow = (j >= 0 && j < a.sel_range) ? j : -1;
                }
                if (wrow >= 0) {
                    off = (long long)wrow * a.d;
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        if (b0 + b < a.B)
                            cf[b] = a.coef[(size_t)(b0 + b) * a.coef_ld + i];
                } else {
                    set_status(a.status, DV_ERR_DEVICE_INDEX);
                }
            }
            for (int rr = 0; rr < nr; rr += U) {
                uint4 v[U];
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    const long long o = __shfl_sync(0xffffffffu, off, (rr + q) & 31);
                    v[q] = (rr + q < nr && o >= 0 && colok)
                               ? ld_stream(W + (size_t)o + col)
                               : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int q = 0; q < U; ++q) {
                    float f[EPC];
                    Elem<T>::unpack(v[q], f);
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const float c = __shfl_sync(0xffffffffu, cf[b], (rr + q) & 31);
#pragma unroll
                        for (int e = 0; e < EPC; ++e)
                            acc[b][e] = fmaf(c, f[e], acc[b][e]);
                    }
                }
            }
        }

        if (G == 1) {
            if (colok) {
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    if (b0 + b >= a.B)
                        break;
                    const float *res = a.res + (size_t)(b0 + b) * a.d + col;
                    float *out = a.out + (size_t)(b0 + b) * a.d + col;
#pragma unroll
                    for (int e = 0; e < EPC; ++e)
                        out[e] = (res[e] + Elem<T>::load(static_cast<const T *>(a.bias),
                                                         (size_t)col + e)) +
                                 acc[b][e];
                }
            }
            continue;
        }
        // publish this group's partial, then let the last group of the slice reduce
        float *pp = a.part + ((size_t)tile * G + g) * NB * a.d;
        if (colok) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int e = 0; e < EPC; e += 4)
                    *reinterpret_cast<float4 *>(pp + (size_t)b * a.d + col + e) =
                        make_float4(acc[b][e], acc[b][e + 1], acc[b][e + 2], acc[b][e + 3]);
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0)
            last = (atomicAdd(&a.cnt[tile * S + s], 1) == G - 1);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last)
            continue;
        __threadfence();
        if (colok) {
            float sum[NB][EPC];
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    sum[b][e] = 0.f;
            const float *base = a.part + (size_t)tile * G * NB * a.d;
            for (int gg = 0; gg < G; ++gg) {
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                    for (int e = 0; e < EPC; e += 4) {
                        const float4 p = __ldcg(reinterpret_cast<const float4 *>(
                            base + ((size_t)gg * NB + b) * a.d + col + e));
                        sum[b][e] += p.x;
                        sum[b][e + 1] += p.y;
                        sum[b][e + 2] += p.z;
                        sum[b][e + 3] += p.w;
                    }
            }
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b0 + b >= a.B)
                    break;
                const float *res = a.res + (size_t)(b0 + b) * a.d + col;
                float *out = a.out + (size_t)(b0 + b) * a.d + col;
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    out[e] = (res[e] + Elem<T>::load(static_cast<const T *>(a.bias),
                                                     (size_t)col + e)) +
                             sum[b][e];
            }
        }
        if (lane == 0)
            a.cnt[tile * S + s] = 0;
    }
}

template <typename T, int NB, int KIND>
cudaError_t launch_one(const ColArgs &a, dim3 grid, cudaStream_t st, bool pdl)
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
    return cudaLaunchKernelEx(&cfg, k_colacc<T, NB, KIND>, a);
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
