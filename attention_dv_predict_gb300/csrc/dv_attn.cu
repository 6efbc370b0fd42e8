// dv_attn.cu -- decode attention over the selected heads' KV cache, and the
// copy probe used for the roofline denominator (sm_103a).
//
// For every batch row b and selected head h ("DejaVu Guide: Contextual
// Sparsity for LLM Inference", "2. Head-Pruned Attention Dispatch": only the
// active heads' KV history is read):
//   o = softmax(q . K[b, h, 0..kv_len]^T) . V[b, h, 0..kv_len]
// with q already scaled by 1/sqrt(dh) and position kv_len just appended.
//
// The kv_len + 1 positions are cut into splits; one warp handles one
// (b, head, split) unit.  A group of dh*sizeof(T)/16 lanes covers one key
// row with 16-byte loads, so a warp scores 32/group keys per step, reduces
// each dot product with xor shuffles inside its group and keeps a running
// max / sum / weighted V (online softmax) per group.  Groups then merge by
// butterfly shuffles, the split writes (max, sum, o) and the last split of
// a (b, head) to arrive combines all splits in split order.
#include "dv_common.cuh"

namespace dv {
namespace {

template <typename T, int LPK>
__global__ void __launch_bounds__(kThreads) k_attn(const AttnArgs a)
{
    constexpr int EPC = Elem<T>::EPC;
    constexpr int KPW = 32 / LPK;  // keys per warp step
    constexpr int UK = 4;          // warp steps in flight
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = lane / LPK, dc = lane % LPK;
    const int dh = a.dh;
    const int ns = min(max(*a.n_sel, 0), a.max_sel);
    const int per_b = ns * a.splits;
    const int units = a.B * per_b;
    const int L1 = a.kv_len + 1;
    const T *Kc = static_cast<const T *>(a.kc);
    const T *Vc = static_cast<const T *>(a.vc);
    const int nw = gridDim.x * kWarpsPerBlock;

    for (int u = blockIdx.x * kWarpsPerBlock + warp; u < units; u += nw) {
        const int b = u / per_b, rem = u - b * per_b;
        const int j = rem / a.splits, sp = rem - j * a.splits;
        const int h = a.sel[j];
        if (h < 0 || h >= a.H) {
            if (lane == 0)
                set_status(a.status, DV_ERR_DEVICE_INDEX);
            continue;
        }
        const int p0 = sp * a.split_len, p1 = min(L1, p0 + a.split_len);
        float q[EPC];
        {
            const float *qp = a.q + ((size_t)b * a.max_sel + j) * dh + dc * EPC;
#pragma unroll
            for (int e = 0; e < EPC; e += 4) {
                const float4 t = *reinterpret_cast<const float4 *>(qp + e);
                q[e] = t.x;
                q[e + 1] = t.y;
                q[e + 2] = t.z;
                q[e + 3] = t.w;
            }
        }
        const size_t base = ((size_t)b * a.H + h) * (size_t)a.kv_cap * dh + (size_t)dc * EPC;
        float m = -INFINITY, l = 0.f, o[EPC];
#pragma unroll
        for (int e = 0; e < EPC; ++e)
            o[e] = 0.f;

        for (int pb = p0; pb < p1; pb += KPW * UK) {
            uint4 kv[UK], vv[UK];
#pragma unroll
            for (int uu = 0; uu < UK; ++uu) {
                const int p = pb + uu * KPW + ks;
                if (p < p1) {
                    kv[uu] = ld_stream(Kc + base + (size_t)p * dh);
                    vv[uu] = ld_stream(Vc + base + (size_t)p * dh);
                } else {
                    kv[uu] = make_uint4(0u, 0u, 0u, 0u);
                    vv[uu] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int uu = 0; uu < UK; ++uu) {
                const int p = pb + uu * KPW + ks;
                float kf[EPC];
                Elem<T>::unpack(kv[uu], kf);
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    dot = fmaf(q[e], kf[e], dot);
#pragma unroll
                for (int off = LPK / 2; off > 0; off >>= 1)
                    dot += __shfl_xor_sync(0xffffffffu, dot, off);
                if (p < p1) {
                    float vf[EPC];
                    Elem<T>::unpack(vv[uu], vf);
                    const float mn = fmaxf(m, dot);
                    const float sc = expf(m - mn);
                    const float pe = expf(dot - mn);
                    l = fmaf(l, sc, pe);
#pragma unroll
                    for (int e = 0; e < EPC; ++e)
                        o[e] = fmaf(o[e], sc, pe * vf[e]);
                    m = mn;
                }
            }
        }
        // merge the key groups of the warp (butterfly: every lane ends with the total)
#pragma unroll
        for (int off = LPK; off < 32; off <<= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
            const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
            const float mn = fmaxf(m, m2);
            const float s1 = (m == -INFINITY) ? 0.f : expf(m - mn);
            const float s2 = (m2 == -INFINITY) ? 0.f : expf(m2 - mn);
            l = l * s1 + l2 * s2;
#pragma unroll
            for (int e = 0; e < EPC; ++e) {
                const float o2 = __shfl_xor_sync(0xffffffffu, o[e], off);
                o[e] = o[e] * s1 + o2 * s2;
            }
            m = mn;
        }
        float *dst = a.o + ((size_t)b * a.max_sel + j) * dh + dc * EPC;
        if (a.splits == 1) {
            if (ks == 0) {
                const float inv = 1.f / l;
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    dst[e] = o[e] * inv;
            }
            continue;
        }
        const int rec = kAttnRec + dh;
        float *recs = a.part + ((size_t)b * a.max_sel + j) * a.splits * rec;
        if (ks == 0) {
            float *r = recs + (size_t)sp * rec;
            if (dc == 0) {
                r[0] = m;
                r[1] = l;
            }
#pragma unroll
            for (int e = 0; e < EPC; ++e)
                r[kAttnRec + dc * EPC + e] = o[e];
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        int *cnt = a.cnt + (size_t)b * a.max_sel + j;
        if (lane == 0)
            last = (atomicAdd(cnt, 1) == a.splits - 1);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last)
            continue;
        __threadfence();
        if (ks == 0) {
            float M = -INFINITY;
            for (int s = 0; s < a.splits; ++s)
                M = fmaxf(M, __ldcg(recs + (size_t)s * rec));
            float Ls = 0.f, O[EPC];
#pragma unroll
            for (int e = 0; e < EPC; ++e)
                O[e] = 0.f;
            for (int s = 0; s < a.splits; ++s) {
                const float *r = recs + (size_t)s * rec;
                const float w = expf(__ldcg(r) - M);
                Ls = fmaf(__ldcg(r + 1), w, Ls);
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    O[e] = fmaf(__ldcg(r + kAttnRec + dc * EPC + e), w, O[e]);
            }
            const float inv = 1.f / Ls;
#pragma unroll
            for (int e = 0; e < EPC; ++e)
                dst[e] = O[e] * inv;
        }
        if (lane == 0)
            *cnt = 0;
    }
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
    case 1: return cudaLaunchKernelEx(&cfg, k_attn<T, 1>, a);
    case 2: return cudaLaunchKernelEx(&cfg, k_attn<T, 2>, a);
    case 4: return cudaLaunchKernelEx(&cfg, k_attn<T, 4>, a);
    case 8: return cudaLaunchKernelEx(&cfg, k_attn<T, 8>, a);
    case 16: return cudaLaunchKernelEx(&cfg, k_attn<T, 16>, a);
    case 32: return cudaLaunchKernelEx(&cfg, k_attn<T, 32>, a);
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
    k_copy<<<grid, kThreads, 0, st>>>(static_cast<uint4 *>(dst), static_cast<const uint4 *>(src),
                                      n16);
    return cudaGetLastError();
}

}  // namespace dv
