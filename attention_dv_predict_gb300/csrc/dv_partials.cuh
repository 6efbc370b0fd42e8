// dv_partials.cuh -- the second half of the one-pass column accumulations
// (sm_103a): out[b][col] = res[b][col] + bias[col] + sum over CTAs c of
// part[c][b][col], the partials added in a fixed order so the result does
// not depend on scheduling (the one-pass MLP: y = h1 + b2 + ...).
#pragma once

#include "dv_common.cuh"

namespace dv {
namespace {

constexpr int kRedSlices = 32;
constexpr int kRedQuads = kThreads / kRedSlices;  // 16 column quads: 64 columns

// CTA (g, b): columns [64 g, 64 g + 64) of batch row b; thread (s, q)
// sums the partials c = s, s + 32, ... of column quad q, all in flight at
// once, then 16 threads add the 32 slices in order.  (Narrow CTAs: at 128
// columns 96 of the 152 SMs worked and each CTA took ~2.6 us.)
template <typename T, int NB>
__global__ void __launch_bounds__(kThreads) k_part_sum(const PartSumArgs a)
{
    unsigned long long *stamps =
        chain_stamps((int)blockIdx.x < a.stamp_ctas ? a.stamps : nullptr);
    __shared__ float4 sred[kRedSlices][kRedQuads];
    const int tid = threadIdx.x, q = tid % kRedQuads, s = tid / kRedQuads;
    const int b = blockIdx.y, col = (blockIdx.x * kRedQuads + q) * 4;
    const bool in = col < a.d && b < a.B;
    float4 base = make_float4(0.f, 0.f, 0.f, 0.f);
    if (in && s == 0) {  // inputs from two launches back or older
        const float4 h = __ldcg(reinterpret_cast<const float4 *>(a.res + (size_t)b * a.d + col));
        const T *bias = static_cast<const T *>(a.bias);
        base = make_float4(h.x + Elem<T>::load(bias, col), h.y + Elem<T>::load(bias, col + 1),
                           h.z + Elem<T>::load(bias, col + 2), h.w + Elem<T>::load(bias, col + 3));
    }
    pdl_wait();
    chain_stamp(stamps, 1);
    pdl_launch_dependents();
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    if (in) {
        constexpr int kBatch = kPartMaxCtas / kRedSlices;
        for (int c0 = s; c0 < a.nparts; c0 += kBatch * kRedSlices) {
            float4 v[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int c = c0 + k * kRedSlices;
                v[k] = c < a.nparts ? __ldcg(reinterpret_cast<const float4 *>(
                                          a.part + ((size_t)c * NB + b) * a.d + col))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                sum.x += v[k].x;
                sum.y += v[k].y;
                sum.z += v[k].z;
                sum.w += v[k].w;
            }
        }
    }
    chain_stamp(stamps, 4);  // partials summed (thread 0's slice)
    sred[s][q] = sum;
    __syncthreads();
    if (s == 0 && in) {
        float4 t = base;
        for (int k = 0; k < kRedSlices; ++k) {
            const float4 v = sred[k][q];
            t.x += v.x;
            t.y += v.y;
            t.z += v.z;
            t.w += v.w;
        }
        *reinterpret_cast<float4 *>(a.out + (size_t)b * a.d + col) = t;
    }
    chain_stamp_end(stamps);
}

template <typename T, int NB>
cudaError_t launch_part_sum_t(const PartSumArgs &a, cudaStream_t st)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(part_sum_groups(a.d), a.B);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_part_sum<T, NB>, a);
}

// Column-accumulate pass of a one-pass kernel: rows [0, nr) of
// this CTA (weight row offsets off[r], -1 = skip; coefficients coef[r][NB]
// in shared memory) times W, thread t owning 16-byte chunks t + 512 j of
// the d columns; a ring of four rows in flight per thread.  w0..w2 hold
// rows 0..2, loaded by the caller (before whatever it waited on).  Stores
// this CTA's partial part[cta][b][d].
template <typename T, int NB, int CJ>
DV_DEV void col_ring_load(const T *W, long long off, int d, uint4 (&v)[CJ])
{
    constexpr int EPC = Elem<T>::EPC;
    const int cpr = d / EPC;
#pragma unroll
    for (int j = 0; j < CJ; ++j) {
        const int c = threadIdx.x + kThreads * j;
        v[j] = (off >= 0 && c < cpr) ? ld_stream(W + off + (size_t)c * EPC)
                                     : make_uint4(0u, 0u, 0u, 0u);
    }
}

template <typename T, int NB, int CJ>
DV_DEV void col_ring(const T *W, const long long *off, const float *coef, int nr, int d,
                     uint4 (&w0)[CJ], uint4 (&w1)[CJ], uint4 (&w2)[CJ], float *part_cta)
{
    constexpr int EPC = Elem<T>::EPC;
    const int cpr = d / EPC;
    float acc[CJ][EPC][NB];
#pragma unroll
    for (int j = 0; j < CJ; ++j)
#pragma unroll
        for (int e = 0; e < EPC; ++e)
#pragma unroll
            for (int b = 0; b < NB; ++b)
                acc[j][e][b] = 0.f;
    auto ld = [&](int r, uint4 (&v)[CJ]) {
        col_ring_load<T, NB, CJ>(W, r < nr ? off[r] : -1, d, v);
    };
    auto use = [&](int r, const uint4 (&v)[CJ]) {
        if (r >= nr)
            return;
        float cf[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b)
            cf[b] = coef[r * NB + b];
#pragma unroll
        for (int j = 0; j < CJ; ++j) {
            float f[EPC];
            Elem<T>::unpack(v[j], f);
#pragma unroll
            for (int e = 0; e < EPC; ++e)
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    acc[j][e][b] = fmaf(cf[b], f[e], acc[j][e][b]);
        }
    };
    uint4 w3[CJ];
    for (int r = 0; r < nr; r += 4) {
        ld(r + 3, w3);
        use(r, w0);
        ld(r + 4, w0);
        use(r + 1, w1);
        ld(r + 5, w1);
        use(r + 2, w2);
        ld(r + 6, w2);
        use(r + 3, w3);
    }
#pragma unroll
    for (int j = 0; j < CJ; ++j) {
        const int c = threadIdx.x + kThreads * j;
        if (c >= cpr)
            continue;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float *o = part_cta + (size_t)b * d + (size_t)c * EPC;
#pragma unroll
            for (int e = 0; e < EPC; e += 4)
                *reinterpret_cast<float4 *>(o + e) =
                    make_float4(acc[j][e][b], acc[j][e + 1][b], acc[j][e + 2][b], acc[j][e + 3][b]);
        }
    }
}

}  // namespace
}  // namespace dv
