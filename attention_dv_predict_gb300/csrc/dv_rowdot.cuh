// dv_rowdot.cuh -- the row-dot GEMV of the sparse layer decode (sm_103a):
// the body shared by its stand-alone kernels (dv_rowdot.cu) and the
// fused steps that the streaming kernel (dv_stream.cu) restates.
//
// One body serves every step whose output element is the dot product of one
// weight row with an activation vector:
//   PRED1  head scores s_h = x_pred . pred_h^T and the low-rank factor
//          u = x_pred . pred_a^T ("DejaVu Guide: Contextual Sparsity for LLM
//          Inference", "1. Mathematical Formulation of Lookahead Predictors");
//   PRED2  neuron scores s_n = u . pred_b^T; every CTA adds its scores to the
//          histogram of the keys' top 11 bits (dv_select.cuh).  In the fused
//          decode its last CTA selects the heads and writes LayerNorm(x)
//          instead of taking rows, then publishes both with a flag;
//   QKV    the selected heads' q, k, v rows on LayerNorm(x), bias, q scaling
//          and the KV append ("2. Head-Pruned Attention Dispatch").  In the
//          fused decode its last CTA runs the whole neuron selection once the
//          stage-2 scores are complete;
//   FC1    the selected neurons' fc1 rows on LayerNorm(h1), bias and ReLU
//          (the guide's listing, DejaVuSparseMLP.forward_sparse, steps 1-2).
//
// Streaming: every weight byte is read once with a 16-byte non-allocating
// load.  Rows are cut into units of at most 32*U chunks (long rows) or packed
// several to a unit (short rows); the units are dealt to all warps of the
// participating CTAs in contiguous, balanced ranges, and each warp keeps two
// units in flight (the next unit's loads are issued before the current one is
// consumed).  The activations are staged once per CTA in shared memory while
// the first weight loads are in flight.  A row split across two or more warp
// ranges is combined by the last warp to finish it (an atomic count of the
// row's units), which sums the partials in warp order: results do not depend
// on scheduling.
//
// Dependencies (Dep, dv_common.cuh): the body issues whatever does not depend
// on the producing step (its first weight loads) before dep.wait(); as a
// stand-alone kernel that is the programmatic-dependent grid wait, after
// which the next kernel may launch, so data two kernels back is always
// complete.
#pragma once

#include "dv_common.cuh"
#include "dv_select.cuh"

namespace dv {
namespace {



// Staged activation layout: for binary16 weights a 16-byte chunk holds 8
// elements; the staged activations are split into the low and high 4 of
// every chunk (two float4 arrays) so each lane's two float4 reads hit
// consecutive addresses across the warp (no bank conflicts).  For binary32
// weights the layout is the natural one.
template <typename T, int NB>
DV_DEV void fma_chunk(const uint4 &v, const float *xs, int K, int gc, float (&acc)[NB])
{
    constexpr int EPC = Elem<T>::EPC;
    float f[EPC];
    Elem<T>::unpack(v, f);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const float *xb = xs + (size_t)b * K;
        if constexpr (EPC == 8) {
            const float4 lo = reinterpret_cast<const float4 *>(xb)[gc];
            const float4 hi = reinterpret_cast<const float4 *>(xb + (K >> 1))[gc];
            float s = acc[b];
            s = fmaf(f[0], lo.x, s);
            s = fmaf(f[1], lo.y, s);
            s = fmaf(f[2], lo.z, s);
            s = fmaf(f[3], lo.w, s);
            s = fmaf(f[4], hi.x, s);
            s = fmaf(f[5], hi.y, s);
            s = fmaf(f[6], hi.z, s);
            s = fmaf(f[7], hi.w, s);
            acc[b] = s;
        } else {
            const float4 xv = reinterpret_cast<const float4 *>(xb)[gc];
            float s = acc[b];
            s = fmaf(f[0], xv.x, s);
            s = fmaf(f[1], xv.y, s);
            s = fmaf(f[2], xv.z, s);
            s = fmaf(f[3], xv.w, s);
            acc[b] = s;
        }
    }
}

// ---------------------------------------------------------------------------
// Activation staging: NB rows [b0, b0 + NB), normalised when asked.  A thread
// owns up to kStageChunks 16-byte chunks of a row (EPC elements each, strided
// by the block size) and keeps them in registers, so x, the norm gain and the
// norm bias are each read once with all loads in flight together; the mean
// and variance come from two block reductions over the registers.
constexpr int kStageChunks = 4;

template <typename T>
DV_DEV void stage_chunk_store(float *dst, int K, int c, const float (&v)[Elem<T>::EPC])
{
    if constexpr (Elem<T>::EPC == 8) {
        reinterpret_cast<float4 *>(dst)[c] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(dst + (K >> 1))[c] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        reinterpret_cast<float4 *>(dst)[c] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// One activation row src[0..K), normalised when g != nullptr, handed chunk
// by chunk to store(c, v) (c = chunk index, v = its EPC values).  Every
// thread of the block calls it; barriers inside.
template <typename T, typename Store>
DV_DEV void norm_row(const float *src, int K, const void *g_, const void *b_, int norm_kind,
                     float eps, float *red, Store store)
{
    constexpr int EPC = Elem<T>::EPC;
    constexpr int CQ = kStageChunks;
    const int nch = K / EPC, tid = threadIdx.x, nt = blockDim.x;
    const bool norm = g_ != nullptr;
    const bool ln = norm_kind == DV_LAYERNORM;
    for (int c0 = 0; c0 < nch; c0 += nt * CQ) {
        // chunks c0 + tid + q*nt of this row (all of it when nch <= nt*CQ)
        float v[CQ][EPC];
        uint4 gv[CQ], bv[CQ];
#pragma unroll
        for (int q = 0; q < CQ; ++q) {
            const int c = c0 + tid + q * nt;
            const bool in = c < nch;
#pragma unroll
            for (int e = 0; e < EPC; e += 4) {
                const float4 t =
                    in ? __ldcg(reinterpret_cast<const float4 *>(src + (size_t)c * EPC) + e / 4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
                v[q][e] = t.x;
                v[q][e + 1] = t.y;
                v[q][e + 2] = t.z;
                v[q][e + 3] = t.w;
            }
            gv[q] = (in && norm) ? reinterpret_cast<const uint4 *>(g_)[c]
                                 : make_uint4(0u, 0u, 0u, 0u);
            bv[q] = (in && norm && ln) ? reinterpret_cast<const uint4 *>(b_)[c]
                                       : make_uint4(0u, 0u, 0u, 0u);
        }
        float mean = 0.f, inv = 1.f;
        if (norm) {
            if (nch > nt * CQ) {
                // long rows: statistics over the whole row first (rare)
                float s = 0.f, ss = 0.f;
                for (int c = tid; c < nch; c += nt)
                    for (int e = 0; e < EPC; ++e)
                        s += __ldcg(src + (size_t)c * EPC + e);
                mean = ln ? block_sum(s, red) / (float)K : 0.f;
                for (int c = tid; c < nch; c += nt)
                    for (int e = 0; e < EPC; ++e) {
                        const float d = __ldcg(src + (size_t)c * EPC + e) - mean;
                        ss = fmaf(d, d, ss);
                    }
                inv = rsqrtf(block_sum(ss, red) / (float)K + eps);
            } else {
                float s = 0.f;
#pragma unroll
                for (int q = 0; q < CQ; ++q)
#pragma unroll
                    for (int e = 0; e < EPC; ++e)
                        s += v[q][e];
                mean = ln ? block_sum(s, red) / (float)K : 0.f;
                float ss = 0.f;
#pragma unroll
                for (int q = 0; q < CQ; ++q) {
                    if (c0 + tid + q * nt >= nch)
                        break;
#pragma unroll
                    for (int e = 0; e < EPC; ++e) {
                        const float d = v[q][e] - mean;
                        ss = fmaf(d, d, ss);
                    }
                }
                inv = rsqrtf(block_sum(ss, red) / (float)K + eps);
            }
        }
#pragma unroll
        for (int q = 0; q < CQ; ++q) {
            const int c = c0 + tid + q * nt;
            if (c >= nch)
                break;
            if (norm) {
                float g[EPC], be[EPC];
                Elem<T>::unpack(gv[q], g);
                if (ln)
                    Elem<T>::unpack(bv[q], be);
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    v[q][e] = (v[q][e] - mean) * inv * g[e] + (ln ? be[e] : 0.f);
            }
            store(c, v[q]);
        }
    }
}

// Statistics of one row src[0..K) (K a multiple of 4, 16-byte aligned) by
// one warp, in one pass over the row (read at L2): (mean, 1/sqrt(var + eps))
// for LayerNorm, (0, 1/sqrt(mean of squares + eps)) for RMSNorm.  For
// LayerNorm each lane sums its values shifted by its own first one, turns
// that into (count, mean, M2) and the lanes merge pairwise (Chan, Golub and
// LeVeque's update); lane 0's result is broadcast.
DV_DEV float2 warp_row_stats(const float *src, int K, bool ln, float eps, int lane)
{
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    const int n4 = K >> 2;
    if (!ln) {
        float ss = 0.f;
#pragma unroll 8
        for (int i = lane; i < n4; i += 32) {
            const float4 t = __ldcg(s4 + i);
            ss = fmaf(t.x, t.x, ss);
            ss = fmaf(t.y, t.y, ss);
            ss = fmaf(t.z, t.z, ss);
            ss = fmaf(t.w, t.w, ss);
        }
        return make_float2(0.f, rsqrtf(warp_sum(ss) / (float)K + eps));
    }
    const float c = lane < n4 ? __ldcg(src + 4 * lane) : 0.f;
    float s1 = 0.f, s2 = 0.f;
#pragma unroll 8
    for (int i = lane; i < n4; i += 32) {
        const float4 t = __ldcg(s4 + i);
        const float dx = t.x - c, dy = t.y - c, dz = t.z - c, dw = t.w - c;
        s1 += (dx + dy) + (dz + dw);
        s2 = fmaf(dx, dx, s2);
        s2 = fmaf(dy, dy, s2);
        s2 = fmaf(dz, dz, s2);
        s2 = fmaf(dw, dw, s2);
    }
    float n = (float)(4 * ((n4 - lane + 31) / 32 > 0 ? (n4 - lane + 31) / 32 : 0));
    float mean = n > 0.f ? c + s1 / n : 0.f;
    float m2 = n > 0.f ? fmaxf(s2 - s1 * (s1 / n), 0.f) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float nb = __shfl_xor_sync(0xffffffffu, n, o);
        const float mb = __shfl_xor_sync(0xffffffffu, mean, o);
        const float m2b = __shfl_xor_sync(0xffffffffu, m2, o);
        const float tot = n + nb;
        if (tot > 0.f) {
            const float delta = mb - mean;
            mean = fmaf(delta, nb / tot, mean);
            m2 = m2 + m2b + delta * delta * (n * nb / tot);
            n = tot;
        }
    }
    mean = __shfl_sync(0xffffffffu, mean, 0);
    m2 = __shfl_sync(0xffffffffu, m2, 0);
    return make_float2(mean, rsqrtf(m2 / (float)K + eps));
}

// Normalised chunk c (EPC values from src + c EPC) with the row statistics st.
template <typename T>
DV_DEV void norm_chunk(const float *src, int c, const void *g_, const void *b_, bool ln, float2 st,
                       float (&v)[Elem<T>::EPC])
{
    constexpr int EPC = Elem<T>::EPC;
    const float4 *s4 = reinterpret_cast<const float4 *>(src + (size_t)c * EPC);
#pragma unroll
    for (int e = 0; e < EPC; e += 4) {
        const float4 t = __ldcg(s4 + e / 4);
        v[e] = t.x;
        v[e + 1] = t.y;
        v[e + 2] = t.z;
        v[e + 3] = t.w;
    }
    if (g_) {
        float g[EPC], be[EPC];
        Elem<T>::unpack(reinterpret_cast<const uint4 *>(g_)[c], g);
        if (ln)
            Elem<T>::unpack(reinterpret_cast<const uint4 *>(b_)[c], be);
#pragma unroll
        for (int e = 0; e < EPC; ++e)
            v[e] = (v[e] - st.x) * st.y * g[e] + (ln ? be[e] : 0.f);
    }
}

template <typename T, int NB>
DV_DEV void stage_acts(const RowArgs &a, float *xs, int b0, float *red)
{
    const int K = a.K;
    if constexpr (NB >= 4) {
        // several rows: their statistics a warp per row, then chunks of any
        // row by every thread
        constexpr int EPC = Elem<T>::EPC;
        __shared__ float2 sstat[NB];
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const bool ln = a.norm_kind == DV_LAYERNORM;
        if (a.norm_g) {
            for (int bi = warp; bi < NB; bi += kWarpsPerBlock)
                if (b0 + bi < a.B) {
                    const float2 st =
                        warp_row_stats(a.x + (size_t)(b0 + bi) * a.x_ld, K, ln, a.eps, lane);
                    if (lane == 0)
                        sstat[bi] = st;
                }
            __syncthreads();
        }
        const int cpr = K / EPC;
        for (int i = threadIdx.x; i < NB * cpr; i += blockDim.x) {
            const int bi = i / cpr, c = i - bi * cpr, b = b0 + bi;
            float v[EPC];
            if (b < a.B) {
                norm_chunk<T>(a.x + (size_t)b * a.x_ld, c, a.norm_g, a.norm_b, ln,
                              a.norm_g ? sstat[bi] : make_float2(0.f, 1.f), v);
            } else {
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    v[e] = 0.f;
            }
            stage_chunk_store<T>(xs + (size_t)bi * K, K, c, v);
        }
        __syncthreads();
        return;
    }
    for (int bi = 0; bi < NB; ++bi) {
        const int b = b0 + bi;
        float *dst = xs + (size_t)bi * K;
        if (b >= a.B) {
            for (int c = threadIdx.x; c < K; c += blockDim.x)
                dst[c] = 0.f;
            continue;
        }
        norm_row<T>(a.x + (size_t)b * a.x_ld, K, a.norm_g, a.norm_b, a.norm_kind, a.eps, red,
                    [&](int c, const float(&v)[Elem<T>::EPC]) {
                        stage_chunk_store<T>(dst, K, c, v);
                    });
    }
    __syncthreads();
}

// Side work of one CTA of the stage-2 predictor kernel in the fused decode:
// select the heads (the head scores come from the previous kernel) and
// write the attention block's normalised input xn = norm(x) to global
// memory, both for the QKV kernel that follows.  The side work may be split
// over nparts CTAs: this one (part) normalises rows part, part + nparts, ...
// and part 0 also selects the heads.  A lone side CTA with kSideWarpRows
// rows or more deals the rows out to its warps; otherwise the whole CTA
// normalises one row after the other (a lone warp per row was slower for
// few rows, and one CTA's L2 bandwidth too little for many).
constexpr int kSideWarpRows = 4;

template <typename T>
__device__ __noinline__ void pred2_side(const RowArgs &a, float *red, int part, int nparts)
{
    __shared__ unsigned wbits[kWarpsPerBlock * kHeadKPL];
    __shared__ unsigned ubits[kHeadKPL];
    const PredSide &p = a.side;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool ln = p.norm_kind == DV_LAYERNORM;
    constexpr int EPC = Elem<T>::EPC;
    const bool by_warp = nparts == 1 && a.B >= kSideWarpRows;
    if (!by_warp) {
        for (int b = part; b < a.B; b += nparts) {
            float *dst = p.xn + (size_t)b * p.d;
            norm_row<T>(p.x + (size_t)b * p.x_ld, p.d, p.g, p.beta, p.norm_kind, p.eps, red,
                        [&](int c, const float(&v)[EPC]) {
#pragma unroll
                            for (int e = 0; e < EPC; e += 4)
                                *reinterpret_cast<float4 *>(dst + (size_t)c * EPC + e) =
                                    make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                        });
        }
    }
    for (int b = warp; b < a.B && by_warp; b += kWarpsPerBlock) {
        const float *src = p.x + (size_t)b * p.x_ld;
        float *dst = p.xn + (size_t)b * p.d;
        const float2 st = p.g ? warp_row_stats(src, p.d, ln, p.eps, lane) : make_float2(0.f, 1.f);
        for (int c = lane; c < p.d / EPC; c += 32) {
            float v[EPC];
            norm_chunk<T>(src, c, p.g, p.beta, ln, st, v);
#pragma unroll
            for (int e = 0; e < EPC; e += 4)
                *reinterpret_cast<float4 *>(dst + (size_t)c * EPC + e) =
                    make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
        }
    }
    if (part == 0)
        head_select_block(p.s_h, a.B, p.H, p.k_h, wbits, ubits, p.idx_h, p.u_h, p.n_u_h);
}

// ---------------------------------------------------------------------------
// Row addressing.
struct RowRef {
    const void *p;  // first element of the row (nullptr: invalid row)
    int j, t, e, h;
};

DV_DEV int sel_at(const RowArgs &a, int j, const int *ssel, int sj0, int sn)
{
    const int o = j - sj0;
    return (o >= 0 && o < sn) ? ssel[o] : ld_cg(a.sel + j);
}

template <typename T, int KIND>
DV_DEV RowRef row_ref(const RowArgs &a, int row, const int *ssel, int sj0, int sn)
{
    RowRef r;
    r.j = r.t = r.e = r.h = 0;
    const T *w0 = static_cast<const T *>(a.w0);
    if constexpr (KIND == RK_PRED1) {
        r.p = row < a.split_rows ? (const void *)(w0 + (size_t)row * a.K)
                                 : (const void *)(static_cast<const T *>(a.w1) +
                                                  (size_t)(row - a.split_rows) * a.K);
    } else if constexpr (KIND == RK_PRED2) {
        r.p = w0 + (size_t)row * a.K;
    } else if constexpr (KIND == RK_QKV) {
        const int per = 3 * a.dh;
        r.j = row / per;
        const int rem = row - r.j * per;
        r.t = rem / a.dh;
        r.e = rem - r.t * a.dh;
        r.h = sel_at(a, r.j, ssel, sj0, sn);
        r.p = (r.h >= 0 && r.h < a.sel_range)
                  ? (const void *)(w0 + (((size_t)r.t * a.H + r.h) * a.dh + r.e) * a.K)
                  : nullptr;
    } else {
        // FC1 (SwiGLU: rows 2j and 2j + 1 are slot j's gate and up rows)
        r.j = row >> a.swiglu;
        r.t = row & a.swiglu;
        r.h = sel_at(a, r.j, ssel, sj0, sn);
        r.p = (r.h >= 0 && r.h < a.sel_range)
                  ? (const void *)(w0 + ((size_t)(r.h << a.swiglu) + r.t) * a.K)
                  : nullptr;
    }
    return r;
}

template <typename T, int U>
DV_DEV void load_unit(const RowRef &r, bool live, int coff, int ucr, int lig, int LG,
                      uint4 (&v)[U])
{
    constexpr int EPC = Elem<T>::EPC;
    const T *p = static_cast<const T *>(r.p);
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const int c = lig + LG * j;
        v[j] = (live && p && c < ucr) ? ld_stream(p + (size_t)(coff + c) * EPC)
                                      : make_uint4(0u, 0u, 0u, 0u);
    }
}

template <typename T, int NB, int U>
DV_DEV void consume_unit(const uint4 (&v)[U], bool live, int coff, int ucr, int lig, int LG,
                         const float *xs, int K, float (&acc)[NB])
{
    if (!live)
        return;
#pragma unroll
    for (int j = 0; j < U; ++j) {
        const int c = lig + LG * j;
        if (c < ucr)
            fma_chunk<T, NB>(v[j], xs, K, coff + c, acc);
    }
}

template <typename T, int NB, int KIND>
DV_DEV void finalize(const RowArgs &a, int row, const RowRef &m, const float (&acc)[NB], int b0,
                     int *shist)
{
#pragma unroll
    for (int bi = 0; bi < NB; ++bi) {
        const int b = b0 + bi;
        if (b >= a.B)
            break;
        float v = acc[bi];
        if constexpr (KIND == RK_PRED1) {
            if (row < a.split_rows) {
                a.out0[(size_t)b * a.split_rows + row] = v;
                if (a.user_scores)
                    a.user_scores[(size_t)b * a.split_rows + row] = v;
            } else {
                const int r = a.max_rows - a.split_rows;
                a.out1[(size_t)b * r + (row - a.split_rows)] = v;
            }
        } else if constexpr (KIND == RK_PRED2) {
            a.out0[(size_t)b * a.max_rows + row] = v;
            if (a.user_scores)
                a.user_scores[(size_t)b * a.max_rows + row] = v;
            atomicAdd(&shist[bi * kTopkBins + (score_key(v) >> 21)], 1);
        } else if constexpr (KIND == RK_QKV) {
            v += Elem<T>::load(static_cast<const T *>(a.bias),
                               ((size_t)m.t * a.H + m.h) * a.dh + m.e);
            if (m.t == 0) {
                a.out0[((size_t)b * a.max_sel + m.j) * a.dh + m.e] = v * a.q_scale;
            } else {
                T *cache = static_cast<T *>(m.t == 1 ? a.kc : a.vc);
                cache[(((size_t)b * a.H + m.h) * a.kv_cap + a.kv_len) * a.dh + m.e] =
                    Elem<T>::from_float(v);
            }
        } else if (a.swiglu) {  // the gate or up value; FC2 forms silu(gate) * up
            v += Elem<T>::load(static_cast<const T *>(a.bias), (size_t)(m.h << 1) + m.t);
            a.out0[(size_t)b * a.max_rows + row] = v;
        } else {
            v += Elem<T>::load(static_cast<const T *>(a.bias), (size_t)m.h);
            a.out0[(size_t)b * a.max_rows + row] = fmaxf(v, 0.f);
        }
    }
}

// Unit range of warp w: [start(w), start(w + 1)).
DV_DEV int range_start(int units, int W, int w) { return (int)((long long)units * w / W); }
// The warp whose range holds unit u.
DV_DEV int warp_of(int units, int W, int u)
{
    return (int)((((long long)u + 1) * W - 1) / units);
}

// ---------------------------------------------------------------------------

template <typename T, int NB, int KIND, int U, class Dep>
DV_DEV void rowdot_body(const RowArgs &a, int cta, int nct, const Dep &dep)
{
    extern __shared__ __align__(16) float smem[];
    __shared__ float red[34];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile = blockIdx.y, b0 = tile * NB;
    const RowGeo g = a.geo;
    float *xs = smem;
    int *shist = reinterpret_cast<int *>(smem + (size_t)NB * a.K);
    // staged gather indices, after the histogram (PRED2) or the activations
    int *ssel = shist + (KIND == RK_PRED2 ? NB * kTopkBins : 0);

    int ncta = nct;  // CTAs that share the rows
    if constexpr (KIND == RK_PRED2) {
        if (a.side_cta) {
            ncta = nct - 1;
            if (cta == ncta) {  // the last CTA does the side work instead
                dep.wait();
                if (tile == 0) {
                    pred2_side<T>(a, red, 0, 1);
                    __threadfence();
                    __syncthreads();
                    if (threadIdx.x == 0 && a.side_flag)
                        st_release_gpu(a.side_flag, 1);
                }
                return;
            }
        }
    }
    if constexpr (KIND == RK_QKV) {
        if (a.side_cta) {
            ncta = nct - a.side_cta;
            if (cta >= ncta) {
                // the last side_cta CTAs select the neurons instead (rows
                // split among them): they need the whole stage-2 grid
                // (scores and histogram)
                dep.wait();
                if (tile == 0) {
                    __shared__ int nscr[48];
                    neuron_select_cta(a.ns, final_smem(smem, a.ns.N, nscr), cta - ncta,
                                      a.side_cta);
                }
                return;
            }
        }
        if (a.side_flag) {
            // the head union and norm(x) come from the previous kernel's side
            // CTA: start as soon as it has published them (bounded polling,
            // then the grid dependency).  The dependents may launch now: the
            // attention kernel reads only flag-published data before its wait.
            __shared__ int s_ready;
            if (threadIdx.x == 0) {
                int ok = 0;
                for (int it = 0; it < kSideSpin && !ok; ++it) {
                    ok = ld_acquire_gpu(a.side_flag);
                    if (!ok)
                        __nanosleep(128);
                }
                s_ready = ok;
            }
            __syncthreads();
            if (!s_ready) {
                dep.wait();
            } else {
                dep.ready();
                dep.trigger();
            }
        } else {  // the head union was given by the caller
            dep.wait();
        }
    }
    int rows = a.max_rows;
    int sj0 = 0, sn = 0;  // staged gather indices: ssel[i] = sel[sj0 + i], i < sn
    if constexpr (KIND == RK_QKV)
        rows = min(max(ld_cg(a.n_sel), 0), a.max_sel) * 3 * a.dh;
    else if constexpr (KIND == RK_FC1)
        rows = min(max(ld_cg(a.n_sel), 0), a.max_sel) << a.swiglu;
    const bool seg = g.nsu > 0;
    const int units = seg ? rows * g.nsu : (rows + g.rpu - 1) / g.rpu;
    const int Wt = ncta * kWarpsPerBlock;
    const int gw = cta * kWarpsPerBlock + warp;
    // at most one segmented row per warp (the stage-1 predictor: 1096 rows
    // of 24 KB at OPT-175B): whole rows per warp, so no row is shared and
    // no partial sums are combined; otherwise equal shares of the units
    const bool whole = seg && rows <= Wt;
    auto ustart = [&](int w) {
        return whole ? (int)((long long)rows * w / Wt) * g.nsu : range_start(units, Wt, w);
    };
    const int ub = ustart(gw), ue = ustart(gw + 1);
    const int LG = 32 / g.rpu;
    const int grp = lane / LG, lig = lane - grp * LG;

    // gather indices of the rows this CTA touches, staged in shared memory
    const bool stage_sel = (KIND == RK_FC1) || (KIND == RK_QKV);
    if (stage_sel) {
        const int cb = ustart(cta * kWarpsPerBlock);
        const int ce = ustart((cta + 1) * kWarpsPerBlock);
        if (ce > cb) {
            const int r0 = seg ? cb / g.nsu : cb * g.rpu;
            const int r1 = seg ? (ce - 1) / g.nsu : min(rows, ce * g.rpu) - 1;
            const int j0 = (KIND == RK_QKV) ? r0 / (3 * a.dh) : r0 >> a.swiglu;
            const int j1 = (KIND == RK_QKV) ? r1 / (3 * a.dh) : r1 >> a.swiglu;
            sj0 = j0;
            sn = min(j1 - j0 + 1, kSelStage);
        }
    }

    // (row, segment) of the warp's first unit; later units advance incrementally
    int r = 0, sg = 0;
    if (ub < ue) {
        if (seg) {
            r = ub / g.nsu;
            sg = ub - r * g.nsu;
        } else {
            r = ub * g.rpu + grp;
        }
    }
    // first unit's loads go out before the activations are staged
    uint4 cur[U];
    RowRef rcur;
    rcur.p = nullptr;
    rcur.j = rcur.t = rcur.e = rcur.h = 0;
    bool lcur = ub < ue && r < rows;
    if (lcur)
        rcur = row_ref<T, KIND>(a, r, ssel, sj0, stage_sel ? 0 : sn);
    load_unit<T, U>(rcur, lcur, sg * g.ucr, g.ucr, lig, LG, cur);
    if (stage_sel)
        for (int i = threadIdx.x; i < sn; i += blockDim.x)
            ssel[i] = ld_cg(a.sel + sj0 + i);
    if constexpr (KIND == RK_PRED2) {
        for (int i = threadIdx.x; i < NB * kTopkBins; i += blockDim.x)
            shist[i] = 0;
    }
    if constexpr (KIND == RK_PRED1 || KIND == RK_PRED2 || KIND == RK_FC1) {
        // activations come from the previous kernel (PRED1: from whatever ran
        // before the call; only its weight rows are read before this point)
        dep.wait();
        if constexpr (KIND == RK_PRED1) {
            if (a.side_flag && cta == 0 && tile == 0 && threadIdx.x == 0)
                *a.side_flag = 0;
        }
    }
    stage_acts<T, NB>(a, xs, b0, red);
    chain_stamp(dep.stamps, 4);  // activations staged

    if (seg) {
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b)
            acc[b] = 0.f;
        int run_cov = 0;
        const int first_row = r;
        for (int u = ub; u < ue; ++u) {
            const bool more = u + 1 < ue;
            int rn = r, sgn = sg + 1;
            if (sgn == g.nsu) {
                sgn = 0;
                rn = r + 1;
            }
            uint4 nxt[U];
            RowRef rnext = rcur;
            if (more && rn != r)
                rnext = row_ref<T, KIND>(a, rn, ssel, sj0, sn);
            load_unit<T, U>(rnext, more, sgn * g.ucr, g.ucr, lig, LG, nxt);
            consume_unit<T, NB, U>(cur, rcur.p != nullptr, sg * g.ucr, g.ucr, lig, LG, xs, a.K,
                                   acc);
            ++run_cov;
            if (!more || rn != r) {
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    acc[b] = warp_sum(acc[b]);
                if (rcur.p == nullptr && lane == 0)
                    set_status(a.status, DV_ERR_DEVICE_INDEX);
                if (run_cov == g.nsu) {
                    if (lane == 0 && rcur.p)
                        finalize<T, NB, KIND>(a, r, rcur, acc, b0, shist);
                } else {
                    const int slot = (r == first_row) ? 0 : 1;
                    float *pp = a.part + (((size_t)tile * Wt + gw) * 2 + slot) * NB;
                    int *cnt = a.rowcnt + (size_t)tile * a.max_rows + r;
                    int last = 0;
                    if (lane == 0) {
#pragma unroll
                        for (int b = 0; b < NB; ++b)
                            pp[b] = acc[b];
                        __threadfence();
                        last = (atomicAdd(cnt, run_cov) + run_cov == g.nsu);
                    }
                    last = __shfl_sync(0xffffffffu, last, 0);
                    if (last && lane == 0) {
                        __threadfence();
                        float s[NB];
#pragma unroll
                        for (int b = 0; b < NB; ++b)
                            s[b] = 0.f;
                        const int wa = warp_of(units, Wt, r * g.nsu);
                        const int wb = warp_of(units, Wt, r * g.nsu + g.nsu - 1);
                        for (int w = wa; w <= wb; ++w) {
                            const int st = range_start(units, Wt, w);
                            if (st >= range_start(units, Wt, w + 1))
                                continue;
                            const int sl = (st / g.nsu == r) ? 0 : 1;
                            const float *q = a.part + (((size_t)tile * Wt + w) * 2 + sl) * NB;
#pragma unroll
                            for (int b = 0; b < NB; ++b)
                                s[b] += ld_cg(q + b);
                        }
                        if (rcur.p)
                            finalize<T, NB, KIND>(a, r, rcur, s, b0, shist);
                        *cnt = 0;
                    }
                }
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    acc[b] = 0.f;
                run_cov = 0;
            }
#pragma unroll
            for (int j = 0; j < U; ++j)
                cur[j] = nxt[j];
            rcur = rnext;
            r = rn;
            sg = sgn;
        }
    } else {
        for (int u = ub; u < ue; ++u) {
            const bool more = u + 1 < ue;
            const int rn = r + g.rpu;
            uint4 nxt[U];
            RowRef rnext;
            rnext.p = nullptr;
            rnext.j = rnext.t = rnext.e = rnext.h = 0;
            const bool lnext = more && rn < rows;
            if (lnext)
                rnext = row_ref<T, KIND>(a, rn, ssel, sj0, sn);
            load_unit<T, U>(rnext, lnext, 0, g.ucr, lig, LG, nxt);
            float acc[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                acc[b] = 0.f;
            consume_unit<T, NB, U>(cur, lcur && rcur.p != nullptr, 0, g.ucr, lig, LG, xs, a.K,
                                   acc);
#pragma unroll
            for (int b = 0; b < NB; ++b)
                for (int off = LG >> 1; off > 0; off >>= 1)
                    acc[b] += __shfl_xor_sync(0xffffffffu, acc[b], off);
            if (lig == 0 && lcur) {
                if (rcur.p)
                    finalize<T, NB, KIND>(a, r, rcur, acc, b0, shist);
                else
                    set_status(a.status, DV_ERR_DEVICE_INDEX);
            }
#pragma unroll
            for (int j = 0; j < U; ++j)
                cur[j] = nxt[j];
            rcur = rnext;
            lcur = lnext;
            r = rn;
        }
    }
    chain_stamp(dep.stamps, 5);  // rows done
    if constexpr (KIND == RK_PRED2) {  // this CTA's scores into the first-digit histogram
        __syncthreads();
        for (int i = threadIdx.x; i < NB * kTopkBins; i += blockDim.x) {
            const int bi = i / kTopkBins;
            const int v = shist[i];
            if (v && b0 + bi < a.B)
                atomicAdd(&a.hist[(size_t)(b0 + bi) * kTopkBins + (i - bi * kTopkBins)], v);
        }
    }
}

}  // namespace
}  // namespace dv
