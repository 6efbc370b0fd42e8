// dv_colacc.cuh -- column-gather GEMV of the sparse layer decode (sm_103a): the
// body of its stand-alone kernels (dv_colacc.cu).
//
//   OPROJ  h1[b] = x[b] + b_o + sum over selected heads h and e < dh of
//          o[b][h][e] * w_oT[h][e][:]       ("DejaVu Guide: Contextual Sparsity
//          for LLM Inference", "2. Head-Pruned Attention Dispatch": inactive
//          heads' output-projection weights are never read);
//   FC2    y[b] = h1[b] + b2 + sum over selected neurons j of a[b][j] * w2T[j][:]
//          (the guide's listing, DejaVuSparseMLP.forward_sparse, steps 3-4: the
//          selected fc2 columns, kept transposed so each is one contiguous row).
//
// Work: the output columns are cut into blocks of CB columns (CB = 32 lanes
// x P chunks of 16 bytes: 1 KB of a binary16 row at P = 2, 512 bytes at
// P = 1; narrow blocks keep the number of CTAs sharing a block, and so the
// final cross-CTA sum, small).  The (block, row) pieces are dealt to the
// CTAs of a persistent grid in contiguous, balanced ranges, block-major.
// Inside a CTA the warps take the rows of a block round-robin, two batches of
// rows in flight per warp, each lane accumulating P strided 16-byte chunks
// (every load instruction reads 512 contiguous bytes, and a warp reads a
// whole piece of a row at once); the 16 warps then reduce in shared memory.  A block covered entirely by one CTA is finished there;
// a block shared by several CTAs is finished by the last of them to arrive
// (atomic count of rows), which sums their partials in CTA order -- results
// do not depend on scheduling.
#pragma once

#include "dv_common.cuh"

namespace dv {
namespace {

constexpr int kStageRows = kColStageRows;  // rows whose offsets and coefficients are staged at once
constexpr int kMaxCover = kColMaxCover;     // CTAs that may share one column block
constexpr int kCoverBatch = 8;   // partials loaded together by the combining CTA
constexpr int kRecBatch = 8;     // attention chunk records loaded together

template <int KIND>
DV_DEV long long row_offset(const ColArgs &a, int i)
{
    const int j = (KIND == CK_OPROJ) ? i / a.dh : i;
    const int h = ld_cg(a.sel + j);
    if (h < 0 || h >= a.sel_range)
        return -1;
    if constexpr (KIND == CK_OPROJ)
        return ((long long)h * a.dh + (i - j * a.dh)) * a.d;
    else
        return (long long)h * a.d;
}

// Coefficient of row i for batch row b.  FC2: the fc1 activation.  OPROJ:
// attention output o[b][j][e] (i = j*dh + e), merged from the attention
// kernel's C chunk records (m, l, weighted V) of head slot j:
//   o = sum_c exp(m_c - M) V_c[e] / sum_c exp(m_c - M) l_c,  M = max_c m_c.
template <int KIND>
DV_DEV float coef_at(const ColArgs &a, int b, int i)
{
    if constexpr (KIND == CK_OPROJ) {
        // the records were written by the previous kernel (read at L2); loads
        // in batches of kRecBatch chunks
        const int j = i / a.dh, e = i - j * a.dh;
        const int C = a.attn_C, rec = kAttnRec + a.dh;
        const float *r = a.attn_rec + ((size_t)b * a.max_sel + j) * C * rec;
        if (C <= kRecBatch) {  // all records in one batch of loads
            float m[kRecBatch], l[kRecBatch], o[kRecBatch];
#pragma unroll
            for (int u = 0; u < kRecBatch; ++u) {
                const float *rc = r + (size_t)u * rec;
                const bool in = u < C;
                m[u] = in ? __ldcg(rc) : -INFINITY;
                l[u] = in ? __ldcg(rc + 1) : 0.f;
                o[u] = in ? __ldcg(rc + kAttnRec + e) : 0.f;
            }
            float MM = m[0];
#pragma unroll
            for (int u = 1; u < kRecBatch; ++u)
                MM = fmaxf(MM, m[u]);
            float LL = 0.f, OO = 0.f;
#pragma unroll
            for (int u = 0; u < kRecBatch; ++u) {
                if (u >= C)
                    break;
                const float w = expf(m[u] - MM);
                LL = fmaf(l[u], w, LL);
                OO = fmaf(o[u], w, OO);
            }
            return OO / LL;
        }
        float MM = -INFINITY;
        for (int c0 = 0; c0 < C; c0 += kRecBatch) {
            float m[kRecBatch];
#pragma unroll
            for (int u = 0; u < kRecBatch; ++u)
                m[u] = c0 + u < C ? __ldcg(r + (size_t)(c0 + u) * rec) : -INFINITY;
#pragma unroll
            for (int u = 0; u < kRecBatch; ++u)
                MM = fmaxf(MM, m[u]);
        }
        float LL = 0.f, OO = 0.f;
        for (int c0 = 0; c0 < C; c0 += kRecBatch) {
            float m[kRecBatch], l[kRecBatch], o[kRecBatch];
#pragma unroll
            for (int u = 0; u < kRecBatch; ++u) {
                const float *rc = r + (size_t)(c0 + u) * rec;
                const bool in = c0 + u < C;
                m[u] = in ? __ldcg(rc) : 0.f;
                l[u] = in ? __ldcg(rc + 1) : 0.f;
                o[u] = in ? __ldcg(rc + kAttnRec + e) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < kRecBatch; ++u) {
                if (c0 + u >= C)
                    break;
                const float w = expf(m[u] - MM);
                LL = fmaf(l[u], w, LL);
                OO = fmaf(o[u], w, OO);
            }
        }
        return OO / LL;
    } else if (a.swiglu) {  // silu(gate) * up of slot i
        const float g = __ldcg(a.coef + (size_t)b * a.coef_ld + 2 * i);
        const float u = __ldcg(a.coef + (size_t)b * a.coef_ld + 2 * i + 1);
        return g / (1.f + expf(-g)) * u;
    } else {
        return __ldcg(a.coef + (size_t)b * a.coef_ld + i);
    }
}

// Work split.  Pieces are (column block, row); CTA c takes pieces [p0, p1).
// With no more column blocks than CTAs, block cb is shared by CTAs
// [first_cta(cb), first_cta(cb + 1)), which split its rows evenly, so no
// CTA straddles two blocks; otherwise every CTA takes whole blocks.
DV_DEV int first_cta(int cb, int nc, int ncb)
{
    return (int)(((long long)cb * nc + ncb - 1) / ncb);
}
DV_DEV void cta_pieces(int c, int nc, int ncb, int rows, long long *p0, long long *p1)
{
    if (ncb <= nc) {
        const int cb = (int)((long long)c * ncb / nc);
        const int f = first_cta(cb, nc, ncb), m = first_cta(cb + 1, nc, ncb) - f;
        const int r = c - f;
        *p0 = (long long)cb * rows + (long long)rows * r / m;
        *p1 = (long long)cb * rows + (long long)rows * (r + 1) / m;
    } else {
        *p0 = (long long)((long long)c * ncb / nc) * rows;
        *p1 = (long long)((long long)(c + 1) * ncb / nc) * rows;
    }
}

template <typename T, int NB, int P>
DV_DEV void write_out(const ColArgs &a, int b0, int col, const float (&v)[NB])
{
    if (col >= a.d)
        return;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        if (b0 + b >= a.B)
            break;
        a.out[(size_t)(b0 + b) * a.d + col] =
            (__ldcg(a.res + (size_t)(b0 + b) * a.d + col) +
             Elem<T>::load(static_cast<const T *>(a.bias), (size_t)col)) +
            v[b];
    }
}

template <typename T, int NB, int KIND, int P, class Dep>
DV_DEV void colacc_body(const ColArgs &a, int cta, int nct, const Dep &dep)
{
    constexpr int EPC = Elem<T>::EPC;
    // rows per batch: 8 loads in flight per lane (4 rows at NB >= 8, whose
    // accumulators take the registers)
    constexpr int R = NB >= 8 ? 4 : 8 / P;
    constexpr int CB = 32 * P * EPC;    // columns per block
    constexpr int CPT = (CB + kThreads - 1) / kThreads;  // block columns per thread
    // dynamic shared memory (colacc_smem_bytes): the warps' block partials,
    // then the stage's row offsets and coefficients and the partial slots of
    // the CTAs sharing a block
    extern __shared__ __align__(16) float red[];  // [kWarpsPerBlock][CB]
    long long *soff = reinterpret_cast<long long *>(red + kWarpsPerBlock * CB);  // [kStageRows]
    float *scoef = reinterpret_cast<float *>(soff + kStageRows);  // [kStageRows][NB]
    int *s_cover = reinterpret_cast<int *>(scoef + kStageRows * NB);  // [kMaxCover]
    __shared__ int s_last, s_ncover;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int tile = blockIdx.y, b0 = tile * NB;
    const int ns = min(max(ld_cg(a.n_sel), 0), a.max_sel);
    const int rows = (KIND == CK_OPROJ) ? ns * a.dh : ns;
    const int ncb = (a.d + CB - 1) / CB;
    const int nc = nct;
    const long long total = (long long)ncb * rows;
    const T *W = static_cast<const T *>(a.w);

    if (total == 0) {  // nothing selected: out = res + bias
        dep.wait();
        for (int col = cta * blockDim.x + tid; col < a.d; col += nc * blockDim.x) {
            float z[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                z[b] = 0.f;
            write_out<T, NB, P>(a, b0, col, z);
        }
        return;
    }

    long long p0, p1;
    cta_pieces(cta, nc, ncb, rows, &p0, &p1);
    const int first_cb = (int)(p0 / rows);
    const int last_cb = p1 > p0 ? (int)((p1 - 1) / rows) : first_cb;
    // residual + bias of the columns of this CTA's first and last column
    // blocks (the ones it may have to finish), read before the grid wait:
    // both are inputs or come from kernels at least two launches back
    float rb0[CPT][NB], rb1[CPT][NB];
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
        const int bc = tid + k * kThreads;
        const int c0 = first_cb * CB + bc, c1 = last_cb * CB + bc;
        const bool in0 = p1 > p0 && bc < CB && c0 < a.d;
        const bool in1 = p1 > p0 && bc < CB && c1 < a.d;
        const float bias0 = in0 ? Elem<T>::load(static_cast<const T *>(a.bias), (size_t)c0) : 0.f;
        const float bias1 = in1 ? Elem<T>::load(static_cast<const T *>(a.bias), (size_t)c1) : 0.f;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const bool bin = b0 + b < a.B;
            rb0[k][b] = (in0 && bin) ? __ldcg(a.res + (size_t)(b0 + b) * a.d + c0) + bias0 : 0.f;
            rb1[k][b] = (in1 && bin) ? __ldcg(a.res + (size_t)(b0 + b) * a.d + c1) + bias1 : 0.f;
        }
    }
    bool waited = false;  // griddepcontrol.wait done (uniform over the CTA)
    for (long long pp = p0; pp < p1;) {
        const int cb = (int)(pp / rows);
        const int i0 = (int)(pp - (long long)cb * rows);
        const int i1 = (int)min((long long)rows, i0 + (p1 - pp));
        pp += i1 - i0;
        float acc[NB][P * EPC];
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int e = 0; e < P * EPC; ++e)
                acc[b][e] = 0.f;

        for (int s0 = i0; s0 < i1; s0 += kStageRows) {
            const int s1 = min(i1, s0 + kStageRows);
            __syncthreads();  // the previous stage is consumed
            for (int i = s0 + tid; i < s1; i += blockDim.x) {
                const long long off = row_offset<KIND>(a, i);
                soff[i - s0] = off;
                if (off < 0)
                    set_status(a.status, DV_ERR_DEVICE_INDEX);
            }
            if (!waited) {
                // the gather indices come from kernels at least two launches
                // back; the coefficients from the previous one
                dep.wait();
                waited = true;
            }
            // FU rows per thread at once, so that their loads overlap
            constexpr int FU = NB <= 2 ? 2 : 1;
            for (int i = s0 + tid; i < s1; i += FU * blockDim.x) {
                float cv[FU][NB];
#pragma unroll
                for (int f = 0; f < FU; ++f)
#pragma unroll
                    for (int b = 0; b < NB; ++b) {
                        const int ii = i + f * (int)blockDim.x;
                        cv[f][b] = (b0 + b < a.B && ii < s1) ? coef_at<KIND>(a, b0 + b, ii) : 0.f;
                    }
#pragma unroll
                for (int f = 0; f < FU; ++f)
                    if (i + f * (int)blockDim.x < s1)
#pragma unroll
                        for (int b = 0; b < NB; ++b)
                            scoef[(i + f * blockDim.x - s0) * NB + b] = cv[f][b];
            }
            __syncthreads();
            if (pp - (i1 - i0) == p0 && s0 == i0)
                chain_stamp(dep.stamps, 4);  // the first stage's coefficients staged
            // warp w takes rows s0 + w + 16 t; R rows per batch, two batches in flight
            const int cnt = (s1 - s0 - warp + kWarpsPerBlock - 1) / kWarpsPerBlock;
            const int nbatch = cnt > 0 ? (cnt + R - 1) / R : 0;
            auto load = [&](int q, uint4 (&v)[R][P]) {
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int t = q * R + r;
                    const int li = warp + kWarpsPerBlock * t;  // row index within the stage
                    const long long off = (t < cnt) ? soff[li] : -1;
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        const int col = cb * CB + (lane + 32 * p) * EPC;
                        v[r][p] = (off >= 0 && col < a.d) ? ld_stream(W + off + col)
                                                          : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            };
            uint4 vc[R][P];
            load(0, vc);
            for (int q = 0; q < nbatch; ++q) {
                uint4 vn[R][P];
                load(q + 1 < nbatch ? q + 1 : nbatch, vn);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    // the row's coefficients, read at use (a broadcast over the warp)
                    const int t = q * R + r;
                    const bool live = t < cnt;
                    const float *cf = scoef + (warp + kWarpsPerBlock * (live ? t : 0)) * NB;
#pragma unroll
                    for (int p = 0; p < P; ++p) {
                        float f[EPC];
                        Elem<T>::unpack(vc[r][p], f);
#pragma unroll
                        for (int b = 0; b < NB; ++b) {
                            const float c = live ? cf[b] : 0.f;
#pragma unroll
                            for (int e = 0; e < EPC; ++e)
                                acc[b][p * EPC + e] = fmaf(c, f[e], acc[b][p * EPC + e]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < R; ++r)
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        vc[r][p] = vn[r][p];
            }
        }

        chain_stamp(dep.stamps, 5);  // this piece's rows consumed
        // reduce the warps in shared memory, one batch row at a time
        const bool whole = (i0 == 0 && i1 == rows);
        const int slot = (cb == first_cb) ? 0 : 1;
        float sum[CPT][NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            __syncthreads();
#pragma unroll
            for (int p = 0; p < P; ++p)
#pragma unroll
                for (int e = 0; e < EPC; e += 4)
                    *reinterpret_cast<float4 *>(red + warp * CB + (lane + 32 * p) * EPC + e) =
                        make_float4(acc[b][p * EPC + e], acc[b][p * EPC + e + 1],
                                    acc[b][p * EPC + e + 2], acc[b][p * EPC + e + 3]);
            __syncthreads();
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int col = tid + k * kThreads;
                float s = 0.f;
                if (col < CB)
                    for (int w = 0; w < kWarpsPerBlock; ++w)
                        s += red[w * CB + col];
                sum[k][b] = s;
            }
        }
        if (whole) {
#pragma unroll
            for (int k = 0; k < CPT; ++k) {
                const int col = tid + k * kThreads;
                if (col < CB)
                    write_out<T, NB, P>(a, b0, cb * CB + col, sum[k]);
            }
            continue;
        }
        // publish this CTA's partial of block cb; the last CTA to finish the block sums them
        float *pp_out = a.part + (((size_t)tile * nc + cta) * 2 + slot) * NB * CB;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int col = tid + k * kThreads;
            if (col < CB)
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    pp_out[b * CB + col] = sum[k][b];
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            int *cntp = a.cnt + (size_t)tile * ncb + cb;
            s_last = (atomicAdd(cntp, i1 - i0) + (i1 - i0) == rows);
        }
        __syncthreads();
        if (!s_last)
            continue;
        chain_stamp(dep.stamps, 6);  // finishing block cb
        __threadfence();
        // the CTAs sharing block cb (each used its slot 0), in CTA order
        if (tid < 32) {
            const int ca = first_cta(cb, nc, ncb), cz = first_cta(cb + 1, nc, ncb) - 1;
            for (int c = ca + tid; c <= cz; c += 32) {
                long long q0, q1;
                cta_pieces(c, nc, ncb, rows, &q0, &q1);
                if (c - ca < kMaxCover)
                    s_cover[c - ca] = q1 > q0 ? c * 2 : -1;
            }
            if (tid == 0)
                s_ncover = min(cz - ca + 1, kMaxCover);
        }
        __syncthreads();
        const int ncover = s_ncover;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int col = tid + k * kThreads;
            if (col >= CB)
                continue;
            float s[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                s[b] = 0.f;
            // kCoverBatch partials loaded at once, then added in CTA order
            for (int c0 = 0; c0 < ncover; c0 += kCoverBatch) {
                float v[kCoverBatch][NB];
                unsigned live = 0u;
#pragma unroll
                for (int u = 0; u < kCoverBatch; ++u) {
                    const int slot = (c0 + u < ncover) ? s_cover[c0 + u] : -1;
                    const float *q =
                        a.part + ((size_t)tile * nc * 2 + (slot < 0 ? 0 : slot)) * NB * CB;
                    live |= (slot >= 0 ? 1u : 0u) << u;
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        v[u][b] = slot >= 0 ? __ldcg(q + b * CB + col) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < kCoverBatch; ++u)
                    if ((live >> u) & 1u)
#pragma unroll
                        for (int b = 0; b < NB; ++b)
                            s[b] += v[u][b];
            }
            const int oc = cb * CB + col;
            if (oc < a.d) {
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    if (b0 + b < a.B)
                        a.out[(size_t)(b0 + b) * a.d + oc] =
                            (cb == first_cb ? rb0[k][b] : rb1[k][b]) + s[b];
            }
        }
        if (tid == 0)
            a.cnt[(size_t)tile * ncb + cb] = 0;
    }
}

}  // namespace
}  // namespace dv
