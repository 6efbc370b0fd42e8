// dv_rowdot.cu -- row-dot GEMV kernels of the sparse layer decode (sm_103a).
//
// One kernel template serves every step whose output element is the dot
// product of one weight row with an activation vector:
//   PRED1  head scores s_h = x_pred . pred_h^T and the low-rank factor
//          u = x_pred . pred_a^T ("DejaVu Guide: Contextual Sparsity for LLM
//          Inference", "1. Mathematical Formulation of Lookahead Predictors"),
//          then the top-k of the heads in the last CTA;
//   PRED2  neuron scores s_n = u . pred_b^T, then the top-k of the neurons in
//          the last CTA (the first radix digit's histogram is built on the
//          way by every CTA);
//   QKV    the selected heads' q, k, v rows on LayerNorm(x), bias, q scaling
//          and the KV append ("2. Head-Pruned Attention Dispatch");
//   FC1    the selected neurons' fc1 rows on LayerNorm(h1), bias and ReLU
//          (listing, DejaVuSparseMLP.forward_sparse, steps 1-2).
//
// Work split: each row is cut into `nseg` equal segments; the (row, segment)
// units are dealt round-robin to all warps of a persistent grid.  A warp
// streams its segment with 16-byte non-allocating loads (8 in flight per
// lane) and dots it with the activations staged once per CTA in shared
// memory.  When a row has several segments, each writes its partial and the
// last to arrive (atomic counter) sums them in segment order and runs the
// epilogue, so results do not depend on scheduling.
#include "dv_common.cuh"

namespace dv {
namespace {

// Position of activation element c in the staged layout.  For binary16
// weights a 16-byte chunk holds 8 elements; the staged activations are split
// into the low and high 4 of every chunk so each lane's two float4 reads hit
// consecutive addresses across the warp (no bank conflicts).
template <typename T>
DV_DEV int xs_index(int c, int K);
template <>
DV_DEV int xs_index<float>(int c, int) { return c; }
template <>
DV_DEV int xs_index<__half>(int c, int K)
{
    const int ch = c >> 3, w = c & 7;
    return (w < 4) ? (ch << 2) + w : (K >> 1) + (ch << 2) + (w - 4);
}

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

// Dot of chunks [c0, c0 + nchunk) of one weight row with the staged
// activations; lane-partial sums (reduce across the warp afterwards).
template <typename T, int NB>
DV_DEV void warp_dot(const T *__restrict__ w, int c0, int nchunk, const float *xs, int K,
                     float (&acc)[NB], int lane)
{
    constexpr int EPC = Elem<T>::EPC;
    constexpr int U = 8;
    int c = lane;
    for (; c + 32 * (U - 1) < nchunk; c += 32 * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = ld_stream(w + (size_t)(c0 + c + 32 * u) * EPC);
#pragma unroll
        for (int u = 0; u < U; ++u)
            fma_chunk<T, NB>(v[u], xs, K, c0 + c + 32 * u, acc);
    }
    if (c < nchunk) {  // fewer than U chunks left for this lane: one guarded batch
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            v[u] = (c + 32 * u < nchunk) ? ld_stream(w + (size_t)(c0 + c + 32 * u) * EPC)
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (c + 32 * u < nchunk)
                fma_chunk<T, NB>(v[u], xs, K, c0 + c + 32 * u, acc);
    }
}

// Stage NB activation rows [b0, b0 + NB) into shared memory, normalised when
// the kind asks for it.  Rows past the batch are zero.
template <typename T, int NB>
DV_DEV void stage_acts(const RowArgs &a, float *xs, int b0, float *red)
{
    const int K = a.K, tid = threadIdx.x, nt = blockDim.x;
    for (int bi = 0; bi < NB; ++bi) {
        const int b = b0 + bi;
        float *dst = xs + (size_t)bi * K;
        const bool live = b < a.B;
        const float *src = a.x + (size_t)(live ? b : 0) * a.x_ld;
        float mean = 0.f, inv = 1.f;
        if (live && a.norm_g) {
            if (a.norm_kind == DV_LAYERNORM) {
                float s = 0.f;
                for (int c = tid; c < K; c += nt)
                    s += src[c];
                mean = block_sum(s, red) / (float)K;
                float v = 0.f;
                for (int c = tid; c < K; c += nt) {
                    const float t = src[c] - mean;
                    v = fmaf(t, t, v);
                }
                inv = rsqrtf(block_sum(v, red) / (float)K + a.eps);
            } else {
                float v = 0.f;
                for (int c = tid; c < K; c += nt)
                    v = fmaf(src[c], src[c], v);
                inv = rsqrtf(block_sum(v, red) / (float)K + a.eps);
            }
        }
        for (int c = tid; c < K; c += nt) {
            float v = 0.f;
            if (live) {
                v = src[c];
                if (a.norm_g) {
                    const float g = Elem<T>::load(static_cast<const T *>(a.norm_g), c);
                    const float bb = (a.norm_kind == DV_LAYERNORM)
                                         ? Elem<T>::load(static_cast<const T *>(a.norm_b), c)
                                         : 0.f;
                    v = (v - mean) * inv * g + bb;
                }
            }
            dst[xs_index<T>(c, K)] = v;
        }
    }
    __syncthreads();
}

struct Meta {
    bool ok;
    int t, h, e, j;
};

template <typename T, int KIND>
DV_DEV const T *row_ptr(const RowArgs &a, int row, Meta &m)
{
    m.ok = true;
    m.t = m.h = m.e = m.j = 0;
    const T *w0 = static_cast<const T *>(a.w0);
    if constexpr (KIND == RK_PRED1) {
        if (row < a.split_rows)
            return w0 + (size_t)row * a.K;
        return static_cast<const T *>(a.w1) + (size_t)(row - a.split_rows) * a.K;
    } else if constexpr (KIND == RK_PRED2) {
        return w0 + (size_t)row * a.K;
    } else if constexpr (KIND == RK_QKV) {
        const int per = 3 * a.dh;
        const int j = row / per, rem = row - j * per;
        m.j = j;
        m.t = rem / a.dh;
        m.e = rem - m.t * a.dh;
        const int h = a.sel[j];
        m.h = h;
        if (h < 0 || h >= a.sel_range) {
            m.ok = false;
            return nullptr;
        }
        return w0 + (((size_t)m.t * a.H + h) * a.dh + m.e) * a.K;
    } else {
        const int j = a.sel[row];
        m.h = j;
        if (j < 0 || j >= a.sel_range) {
            m.ok = false;
            return nullptr;
        }
        return w0 + (size_t)j * a.K;
    }
}

template <typename T, int NB, int KIND>
DV_DEV void finalize(const RowArgs &a, int row, const Meta &m, const float (&acc)[NB], int b0,
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
        } else {
            v += Elem<T>::load(static_cast<const T *>(a.bias), (size_t)m.h);
            a.out0[(size_t)b * a.max_sel + row] = fmaxf(v, 0.f);
        }
    }
}

// ---------------------------------------------------------------------------
// Block-wide exact top-k of one row of binary32 scores (all threads of the
// block).  Keys are order-preserving integers (score_key); a three-pass
// radix select (11, 11, 10 bits) finds the k-th largest key T and how many
// keys equal to T are kept; the output pass keeps every key > T and the
// lowest-index keys == T, writing indices in ascending order.
DV_DEV void find_bin(const int *hist, int nb, int krem, int *scr)
{
    const int nt = blockDim.x, tid = threadIdx.x;
    const int per = (nb + nt - 1) / nt;
    const int top = nb - 1 - tid * per;
    int c = 0;
    for (int q = 0; q < per; ++q) {
        const int bin = top - q;
        if (bin >= 0)
            c += hist[bin];
    }
    int tot;
    const int before = block_excl_scan(c, scr + 4, &tot);
    if (before < krem && krem <= before + c) {
        int acc = before;
        for (int q = 0; q < per; ++q) {
            const int bin = top - q;
            if (bin < 0)
                break;
            const int h = hist[bin];
            if (krem <= acc + h) {
                scr[0] = bin;
                scr[1] = krem - acc;
                break;
            }
            acc += h;
        }
    }
    __syncthreads();
}

DV_DEV void block_topk_row(const float *s, int n, int k, int *ghist, int32_t *out,
                           unsigned *bitmap, int *hist, int *scr)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    unsigned prefix = 0u, pmask = 0u;
    int krem = k;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = shifts[pass], nbins = 1 << widths[pass];
        if (pass == 0 && ghist) {
            for (int i = tid; i < nbins; i += nt) {
                hist[i] = ld_cg(ghist + i);
                ghist[i] = 0;  // leave the global histogram zero for the next call
            }
        } else {
            for (int i = tid; i < nbins; i += nt)
                hist[i] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += nt) {
                const unsigned key = score_key(ld_cg(s + i));
                if ((key & pmask) == prefix)
                    atomicAdd(&hist[(key >> shift) & (unsigned)(nbins - 1)], 1);
            }
        }
        __syncthreads();
        find_bin(hist, nbins, krem, scr);
        prefix |= (unsigned)scr[0] << shift;
        pmask |= (unsigned)(nbins - 1) << shift;
        krem = scr[1];
        __syncthreads();
    }
    const unsigned T = prefix;
    const int need_eq = krem;
    const int per = (n + nt - 1) / nt;
    const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
    int gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
        const unsigned key = score_key(ld_cg(s + i));
        gt += key > T;
        eq += key == T;
    }
    int tot;
    const int eq_before = block_excl_scan(eq, scr + 4, &tot);
    const int take_eq = min(max(need_eq - eq_before, 0), eq);
    int pos = block_excl_scan(gt + take_eq, scr + 4, &tot);
    int eq_seen = 0;
    for (int i = i0; i < i1; ++i) {
        const unsigned key = score_key(ld_cg(s + i));
        bool keep = key > T;
        if (key == T) {
            keep = eq_seen < take_eq;
            ++eq_seen;
        }
        if (keep) {
            out[pos++] = i;
            atomicOr(&bitmap[i >> 5], 1u << (i & 31));
        }
    }
    __syncthreads();
}

template <int KIND, int NB>
DV_DEV void topk_tail(const RowArgs &a, float *smem, int *shist, int b0)
{
    __shared__ int s_last;
    __shared__ int scr[48];
    if constexpr (KIND == RK_PRED2) {
        __syncthreads();
        for (int i = threadIdx.x; i < NB * kTopkBins; i += blockDim.x) {
            const int bi = i / kTopkBins;
            const int v = shist[i];
            if (v && b0 + bi < a.B)
                atomicAdd(&a.hist[(size_t)(b0 + bi) * kTopkBins + (i - bi * kTopkBins)], v);
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int total = gridDim.x * gridDim.y;
        s_last = (atomicAdd(a.done, 1) == total - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();
    int *hist = reinterpret_cast<int *>(smem);
    unsigned *bitmap = reinterpret_cast<unsigned *>(hist + kTopkBins);
    const int n = a.topk_n, k = a.topk_k, W = (n + 31) / 32;
    for (int i = threadIdx.x; i < W; i += blockDim.x)
        bitmap[i] = 0u;
    __syncthreads();
    for (int b = 0; b < a.B; ++b)
        block_topk_row(a.out0 + (size_t)b * n, n, k,
                       KIND == RK_PRED2 ? a.hist + (size_t)b * kTopkBins : nullptr,
                       a.idx_out + (size_t)b * k, bitmap, hist, scr);
    // union of the rows, ascending
    const int nt = blockDim.x, tid = threadIdx.x;
    const int per = (W + nt - 1) / nt;
    const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w)
        cnt += __popc(bitmap[w]);
    int tot;
    int pos = block_excl_scan(cnt, scr + 4, &tot);
    for (int w = w0; w < w1; ++w) {
        unsigned bits = bitmap[w];
        while (bits) {
            const int bit = __ffs(bits) - 1;
            a.u_out[pos++] = w * 32 + bit;
            bits &= bits - 1u;
        }
    }
    if (tid == 0) {
        *a.n_u_out = tot;
        *a.done = 0;
    }
}

template <typename T, int NB, int KIND>
__global__ void __launch_bounds__(kThreads, 1) k_rowdot(const RowArgs a)
{
    extern __shared__ __align__(16) float smem[];
    __shared__ float red[34];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int tile = blockIdx.y, b0 = tile * NB;
    float *xs = smem;
    int *shist = reinterpret_cast<int *>(smem + (size_t)NB * a.K);
    if constexpr (KIND == RK_PRED2) {
        for (int i = threadIdx.x; i < NB * kTopkBins; i += blockDim.x)
            shist[i] = 0;
    }
    stage_acts<T, NB>(a, xs, b0, red);

    int rows = a.max_rows;
    if constexpr (KIND == RK_QKV || KIND == RK_FC1) {
        const int ns = min(max(*a.n_sel, 0), a.max_sel);
        rows = (KIND == RK_QKV) ? ns * 3 * a.dh : ns;
    }
    constexpr int EPC = Elem<T>::EPC;
    const int segc = a.seglen / EPC;
    const long long units = (long long)rows * a.nseg;
    const long long nw = (long long)gridDim.x * kWarpsPerBlock;
    for (long long u = (long long)blockIdx.x * kWarpsPerBlock + warp; u < units; u += nw) {
        const int row = (int)(u / a.nseg), seg = (int)(u - (long long)row * a.nseg);
        Meta m;
        const T *wrow = row_ptr<T, KIND>(a, row, m);
        float acc[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b)
            acc[b] = 0.f;
        if (m.ok)
            warp_dot<T, NB>(wrow, seg * segc, segc, xs, a.K, acc, lane);
        else if (lane == 0)
            set_status(a.status, DV_ERR_DEVICE_INDEX);
#pragma unroll
        for (int b = 0; b < NB; ++b)
            acc[b] = warp_sum(acc[b]);
        if (a.nseg == 1) {
            if (m.ok && lane == 0)
                finalize<T, NB, KIND>(a, row, m, acc, b0, shist);
            continue;
        }
        const size_t slot = (size_t)tile * a.max_rows + row;
        float *pp = a.part + (slot * a.nseg + seg) * NB;
        int last = 0;
        if (lane == 0) {
#pragma unroll
            for (int b = 0; b < NB; ++b)
                pp[b] = acc[b];
            __threadfence();
            last = (atomicAdd(&a.rowcnt[slot], 1) == a.nseg - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last && lane == 0) {
            __threadfence();
            float s[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                s[b] = 0.f;
            const float *base = a.part + slot * a.nseg * NB;
            for (int sg = 0; sg < a.nseg; ++sg)
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    s[b] += ld_cg(base + sg * NB + b);
            if (m.ok)
                finalize<T, NB, KIND>(a, row, m, s, b0, shist);
            a.rowcnt[slot] = 0;
        }
    }
    if constexpr (KIND == RK_PRED1 || KIND == RK_PRED2)
        topk_tail<KIND, NB>(a, smem, shist, b0);
}

template <typename T, int NB, int KIND>
cudaError_t launch_one(const RowArgs &a, dim3 grid, size_t smem, cudaStream_t st, bool pdl)
{
    auto kern = k_rowdot<T, NB, KIND>;
    // Opt in to the shared-memory budget once per device (not per launch, so
    // later launches may be captured into a CUDA graph).
    static bool configured[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSmemCap);
        if (e != cudaSuccess)
            return e;
        configured[dev] = true;
    }
    if (smem > kSmemCap)
        return cudaErrorInvalidValue;
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
cudaError_t dispatch_nb(int nb, const RowArgs &a, dim3 grid, size_t smem, cudaStream_t st,
                        bool pdl)
{
    switch (nb) {
    case 1: return launch_one<T, 1, KIND>(a, grid, smem, st, pdl);
    case 2: return launch_one<T, 2, KIND>(a, grid, smem, st, pdl);
    case 4: return launch_one<T, 4, KIND>(a, grid, smem, st, pdl);
    case 8: return launch_one<T, 8, KIND>(a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
    }
}

template <typename T>
cudaError_t dispatch_kind(int kind, int nb, const RowArgs &a, dim3 grid, size_t smem,
                          cudaStream_t st, bool pdl)
{
    switch (kind) {
    case RK_PRED1: return dispatch_nb<T, RK_PRED1>(nb, a, grid, smem, st, pdl);
    case RK_PRED2: return dispatch_nb<T, RK_PRED2>(nb, a, grid, smem, st, pdl);
    case RK_QKV: return dispatch_nb<T, RK_QKV>(nb, a, grid, smem, st, pdl);
    case RK_FC1: return dispatch_nb<T, RK_FC1>(nb, a, grid, smem, st, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int rowdot_nb(int B, int K, int kind)
{
    int nb = 1;
    while (nb < B && nb < 8)
        nb <<= 1;
    const size_t extra = (kind == RK_PRED2) ? (size_t)kTopkBins * 4 : 0;
    while (nb > 1 && (size_t)nb * ((size_t)K * 4 + extra) > kSmemCap)
        nb >>= 1;
    return nb;
}

size_t rowdot_smem(int kind, int nb, int K, int topk_n)
{
    size_t main = (size_t)nb * K * 4 + (kind == RK_PRED2 ? (size_t)nb * kTopkBins * 4 : 0);
    size_t tail = 0;
    if (kind == RK_PRED1 || kind == RK_PRED2)
        tail = ((size_t)kTopkBins + (size_t)(topk_n + 31) / 32) * 4;
    return main > tail ? main : tail;
}

cudaError_t launch_rowdot(int kind, int dtype, int nb, const RowArgs &a, dim3 grid, size_t smem,
                          cudaStream_t st, bool pdl)
{
    if (dtype == DV_F16)
        return dispatch_kind<__half>(kind, nb, a, grid, smem, st, pdl);
    return dispatch_kind<float>(kind, nb, a, grid, smem, st, pdl);
}

}  // namespace dv
