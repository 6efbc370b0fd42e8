// dv_attn.cuh -- decode attention over the selected heads' KV cache (sm_103a):
// the body of its stand-alone kernel (dv_attn.cu).
//
// For every batch row b and selected head h ("DejaVu Guide: Contextual
// Sparsity for LLM Inference", "2. Head-Pruned Attention Dispatch": only the
// active heads' KV history is read):
//   o = softmax(q . K[b, h, 0..kv_len]^T) . V[b, h, 0..kv_len]
// with q already scaled by 1/sqrt(dh) and position kv_len just appended.
//
// The kv_len + 1 positions of a (batch row, head) are cut into C chunks, one
// CTA each, and a chunk's positions are split among the CTA's 16 warps.  A
// group of dh*sizeof(T)/16 lanes covers one key row with 16-byte loads, so a
// warp scores 32/group keys per step (two batches of steps in flight),
// reduces each dot product with xor shuffles inside its group and keeps a
// running max / sum / weighted V (online softmax) per group.  Groups merge by
// butterfly shuffles and the warps of the CTA merge in shared memory into one
// chunk record (max m, weight sum l, weighted V, not yet divided); the
// out-projection kernel merges the C records of a head while it stages its
// coefficients.
//
// The head list was published before the previous kernel ran (flag) or
// given by the caller, so the CTAs read it and place their work before the
// grid wait.  q and the appended position come from the QKV kernel: the warp
// whose range holds the appended position loads after the wait, the other
// warps issue their first two batches of older positions before it (hiding
// the first round trip: measured 2 us per OPT-175B decode).
#pragma once

#include "dv_common.cuh"

namespace dv {
namespace {

// K/V rows are streamed through the non-coherent path: the cache's older
// positions are inputs, never written while this kernel runs.  Position
// kv_len was just written by the QKV kernel, which may still have been running
// when this grid started (programmatic dependent launch), and reading it
// through the non-coherent path returned stale data in about 1 of 25
// decodes; the warp whose range holds it reads all its rows at L2 instead.

template <typename T, int LPK, class Dep>
DV_DEV void attn_body(const AttnArgs &a, int cta, int nct, const Dep &dep)
{
    constexpr int EPC = Elem<T>::EPC;
    constexpr int KPW = 32 / LPK;  // keys per warp step
    constexpr int UK = 4;          // warp steps per batch (two batches in flight)
    constexpr int DH = LPK * EPC;  // head dimension
    __shared__ float wm[kWarpsPerBlock], wl[kWarpsPerBlock];
    extern __shared__ __align__(16) float attn_smem[];
    float(*wo)[DH] = reinterpret_cast<float(*)[DH]>(attn_smem);  // [kWarpsPerBlock][DH]
    __shared__ int s_ready;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = lane / LPK, dc = lane % LPK;
    const int C = a.splits;  // chunks per (row, head)
    const int L1 = a.kv_len + 1;
    const T *Kc = static_cast<const T *>(a.kc);
    const T *Vc = static_cast<const T *>(a.vc);
    bool waited = false;
    if (a.side_flag) {
        // the head union is published by the stage-2 predictor's side CTA
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
            waited = true;
        }
    }
    const int ns = min(max(ld_cg(a.n_sel), 0), a.max_sel);
    const int units = a.B * ns * C;

    for (int cu = cta; cu < units; cu += nct) {
        const int per_b = ns * C;
        const int b = cu / per_b, rem = cu - b * per_b;
        const int j = rem / C, c = rem - j * C;
        const int h = ld_cg(a.sel + j);
        if (h < 0 || h >= a.H) {  // uniform over the CTA
            if (threadIdx.x == 0)
                set_status(a.status, DV_ERR_DEVICE_INDEX);
            continue;
        }
        const int c0 = (int)((long long)L1 * c / C), c1 = (int)((long long)L1 * (c + 1) / C);
        const int p0 = c0 + (int)((long long)(c1 - c0) * warp / kWarpsPerBlock);
        const int p1 = c0 + (int)((long long)(c1 - c0) * (warp + 1) / kWarpsPerBlock);
        const size_t base = ((size_t)b * a.H + h) * (size_t)a.kv_cap * DH + (size_t)dc * EPC;
        const int nbatch = (p1 - p0 + KPW * UK - 1) / (KPW * UK);
        // the warp whose range holds position kv_len reads all its rows at L2
        const bool coh = p0 <= a.kv_len && a.kv_len < p1;  // uniform over the warp
        // q and the appended K/V come from the previous kernel: the warp
        // holding position kv_len waits before its loads; the others load
        // their older positions (inputs no kernel writes) first
        if (!waited && coh) {
            dep.wait();
            waited = true;
        }
        auto ldkv = [&](const T *row) { return coh ? ld_stream_coherent(row) : ld_stream(row); };
        uint4 kc[UK], vc[UK], kn[UK], vn[UK];
#pragma unroll
        for (int uu = 0; uu < UK; ++uu) {
            const int p = p0 + uu * KPW + ks;
            kc[uu] = p < p1 ? ldkv(Kc + base + (size_t)p * DH) : make_uint4(0u, 0u, 0u, 0u);
            vc[uu] = p < p1 ? ldkv(Vc + base + (size_t)p * DH) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int uu = 0; uu < UK; ++uu) {
            const int p = p0 + (UK + uu) * KPW + ks;
            kn[uu] = p < p1 ? ldkv(Kc + base + (size_t)p * DH) : make_uint4(0u, 0u, 0u, 0u);
            vn[uu] = p < p1 ? ldkv(Vc + base + (size_t)p * DH) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (!waited) {
            dep.wait();
            waited = true;
        }
        float q[EPC];
        {
            const float *qp = a.q + ((size_t)b * a.max_sel + j) * DH + dc * EPC;
#pragma unroll
            for (int e = 0; e < EPC; e += 4) {
                const float4 t = __ldcg(reinterpret_cast<const float4 *>(qp + e));
                q[e] = t.x;
                q[e + 1] = t.y;
                q[e + 2] = t.z;
                q[e + 3] = t.w;
            }
        }
        float m = -INFINITY, l = 0.f, o[EPC];
#pragma unroll
        for (int e = 0; e < EPC; ++e)
            o[e] = 0.f;

        for (int bt = 0; bt < nbatch; ++bt) {
            if (bt == 1)
                chain_stamp(dep.stamps, 4);  // warp 0's first batch consumed
            const int pb = p0 + bt * KPW * UK;
#pragma unroll
            for (int uu = 0; uu < UK; ++uu) {
                const int p = pb + uu * KPW + ks;
                float kf[EPC];
                Elem<T>::unpack(kc[uu], kf);
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < EPC; ++e)
                    dot = fmaf(q[e], kf[e], dot);
#pragma unroll
                for (int off = LPK / 2; off > 0; off >>= 1)
                    dot += __shfl_xor_sync(0xffffffffu, dot, off);
                if (p < p1) {
                    float vf[EPC];
                    Elem<T>::unpack(vc[uu], vf);
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
            // the next batch moves up; the one after it is loaded (the waited
            // state holds here, so every position may be read)
#pragma unroll
            for (int uu = 0; uu < UK; ++uu) {
                kc[uu] = kn[uu];
                vc[uu] = vn[uu];
                const int p = pb + 2 * KPW * UK + uu * KPW + ks;
                kn[uu] = p < p1 ? ldkv(Kc + base + (size_t)p * DH) : make_uint4(0u, 0u, 0u, 0u);
                vn[uu] = p < p1 ? ldkv(Vc + base + (size_t)p * DH) : make_uint4(0u, 0u, 0u, 0u);
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
        chain_stamp(dep.stamps, 5);  // warp 0's keys done
        if (ks == 0) {
#pragma unroll
            for (int e = 0; e < EPC; ++e)
                wo[warp][dc * EPC + e] = o[e];
        }
        if (lane == 0) {
            wm[warp] = m;
            wl[warp] = l;
        }
        __syncthreads();
        // combine the warps of the CTA (thread t owns dimension t) into the record
        float M = -INFINITY;
        for (int w = 0; w < kWarpsPerBlock; ++w)
            M = fmaxf(M, wm[w]);
        float Ls = 0.f;
        for (int w = 0; w < kWarpsPerBlock; ++w)
            Ls += (wm[w] == -INFINITY) ? 0.f : wl[w] * expf(wm[w] - M);
        const int t = threadIdx.x;
        float Ot = 0.f;
        if (t < DH)
            for (int w = 0; w < kWarpsPerBlock; ++w)
                Ot += (wm[w] == -INFINITY) ? 0.f : wo[w][t] * expf(wm[w] - M);
        const int rec = kAttnRec + DH;
        float *r = a.part + (((size_t)b * a.max_sel + j) * C + c) * rec;
        if (t < DH)
            r[kAttnRec + t] = Ot;
        if (t == 0) {
            r[0] = M;
            r[1] = Ls;
        }
        chain_stamp(dep.stamps, 6);  // record written (thread 0)
        __syncthreads();
    }
    if (!waited) {  // no unit: still order this grid after the previous one
        dep.wait();
    }
}

}  // namespace
}  // namespace dv
