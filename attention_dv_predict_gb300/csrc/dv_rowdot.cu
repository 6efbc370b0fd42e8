// dv_rowdot.cu -- stand-alone row-dot kernels of the sparse layer decode
// (sm_103a): the CUDA-core body of dv_rowdot.cuh as one kernel per step, the
// tensor-core variant for batch tiles of 8, and their launchers.
#include "dv_rowdot.cuh"

namespace dv {
namespace {

template <typename T, int NB, int KIND, int U>
__global__ void __launch_bounds__(kThreads, 1) k_rowdot(const RowArgs a)
{
    unsigned long long *s = chain_stamps(a.stamps);
    rowdot_body<T, NB, KIND, U>(a, blockIdx.x, gridDim.x, PdlDep{s});
    chain_stamp_end(s);
}

// ---------------------------------------------------------------------------
// Tensor-core variant for batch tiles of 8 rows (binary16 weights; every kind).
//
// out[b][row] = sum_k W[row][k] x[b][k] as mma.sync m16n8k16 (f32 accumulate):
// A = 16 weight rows x 16 k, B = 16 k x 8 batch rows.  A lane loads 16
// contiguous bytes (8 k) of row g and of row g + 8 (g = lane / 4, t = lane % 4,
// k = 8t .. 8t + 7 of a 32-k block); the first 4 k feed one mma, the last 4
// the next, so the fragments' k order is a fixed permutation of the block
// that A and B share (the sum over k does not depend on it).  Activations
// are split into binary16 hi = rn(x) and lo = rn(x - hi), each multiplied
// separately, so the products keep binary32 accuracy.  K is cut into S
// segments so one segment's hi/lo activations fit in shared memory; the
// CTAs of segment s split the 16-row groups, and a group's S partial sums
// are added in segment order by the last warp to finish it.  K need only be
// a multiple of 8 (whole 16-byte chunks): the last 32-k block is padded with
// zero weights and zero activations.

constexpr int kMmaBK = 4;  // 32-k blocks per load batch (two batches in flight)

DV_DEV void mma16816(float (&d)[4], unsigned a0, unsigned a1, unsigned a2, unsigned a3,
                     unsigned b0, unsigned b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One output of row `row` (metadata m) for batch row b.
template <typename T, int KIND>
DV_DEV void finalize_one(const RowArgs &a, int row, const RowRef &m, int b, float v)
{
    if constexpr (KIND == RK_PRED1) {
        if (row < a.split_rows) {
            a.out0[(size_t)b * a.split_rows + row] = v;
            if (a.user_scores)
                a.user_scores[(size_t)b * a.split_rows + row] = v;
        } else {
            a.out1[(size_t)b * (a.max_rows - a.split_rows) + (row - a.split_rows)] = v;
        }
    } else if constexpr (KIND == RK_PRED2) {  // the histogram is added by the caller
        a.out0[(size_t)b * a.max_rows + row] = v;
        if (a.user_scores)
            a.user_scores[(size_t)b * a.max_rows + row] = v;
    } else if constexpr (KIND == RK_QKV) {
        v += Elem<T>::load(static_cast<const T *>(a.bias), ((size_t)m.t * a.H + m.h) * a.dh + m.e);
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

template <int KIND, int NT>
__global__ void __launch_bounds__(kThreads, 1) k_rowdot_mma(const RowArgs a)
{
    using T = __half;
    unsigned long long *stamps = chain_stamps(a.stamps);
    extern __shared__ __align__(16) float smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // NT batch tiles of 8 rows per weight pass: every weight fragment feeds
    // the MMAs of all of them
    const int tile = blockIdx.y, b0 = tile * 8 * NT;
    int ncta = gridDim.x;
    if constexpr (KIND == RK_PRED2) {
        if (a.side_cta) {
            // the last side_cta CTAs: the head selection and norm(x), rows
            // split among them; the last to finish publishes the flag
            ncta = gridDim.x - a.side_cta;
            if ((int)blockIdx.x >= ncta) {
                pdl_wait();
                chain_stamp(stamps, 1);
                pdl_launch_dependents();
                if (tile == 0) {
                    __shared__ float sred[34];
                    pred2_side<T>(a, sred, blockIdx.x - ncta, a.side_cta);
                    __threadfence();
                    __syncthreads();
                    if (threadIdx.x == 0) {
                        const bool last = a.side_cta == 1 ||
                                          atomicAdd(a.side_done, 1) == a.side_cta - 1;
                        if (last) {
                            __threadfence();
                            if (a.side_cta > 1)
                                *a.side_done = 0;
                            if (a.side_flag)
                                st_release_gpu(a.side_flag, 1);
                        }
                    }
                    chain_stamp(stamps, 6);  // side work done
                }
                chain_stamp_end(stamps);
                return;
            }
        }
    }
    if constexpr (KIND == RK_QKV) {
        if (a.side_cta) {
            ncta = gridDim.x - a.side_cta;
            if ((int)blockIdx.x >= ncta) {  // the neuron selection (as in k_rowdot)
                pdl_wait();
                chain_stamp(stamps, 1);
                pdl_launch_dependents();
                if (tile == 0) {
                    __shared__ int nscr[48];
                    neuron_select_cta(a.ns, final_smem(smem, a.ns.N, nscr), blockIdx.x - ncta,
                                      a.side_cta);
                    chain_stamp(stamps, 6);  // selection done
                }
                chain_stamp_end(stamps);
                return;
            }
        }
        if (a.side_flag) {
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
            if (!s_ready)
                pdl_wait();
            chain_stamp(stamps, 1);
            pdl_launch_dependents();
        } else {
            pdl_wait();
            chain_stamp(stamps, 1);
            pdl_launch_dependents();
        }
    }
    const int K = a.K;
    int rows;
    if constexpr (KIND == RK_QKV)
        rows = min(max(ld_cg(a.n_sel), 0), a.max_sel) * 3 * a.dh;
    else if constexpr (KIND == RK_FC1)
        rows = min(max(ld_cg(a.n_sel), 0), a.max_sel);
    else
        rows = a.max_rows;
    const int ngroups = (rows + 15) >> 4;
    const int S = a.mma_seg;
    // segment of this CTA, its CTAs, and this CTA's share of the row groups
    const int sgm = (int)((long long)blockIdx.x * S / ncta);
    const int cf = (int)(((long long)sgm * ncta + S - 1) / S);
    const int cl = (int)(((long long)(sgm + 1) * ncta + S - 1) / S);
    const int r = blockIdx.x - cf, m = cl - cf;
    const int g0 = (int)((long long)ngroups * r / m), g1 = (int)((long long)ngroups * (r + 1) / m);
    const int wg0 = g0 + (int)((long long)(g1 - g0) * warp / kWarpsPerBlock);
    const int wg1 = g0 + (int)((long long)(g1 - g0) * (warp + 1) / kWarpsPerBlock);
    const int k0 = sgm * a.mma_ks;
    const int kn = min(a.mma_ks, K - k0);  // multiple of 8
    const int nblk = (kn + 31) >> 5;       // 32-k blocks, the last one zero-padded
    const int ldx = rowdot_mma_ldx(a.mma_ks);  // staged row stride in halves

    if constexpr (KIND != RK_QKV) {  // the activations come from the previous kernel
        pdl_wait();
        chain_stamp(stamps, 1);
        pdl_launch_dependents();
        if constexpr (KIND == RK_PRED1) {
            if (a.side_flag && blockIdx.x == 0 && tile == 0 && threadIdx.x == 0)
                *a.side_flag = 0;
        }
    }
    // this segment's activations of batch rows b0 .. b0 + 8 NT - 1: hi and lo
    // halves.  The rows' statistics first (a warp per row, over the whole
    // row), then every thread normalises and splits chunks of any row.
    __half *xh = reinterpret_cast<__half *>(smem);
    __half *xl = xh + 8 * NT * ldx;
    {
        __shared__ float2 sstat[8 * NT];
        const bool ln = a.norm_kind == DV_LAYERNORM;
        if (a.norm_g) {
            for (int bi = warp; bi < 8 * NT; bi += kWarpsPerBlock) {
                const int b = b0 + bi;
                if (b < a.B) {
                    const float2 st = warp_row_stats(a.x + (size_t)b * a.x_ld, K, ln, a.eps, lane);
                    if (lane == 0)
                        sstat[bi] = st;
                }
            }
            __syncthreads();
        }
        const int cps = nblk * 4;  // 8-element chunks of the segment per row
        for (int i = threadIdx.x; i < 8 * NT * cps; i += blockDim.x) {
            const int bi = i / cps, c = i - bi * cps, b = b0 + bi;
            float v[8];
            if (b < a.B && 8 * c < kn) {
                norm_chunk<T>(a.x + (size_t)b * a.x_ld, (k0 >> 3) + c, a.norm_g, a.norm_b, ln,
                              a.norm_g ? sstat[bi] : make_float2(0.f, 1.f), v);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = 0.f;
            }
            __align__(16) __half hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                hi[e] = __float2half_rn(v[e]);
                lo[e] = __float2half_rn(v[e] - __half2float(hi[e]));
            }
            *reinterpret_cast<uint4 *>(xh + bi * ldx + 8 * c) = *reinterpret_cast<const uint4 *>(hi);
            *reinterpret_cast<uint4 *>(xl + bi * ldx + 8 * c) = *reinterpret_cast<const uint4 *>(lo);
        }
    }
    __syncthreads();
    chain_stamp(stamps, 4);  // activations staged

    const int g = lane >> 2, t = lane & 3;
    const int nlive = (kn - 8 * t + 31) >> 5;  // blocks whose chunk t is inside the segment
    const __half *xhr = xh + g * ldx + 8 * t, *xlr = xl + g * ldx + 8 * t;
    for (int grp = wg0; grp < wg1; ++grp) {
        const int ra = grp * 16 + g, rb = ra + 8;
        RowRef ma, mb;
        ma.p = mb.p = nullptr;
        ma.j = ma.t = ma.e = ma.h = mb.j = mb.t = mb.e = mb.h = 0;
        if (ra < rows)
            ma = row_ref<T, KIND>(a, ra, nullptr, 0, 0);
        if (rb < rows)
            mb = row_ref<T, KIND>(a, rb, nullptr, 0, 0);
        if ((ra < rows && !ma.p) || (rb < rows && !mb.p))
            set_status(a.status, DV_ERR_DEVICE_INDEX);
        const T *pa = ma.p ? static_cast<const T *>(ma.p) + k0 + 8 * t : nullptr;
        const T *pb = mb.p ? static_cast<const T *>(mb.p) + k0 + 8 * t : nullptr;
        float acc[NT][4];
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
            acc[tt][0] = acc[tt][1] = acc[tt][2] = acc[tt][3] = 0.f;
        uint4 wa[kMmaBK], wb[kMmaBK];
#pragma unroll
        for (int i = 0; i < kMmaBK; ++i) {
            wa[i] = (i < nlive && pa) ? ld_stream(pa + i * 32) : make_uint4(0u, 0u, 0u, 0u);
            wb[i] = (i < nlive && pb) ? ld_stream(pb + i * 32) : make_uint4(0u, 0u, 0u, 0u);
        }
        for (int blk0 = 0; blk0 < nblk; blk0 += kMmaBK) {
            uint4 na[kMmaBK], nb[kMmaBK];
#pragma unroll
            for (int i = 0; i < kMmaBK; ++i) {
                const int blk = blk0 + kMmaBK + i;
                na[i] = (blk < nlive && pa) ? ld_stream(pa + blk * 32) : make_uint4(0u, 0u, 0u, 0u);
                nb[i] = (blk < nlive && pb) ? ld_stream(pb + blk * 32) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int i = 0; i < kMmaBK; ++i) {
                const int blk = blk0 + i;
                if (blk < nblk) {
#pragma unroll
                    for (int tt = 0; tt < NT; ++tt) {
                        const size_t to = (size_t)tt * 8 * ldx + blk * 32;
                        const uint4 h4 = *reinterpret_cast<const uint4 *>(xhr + to);
                        const uint4 l4 = *reinterpret_cast<const uint4 *>(xlr + to);
                        mma16816(acc[tt], wa[i].x, wb[i].x, wa[i].y, wb[i].y, h4.x, h4.y);
                        mma16816(acc[tt], wa[i].x, wb[i].x, wa[i].y, wb[i].y, l4.x, l4.y);
                        mma16816(acc[tt], wa[i].z, wb[i].z, wa[i].w, wb[i].w, h4.z, h4.w);
                        mma16816(acc[tt], wa[i].z, wb[i].z, wa[i].w, wb[i].w, l4.z, l4.w);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < kMmaBK; ++i) {
                wa[i] = na[i];
                wb[i] = nb[i];
            }
        }
        // acc[tt]: (row ra, batch 2t), (ra, 2t+1), (rb, 2t), (rb, 2t+1) of tile tt
        if (S > 1) {
            float *pp = a.mma_part + (((size_t)tile * a.mma_groups + grp) * S + sgm) * 128 * NT;
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                pp[tt * 128 + g * 8 + 2 * t] = acc[tt][0];
                pp[tt * 128 + g * 8 + 2 * t + 1] = acc[tt][1];
                pp[tt * 128 + (g + 8) * 8 + 2 * t] = acc[tt][2];
                pp[tt * 128 + (g + 8) * 8 + 2 * t + 1] = acc[tt][3];
            }
            __threadfence();
            int last = 0;
            int *cnt = a.mma_cnt + (size_t)tile * a.mma_groups + grp;
            if (lane == 0)
                last = (atomicAdd(cnt, 1) == S - 1);
            last = __shfl_sync(0xffffffffu, last, 0);
            if (!last)
                continue;
            __threadfence();
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                // the S partials in segment order, kSumBatch of them loaded at once
                constexpr int kSumBatch = 8;
                float sum[4] = {0.f, 0.f, 0.f, 0.f};
                for (int q0 = 0; q0 < S; q0 += kSumBatch) {
                    float v[kSumBatch][4];
#pragma unroll
                    for (int u = 0; u < kSumBatch; ++u) {
                        const float *qp = a.mma_part +
                                          (((size_t)tile * a.mma_groups + grp) * S + q0 + u) *
                                              128 * NT +
                                          tt * 128;
                        const bool in = q0 + u < S;
                        v[u][0] = in ? __ldcg(qp + g * 8 + 2 * t) : 0.f;
                        v[u][1] = in ? __ldcg(qp + g * 8 + 2 * t + 1) : 0.f;
                        v[u][2] = in ? __ldcg(qp + (g + 8) * 8 + 2 * t) : 0.f;
                        v[u][3] = in ? __ldcg(qp + (g + 8) * 8 + 2 * t + 1) : 0.f;
                    }
#pragma unroll
                    for (int u = 0; u < kSumBatch; ++u)
                        if (q0 + u < S)
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                sum[i] += v[u][i];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    acc[tt][i] = sum[i];
            }
            if (lane == 0)
                *cnt = 0;
        }
#pragma unroll
        for (int tt = 0; tt < NT; ++tt) {
            const int bt = b0 + tt * 8 + 2 * t;
            if (ma.p) {
                if (bt < a.B)
                    finalize_one<T, KIND>(a, ra, ma, bt, acc[tt][0]);
                if (bt + 1 < a.B)
                    finalize_one<T, KIND>(a, ra, ma, bt + 1, acc[tt][1]);
            }
            if (mb.p) {
                if (bt < a.B)
                    finalize_one<T, KIND>(a, rb, mb, bt, acc[tt][2]);
                if (bt + 1 < a.B)
                    finalize_one<T, KIND>(a, rb, mb, bt + 1, acc[tt][3]);
            }
            if constexpr (KIND == RK_PRED2) {
                // first-digit histogram: the lanes holding the same (batch
                // row, digit) add their count once
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int b = bt + (i & 1);
                    const bool live = (i < 2 ? ma.p : mb.p) != nullptr && b < a.B;
                    const unsigned dig = score_key(acc[tt][i]) >> 21;
                    const unsigned key = live ? ((unsigned)b << 11) | dig : 0xffffffffu;
                    const unsigned same = __match_any_sync(0xffffffffu, key);
                    if (live && lane == __ffs(same) - 1)
                        atomicAdd(a.hist + (size_t)b * kTopkBins + dig, __popc(same));
                }
            }
        }
    }
    chain_stamp(stamps, 5);  // groups done
    chain_stamp_end(stamps);
}

// ---------------------------------------------------------------------------
// tcgen05 variant of the fc1 row kernel (binary16, batch tiles of 16 or 32
// rows per weight pass).
//
// D (128 gathered fc1 rows x N) accumulates in tensor memory, N = 2 BT
// columns: the binary16 hi parts of the BT batch rows, then their lo parts
// (the two are added in the epilogue, as in the mma.sync kernel).  A = 128
// gathered weight rows x 64 k per stage, copied by cp.async into a ring of
// shared-memory stages laid out as the 128-byte-swizzled K-major canonical
// form (row r at r * 128 bytes, its 16-byte chunk j at slot j ^ (r % 8));
// B = this CTA's K segment of the normalised activations, split and
// swizzled the same way once per CTA.  One thread issues four
// tcgen05.mma.kind::f16 (K = 16 each) per stage and commits them to the
// stage's mbarrier, which frees the slot for the next copy.  K is cut into
// S segments (B operand <= 128 KB); CTAs of a segment split the 128-row
// tiles, and a tile's S partials are added in segment order by the CTA
// that finishes it last.  Every wait is bounded (DV_ERR_TIMEOUT, the CTA
// then skips its work, waits for its own MMAs and frees its tensor memory).

constexpr int kTcThreads = 256;
constexpr int kTcStages = 4;              // ring slots of 128 rows x 128 bytes
constexpr int kTcSlot = 128 * 128;        // bytes per slot
constexpr int kTcBBytes = 128 * 1024;     // B operand budget
constexpr long long kTcSpin = 1LL << 22;  // polls of an mbarrier before giving up

DV_DEV uint32_t tc_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

DV_DEV void tc_bar_init(uint64_t *b)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tc_smem(b)) : "memory");
}
// true once the phase with this parity has completed; false after kTcSpin polls
DV_DEV bool tc_bar_wait(uint64_t *b, uint32_t parity)
{
    for (long long it = 0; it < kTcSpin; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(tc_smem(b)), "r"(parity)
            : "memory");
        if (ok)
            return true;
    }
    return false;
}
DV_DEV void tc_cp16(uint32_t dst, const void *src, bool valid)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
// Shared-memory matrix descriptor: 128-byte swizzle, K-major, 8-row groups
// 1024 bytes apart.
DV_DEV uint64_t tc_desc(uint32_t saddr)
{
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16: f32 accumulate, f16 A and B, both
// K-major, M = 128, N columns.
__host__ __device__ constexpr uint32_t tc_idesc(int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
DV_DEV void tc_mma(uint32_t tmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
        : "memory");
}
DV_DEV void tc_commit(uint64_t *b)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     tc_smem(b))
                 : "memory");
}
DV_DEV void tc_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = __uint_as_float(r[i]);
}
DV_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DV_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
DV_DEV void tc_fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// The B operand holds N rows; byte offset of 16-byte chunk (row n, k / 8 = c8)
// in the swizzled layout (64-k regions of N x 128 bytes).
DV_DEV uint32_t tc_b_off(int N, int n, int c8)
{
    return (uint32_t)((c8 >> 3) * N * 128 + n * 128 + (((c8 & 7) ^ (n & 7)) << 4));
}

template <int BT>
__global__ void __launch_bounds__(kTcThreads, 1) k_rowdot_tc(const RowArgs a)
{
    using T = __half;
    constexpr int N = 2 * BT;
    constexpr int TCOLS = N < 32 ? 32 : N;  // tensor-memory columns (power of 2)
    constexpr uint32_t IDESC = tc_idesc(N);
    unsigned long long *stamps = chain_stamps(a.stamps);
    extern __shared__ __align__(16) unsigned char tc_raw[];
    unsigned char *sm = tc_raw + ((1024 - (tc_smem(tc_raw) & 1023)) & 1023);
    unsigned char *xb = sm;                // B operand: ks / 64 regions of N x 128 bytes
    unsigned char *ring = sm + kTcBBytes;  // kTcStages slots of 128 x 128 bytes
    __shared__ __align__(8) uint64_t bar[kTcStages];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort, s_last;
    __shared__ long long s_off[128];
    __shared__ float2 sstat[BT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile_b = blockIdx.y, b0 = tile_b * BT;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         tc_smem(&s_tmem)),
                     "r"(TCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < kTcStages; ++i)
            tc_bar_init(&bar[i]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        s_abort = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    pdl_wait();  // h1 comes from the previous kernel
    chain_stamp(stamps, 1);
    pdl_launch_dependents();

    const int K = a.K, S = a.mma_seg, ks = a.mma_ks;
    const int rows = (min(max(ld_cg(a.n_sel), 0), a.max_sel)) << a.swiglu;
    const int ntiles = (rows + 127) >> 7;
    const int ncta = gridDim.x;
    const int sgm = (int)((long long)blockIdx.x * S / ncta);
    const int cf = (int)(((long long)sgm * ncta + S - 1) / S);
    const int cl = (int)(((long long)(sgm + 1) * ncta + S - 1) / S);
    const int t0 = (int)((long long)ntiles * (blockIdx.x - cf) / (cl - cf));
    const int t1 = (int)((long long)ntiles * (blockIdx.x - cf + 1) / (cl - cf));
    const int k0 = sgm * ks;
    const int kn = min(ks, K - k0);        // multiple of 64
    const int nkc = kn >> 6;               // 64-k chunks of this segment

    // B operand: norm(h1) of batch rows b0 .. b0 + BT - 1 over this segment,
    // hi parts in rows 0 .. BT - 1, lo parts in rows BT .. 2 BT - 1
    {
        const bool ln = a.norm_kind == DV_LAYERNORM;
        if (a.norm_g) {
            for (int bi = warp; bi < BT; bi += kTcThreads / 32) {
                const int b = b0 + bi;
                if (b < a.B) {
                    const float2 st = warp_row_stats(a.x + (size_t)b * a.x_ld, K, ln, a.eps, lane);
                    if (lane == 0)
                        sstat[bi] = st;
                }
            }
            __syncthreads();
        }
        const int cps = nkc * 8;  // 8-element chunks per row
        for (int i = tid; i < BT * cps; i += kTcThreads) {
            const int bi = i / cps, c = i - bi * cps, b = b0 + bi;
            float v[8];
            if (b < a.B) {
                norm_chunk<T>(a.x + (size_t)b * a.x_ld, (k0 >> 3) + c, a.norm_g, a.norm_b, ln,
                              a.norm_g ? sstat[bi] : make_float2(0.f, 1.f), v);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = 0.f;
            }
            __align__(16) __half hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                hi[e] = __float2half_rn(v[e]);
                lo[e] = __float2half_rn(v[e] - __half2float(hi[e]));
            }
            *reinterpret_cast<uint4 *>(xb + tc_b_off(N, bi, c)) = *reinterpret_cast<const uint4 *>(hi);
            *reinterpret_cast<uint4 *>(xb + tc_b_off(N, BT + bi, c)) =
                *reinterpret_cast<const uint4 *>(lo);
        }
    }
    tc_fence_async_smem();
    __syncthreads();
    chain_stamp(stamps, 4);  // activations staged

    const T *W = static_cast<const T *>(a.w0);
    const int cr = tid >> 1, ch = (tid & 1) * 4;  // copy: row cr, 16-byte chunks ch .. ch + 3
    // Chunks are numbered q = 0, 1, ... over the CTA's tiles; chunk q uses
    // ring slot q % kTcStages and completes phase q / kTcStages of its
    // mbarrier.  Each tile: its row offsets, kTcStages - 1 copies ahead, then
    // per chunk: wait for its copies, one thread issues the MMAs and commits,
    // every thread issues the copy kTcStages - 1 chunks ahead into the slot
    // the previous chunk's MMAs have released.  One cp.async group per chunk
    // slot (empty groups keep the count), so wait_group(kTcStages - 2) means
    // "this chunk has landed".
    int q = 0;
    for (int t = t0; t < t1; ++t) {
        __syncthreads();
        const bool stop = s_abort != 0;  // read by all between two barriers: uniform
        __syncthreads();
        if (stop)
            break;
        if (tid < 128) {  // gather offsets of the tile's rows
            const int row = t * 128 + tid;
            long long off = -1;
            if (row < rows) {
                const RowRef m = row_ref<T, RK_FC1>(a, row, nullptr, 0, 0);
                if (m.p)
                    off = (long long)(static_cast<const T *>(m.p) - W);
                else
                    set_status(a.status, DV_ERR_DEVICE_INDEX);
            }
            s_off[tid] = off;
        }
        __syncthreads();
        const long long off = s_off[cr];
        auto copy = [&](int c, int qq) {  // chunk c of this tile into slot qq % kTcStages
            if (c < nkc) {
                const uint32_t dst = tc_smem(ring + (qq % kTcStages) * kTcSlot + cr * 128);
#pragma unroll
                for (int j = ch; j < ch + 4; ++j) {
                    const bool ok = off >= 0;
                    tc_cp16(dst + ((j ^ (cr & 7)) << 4),
                            ok ? (const void *)(W + off + k0 + c * 64 + j * 8) : (const void *)W,
                            ok);
                }
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        // the previous tile's MMAs are all complete (waited below), so the
        // first slots are free
        for (int i = 0; i < kTcStages - 1; ++i)
            copy(i, q + i);
        for (int c = 0; c < nkc; ++c, ++q) {
            asm volatile("cp.async.wait_group %0;" ::"n"(kTcStages - 2) : "memory");
            tc_fence_async_smem();
            __syncthreads();
            if (tid == 0) {
                tc_fence_after();
                const uint32_t aaddr = tc_smem(ring + (q % kTcStages) * kTcSlot);
                const uint32_t baddr = tc_smem(xb + c * N * 128);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma(tmem, tc_desc(aaddr + 32 * kk), tc_desc(baddr + 32 * kk), IDESC,
                           (c > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&bar[q % kTcStages]);
            }
            // slot (q + kTcStages - 1) % kTcStages was chunk q - 1's
            if (c + kTcStages - 1 < nkc && c >= 1 &&
                !tc_bar_wait(&bar[(q - 1) % kTcStages], ((q - 1) / kTcStages) & 1))
                s_abort = 1;
            copy(c + kTcStages - 1, q + kTcStages - 1);
        }
        // the tile's last MMAs (and so all of them) are complete (on a
        // timeout the status is set and the tile finishes with what it has,
        // so every thread meets the same barriers; the next tile stops)
        if (!tc_bar_wait(&bar[(q - 1) % kTcStages], ((q - 1) / kTcStages) & 1))
            s_abort = 1;
        tc_fence_after();
        // warp w reads TMEM lanes 32 (w % 4) + lane (the tile's rows); warps
        // 0-3 take batch rows 0 .. BT/2 - 1, warps 4-7 the rest
        const int rl = 32 * (warp & 3) + lane, bh = (warp >> 2) * (BT / 2);
        float v[BT / 2];
#pragma unroll
        for (int g = 0; g < BT / 2; g += 8) {
            float h[8], l[8];
            const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
            tc_ld8(tmem + lanes + (uint32_t)(bh + g), h);
            tc_ld8(tmem + lanes + (uint32_t)(BT + bh + g), l);
#pragma unroll
            for (int e = 0; e < 8; ++e)
                v[g + e] = h[e] + l[e];
        }
        tc_fence_before();
        const int row = t * 128 + rl;
        const size_t pbase = (((size_t)tile_b * a.mma_groups + t) * S) * 128 * BT;
        bool fin = S == 1;
        if (S > 1) {  // this segment's partial; the last of the S CTAs adds them in order
            float *pp = a.mma_part + pbase + (size_t)sgm * 128 * BT + (size_t)rl * BT + bh;
#pragma unroll
            for (int e = 0; e < BT / 2; ++e)
                pp[e] = v[e];
            __threadfence();
            __syncthreads();
            if (tid == 0)
                s_last = atomicAdd(a.mma_cnt + (size_t)tile_b * a.mma_groups + t, 1) == S - 1;
            __syncthreads();
            fin = s_last != 0;
            if (fin) {
                __threadfence();
#pragma unroll
                for (int e = 0; e < BT / 2; ++e)
                    v[e] = 0.f;
                for (int sg = 0; sg < S; ++sg) {
                    const float *qp =
                        a.mma_part + pbase + (size_t)sg * 128 * BT + (size_t)rl * BT + bh;
#pragma unroll
                    for (int e = 0; e < BT / 2; ++e)
                        v[e] += __ldcg(qp + e);
                }
                if (tid == 0)
                    a.mma_cnt[(size_t)tile_b * a.mma_groups + t] = 0;
            }
        }
        if (fin && row < rows) {
            const RowRef m = row_ref<T, RK_FC1>(a, row, nullptr, 0, 0);
            if (m.p)
#pragma unroll
                for (int e = 0; e < BT / 2; ++e)
                    if (b0 + bh + e < a.B)
                        finalize_one<T, RK_FC1>(a, row, m, b0 + bh + e, v[e]);
        }
        // (the loop's first barrier keeps the next tile's MMAs behind these reads)
    }
    if (s_abort && tid == 0)
        set_status(a.status, DV_ERR_TIMEOUT);
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    // on the abort path, wait (bounded) for the MMAs already committed
    if (s_abort && tid == 0 && q > 0)
        tc_bar_wait(&bar[(q - 1) % kTcStages], ((q - 1) / kTcStages) & 1);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TCOLS)
                     : "memory");
    }
    chain_stamp(stamps, 5);
    chain_stamp_end(stamps);
}

template <typename T, int NB, int KIND>
cudaError_t launch_one(const RowArgs &a, dim3 grid, size_t smem, cudaStream_t st, bool pdl)
{
    constexpr int U = NB <= 2 ? 8 : 4;
    auto kern = k_rowdot<T, NB, KIND, U>;
    // Opt in to the shared-memory budget once per device (not per launch, so
    // later launches may be captured into a CUDA graph).
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemCap);
    });
    if (e != cudaSuccess)
        return e;
    if (smem > kSmemCap || a.geo.U != U)
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

RowGeo rowdot_geometry(int K, int dtype, int nb)
{
    RowGeo g;
    const int epc = dtype == DV_F16 ? 8 : 4;
    g.U = nb <= 2 ? 8 : 4;
    const int lim = 32 * g.U;  // chunks one warp has in flight per unit
    g.cpr = K / epc;
    if (g.cpr >= lim) {
        // segment mode: the largest divisor of cpr not above lim
        int uc = lim;
        while (uc > 1 && g.cpr % uc != 0)
            --uc;
        g.ucr = uc;
        g.nsu = g.cpr / uc;
        g.rpu = 1;
    } else {
        int rpu = 1;
        while (rpu < 4 && g.cpr * rpu * 2 <= lim)
            rpu <<= 1;
        g.rpu = rpu;
        g.ucr = g.cpr;
        g.nsu = 0;
    }
    return g;
}

int rowdot_nb(int B, int K, int kind)
{
    int nb = 1;
    while (nb < B && nb < 8)
        nb <<= 1;
    while (nb > 1 && rowdot_smem(kind, nb, K) > kSmemCap)
        nb >>= 1;
    return nb;
}

// Activations [nb][K] floats, the first-digit histogram (PRED2) and the
// staged gather indices.
size_t rowdot_smem(int kind, int nb, int K)
{
    return (size_t)nb * K * 4 + (kind == RK_PRED2 ? (size_t)nb * kTopkBins * 4 : 0) +
           (size_t)kSelStage * 4;
}

cudaError_t launch_rowdot(int kind, int dtype, int nb, const RowArgs &a, dim3 grid, size_t smem,
                          cudaStream_t st, bool pdl)
{
    if (dtype == DV_F16)
        return dispatch_kind<__half>(kind, nb, a, grid, smem, st, pdl);
    return dispatch_kind<float>(kind, nb, a, grid, smem, st, pdl);
}

namespace {

template <int KIND, int NT>
cudaError_t launch_rowdot_mma_t(const cudaLaunchConfig_t &cfg, const RowArgs &a)
{
    auto kern = k_rowdot_mma<KIND, NT>;
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemCap);
    });
    if (e != cudaSuccess)
        return e;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int KIND>
cudaError_t dispatch_nt(int nt, const cudaLaunchConfig_t &cfg, const RowArgs &a)
{
    switch (nt) {
    case 1: return launch_rowdot_mma_t<KIND, 1>(cfg, a);
    case 2: return launch_rowdot_mma_t<KIND, 2>(cfg, a);
    case 4: return launch_rowdot_mma_t<KIND, 4>(cfg, a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

int rowdot_mma_tiles(int B) { return B <= 8 ? 1 : (B <= 16 ? 2 : 4); }

// tcgen05 fc1 kernel: K segments whose hi/lo activations (2 bt rows of
// binary16 per k) fit the B-operand budget, multiples of 64.
void rowdot_tc_plan(int K, int bt, int *S, int *ks)
{
    int len = kTcBBytes / (2 * 2 * bt);
    len = len / 64 * 64;
    if (len > K)
        len = (K + 63) / 64 * 64;
    *ks = len;
    *S = (K + len - 1) / len;
}
size_t rowdot_tc_smem() { return (size_t)kTcBBytes + (size_t)kTcStages * kTcSlot + 1024; }

cudaError_t launch_rowdot_tc(const RowArgs &a, dim3 grid, cudaStream_t st, bool pdl)
{
    if (a.mma_nt != 2 && a.mma_nt != 4)
        return cudaErrorInvalidValue;
    auto kern = a.mma_nt == 2 ? k_rowdot_tc<16> : k_rowdot_tc<32>;
    static DeviceOnce once[2];
    const size_t smem = rowdot_tc_smem();
    cudaError_t e = once[a.mma_nt == 2 ? 0 : 1].run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

cudaError_t launch_rowdot_mma(int kind, const RowArgs &a, dim3 grid, size_t smem,
                              cudaStream_t st, bool pdl)
{
    if (kind < RK_PRED1 || kind > RK_FC1)
        return cudaErrorInvalidValue;
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
    const int nt = a.mma_nt;
    switch (kind) {
    case RK_PRED1: return dispatch_nt<RK_PRED1>(nt, cfg, a);
    case RK_PRED2: return dispatch_nt<RK_PRED2>(nt, cfg, a);
    case RK_QKV: return dispatch_nt<RK_QKV>(nt, cfg, a);
    default: return dispatch_nt<RK_FC1>(nt, cfg, a);
    }
}

// K segments and their length for the tensor-core variant: each segment's
// hi/lo activations of 8 nt batch rows (32 nt bytes per k, plus padding)
// must fit the shared-memory budget.
void rowdot_mma_plan(int K, int nt, int *S, int *ks)
{
    const size_t budget = 160 * 1024;
    int s = 1, len = 0;
    for (;; ++s) {
        len = ((K + s - 1) / s + 31) / 32 * 32;
        if ((size_t)32 * nt * rowdot_mma_ldx(len) <= budget || len <= 32)
            break;
    }
    *ks = len;
    *S = (K + len - 1) / len;
}

size_t rowdot_mma_smem(int ks, int nt) { return (size_t)32 * nt * rowdot_mma_ldx(ks); }

}  // namespace dv
