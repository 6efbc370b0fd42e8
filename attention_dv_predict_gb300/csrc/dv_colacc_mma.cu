// dv_colacc_mma.cu -- tensor-core variant of the column-gather GEMV for batch
// tiles of 8 rows, one, two or four tiles per weight pass (binary16 weights;
// out-projection and fc2), sm_103a.
//
//   out[b][c] = res[b][c] + bias[c] + sum_i coef[b][i] * W[row(i)][c]
// (the kernels of dv_colacc.cuh, same gather, coefficients and residual).
//
// From a few batch rows on, the CUDA-core kernel is bound by instruction
// issue: every 16-byte weight chunk costs 8 x NB multiply-adds plus its
// conversions.  Here the sum over gathered rows i is the K dimension of
// mma.sync m16n8k16 (f16 in, f32 accumulate):
//   A (16 x 16) = coefficients: rows 0-7 the binary16 hi part of batch rows
//                 b0 .. b0+7, rows 8-15 the lo part (coef - hi), so one MMA
//                 carries both and the products keep ~22 bits;
//   B (16 x 8)  = 16 gathered weight rows x 8 columns;
//   D (16 x 8)  = hi and lo partial sums, added at the end.
// A CTA takes NT tiles of 8 batch rows (NT = 2 above 8 rows, 4 above 16): the B
// fragments of each weight group feed the MMAs of every tile, so the
// weights are read once per 8 NT batch rows.
// Each warp owns 32 columns of a 512-column block.  The CTA copies groups of
// 16 gathered rows x 1 KB into a shared-memory ring with cp.async (warp w
// copies row w of the group, 512 contiguous bytes per instruction; no
// register staging, kCmStages groups in flight; one barrier per group), and
// every warp reads its 32 columns back transposed with ldmatrix.trans, which
// yields B fragments directly.
// The coefficients of a stage of rows are staged once per CTA, already laid
// out as A fragments.  Warps own disjoint columns, so there is no reduction
// across warps.  The (block, row) pieces are split evenly over the CTAs in
// block-major order (a CTA may end one block and start the next: two
// partial slots); the last CTA to finish a block adds the partials of the
// CTAs that share it in CTA order, 8 consecutive outputs per thread with
// 16-byte loads.
#include "dv_colacc.cuh"

namespace dv {
namespace {

constexpr int kCmCB = 32 * kWarpsPerBlock;  // columns per block (512)
constexpr int kCmStages = 6;                // 16-row groups in flight per CTA
constexpr int kCmSRT = 2048;                // rows x tiles staged at once (NT x rows <= 2048)
constexpr int kCmLd = kCmCB + 8;            // halves per staged row (16-byte pad: ldmatrix
                                            // rows of a warp fall in distinct banks)
constexpr size_t kCmRing = (size_t)kCmStages * 16 * kCmLd * 2;
constexpr size_t kCmFrag = (size_t)(kCmSRT / 16) * 32 * 16;
constexpr size_t kCmOff = (size_t)kCmSRT * 8;
constexpr size_t kCmSmem = kCmRing + kCmFrag + kCmOff + (size_t)kMaxCover * 4;
constexpr int kCmFill = 8;   // coefficients in flight per thread while staging
constexpr int kCmCover = 4;  // CTA partials loaded together by the combining CTA
static_assert(kCmCB == kThreads, "the combine gives each thread 8 outputs of each tile");

// CTA c takes pieces [total c / nc, total (c + 1) / nc).
DV_DEV long long cm_piece0(int c, int nc, long long total) { return total * c / nc; }
// The CTA whose range holds piece x.
DV_DEV int cm_cta_of(long long x, int nc, long long total)
{
    int c = (int)(x * nc / total);
    while (c + 1 < nc && cm_piece0(c + 1, nc, total) <= x)
        ++c;
    while (c > 0 && cm_piece0(c, nc, total) > x)
        --c;
    return c;
}

DV_DEV void cp_async16(void *dst, const void *src, bool valid)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;" ::"r"(s), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
DV_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DV_DEV void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

DV_DEV void ldsm_x4_trans(unsigned (&r)[4], const void *p)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(s)
                 : "memory");
}

DV_DEV void mma_f16(float (&d)[4], const uint4 &a, unsigned b0, unsigned b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b0), "r"(b1));
}

template <int KIND, int NT, class Dep>
DV_DEV void colacc_mma_body(const ColArgs &a, int cta, int nct, const Dep &dep)
{
    constexpr int NB = 8 * NT, CB = kCmCB;
    constexpr int SR = kCmSRT / NT;  // rows staged at once
    extern __shared__ __align__(16) unsigned char cm_smem[];
    __half *ring = reinterpret_cast<__half *>(cm_smem);
    uint4 *frag = reinterpret_cast<uint4 *>(cm_smem + kCmRing);  // [group][tile][lane]
    long long *soff = reinterpret_cast<long long *>(cm_smem + kCmRing + kCmFrag);
    int *s_cover = reinterpret_cast<int *>(cm_smem + kCmRing + kCmFrag + kCmOff);
    __shared__ int s_last, s_ncover;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    const int g = lane >> 2, t = lane & 3;
    const int tile = blockIdx.y, b0 = tile * NB;
    const int ns = min(max(ld_cg(a.n_sel), 0), a.max_sel);
    const int rows = (KIND == CK_OPROJ) ? ns * a.dh : ns;
    const int ncb = (a.d + CB - 1) / CB;
    const int nc = nct;
    const long long total = (long long)ncb * rows;
    const __half *W = static_cast<const __half *>(a.w);
    const __half *bias = static_cast<const __half *>(a.bias);

    if (total == 0) {  // nothing selected: out = res + bias
        dep.wait();
        for (int col = cta * blockDim.x + tid; col < a.d; col += nc * blockDim.x)
            for (int b = 0; b < NB && b0 + b < a.B; ++b)
                a.out[(size_t)(b0 + b) * a.d + col] =
                    __ldcg(a.res + (size_t)(b0 + b) * a.d + col) + __half2float(bias[col]);
        return;
    }

    const long long p0 = cm_piece0(cta, nc, total), p1 = cm_piece0(cta + 1, nc, total);
    const int first_cb = p1 > p0 ? (int)(p0 / rows) : 0;
    bool waited = false;
    for (long long pp = p0; pp < p1;) {
        const int cb = (int)(pp / rows);
        const int i0 = (int)(pp - (long long)cb * rows);
        const int i1 = (int)min((long long)rows, i0 + (p1 - pp));
        pp += i1 - i0;
        const int col0 = cb * CB + 32 * warp;  // this warp's first column
        float acc[NT][4][4];
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[n][j][e] = 0.f;

        for (int s0 = i0; s0 < i1; s0 += SR) {
            const int s1 = min(i1, s0 + SR);
            const int ngr = (s1 - s0 + 15) >> 4;
            __syncthreads();  // the previous stage's offsets and fragments are consumed
            for (int i = tid; i < ngr * 16; i += blockDim.x) {
                long long off = -1;
                if (s0 + i < s1) {
                    off = row_offset<KIND>(a, s0 + i);
                    if (off < 0)
                        set_status(a.status, DV_ERR_DEVICE_INDEX);
                }
                soff[i] = off;
            }
            __syncthreads();
            // group q of the stage into ring slot q % kCmStages: warp w copies
            // row w (two 512-byte halves, 16 bytes a lane); one commit per
            // call, so the wait count stays uniform (empty groups past the end)
            auto issue = [&](int q) {
                if (q < ngr) {
                    __half *dst = ring + ((q % kCmStages) * 16 + warp) * kCmLd;
                    const long long off = soff[q * 16 + warp];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int cc = 256 * h + 8 * lane;
                        const int col = cb * CB + cc;
                        const bool ok = off >= 0 && col < a.d;
                        cp_async16(dst + cc, ok ? (const void *)(W + off + col) : a.w, ok);
                    }
                }
                cp_async_commit();
            };
            // weights are constant and the gather list comes from kernels at
            // least two launches back: the first groups go out before the wait
#pragma unroll
            for (int q = 0; q < kCmStages - 1; ++q)
                issue(q);
            if (!waited) {  // the coefficients come from the previous kernel
                dep.wait();
                waited = true;
            }
            // coefficients as A fragments: for row k of group q and batch row
            // 8n + b (tile n), lane 4b + (k & 7) / 2 of fragment (q, n) holds
            // hi in halves (k >= 8 ? 4 : 0) + (k & 1) and lo two halves further
            const int nitems = ngr * 16 * NB;
            for (int base = tid; base < nitems; base += kCmFill * blockDim.x) {
                float cv[kCmFill];
#pragma unroll
                for (int u = 0; u < kCmFill; ++u) {
                    const int it = base + u * blockDim.x;
                    const int i = it / NB, b = it - i * NB;
                    cv[u] = (it < nitems && s0 + i < s1 && b0 + b < a.B && soff[i] >= 0)
                                ? coef_at<KIND>(a, b0 + b, s0 + i)
                                : 0.f;
                }
#pragma unroll
                for (int u = 0; u < kCmFill; ++u) {
                    const int it = base + u * blockDim.x;
                    if (it >= nitems)
                        break;
                    const int i = it / NB, bb = it - i * NB;
                    const int n = bb >> 3, b = bb & 7;
                    const int q = i >> 4, k = i & 15;
                    const __half hi = __float2half_rn(cv[u]);
                    const __half lo = __float2half_rn(cv[u] - __half2float(hi));
                    __half *fh = reinterpret_cast<__half *>(frag + (q * NT + n) * 32 + 4 * b +
                                                            ((k & 7) >> 1));
                    const int ho = ((k >> 3) ? 4 : 0) + (k & 1);
                    fh[ho] = hi;
                    fh[ho + 2] = lo;
                }
            }
            __syncthreads();
            // ldmatrix: lane l addresses row l & 7 of matrix l >> 3; matrix m
            // of a call for column tiles (j, j + 1) is (rows 8(m & 1) .. +7,
            // tile j + (m >> 1)), giving b0, b1 of tile j and b0, b1 of j + 1
            const int mrow = ((lane >> 3) & 1) * 8 + (lane & 7), mcol = 32 * warp + 8 * (lane >> 4);
            for (int q = 0; q < ngr; ++q) {
                // this thread's copies of group q are done; the barrier makes
                // every warp's visible and frees the slot read at q - 1
                cp_async_wait<kCmStages - 2>();
                __syncthreads();
                issue(q + kCmStages - 1);
                uint4 af[NT];
#pragma unroll
                for (int n = 0; n < NT; ++n)
                    af[n] = frag[(q * NT + n) * 32 + lane];
                const __half *slot = ring + (q % kCmStages) * 16 * kCmLd + mrow * kCmLd + mcol;
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {
                    unsigned bf[4];
                    ldsm_x4_trans(bf, slot + 16 * jp);
#pragma unroll
                    for (int n = 0; n < NT; ++n) {
                        mma_f16(acc[n][2 * jp], af[n], bf[0], bf[1]);
                        mma_f16(acc[n][2 * jp + 1], af[n], bf[2], bf[3]);
                    }
                }
            }
            cp_async_wait<0>();
        }

        // this piece's sums: batch row 8n + g, columns col0 + 8j + 2t (+1)
        const bool whole = (i0 == 0 && i1 == rows);
        const int slot = (cb == first_cb) ? 0 : 1;
        if (whole) {
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int b = b0 + 8 * n + g;
                if (b >= a.B)
                    continue;
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = col0 + 8 * j + 2 * t + e;
                        if (col < a.d)
                            a.out[(size_t)b * a.d + col] =
                                (__ldcg(a.res + (size_t)b * a.d + col) + __half2float(bias[col])) +
                                (acc[n][j][e] + acc[n][j][e + 2]);
                    }
            }
            continue;
        }
        float *pp_out = a.part + (((size_t)tile * nc + cta) * 2 + slot) * NB * CB;
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    pp_out[(8 * n + g) * CB + 32 * warp + 8 * j + 2 * t + e] =
                        acc[n][j][e] + acc[n][j][e + 2];
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            int *cntp = a.cnt + (size_t)tile * ncb + cb;
            s_last = (atomicAdd(cntp, i1 - i0) + (i1 - i0) == rows);
        }
        __syncthreads();
        if (!s_last)
            continue;
        __threadfence();
        if (tid < 32) {  // the CTAs sharing block cb, in CTA order, and their slots
            const int ca = cm_cta_of((long long)cb * rows, nc, total);
            const int cz = cm_cta_of((long long)(cb + 1) * rows - 1, nc, total);
            for (int c = ca + tid; c <= cz; c += 32) {
                const long long q0 = cm_piece0(c, nc, total), q1 = cm_piece0(c + 1, nc, total);
                if (c - ca < kMaxCover)
                    s_cover[c - ca] = q1 > q0 ? c * 2 + (q0 / rows == cb ? 0 : 1) : -1;
            }
            if (tid == 0)
                s_ncover = min(cz - ca + 1, kMaxCover);
        }
        __syncthreads();
        for (int n = 0; n < NT; ++n) {
            const int ncover = s_ncover;
            const int e0 = n * 8 * CB + tid * 8;  // outputs e0 .. e0 + 7: batch row e0 / CB
            float sum[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
                sum[e] = 0.f;
            for (int c0 = 0; c0 < ncover; c0 += kCmCover) {
                float4 v[kCmCover][2];
#pragma unroll
                for (int u = 0; u < kCmCover; ++u) {
                    const int sl = (c0 + u < ncover) ? s_cover[c0 + u] : -1;
                    const float4 *q = reinterpret_cast<const float4 *>(
                        a.part + ((size_t)tile * nc * 2 + (sl < 0 ? 0 : sl)) * NB * CB + e0);
                    v[u][0] = sl >= 0 ? __ldcg(q) : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[u][1] = sl >= 0 ? __ldcg(q + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < kCmCover; ++u) {
                    sum[0] += v[u][0].x;
                    sum[1] += v[u][0].y;
                    sum[2] += v[u][0].z;
                    sum[3] += v[u][0].w;
                    sum[4] += v[u][1].x;
                    sum[5] += v[u][1].y;
                    sum[6] += v[u][1].z;
                    sum[7] += v[u][1].w;
                }
            }
            const int b = e0 / CB, cc = e0 - b * CB;
            if (b0 + b < a.B) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int col = cb * CB + cc + e;
                    if (col < a.d)
                        a.out[(size_t)(b0 + b) * a.d + col] =
                            (__ldcg(a.res + (size_t)(b0 + b) * a.d + col) + __half2float(bias[col])) +
                            sum[e];
                }
            }
        }
        if (tid == 0)
            a.cnt[(size_t)tile * ncb + cb] = 0;
    }
    if (!waited)
        dep.wait();
}

template <int KIND, int NT>
__global__ void __launch_bounds__(kThreads, 1) k_colacc_mma(const ColArgs a)
{
    unsigned long long *s = chain_stamps(a.stamps);
    colacc_mma_body<KIND, NT>(a, blockIdx.x, gridDim.x, PdlDep{s});
    chain_stamp_end(s);
}

}  // namespace

size_t colacc_mma_smem() { return kCmSmem; }

// Four tiles a pass (above 16 rows) only for fc2: the out-projection's
// coefficient staging (the attention records' merge) spills at four tiles
// and measured slower than two passes of two (batch 32: +25 us; fc2: -22).
int colacc_mma_tiles(int B, int kind)
{
    return B > 16 && kind == CK_FC2 ? 4 : (B > 8 ? 2 : 1);
}

cudaError_t launch_colacc_mma(int kind, int nt, const ColArgs &a, dim3 grid, cudaStream_t st,
                              bool pdl)
{
    if ((kind != CK_OPROJ && kind != CK_FC2) || (nt != 1 && nt != 2 && nt != 4))
        return cudaErrorInvalidValue;
    void (*const table[2][3])(ColArgs) = {
        {k_colacc_mma<CK_OPROJ, 1>, k_colacc_mma<CK_OPROJ, 2>, k_colacc_mma<CK_OPROJ, 4>},
        {k_colacc_mma<CK_FC2, 1>, k_colacc_mma<CK_FC2, 2>, k_colacc_mma<CK_FC2, 4>}};
    const int ki = kind == CK_OPROJ ? 0 : 1, ti = nt == 4 ? 2 : nt - 1;
    void (*kern)(ColArgs) = table[ki][ti];
    static DeviceOnce once[2][3];
    cudaError_t e = once[ki][ti].run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kCmSmem);
    });
    if (e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kCmSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace dv
