// dv_stream.cu -- the whole sparse layer decode as one persistent streaming
// kernel (sm_103a), for binary16 layers with 128-wide heads at batches of 1
// and 2.
//
// The step ("DejaVu Guide: Contextual Sparsity for LLM Inference", listing
// DejaVuTransformerLayer.forward; "Core Innovation 1" and "Core Innovation
// 2") reads about 519 MB per decode at the OPT-175B shape, almost all of it
// gathered weight rows that are used once.  As a chain of kernels the HBM
// idles at every boundary (a kernel's CTAs start only when the previous
// kernel's leave, then wait for its results); here it does not:
//
//  * One CTA per SM, 17 warps.  Warp 16 is the PRODUCER: its lane 0 walks the
//    CTA's share of every phase's weight rows in order and copies them with
//    1-D bulk copies (cp.async.bulk, completion counted on an mbarrier) into
//    a ring of 16 KB stages in shared memory.  The addresses depend only on
//    the selections, which are known early (heads after the first predictor
//    stage, neurons before QKV ends), so the producer runs ahead of the
//    computation by up to the whole ring (160 KB per SM, ~3.5 us of the SM's
//    share of HBM bandwidth) -- across the phase boundaries where the
//    consumers wait for each other.
//  * Warps 0-15 are CONSUMERS.  Each thread owns fixed 16-byte chunks of a
//    row (row-dot phases: its activations stay in registers) or fixed output
//    columns (column phases: its accumulators stay in registers), so a weight
//    byte is read once from HBM and once from shared memory.
//  * Phases hand over through counters in the workspace control block
//    (release add after a group barrier, acquire poll by one thread).  Every
//    wait is bounded: one that runs out records DV_ERR_TIMEOUT, the CTA skips
//    its remaining work but still arrives at every counter and waits for its
//    own copies in flight before it exits.
//
// Phases (G CTAs; "rows" are weight rows of d binary16 values):
//  PRED1  head scores and the low-rank factor u (rows of pred_h and pred_a) on
//         x_pred; row segments of 512 chunks are dealt to all CTAs, each
//         segment's dot product goes to part1.  The last CTA to finish sums
//         the head scores and selects the heads.
//  PRED2  neuron scores s_n = u . pred_b^T (short rows, a warp per row) and the
//         histogram of their keys' top 11 bits; then every CTA runs its share
//         of the neuron selection pass (dv_select.cuh) and the last CTA
//         finishes the selection beside QKV.
//  QKV    the selected heads' q, k, v rows on LayerNorm(x) (CTAs 0 .. G-2).
//  ATTN   split-KV attention over the selected heads (q, the new k and v from
//         the QKV segment sums; the new k, v appended to the cache); chunk
//         records (max, weight sum, weighted V).
//  OPROJ  column groups: the G CTAs form ncg groups of gm; group g owns a run
//         of about d / ncg columns (whole 16-byte chunks) and its CTAs split
//         the selected heads' out-projection rows, each accumulating its
//         columns in registers;
//         then each CTA adds the group's partials for a slice of the columns
//         (h1 = x + b_o + sum) and the slice's norm statistics.
//  FC1    the selected neurons' fc1 rows on LayerNorm(h1) (statistics merged
//         from every CTA's records), segment sums to partF.
//  FC2    column groups as OPROJ, coefficients ReLU(fc1 + b1); then y.
#include <algorithm>

#include "dv_select.cuh"

namespace dv {
namespace {

constexpr int kCW = kConsumers / 32;  // consumer warps
constexpr int kSeg = kStreamUnitBytes / 16;  // chunks of a row segment (512)
constexpr int kRU = 16;               // row-dot segments per batch of partial sums
constexpr int kNR = 4;                // u chunks per lane in PRED2 (rank <= 1024)
constexpr int kNJ = 4;                // columns per thread and group in the column phases / 512
constexpr int kDH = 128;              // head dimension served
constexpr int kIdxWin = 1024;         // producer's window of gathered indices

// Fixed part of the dynamic shared memory.
constexpr int kOffBar = 0;     // full[16], empty[16]
constexpr int kOffMisc = 256;  // ints, see the kM* indices
constexpr int kOffRed = 768;   // [2][kRU][kCW][2] floats
constexpr int kOffIdx = kOffRed + 2 * kRU * kCW * 2 * 4;     // producer: u_h[256], window
constexpr int kOffUni = kOffIdx + (256 + kIdxWin) * 4;       // phase scratch
static_assert(kOffUni % 128 == 0, "union region alignment");

// Indices into the misc ints.
enum Misc {
    kMAbort = 0,    // raised by the first wait of the CTA that gives up
    kMBudget = 1,   // wait budget, microseconds
    kMHold = 2,     // test hook: the wait id made never to complete
    kMOk = 3,       // broadcast of a wait's result
    kMCount = 4,    // broadcast of a union length
    kMAgree = 5,    // broadcast of the abort flag
    kMOld = 8,      // broadcast of a counter's previous value
    kMLast = 9,     // this CTA is the last at the exit counter
    kMScr = 16,     // [48] scratch of the group helpers
    kMSb1 = 64,     // [8] neuron pass: bins of the k-th keys
    kMNorm = 72,    // [8] (mean, rstd) per batch row
};

DV_DEV uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier and bulk-copy primitives.
DV_DEV void mbar_init(uint64_t *b, int count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count)
                 : "memory");
}
DV_DEV void mbar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b))
                 : "memory");
}
DV_DEV void mbar_expect_tx(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(b)),
                 "r"(bytes)
                 : "memory");
}
DV_DEV bool mbar_try_wait(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Copy `bytes` (a multiple of 16; both addresses 16-byte aligned) from global
// to this CTA's shared memory; completion is counted on mbarrier b.
DV_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *b)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(b))
        : "memory");
}

DV_DEV int atom_add_acq_rel(int *p, int v)
{
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
                 : "memory");
    return old;
}
DV_DEV void red_add_release(int *p, int v)
{
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------------------
// Bounded waits.  Each gives up when the CTA's abort flag is raised or after
// `budget_ns` (globaltimer), and has an iteration cap besides.
struct Bound {
    unsigned long long budget_ns;
    volatile int *abort;  // shared: raised by the first wait of the CTA that gives up
    int *status;
};

DV_DEV void give_up(const Bound &bd)
{
    set_status(bd.status, DV_ERR_TIMEOUT);
    *bd.abort = 1;
}

DV_DEV bool mbar_wait(uint64_t *b, uint32_t parity, const Bound &bd)
{
    if (mbar_try_wait(b, parity))
        return true;
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < (1 << 26); ++it) {
        if (mbar_try_wait(b, parity))
            return true;
        if (*bd.abort)
            return false;
        if ((it & 7) == 7 && global_ns() - t0 > bd.budget_ns) {
            give_up(bd);
            return false;
        }
    }
    give_up(bd);
    return false;
}

DV_DEV bool poll_ge(const int *p, int target, const Bound &bd)
{
    const unsigned long long t0 = global_ns();
    for (int it = 0; it < (1 << 26); ++it) {
        if (ld_acquire_gpu(p) >= target)
            return true;
        if (*bd.abort)
            return false;
        if ((it & 7) == 7 && global_ns() - t0 > bd.budget_ns) {
            give_up(bd);
            return false;
        }
        __nanosleep(32);
    }
    give_up(bd);
    return false;
}

// ---------------------------------------------------------------------------
// The ring.  Stage k lives in slot k % n; its full barrier's phase parity is
// (k / n) & 1.  Every consumer warp waits for and releases every stage.
struct Ring {
    unsigned char *base;
    uint64_t *full, *empty;
    int n;
    int k;  // next stage
    DV_DEV int slot() const { return k % n; }
    DV_DEV uint32_t par() const { return (uint32_t)((k / n) & 1); }
    DV_DEV unsigned char *buf() const { return base + (size_t)slot() * kStreamStageBytes; }
};

// Consumer warp: wait for the next stage (false: the CTA gave up).
DV_DEV const unsigned char *cons_acquire(Ring &R, const Bound &bd)
{
    const bool good = mbar_wait(&R.full[R.slot()], R.par(), bd);
    // the warp goes on only if every lane saw the stage (all wait, so each
    // lane's reads are ordered after the copy's completion)
    if (!__all_sync(0xffffffffu, good))
        return nullptr;
    return R.buf();
}
DV_DEV void cons_release(Ring &R)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        mbar_arrive(&R.empty[R.slot()]);
    ++R.k;
}

// ---------------------------------------------------------------------------
// Work split helpers (the producer and the consumers derive the same ranges).
DV_DEV int share(long long total, int part, int parts) { return (int)(total * part / parts); }

// Columns [col0, col0 + ncol) of column group g: the row's 16-byte chunks
// split into ncg nearly equal runs.
struct GroupCols {
    int col0, ncol;
};
DV_DEV GroupCols group_cols(int d, int g, int ncg)
{
    const int cpr = d / 8;
    const int c0 = share(cpr, g, ncg), c1 = share(cpr, g + 1, ncg);
    return GroupCols{8 * c0, 8 * (c1 - c0)};
}

// Activation chunks of a row (x_pred, LayerNorm(x), LayerNorm(h1)): thread t
// holds chunks t + 512 i, i < NI, of each batch row.
template <int NB, int NI>
struct Acts {
    float v[NI][NB][8];
};

// ---------------------------------------------------------------------------
// Kernel context shared by the consumer functions.
template <int NB, int NI>
struct Cons {
    const StreamArgs &a;
    Ring R;
    Bound bd;
    float *red;       // [2][kRU][kCW][NB]
    int *misc;        // [16..64) scratch of the group helpers
    unsigned char *uni;
    int cta, tid, lane, warp;
    // The CTA has not given up.  Uniform over the consumers wherever it
    // decides anything that holds a group barrier: it is set only from
    // broadcasts (wait, agree); inside a stage loop a warp may clear its own
    // copy, and the loop then still runs every barrier it would have run.
    bool ok;

    DV_DEV int *ctl(int w) const { return a.ctl + w; }

    // After a stage loop: every consumer takes the CTA's abort flag.
    DV_DEV void agree()
    {
        ConsumerGroup::sync();
        if (tid == 0)
            misc[kMAgree] = *bd.abort ? 0 : 1;
        ConsumerGroup::sync();
        ok = misc[kMAgree] != 0;
    }

    // The group (512 consumer threads) arrives at control word w, whether or
    // not the CTA gave up (so that no other CTA waits for it in vain).
    // Returns the previous count when `want_old`, else 0.
    DV_DEV int arrive(int w, bool want_old = false)
    {
        ConsumerGroup::sync();
        if (tid == 0) {
            int old = 0;
            __threadfence();
            if (want_old)
                old = atom_add_acq_rel(ctl(w), 1);
            else
                red_add_release(ctl(w), 1);
            misc[kMOld] = old;
        }
        ConsumerGroup::sync();
        return misc[kMOld];
    }

    // Wait (all consumers) until control word w reaches target; false if the
    // CTA gave up.  The test hook makes the wait with id == hold never
    // complete, so that it runs out.
    DV_DEV bool wait(int w, int target, int id)
    {
        if (tid == 0) {
            const int hold = misc[kMHold];
            const bool good =
                !*bd.abort && poll_ge(ctl(w), hold == id ? INT_MAX : target, bd);
            misc[kMOk] = good ? 1 : 0;
        }
        ConsumerGroup::sync();
        ok = misc[kMOk] != 0;
        return ok;
    }

    // Poll a flag and read a union length (clamped) behind it.
    DV_DEV int flag_count(int w, const int32_t *count, int max_count)
    {
        if (tid == 0) {
            const bool good = !*bd.abort && poll_ge(ctl(w), 1, bd);
            misc[kMCount] = good ? min(max(__ldcg(count), 0), max_count) : 0;
            misc[kMOk] = good ? 1 : 0;
        }
        ConsumerGroup::sync();
        ok = misc[kMOk] != 0;
        return misc[kMCount];
    }
};

// ---------------------------------------------------------------------------
// Row-dot stages of row segments [u0, u1) (two per stage, 8 KB apart): thread
// t multiplies chunk t of each segment with its activations; the warps' sums
// go to `red`, and after every kRU segments the group adds the kCW warp sums
// of each in warp order and stores part[b * bstride + segment].
template <int NB, int NI>
DV_DEV bool rowdot_stages(Cons<NB, NI> &C, int u0, int u1, int nseg, int cpr,
                          const Acts<NB, NI> &x, float *part, long long bstride)
{
    const int tid = C.tid, lane = C.lane, warp = C.warp;
    int nb = 0, buf = 0, ubase = u0;
    auto flush = [&]() {
        ConsumerGroup::sync();
        for (int i = tid; i < nb * NB; i += kConsumers) {
            const int q = i / NB, b = i - q * NB;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w)
                s += C.red[((buf * kRU + q) * kCW + w) * NB + b];
            part[(size_t)b * bstride + ubase + q] = s;
        }
    };
    for (int u = u0; u < u1; u += 2) {
        const unsigned char *st = C.ok ? cons_acquire(C.R, C.bd) : nullptr;
        if (!st)
            C.ok = false;  // this warp skips the data from here on
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int uu = u + q;
            if (uu >= u1)
                break;
            if (!st) {  // keep the batch count, and so every barrier, unchanged
                if (++nb == kRU) {
                    flush();
                    nb = 0;
                    buf ^= 1;
                    ubase = uu + 1;
                }
                continue;
            }
            const int seg = uu % nseg;
            const int nch = min(kSeg, cpr - seg * kSeg);
            uint4 w = make_uint4(0u, 0u, 0u, 0u);
            if (tid < nch)
                w = *reinterpret_cast<const uint4 *>(st + q * kStreamUnitBytes + tid * 16);
            float f[8];
            Elem<__half>::unpack(w, f);
            float s[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                s[b] = 0.f;
#pragma unroll
            for (int i = 0; i < NI; ++i)
                if (i == seg)
#pragma unroll
                    for (int b = 0; b < NB; ++b)
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            s[b] = fmaf(f[e], x.v[i][b][e], s[b]);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                s[b] = warp_sum(s[b]);
                if (lane == 0)
                    C.red[((buf * kRU + nb) * kCW + warp) * NB + b] = s[b];
            }
            if (++nb == kRU) {
                flush();
                nb = 0;
                buf ^= 1;
                ubase = uu + 1;
            }
        }
        if (st)
            cons_release(C.R);
    }
    if (nb)
        flush();
    C.agree();
    return C.ok;
}

// Load activation chunks of rows src[b * ld ..] (binary32), optionally
// normalised with (mean, rstd) per batch row and gain/bias (binary16).
template <int NB, int NI>
DV_DEV void load_acts(Acts<NB, NI> &x, const float *src, int ld, int cpr, const float *mean,
                      const float *rstd, const __half *g, const __half *beta, bool coherent)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < NI; ++i) {
        const int c = tid + i * kConsumers;
        const bool in = c < cpr;
        float gf[8], bf[8];
        if (g) {
            const uint4 gv = in ? *reinterpret_cast<const uint4 *>(g + (size_t)c * 8)
                                : make_uint4(0u, 0u, 0u, 0u);
            Elem<__half>::unpack(gv, gf);
            const uint4 bv = (in && beta) ? *reinterpret_cast<const uint4 *>(beta + (size_t)c * 8)
                                          : make_uint4(0u, 0u, 0u, 0u);
            Elem<__half>::unpack(bv, bf);
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
            if (in) {
                const float4 *p = reinterpret_cast<const float4 *>(src + (size_t)b * ld + c * 8);
                lo = coherent ? __ldcg(p) : p[0];
                hi = coherent ? __ldcg(p + 1) : p[1];
            }
            float v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float t = v[e];
                if (g)
                    t = in ? (t - mean[b]) * rstd[b] * gf[e] + bf[e] : 0.f;
                x.v[i][b][e] = t;
            }
        }
    }
}

// LayerNorm / RMSNorm statistics of x's rows (binary32, length d) over the
// consumer group.  mean[b] is 0 for RMSNorm.
template <int NB, int NI>
DV_DEV void row_stats(Cons<NB, NI> &C, const Acts<NB, NI> &x, int d, float (&mean)[NB],
                      float (&rstd)[NB])
{
    float *scr = reinterpret_cast<float *>(C.misc + kMScr);
    const bool ln = C.a.norm_kind == DV_LAYERNORM;
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                s += x.v[i][b][e];
        const float mu = ln ? block_sum<ConsumerGroup>(s, scr) / (float)d : 0.f;
        float ss = 0.f;
        const int cpr = d / 8;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (C.tid + i * kConsumers >= cpr)
                break;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float t = x.v[i][b][e] - mu;
                ss = fmaf(t, t, ss);
            }
        }
        mean[b] = mu;
        rstd[b] = rsqrtf(block_sum<ConsumerGroup>(ss, scr) / (float)d + C.a.eps);
    }
}

// Column stages: rows [q0, q1) of the CTA's column group, pps pieces of cg
// binary16 columns per stage; coef[(q - q0) * NB + b] in shared memory.
// Thread t accumulates columns t + 512 j of the group.
template <int NB, int NI>
DV_DEV bool column_stages(Cons<NB, NI> &C, int q0, int q1, int pps, int cg, const float *coef,
                          float (&acc)[kNJ][NB])
{
    const int tid = C.tid;
#pragma unroll
    for (int j = 0; j < kNJ; ++j)
#pragma unroll
        for (int b = 0; b < NB; ++b)
            acc[j][b] = 0.f;
    for (int q = q0; q < q1 && C.ok; q += pps) {
        const unsigned char *st = cons_acquire(C.R, C.bd);
        if (!st) {
            C.ok = false;
            break;
        }
        const int n = min(pps, q1 - q);
        for (int p = 0; p < n; ++p) {
            const __half *piece = reinterpret_cast<const __half *>(st + (size_t)p * cg * 2);
            float cf[NB];
#pragma unroll
            for (int b = 0; b < NB; ++b)
                cf[b] = coef[(q - q0 + p) * NB + b];
#pragma unroll
            for (int j = 0; j < kNJ; ++j) {
                const int col = tid + j * kConsumers;
                if (col < cg) {
                    const float w = __half2float(piece[col]);
#pragma unroll
                    for (int b = 0; b < NB; ++b)
                        acc[j][b] = fmaf(cf[b], w, acc[j][b]);
                }
            }
        }
        cons_release(C.R);
    }
    C.agree();
    return C.ok;
}

// ---------------------------------------------------------------------------
// Attention of one (batch row b, head slot j, chunk c): positions
// [c0, c1) of kv_len + 1.  q and (for the chunk holding position kv_len) the
// new k and v come from the QKV segment sums; the new k, v are rounded to
// binary16, appended to the cache, and used from shared memory.
struct AttnSmem {
    float q[kDH];
    __half kv[2][kDH];
    float wm[kCW], wl[kCW];
    float wo[kCW][kDH];
};

template <int NB, int NI>
DV_DEV void attn_unit(Cons<NB, NI> &C, int b, int j, int c, int h, int nuh)
{
    const StreamArgs &a = C.a;
    AttnSmem &S = *reinterpret_cast<AttnSmem *>(C.uni);
    const int tid = C.tid, lane = C.lane, warp = C.warp;
    const int nseg = a.nseg, L = a.kv_len, L1 = L + 1, Ch = a.attn_C;
    const __half *bq = static_cast<const __half *>(a.b_qkv);
    const bool last = c == Ch - 1;
    // q, and the new k, v (threads 0..383: type t = tid / 128, element e)
    if (tid < (last ? 3 : 1) * kDH) {
        const int t = tid / kDH, e = tid - t * kDH;
        const long long row = (long long)j * 3 * kDH + t * kDH + e;
        const float *pp = a.partQ + (size_t)b * 3 * a.max_u_h * kDH * nseg + row * nseg;
        float s = 0.f;
        for (int g = 0; g < nseg; ++g)
            s += __ldcg(pp + g);
        s += __half2float(bq[((size_t)t * a.H + h) * kDH + e]);
        if (t == 0) {
            S.q[e] = s * a.q_scale;
        } else {
            const __half hv = __float2half_rn(s);
            S.kv[t - 1][e] = hv;
            __half *cache = static_cast<__half *>(t == 1 ? a.kc : a.vc);
            cache[(((size_t)b * a.H + h) * a.kv_cap + L) * kDH + e] = hv;
        }
    }
    ConsumerGroup::sync();
    const int c0 = share(L1, c, Ch), c1 = share(L1, c + 1, Ch);
    const int p0 = c0 + share(c1 - c0, warp, kCW), p1 = c0 + share(c1 - c0, warp + 1, kCW);
    const int ks = lane >> 4, dc = lane & 15;  // key of the pair, 8-dim chunk
    const __half *Kc = static_cast<const __half *>(a.kc);
    const __half *Vc = static_cast<const __half *>(a.vc);
    const size_t base = ((size_t)b * a.H + h) * (size_t)a.kv_cap * kDH + (size_t)dc * 8;
    float q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        q[e] = S.q[dc * 8 + e];
    auto ldkv = [&](int p, int which) -> uint4 {
        if (p >= p1)
            return make_uint4(0u, 0u, 0u, 0u);
        if (p == L)
            return *reinterpret_cast<const uint4 *>(&S.kv[which][dc * 8]);
        return ld_stream((which ? Vc : Kc) + base + (size_t)p * kDH);
    };
    constexpr int UK = 4;  // key pairs per batch; two batches in flight
    uint4 kc[UK], vc[UK], kn[UK], vn[UK];
#pragma unroll
    for (int uu = 0; uu < UK; ++uu) {
        kc[uu] = ldkv(p0 + 2 * uu + ks, 0);
        vc[uu] = ldkv(p0 + 2 * uu + ks, 1);
        kn[uu] = ldkv(p0 + 2 * (UK + uu) + ks, 0);
        vn[uu] = ldkv(p0 + 2 * (UK + uu) + ks, 1);
    }
    float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        o[e] = 0.f;
    for (int pb = p0; pb < p1; pb += 2 * UK) {
#pragma unroll
        for (int uu = 0; uu < UK; ++uu) {
            const int p = pb + 2 * uu + ks;
            float kf[8];
            Elem<__half>::unpack(kc[uu], kf);
            float dot = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                dot = fmaf(q[e], kf[e], dot);
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
                dot += __shfl_xor_sync(0xffffffffu, dot, off);
            if (p < p1) {
                float vf[8];
                Elem<__half>::unpack(vc[uu], vf);
                const float mn = fmaxf(m, dot);
                const float sc = expf(m - mn);
                const float pe = expf(dot - mn);
                l = fmaf(l, sc, pe);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    o[e] = fmaf(o[e], sc, pe * vf[e]);
                m = mn;
            }
        }
#pragma unroll
        for (int uu = 0; uu < UK; ++uu) {
            kc[uu] = kn[uu];
            vc[uu] = vn[uu];
            kn[uu] = ldkv(pb + 2 * (2 * UK + uu) + ks, 0);
            vn[uu] = ldkv(pb + 2 * (2 * UK + uu) + ks, 1);
        }
    }
    {  // merge the two keys of the warp
        const float m2 = __shfl_xor_sync(0xffffffffu, m, 16);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, 16);
        const float mn = fmaxf(m, m2);
        const float s1 = (m == -INFINITY) ? 0.f : expf(m - mn);
        const float s2 = (m2 == -INFINITY) ? 0.f : expf(m2 - mn);
        l = l * s1 + l2 * s2;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float o2 = __shfl_xor_sync(0xffffffffu, o[e], 16);
            o[e] = o[e] * s1 + o2 * s2;
        }
        m = mn;
    }
    if (ks == 0)
#pragma unroll
        for (int e = 0; e < 8; ++e)
            S.wo[warp][dc * 8 + e] = o[e];
    if (lane == 0) {
        S.wm[warp] = m;
        S.wl[warp] = l;
    }
    ConsumerGroup::sync();
    if (tid < kDH) {
        float M = -INFINITY;
        for (int w = 0; w < kCW; ++w)
            M = fmaxf(M, S.wm[w]);
        float Ls = 0.f, Ot = 0.f;
        for (int w = 0; w < kCW; ++w) {
            if (S.wm[w] == -INFINITY)
                continue;
            const float f = expf(S.wm[w] - M);
            Ls = fmaf(S.wl[w], f, Ls);
            Ot = fmaf(S.wo[w][tid], f, Ot);
        }
        float *rec = a.attn_rec + (((size_t)b * a.max_u_h + j) * Ch + c) * (kAttnRec + kDH);
        rec[kAttnRec + tid] = Ot;
        if (tid == 0) {
            rec[0] = M;
            rec[1] = Ls;
        }
    }
    ConsumerGroup::sync();
}

// Attention output o[b][j][e] from the chunk records of head slot j.
DV_DEV float attn_merge(const StreamArgs &a, int b, int j, int e)
{
    const int Ch = a.attn_C, rec = kAttnRec + kDH;
    const float *r = a.attn_rec + ((size_t)b * a.max_u_h + j) * Ch * rec;
    float M = -INFINITY;
    for (int c = 0; c < Ch; ++c)
        M = fmaxf(M, __ldcg(r + (size_t)c * rec));
    float Ls = 0.f, Os = 0.f;
    for (int c = 0; c < Ch; ++c) {
        const float mc = __ldcg(r + (size_t)c * rec);
        if (mc == -INFINITY)
            continue;
        const float f = expf(mc - M);
        Ls = fmaf(__ldcg(r + (size_t)c * rec + 1), f, Ls);
        Os = fmaf(__ldcg(r + (size_t)c * rec + kAttnRec + e), f, Os);
    }
    return Os / Ls;
}

// Norm statistics record (count, mean, sum of squared deviations) merge
// (Chan et al.): a then b.
struct Stat {
    float n, mean, m2;
};
DV_DEV Stat stat_merge(Stat x, Stat y)
{
    if (x.n == 0.f)
        return y;
    if (y.n == 0.f)
        return x;
    const float n = x.n + y.n;
    const float dl = y.mean - x.mean;
    Stat r;
    r.n = n;
    r.mean = x.mean + dl * (y.n / n);
    r.m2 = x.m2 + y.m2 + dl * dl * (x.n * y.n / n);
    return r;
}

// ---------------------------------------------------------------------------
// Column-group reduction: the CTA (group g, member m) adds the group's gm
// partials for its slice of the group's columns, in member order, plus
// res + bias; writes out[b][col] and returns (in `vals`, shared) the values.
template <int NB, int NI>
DV_DEV void group_reduce(Cons<NB, NI> &C, const float *part, const float *res, bool res_coherent,
                         const __half *bias, float *out, float *vals, int *ncols_out)
{
    const StreamArgs &a = C.a;
    const int g = C.cta / a.gm, m = C.cta - g * a.gm;
    const GroupCols gc = group_cols(a.d, g, a.ncg);
    const int s0 = share(gc.ncol, m, a.gm), s1 = share(gc.ncol, m + 1, a.gm);
    const int nc = s1 - s0;
    for (int i = C.tid; i < nc * NB; i += kConsumers) {
        const int b = i / nc, cc = i - b * nc;
        const int col = gc.col0 + s0 + cc;
        float s = 0.f;
        for (int mm = 0; mm < a.gm; ++mm)
            s += __ldcg(part + ((size_t)(g * a.gm + mm) * NB + b) * a.cg + s0 + cc);
        const float rv = res_coherent ? __ldcg(res + (size_t)b * a.d + col) : res[(size_t)b * a.d + col];
        const float v = rv + __half2float(bias[col]) + s;
        out[(size_t)b * a.d + col] = v;
        if (vals)
            vals[i] = v;
    }
    *ncols_out = nc;
}

// ---------------------------------------------------------------------------
// The consumers' sequence of phases.  Every branch that holds a group barrier
// depends only on values that are uniform over the consumers (C.ok after a
// broadcast, the CTA index, counts read by one thread and broadcast), and
// every phase ends with an arrival whether or not the CTA gave up.
template <int NB, int NI>
DV_DEV void consumer(Cons<NB, NI> &C)
{
    const StreamArgs &a = C.a;
    const int G = a.G, cta = C.cta, tid = C.tid;
    const int d = a.d, cpr = d / 8, nseg = a.nseg, H = a.H;
    const int rows1 = H + a.r;
    int *misc = C.misc;
    const __half *g1 = static_cast<const __half *>(a.ln1_g);
    const __half *be1 = static_cast<const __half *>(a.ln1_b);
    const __half *g2 = static_cast<const __half *>(a.ln2_g);
    const __half *be2 = static_cast<const __half *>(a.ln2_b);
    const bool ln = a.norm_kind == DV_LAYERNORM;

    // ---- PRED1: head scores and u on x_pred
    Acts<NB, NI> x;
    load_acts(x, a.x_pred, d, cpr, nullptr, nullptr, nullptr, nullptr, false);
    {
        const long long U = (long long)rows1 * nseg;
        rowdot_stages(C, share(U, cta, G), share(U, cta + 1, G), nseg, cpr, x, a.part1,
                      (long long)rows1 * nseg);
    }
    const int before = C.arrive(kSwPred1, true);
    if (before == G - 1 && C.warp == 0) {
        // the last CTA to finish: head scores from the segment sums, then the
        // head selection (skipped if the CTA gave up; the flag is raised
        // either way so that no CTA waits for it in vain)
        if (C.ok) {
            for (int i = C.lane; i < NB * H; i += 32) {
                const int b = i / H, hh = i - b * H;
                const float *pp = a.part1 + (size_t)b * rows1 * nseg + (size_t)hh * nseg;
                float s = 0.f;
                for (int q = 0; q < nseg; ++q)
                    s += __ldcg(pp + q);
                a.s_h[i] = s;
            }
            __syncwarp();
            __threadfence();
            unsigned *hb = reinterpret_cast<unsigned *>(C.uni);
            int32_t *hs = reinterpret_cast<int32_t *>(C.uni + 2 * kHeadKPL * 4);
            head_select(a.s_h, NB, H, a.k_h, hb, hs, true, a.idx_h, a.u_h, a.n_u_h, C.lane);
            __syncwarp();
        }
        if (C.lane == 0) {
            __threadfence();
            st_release_gpu(C.ctl(kSwHeads), 1);
        }
    }

    // ---- PRED2: neuron scores (a warp per row), histogram of the keys
    int *shist = reinterpret_cast<int *>(C.uni);  // [NB][kTopkBins]
    if (C.ok && C.wait(kSwPred1, G, 1)) {
        const int rc = a.r / 8;
        float ua[kNR][NB][8];
#pragma unroll
        for (int i = 0; i < kNR; ++i) {
            const int c = C.lane + 32 * i;
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float s = 0.f;
                    if (c < rc) {
                        const float *pp =
                            a.part1 + (size_t)b * rows1 * nseg + (size_t)(H + c * 8 + e) * nseg;
                        for (int q = 0; q < nseg; ++q)
                            s += __ldcg(pp + q);
                    }
                    ua[i][b][e] = s;
                }
        }
        for (int i = tid; i < NB * kTopkBins; i += kConsumers)
            shist[i] = 0;
        ConsumerGroup::sync();
        const int j0 = share(a.N, cta, G), j1 = share(a.N, cta + 1, G);
        const int rps = kStreamStageBytes / (a.r * 2);
        bool wok = true;
        for (int j = j0; j < j1 && wok; j += rps) {
            const unsigned char *st = cons_acquire(C.R, C.bd);
            if (!st) {
                wok = false;
                break;
            }
            const int n = min(rps, j1 - j);
            for (int rr = C.warp; rr < n; rr += kCW) {  // short rows: several per warp
                const unsigned char *row = st + (size_t)rr * a.r * 2;
                float sv[NB];
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    sv[b] = 0.f;
#pragma unroll
                for (int i = 0; i < kNR; ++i) {
                    const int c = C.lane + 32 * i;
                    if (c < rc) {
                        float f[8];
                        Elem<__half>::unpack(*reinterpret_cast<const uint4 *>(row + c * 16), f);
#pragma unroll
                        for (int b = 0; b < NB; ++b)
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                sv[b] = fmaf(f[e], ua[i][b][e], sv[b]);
                    }
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const float v = warp_sum(sv[b]);
                    if (C.lane == 0) {
                        a.s_n[(size_t)b * a.N + j + rr] = v;
                        atomicAdd(&shist[b * kTopkBins + (score_key(v) >> 21)], 1);
                    }
                }
            }
            cons_release(C.R);
        }
        C.agree();
        if (C.ok)
            for (int i = tid; i < NB * kTopkBins; i += kConsumers) {
                const int v = shist[i];
                if (v)
                    atomicAdd(&a.hist[i], v);
            }
    }
    C.arrive(kSwPred2);

    // ---- neuron selection pass over this CTA's bitmap words
    NeuronSel ns;
    ns.s_n = a.s_n;
    ns.B = NB;
    ns.N = a.N;
    ns.k = a.k_n;
    ns.hist = a.hist;
    ns.rowbits = a.rowbits;
    ns.cand_key = a.cand_key;
    ns.cand_idx = a.cand_idx;
    ns.cand_cnt = a.cand_cnt;
    ns.idx_n = a.idx_n;
    ns.u_n = a.u_n;
    ns.n_u_n = a.n_u_n;
    ns.status = a.ctl;
    if (C.ok && C.wait(kSwPred2, G, 2)) {
        const int W = (a.N + 31) >> 5;
        neuron_pass<ConsumerGroup>(ns, share(W, cta, G), share(W, cta + 1, G), misc + kMSb1,
                                   shist, misc + kMScr);
    }
    C.arrive(kSwPass);

    // ---- the head union, LN1(x), QKV (CTAs 0 .. G-2)
    const int nuh = C.ok ? C.flag_count(kSwHeads, a.n_u_h, a.max_u_h) : 0;
    if (cta < G - 1) {
        if (C.ok) {
            load_acts(x, a.x, d, cpr, nullptr, nullptr, nullptr, nullptr, false);
            float mean[NB], rstd[NB];
            row_stats(C, x, d, mean, rstd);
            load_acts(x, a.x, d, cpr, mean, rstd, g1, ln ? be1 : nullptr, false);
            const long long U = (long long)3 * nuh * kDH * nseg;
            rowdot_stages(C, share(U, cta, G - 1), share(U, cta + 1, G - 1), nseg, cpr, x, a.partQ,
                          (long long)3 * a.max_u_h * kDH * nseg);
        }
        C.arrive(kSwQkv);
        // ---- attention units (batch row, head slot, chunk) over CTAs 0 .. G-2
        if (C.ok && C.wait(kSwQkv, G - 1, 4)) {
            const int units = NB * nuh * a.attn_C;
            for (int u = cta; u < units; u += G - 1) {
                const int b = u / (nuh * a.attn_C), rem = u - b * nuh * a.attn_C;
                const int j = rem / a.attn_C, c = rem - j * a.attn_C;
                const int h = __ldcg(a.u_h + j);  // uniform
                if (h < 0 || h >= H) {
                    if (tid == 0)
                        set_status(a.ctl, DV_ERR_DEVICE_INDEX);
                    continue;
                }
                attn_unit(C, b, j, c, h, nuh);
            }
        }
        C.arrive(kSwAttn);
    } else {
        // the last CTA takes no QKV rows and no attention: it finishes the
        // neuron selection beside them (the flag is raised either way)
        C.arrive(kSwAttn);
        if (C.ok && C.wait(kSwPass, G, 3))
            neuron_final<ConsumerGroup>(ns, final_smem(C.uni, a.N, misc + kMScr));
        ConsumerGroup::sync();
        if (tid == 0) {
            __threadfence();
            st_release_gpu(C.ctl(kSwNeurons), 1);
        }
    }

    // ---- out-projection: coefficients (merged attention records), columns
    const int g = cta / a.gm, mem = cta - g * a.gm;
    const GroupCols gcol = group_cols(d, g, a.ncg);
    const int pps = min(16, kStreamStageBytes / (gcol.ncol * 2));
    float acc[kNJ][NB];
    if (C.ok && C.wait(kSwAttn, G, 5)) {
        const int RO = nuh * kDH;
        const int q0 = share(RO, mem, a.gm), q1 = share(RO, mem + 1, a.gm);
        float *coef = reinterpret_cast<float *>(C.uni);
        for (int i = tid; i < (q1 - q0) * NB; i += kConsumers) {
            const int qq = i / NB, b = i - qq * NB;
            const int q = q0 + qq;
            coef[i] = attn_merge(a, b, q / kDH, q % kDH);
        }
        ConsumerGroup::sync();
        if (column_stages(C, q0, q1, pps, gcol.ncol, coef, acc)) {
            for (int j = 0; j < kNJ; ++j) {
                const int col = tid + j * kConsumers;
                if (col < gcol.ncol)
                    for (int b = 0; b < NB; ++b)
                        a.partO[((size_t)cta * NB + b) * a.cg + col] = acc[j][b];
            }
        }
    }
    C.arrive(kSwOproj + g);

    // ---- h1 on this CTA's slice of its group's columns, and the slice's
    // norm statistics (count, mean, sum of squared deviations)
    {
        float *vals = reinterpret_cast<float *>(C.uni);
        float *scr = reinterpret_cast<float *>(misc + kMScr);
        if (C.ok && C.wait(kSwOproj + g, a.gm, 6)) {
            int nc = 0;
            group_reduce(C, a.partO, a.x, false, static_cast<const __half *>(a.b_o), a.h1, vals,
                         &nc);
            ConsumerGroup::sync();
            for (int b = 0; b < NB; ++b) {
                float s = 0.f;
                for (int i = tid; i < nc; i += kConsumers)
                    s += vals[b * nc + i];
                const float mu = block_sum<ConsumerGroup>(s, scr) / (float)max(nc, 1);
                float ss = 0.f;
                for (int i = tid; i < nc; i += kConsumers) {
                    const float t = vals[b * nc + i] - mu;
                    ss = fmaf(t, t, ss);
                }
                ss = block_sum<ConsumerGroup>(ss, scr);
                if (tid == 0) {
                    float *st = a.stats + ((size_t)cta * NB + b) * 4;
                    st[0] = (float)nc;
                    st[1] = mu;
                    st[2] = ss;
                }
            }
        }
        C.arrive(kSwNorm2);
    }

    // ---- LN2 from every CTA's records (merged in a fixed order), fc1
    int nun = 0;
    if (C.ok && C.wait(kSwNorm2, G, 7)) {
        float *sres = reinterpret_cast<float *>(misc + kMNorm);  // [NB][2]
        if (C.warp < NB) {
            const int b = C.warp;
            Stat st = {0.f, 0.f, 0.f};
            const int r0 = share(G, C.lane, 32), r1 = share(G, C.lane + 1, 32);
            for (int i = r0; i < r1; ++i) {
                const float *rp = a.stats + ((size_t)i * NB + b) * 4;
                st = stat_merge(st, Stat{__ldcg(rp), __ldcg(rp + 1), __ldcg(rp + 2)});
            }
            for (int off = 1; off < 32; off <<= 1) {  // lane l takes lane l + off
                Stat o;
                o.n = __shfl_down_sync(0xffffffffu, st.n, off);
                o.mean = __shfl_down_sync(0xffffffffu, st.mean, off);
                o.m2 = __shfl_down_sync(0xffffffffu, st.m2, off);
                if ((C.lane & (2 * off - 1)) == 0)
                    st = stat_merge(st, o);
            }
            if (C.lane == 0) {
                const float var = st.m2 / (float)d;
                sres[2 * b] = ln ? st.mean : 0.f;
                sres[2 * b + 1] = rsqrtf((ln ? var : var + st.mean * st.mean) + a.eps);
            }
        }
        ConsumerGroup::sync();
        float mean[NB], rstd[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            mean[b] = sres[2 * b];
            rstd[b] = sres[2 * b + 1];
        }
        load_acts(x, a.h1, d, cpr, mean, rstd, g2, ln ? be2 : nullptr, true);
        nun = C.flag_count(kSwNeurons, a.n_u_n, a.max_u_n);
        if (C.ok) {
            const long long U = (long long)nun * nseg;
            rowdot_stages(C, share(U, cta, G), share(U, cta + 1, G), nseg, cpr, x, a.partF,
                          (long long)a.max_u_n * nseg);
        }
    }
    C.arrive(kSwFc1);

    // ---- fc2: coefficients ReLU(fc1 + b1), column stages, then y
    if (C.ok && C.wait(kSwFc1, G, 8)) {
        const int i0 = share(nun, mem, a.gm), i1 = share(nun, mem + 1, a.gm);
        float *coef = reinterpret_cast<float *>(C.uni);
        const __half *b1 = static_cast<const __half *>(a.b1);
        for (int i = tid; i < (i1 - i0) * NB; i += kConsumers) {
            const int ii = i / NB, b = i - ii * NB;
            const int row = i0 + ii;
            const int jn = __ldcg(a.u_n + row);
            const float *pp = a.partF + (size_t)b * a.max_u_n * nseg + (size_t)row * nseg;
            float s = 0.f;
            for (int q = 0; q < nseg; ++q)
                s += __ldcg(pp + q);
            const float bias = (jn >= 0 && jn < a.N) ? __half2float(b1[jn]) : 0.f;
            coef[i] = fmaxf(s + bias, 0.f);
        }
        ConsumerGroup::sync();
        if (column_stages(C, i0, i1, pps, gcol.ncol, coef, acc)) {
            for (int j = 0; j < kNJ; ++j) {
                const int col = tid + j * kConsumers;
                if (col < gcol.ncol)
                    for (int b = 0; b < NB; ++b)
                        a.partY[((size_t)cta * NB + b) * a.cg + col] = acc[j][b];
            }
        }
    }
    C.arrive(kSwFc2 + g);
    if (C.ok && C.wait(kSwFc2 + g, a.gm, 9)) {
        int nc = 0;
        group_reduce(C, a.partY, a.h1, true, static_cast<const __half *>(a.b2), a.y, nullptr, &nc);
    }
}

// ---------------------------------------------------------------------------
// Producer: lane 0 of warp 16 issues the bulk copies of every stage, in the
// consumers' order; the warp's other lanes help load index lists.
struct Prod {
    const StreamArgs &a;
    Ring R;
    Bound bd;
    int *uh_s;   // [256] head union
    int *win;    // [kIdxWin] window of the neuron union
    int win0, win1;
    int lane;
    bool ok;

    // Begin a stage: wait for its slot, announce `bytes`.
    DV_DEV unsigned char *begin(uint32_t bytes)
    {
        bool good = ok;
        if (lane == 0 && good) {
            good = mbar_wait(&R.empty[R.slot()], R.par() ^ 1u, bd);
            if (good)
                mbar_expect_tx(&R.full[R.slot()], bytes);
        }
        ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
        return ok ? R.buf() : nullptr;
    }
    DV_DEV void copy(unsigned char *dst, const void *src, uint32_t bytes)
    {
        if (lane == 0)
            bulk_g2s(dst, src, bytes, &R.full[R.slot()]);
    }
    DV_DEV void end() { ++R.k; }

    // u_n[i] through the window (all lanes call it with the same i)
    DV_DEV int neuron(int i, int nun)
    {
        if (i < win0 || i >= win1) {
            win0 = i;
            win1 = min(nun, i + kIdxWin);
            for (int q = lane; q < win1 - win0; q += 32)
                win[q] = __ldcg(a.u_n + win0 + q);
            __syncwarp();
        }
        return win[i - win0];
    }
};

DV_DEV const __half *hp(const void *p) { return static_cast<const __half *>(p); }

template <int NB>
DV_DEV void producer(Prod &P)
{
    const StreamArgs &a = P.a;
    const int G = a.G, cta = blockIdx.x, lane = P.lane;
    const int d = a.d, cpr = d / 8, nseg = a.nseg, H = a.H;
    int *status = a.ctl;

    // row-dot segments [u0, u1), two per stage; row_ptr(row) -> row start
    auto rows = [&](long long u0, long long u1, auto row_ptr) {
        for (long long u = u0; u < u1 && P.ok; u += 2) {
            uint32_t bytes = 0;
            const __half *src[2];
            uint32_t nb[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                src[q] = nullptr;
                nb[q] = 0;
                const long long uu = u + q;
                if (uu >= u1)
                    continue;
                const int row = (int)(uu / nseg), seg = (int)(uu - (long long)row * nseg);
                const int nch = min(kSeg, cpr - seg * kSeg);
                src[q] = row_ptr(row) + (size_t)seg * kSeg * 8;
                nb[q] = (uint32_t)nch * 16;
                bytes += nb[q];
            }
            unsigned char *dst = P.begin(bytes);
            if (!dst)
                break;
#pragma unroll
            for (int q = 0; q < 2; ++q)
                if (nb[q])
                    P.copy(dst + q * kStreamUnitBytes, src[q], nb[q]);
            P.end();
        }
    };

    // ---- PRED1
    {
        const long long U = (long long)(H + a.r) * nseg;
        rows(share(U, cta, G), share(U, cta + 1, G), [&](int row) {
            return row < H ? hp(a.pred_h) + (size_t)row * d : hp(a.pred_a) + (size_t)(row - H) * d;
        });
    }
    // ---- PRED2: contiguous rows of pred_b
    {
        const int j0 = share(a.N, cta, G), j1 = share(a.N, cta + 1, G);
        const int rps = kStreamStageBytes / (a.r * 2);
        for (int j = j0; j < j1 && P.ok; j += rps) {
            const int n = min(rps, j1 - j);
            const uint32_t bytes = (uint32_t)n * a.r * 2;
            unsigned char *dst = P.begin(bytes);
            if (!dst)
                break;
            P.copy(dst, hp(a.pred_b) + (size_t)j * a.r, bytes);
            P.end();
        }
    }
    // ---- the head union
    int nuh = 0;
    if (P.ok) {
        int good = 1;
        if (lane == 0)
            good = poll_ge(a.ctl + kSwHeads, 1, P.bd) ? 1 : 0;
        P.ok = __shfl_sync(0xffffffffu, good, 0) != 0;
        if (P.ok) {
            nuh = min(max(__ldcg(a.n_u_h), 0), a.max_u_h);
            for (int j = lane; j < nuh; j += 32) {
                int h = __ldcg(a.u_h + j);
                if (h < 0 || h >= H) {
                    set_status(status, DV_ERR_DEVICE_INDEX);
                    h = 0;  // a valid row; the result is flagged
                }
                P.uh_s[j] = h;
            }
            __syncwarp();
        }
    }
    // ---- QKV (CTAs 0 .. G-2)
    if (cta < G - 1) {
        const long long U = (long long)3 * nuh * kDH * nseg;
        rows(share(U, cta, G - 1), share(U, cta + 1, G - 1), [&](int q) {
            const int j = q / (3 * kDH), rem = q - j * 3 * kDH;
            const int t = rem / kDH, e = rem - t * kDH;
            return hp(a.w_qkv) + (((size_t)t * H + P.uh_s[j]) * kDH + e) * d;
        });
    }
    // ---- out-projection pieces: rows [q0, q1) of group g's columns
    const int g = cta / a.gm, mem = cta - g * a.gm;
    const GroupCols gcol = group_cols(d, g, a.ncg);
    const int pps = min(16, kStreamStageBytes / (gcol.ncol * 2));
    const uint32_t pb = (uint32_t)gcol.ncol * 2;
    {
        const int RO = nuh * kDH;
        const int q0 = share(RO, mem, a.gm), q1 = share(RO, mem + 1, a.gm);
        for (int q = q0; q < q1 && P.ok; q += pps) {
            const int n = min(pps, q1 - q);
            unsigned char *dst = P.begin(pb * n);
            if (!dst)
                break;
            for (int p = 0; p < n; ++p) {
                const int qq = q + p, j = qq / kDH, e = qq - j * kDH;
                P.copy(dst + (size_t)p * pb,
                       hp(a.w_oT) + ((size_t)P.uh_s[j] * kDH + e) * d + gcol.col0, pb);
            }
            P.end();
        }
    }
    // ---- the neuron union
    int nun = 0;
    if (P.ok) {
        int good = 1;
        if (lane == 0)
            good = poll_ge(a.ctl + kSwNeurons, 1, P.bd) ? 1 : 0;
        P.ok = __shfl_sync(0xffffffffu, good, 0) != 0;
        if (P.ok)
            nun = min(max(__ldcg(a.n_u_n), 0), a.max_u_n);
    }
    auto neuron_row = [&](int i) {
        int jn = P.neuron(i, nun);
        if (jn < 0 || jn >= a.N) {
            if (lane == 0)
                set_status(status, DV_ERR_DEVICE_INDEX);
            jn = 0;
        }
        return jn;
    };
    // ---- FC1
    {
        const long long U = (long long)nun * nseg;
        rows(share(U, cta, G), share(U, cta + 1, G),
             [&](int i) { return hp(a.w1) + (size_t)neuron_row(i) * d; });
    }
    // ---- FC2 pieces
    {
        const int i0 = share(nun, mem, a.gm), i1 = share(nun, mem + 1, a.gm);
        for (int i = i0; i < i1 && P.ok; i += pps) {
            const int n = min(pps, i1 - i);
            unsigned char *dst = P.begin(pb * n);
            if (!dst)
                break;
            for (int p = 0; p < n; ++p) {
                const int jn = neuron_row(i + p);  // every lane (the window is shared)
                P.copy(dst + (size_t)p * pb, hp(a.w2T) + (size_t)jn * d + gcol.col0, pb);
            }
            P.end();
        }
    }
}

// ---------------------------------------------------------------------------
template <int NB, int NI>
__global__ void __launch_bounds__(kStreamThreads, 1)
    k_stream(const __grid_constant__ StreamArgs a)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    uint64_t *empty = full + kStreamMaxStages;
    int *misc = reinterpret_cast<int *>(smem + kOffMisc);
    const int tid = threadIdx.x;
    const size_t ring_off = (size_t)kOffUni + (((size_t)a.uni_bytes + 1023) / 1024) * 1024;

    if (tid == 0) {
        for (int s = 0; s < a.nstages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        misc[kMAbort] = 0;
        const int bus = __ldcg(a.ctl + kSwBudget);
        misc[kMBudget] = bus > 0 ? bus : 50000;  // microseconds
        misc[kMHold] = __ldcg(a.ctl + kSwHold);
    }
    __syncthreads();
    Bound bd;
    bd.budget_ns = (unsigned long long)misc[kMBudget] * 1000ull;
    bd.abort = misc + kMAbort;
    bd.status = a.ctl;
    Ring R;
    R.base = smem + ring_off;
    R.full = full;
    R.empty = empty;
    R.n = a.nstages;
    R.k = 0;

    if (tid < kConsumers) {
        Cons<NB, NI> C{a,      R,   bd,       reinterpret_cast<float *>(smem + kOffRed),
                       misc,   smem + kOffUni, (int)blockIdx.x, tid, tid & 31, tid >> 5, true};
        consumer(C);
    } else {
        Prod P{a,
               R,
               bd,
               reinterpret_cast<int *>(smem + kOffIdx),
               reinterpret_cast<int *>(smem + kOffIdx) + 256,
               0,
               0,
               tid & 31,
               true};
        producer<NB>(P);
        // after a give-up, copies may still be in flight into stages nobody
        // consumes: wait (bounded) for the last ring's worth to land
        if (*bd.abort && (tid & 31) == 0) {
            volatile int never = 0;
            Bound drain = bd;
            drain.abort = &never;
            for (int k = max(0, P.R.k - a.nstages); k < P.R.k; ++k) {
                Ring Q = P.R;
                Q.k = k;
                mbar_wait(&Q.full[Q.slot()], Q.par(), drain);
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        misc[kMLast] = atom_add_acq_rel(a.ctl + kSwExit, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (misc[kMLast]) {
        // every CTA has passed its last wait.  After a give-up the neuron
        // selection may not have cleared its histogram and candidate counts:
        // clear them for the next call.
        if (__ldcg(a.ctl) != 0) {
            for (int i = tid; i < NB * kTopkBins; i += blockDim.x)
                a.hist[i] = 0;
            if (tid < NB)
                a.cand_cnt[tid] = 0;
        }
        __syncthreads();
        if (tid == 0) {
            for (int w = kSwPred1; w < kSwEnd; ++w)
                a.ctl[w] = 0;
            __threadfence();
        }
    }
}

template <int NB, int NI>
cudaError_t launch_t(const StreamArgs &a, size_t smem, cudaStream_t st)
{
    auto kern = k_stream<NB, NI>;
    static DeviceOnce once;
    cudaError_t e = once.run([&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kStreamSmemMax);
    });
    if (e != cudaSuccess)
        return e;
    if (smem > kStreamSmemMax)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.G);
    cfg.blockDim = dim3(kStreamThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int NB, int NI>
int ctas_t(size_t smem)
{
    auto kern = k_stream<NB, NI>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kStreamSmemMax) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kStreamThreads, smem) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace
}  // namespace dv

namespace dv {

size_t stream_smem_bytes(int uni_bytes, int nstages)
{
    return (size_t)kOffUni + (((size_t)uni_bytes + 1023) / 1024) * 1024 +
           (size_t)nstages * kStreamStageBytes;
}

size_t stream_fixed_smem() { return (size_t)kOffUni; }

size_t stream_union_bytes(int B, int N, int max_u_h, int max_u_n, int cg, int gm)
{
    const size_t W = (size_t)(N + 31) / 32;
    size_t u = neuron_final_smem_bytes(N);                       // neuron selection finish
    u = std::max(u, (size_t)B * kTopkBins * 4);                  // score histogram, pass
    u = std::max(u, sizeof(AttnSmem));                           // attention
    u = std::max(u, (size_t)(2 * kHeadKPL + kHeadTopkMax) * 4);  // head selection
    u = std::max(u, (((size_t)max_u_h * kDH + gm - 1) / gm) * B * 4);  // out-proj coefficients
    u = std::max(u, (((size_t)max_u_n + gm - 1) / gm) * B * 4);        // fc2 coefficients
    u = std::max(u, (((size_t)cg + gm - 1) / gm) * B * 4);             // a CTA's h1 slice
    (void)W;
    return u;
}

#define DV_STREAM_SWITCH(F, ...)                                                              \
    switch (nb * 8 + ni) {                                                                    \
    case 9: return F<1, 1>(__VA_ARGS__);                                                      \
    case 10: return F<1, 2>(__VA_ARGS__);                                                     \
    case 11: return F<1, 3>(__VA_ARGS__);                                                     \
    case 12: return F<1, 4>(__VA_ARGS__);                                                     \
    case 17: return F<2, 1>(__VA_ARGS__);                                                     \
    case 18: return F<2, 2>(__VA_ARGS__);                                                     \
    case 19: return F<2, 3>(__VA_ARGS__);                                                     \
    case 20: return F<2, 4>(__VA_ARGS__);                                                     \
    default: break;                                                                           \
    }

cudaError_t launch_stream(int nb, int ni, const StreamArgs &a, size_t smem, cudaStream_t st)
{
    DV_STREAM_SWITCH(launch_t, a, smem, st)
    return cudaErrorInvalidValue;
}

int stream_ctas_per_sm(int nb, int ni, size_t smem)
{
    DV_STREAM_SWITCH(ctas_t, smem)
    return 0;
}

}  // namespace dv
