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
//  * One CTA per SM, 13 warps.  Warp 12 is the PRODUCER: its lane 0 walks the
//    CTA's share of every phase's weight rows in order and copies them with
//    1-D bulk copies (cp.async.bulk, completion counted on an mbarrier) into
//    a ring of 32 KB stages in shared memory.  The addresses depend only on
//    the selections, which are known early (heads after the first predictor
//    stage, neurons before QKV ends), so the producer runs ahead of the
//    computation by up to the whole ring (160 KB per SM, ~3.5 us of the SM's
//    share of HBM bandwidth) -- across the phase boundaries where the
//    consumers wait for each other.
//  * Warps 0-11 are CONSUMERS (13 warps keep at most four on an SM
//    sub-partition, so a thread may hold 128 registers).  Each thread owns fixed 16-byte chunks of a
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
//         x_pred; row segments of 384 chunks are dealt to all CTAs, each
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
constexpr int kSeg = kStreamUnitBytes / 16;  // chunks of a row segment (one per consumer thread)
static_assert(kSeg == kConsumers, "thread t of the consumers takes chunk t of a segment");
constexpr int kRU = 32;               // row-dot segments per batch of partial sums
constexpr int kNR = 4;                // u chunks per lane in PRED2 (rank <= 1024)
constexpr int kNJ = 6;                // columns a consumer thread owns per group (<= 2048 / 384)
constexpr int kDH = 128;              // head dimension served
constexpr int kIdxCache = 1024;       // producer: cached neuron-union entries per mlp phase
constexpr int kUnitsPerStage = 8;     // row segments a stage holds at most
constexpr int kPfAhead = 0;  // producer: L2 prefetch this far past the ring (bytes)

// Fixed part of the dynamic shared memory.
constexpr int kOffBar = 0;     // full[16], empty[16]
constexpr int kOffMisc = 256;  // ints, see the kM* indices (128), then [2][kRU] segment ids
constexpr int kOffRed = 1024;  // [2][kRU][kCW][2] floats
constexpr int kOffIdx = kOffRed + 2 * kRU * kCW * 2 * 4;  // producer: u_h[256], u_n caches
constexpr int kOffUni = kOffIdx + (256 + 2 * kIdxCache) * 4;  // phase scratch
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
constexpr int kOffUid = 4 * 128;  // misc byte offset of [2][kRU] row-dot segment ids (ints)

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
// The same with a suspend-time hint: a thread whose phase is not complete
// sleeps (up to the hint, in ns) instead of spinning.
DV_DEV bool mbar_try_wait_sleep(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity), "r"(100000u)
        : "memory");
    return ok != 0;
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
// Fetch `bytes` (a multiple of 16, 16-byte aligned) from global memory into L2.
DV_DEV void prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
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
        if (mbar_try_wait_sleep(b, parity))
            return true;
        if ((it & 15) == 15) {
            if (*bd.abort)
                return false;
            if (global_ns() - t0 > bd.budget_ns) {
                give_up(bd);
                return false;
            }
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

// Consumer warp: wait for the next stage (nullptr: the CTA gave up).
DV_DEV const unsigned char *cons_acquire(Ring &R, const Bound &bd)
{
    // lane 0 polls (one thread per warp, not 32, touches the barrier while
    // the copy lands); then every lane checks the completed phase once, so
    // that its own reads are ordered after the copy
    int good = 1;
    if ((threadIdx.x & 31) == 0)
        good = mbar_wait(&R.full[R.slot()], R.par(), bd) ? 1 : 0;
    if (!__shfl_sync(0xffffffffu, good, 0))
        return nullptr;
    const bool seen = mbar_try_wait(&R.full[R.slot()], R.par());
    if (!__all_sync(0xffffffffu, seen))
        return nullptr;  // cannot happen once lane 0 saw the phase complete
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
// Work split helpers (the producer and the consumers derive the same ranges
// and the same stage packing).
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

// Row segments: unit u is segment u % nseg of row u / nseg (384 chunks of 16
// bytes, the last one of a row shorter).
DV_DEV int seg_chunks(int seg, int cpr) { return min(kSeg, cpr - seg * kSeg); }
// Rows of pred_b a stage holds, and column pieces a stage holds.
DV_DEV int pred2_rows_per_stage(int r)
{
    const int fit = kStreamStageBytes / (r * 2);
    return fit >= kCW ? fit / kCW * kCW : fit;  // whole rounds of the consumer warps
}
DV_DEV int pieces_per_stage(int ncol) { return min(16, kStreamStageBytes / (ncol * 2)); }

// Sum of n <= kMaxSeg segment partials p[0 .. n), added in order; the loads
// are issued together (they are independent), not one round trip after
// another.
constexpr int kMaxSeg = 6;
DV_DEV float sum_segs(const float *p, int n)
{
    float v[kMaxSeg];
#pragma unroll
    for (int q = 0; q < kMaxSeg; ++q)
        v[q] = q < n ? __ldcg(p + q) : 0.f;
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < kMaxSeg; ++q)
        if (q < n)
            s += v[q];
    return s;
}

// Phase timeline (optional): globaltimer at point i of this CTA.
DV_DEV void stamp(const StreamArgs &a, int i)
{
    if (a.stamps && (threadIdx.x == 0 || threadIdx.x == kConsumers))
        a.stamps[(size_t)blockIdx.x * kStreamStamps + i] = global_ns();
}

// ---------------------------------------------------------------------------
// Kernel context shared by the consumer functions.
template <int NB, int NI>
struct Cons {
    const StreamArgs &a;
    Ring R;
    Bound bd;
    float *red;       // [2][kRU][kCW][NB]
    int *misc;
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

    // The group (the consumer threads) arrives at control word w, whether or
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
// Row-dot phases.  A CTA's share of a phase is a contiguous range [u0, u1) of
// row segments (unit u = segment u % nseg of row u / nseg), taken
// SEGMENT-MAJOR: all its rows' segment 0, then segment 1, ...  A consumer
// thread then needs the activations of one segment at a time (8 values per
// batch row, the chunk it owns), plus the next segment's, loaded early.
// Within a segment a stage holds up to seg_units() consecutive rows.

// Rows [*ra, *rb] of segment s in the range [u0, u1) (*rb < *ra: none).
DV_DEV void seg_rows(int u0, int u1, int nseg, int s, int *ra, int *rb)
{
    if (u1 <= u0) {
        *ra = 0;
        *rb = -1;
        return;
    }
    const int r0 = u0 / nseg, s0 = u0 - r0 * nseg;
    const int r1 = (u1 - 1) / nseg, s1 = (u1 - 1) - r1 * nseg;
    *ra = r0 + (s < s0 ? 1 : 0);
    *rb = r1 - (s > s1 ? 1 : 0);
}
// Units of segment s a stage holds.
DV_DEV int seg_units(int s, int cpr)
{
    return min(kUnitsPerStage, kStreamStageBytes / (seg_chunks(s, cpr) * 16));
}

// Where a row segment's activations come from: rows src[b * ld ..] of
// binary32, optionally normalised per batch row with (mean, rstd), gain g and
// bias beta (binary16; beta NULL: none).
template <int NB>
struct ActSrc {
    const float *x;
    int ld;
    bool coherent;  // written by this kernel: read at L2
    bool norm;
    float mean[NB], rstd[NB];
    const __half *g, *beta;
};

// Activation chunk c (8 values per batch row) into v; zero past the row.
template <int NB>
DV_DEV void load_chunk(const ActSrc<NB> &A, int c, int cpr, float (&v)[NB][8])
{
    const bool in = c < cpr;
    float gf[8], bf[8];
    if (A.norm) {
        Elem<__half>::unpack(in ? *reinterpret_cast<const uint4 *>(A.g + (size_t)c * 8)
                                : make_uint4(0u, 0u, 0u, 0u),
                             gf);
        Elem<__half>::unpack((in && A.beta)
                                 ? *reinterpret_cast<const uint4 *>(A.beta + (size_t)c * 8)
                                 : make_uint4(0u, 0u, 0u, 0u),
                             bf);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
        if (in) {
            const float4 *p = reinterpret_cast<const float4 *>(A.x + (size_t)b * A.ld + c * 8);
            lo = A.coherent ? __ldcg(p) : p[0];
            hi = A.coherent ? __ldcg(p + 1) : p[1];
        }
        const float t[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
            v[b][e] = (A.norm && in) ? (t[e] - A.mean[b]) * A.rstd[b] * gf[e] + bf[e] : t[e];
    }
}

// Sum of each of the 8 values v[q] over the warp: lane l ends with the total
// of value (l >> 2) & 7 (a butterfly that halves the values a lane keeps at
// each of the first three steps: 9 shuffles instead of 40).  Fixed pairing,
// so the result does not depend on scheduling.
DV_DEV float warp_sum8(const float (&v)[8], int lane)
{
    const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4;
    float w[4], x[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = h4 ? v[i] : v[i + 4];
        w[i] = (h4 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = h3 ? w[i] : w[i + 2];
        x[i] = (h3 ? w[i + 2] : w[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    const float send = h2 ? x[0] : x[1];
    float y = (h2 ? x[1] : x[0]) + __shfl_xor_sync(0xffffffffu, send, 4);
    y += __shfl_xor_sync(0xffffffffu, y, 2);
    y += __shfl_xor_sync(0xffffffffu, y, 1);
    return y;
}

// Row-dot stages of this CTA's row segments [u0, u1): thread t multiplies
// chunk t of each segment of a stage with its activations, the stage's
// segments are summed over the warp together (warp_sum8), and the warps'
// sums go to `red`; once more than kRU - kUnitsPerStage segments are
// pending, the group adds the kCW warp sums of each in warp order and stores
// part[b * bstride + segment].
template <int NB, int NI>
DV_DEV bool rowdot_stages(Cons<NB, NI> &C, int u0, int u1, int nseg, int cpr,
                          const ActSrc<NB> &A, float *part, long long bstride)
{
    static_assert(kUnitsPerStage == 8, "warp_sum8 reduces one stage");
    const int tid = C.tid, lane = C.lane, warp = C.warp;
    int *uid = reinterpret_cast<int *>(reinterpret_cast<unsigned char *>(C.misc) + kOffUid);
    int nb = 0, buf = 0;
    auto flush = [&]() {
        ConsumerGroup::sync();
        for (int i = tid; i < nb * NB; i += kConsumers) {
            const int q = i / NB, b = i - q * NB;
            float s = 0.f;
#pragma unroll
            for (int w = 0; w < kCW; ++w)
                s += C.red[((buf * kRU + q) * kCW + w) * NB + b];
            part[(size_t)b * bstride + uid[buf * kRU + q]] = s;
        }
    };
    float cur[NB][8], nxt[NB][8];
    load_chunk(A, tid, cpr, cur);
    for (int sg = 0; sg < nseg; ++sg) {
        if (sg + 1 < nseg)  // the next segment's chunk, in flight meanwhile
            load_chunk(A, tid + (sg + 1) * kConsumers, cpr, nxt);
        int ra, rb;
        seg_rows(u0, u1, nseg, sg, &ra, &rb);
        const int nch = seg_chunks(sg, cpr), ups = seg_units(sg, cpr);
        for (int row = ra; row <= rb; row += ups) {
            const int n = min(ups, rb - row + 1);
            const unsigned char *st = C.ok ? cons_acquire(C.R, C.bd) : nullptr;
            if (!st)
                C.ok = false;  // this warp skips the data from here on
            float acc[NB][8];
            uint4 wv[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)  // all of the stage's loads first
                wv[q] = (st && q < n && tid < nch)
                            ? *reinterpret_cast<const uint4 *>(st + q * nch * 16 + tid * 16)
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float f[8];
                Elem<__half>::unpack(wv[q], f);
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    float sv = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        sv = fmaf(f[e], cur[b][e], sv);
                    acc[b][q] = sv;
                }
            }
            if (st)  // every loaded value has been used: the slot can refill
                cons_release(C.R);
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                const float sum = warp_sum8(acc[b], lane);
                const int q = (lane >> 2) & 7;
                if ((lane & 3) == 0 && q < n)
                    C.red[((buf * kRU + nb + q) * kCW + warp) * NB + b] = sum;
            }
            if (tid < n)
                uid[buf * kRU + nb + tid] = (row + tid) * nseg + sg;
            nb += n;
            if (nb > kRU - kUnitsPerStage) {  // uniform: the same on every path
                flush();
                nb = 0;
                buf ^= 1;
            }
        }
        if (sg + 1 < nseg)
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    cur[b][e] = nxt[b][e];
    }
    if (nb)
        flush();
    C.agree();
    return C.ok;
}

// LayerNorm / RMSNorm statistics of rows src[b * ld ..] (binary32, length d)
// over the consumer group: every chunk's loads issued together, then two
// passes over the registers (the mean, then the squared deviations from it).
// mean[b] is 0 for RMSNorm (rstd then from the mean square).

template <int NB, int NI>
DV_DEV void row_stats(Cons<NB, NI> &C, const float *src, int ld, bool coherent, int d,
                      float (&mean)[NB], float (&rstd)[NB])
{
    const int cpr = d / 8, tid = C.tid;
    const bool ln = C.a.norm_kind == DV_LAYERNORM;
    float *scr = reinterpret_cast<float *>(C.misc + kMScr);
    ActSrc<NB> A;
    A.x = src;
    A.ld = ld;
    A.coherent = coherent;
    A.norm = false;
    A.g = A.beta = nullptr;
    float v[NI][NB][8];
#pragma unroll
    for (int i = 0; i < NI; ++i)  // every chunk's loads in flight together
        load_chunk(A, tid + i * kConsumers, cpr, v[i]);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                s += v[i][b][e];
        const float mu = ln ? block_sum<ConsumerGroup>(s, scr) / (float)d : 0.f;
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
            if (tid + i * kConsumers < cpr)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float t = v[i][b][e] - mu;
                    ss = fmaf(t, t, ss);
                }
        }
        mean[b] = mu;
        rstd[b] = rsqrtf(block_sum<ConsumerGroup>(ss, scr) / (float)d + C.a.eps);
    }
}

// Column stages: rows [q0, q1) of the CTA's column group, pps pieces of cg
// binary16 columns per stage; coef[(q - q0) * NB + b] in shared memory.
// Thread t accumulates columns t + 384 j of the group.
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
    int k = 0;
    for (int q = q0; q < q1; q += pps, ++k) {
        // every 4th stage the consumer warps meet: warps that drift apart
        // over the ring starve it (measured: ~2 TB/s without, ~5.7 with)
        if ((k & 3) == 3)
            ConsumerGroup::sync();
        const unsigned char *st = C.ok ? cons_acquire(C.R, C.bd) : nullptr;
        if (!st) {
            C.ok = false;  // this warp skips the data from here on (same barriers)
            continue;
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

// Not inlined: its registers (two batches of K and V rows in flight) are its
// own, not added to those the rest of the consumer code keeps live.
__device__ __noinline__ void attn_unit(const StreamArgs &a, unsigned char *uni, int b, int j,
                                       int c, int h)
{
    AttnSmem &S = *reinterpret_cast<AttnSmem *>(uni);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nseg = a.nseg, L = a.kv_len, L1 = L + 1, Ch = a.attn_C;
    const __half *bq = static_cast<const __half *>(a.b_qkv);
    const bool last = c == Ch - 1;
    // q, and the new k, v (threads 0..383: type t = tid / 128, element e)
    if (tid < (last ? 3 : 1) * kDH) {
        const int t = tid / kDH, e = tid - t * kDH;
        const long long row = (long long)j * 3 * kDH + t * kDH + e;
        const float *pp = a.partQ + (size_t)b * 3 * a.max_u_h * kDH * nseg + row * nseg;
        float s = sum_segs(pp, nseg);
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

// Attention merge, step 1: for head slot j of batch row b, the weight of
// each chunk record c: exp(m_c - M) / sum_c' exp(m_c' - M) l_c'.
DV_DEV void attn_chunk_weights(const StreamArgs &a, int b, int j, float *wgt)
{
    const int Ch = a.attn_C, rec = kAttnRec + kDH;
    const float *r = a.attn_rec + ((size_t)b * a.max_u_h + j) * Ch * rec;
    for (int c = 0; c < Ch; ++c)  // independent loads: (m_c, l_c) into the output first
        wgt[c] = __ldcg(r + (size_t)c * rec);
    float M = -INFINITY;
    for (int c = 0; c < Ch; ++c)
        M = fmaxf(M, wgt[c]);
    float Ls = 0.f;
    for (int c = 0; c < Ch; ++c)
        if (wgt[c] != -INFINITY)
            Ls = fmaf(__ldcg(r + (size_t)c * rec + 1), expf(wgt[c] - M), Ls);
    for (int c = 0; c < Ch; ++c)
        wgt[c] = wgt[c] == -INFINITY ? 0.f : expf(wgt[c] - M) / Ls;
}

// Step 2: o[b][j][e] = sum_c wgt[c] o_c[e] (the chunks' loads in flight together).
DV_DEV float attn_merge(const StreamArgs &a, int b, int j, int e, const float *wgt)
{
    const int Ch = a.attn_C, rec = kAttnRec + kDH;
    const float *r = a.attn_rec + ((size_t)b * a.max_u_h + j) * Ch * rec + kAttnRec + e;
    float s = 0.f;
    for (int c0 = 0; c0 < Ch; c0 += 8) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
            v[u] = c0 + u < Ch ? __ldcg(r + (size_t)(c0 + u) * rec) : 0.f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
            if (c0 + u < Ch)
                s = fmaf(wgt[c0 + u], v[u], s);
    }
    return s;
}

// ---------------------------------------------------------------------------
// Column-group reduction: the CTA (group g, member m) adds the group's gm
// partials for its slice of the group's columns, in member order, plus
// res + bias, and writes out[b][col].
template <int NB, int NI>
DV_DEV void group_reduce(Cons<NB, NI> &C, const float *part, const float *res, bool res_coherent,
                         const __half *bias, float *out)
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
        for (int m0 = 0; m0 < a.gm; m0 += 16) {  // sixteen members' loads in flight, added in order
            float v[16];
#pragma unroll
            for (int u = 0; u < 16; ++u)
                v[u] = m0 + u < a.gm
                           ? __ldcg(part + ((size_t)(g * a.gm + m0 + u) * NB + b) * a.cg + s0 + cc)
                           : 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (m0 + u < a.gm)
                    s += v[u];
        }
        const float rv = res_coherent ? __ldcg(res + (size_t)b * a.d + col) : res[(size_t)b * a.d + col];
        const float v = rv + __half2float(bias[col]) + s;
        out[(size_t)b * a.d + col] = v;
    }
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

    // ---- LN1 statistics of x now (while the first stages arrive), then
    // PRED1: head scores and u on x_pred
    stamp(a, 0);
    float mean1[NB], rstd1[NB];
    {
        ActSrc<NB> A;
        A.x = a.x_pred;
        A.ld = d;
        A.coherent = false;
        A.norm = false;
        A.g = A.beta = nullptr;
        const long long U = (long long)rows1 * nseg;
        rowdot_stages(C, share(U, cta, G), share(U, cta + 1, G), nseg, cpr, A, a.part1,
                      (long long)rows1 * nseg);
    }
    stamp(a, 1);
    const int before = C.arrive(kSwPred1, true);
    // LN1 statistics of x, beside the hand-off to the second predictor stage
    row_stats(C, a.x, d, false, d, mean1, rstd1);
    if (before == G - 1 && C.warp == 0) {
        // the last CTA to finish: head scores from the segment sums (into
        // shared memory), then the head selection (skipped if the CTA gave
        // up; the flag is raised either way so that no CTA waits in vain)
        if (C.ok) {
            float *sh = reinterpret_cast<float *>(C.uni);            // [NB][H]
            unsigned *hb = reinterpret_cast<unsigned *>(sh + NB * kHeadTopkMax);
            int32_t *hs = reinterpret_cast<int32_t *>(hb + 2 * kHeadKPL);
            for (int i = C.lane; i < NB * H; i += 32) {
                const int b = i / H, hh = i - b * H;
                sh[i] = sum_segs(a.part1 + (size_t)b * rows1 * nseg + (size_t)hh * nseg, nseg);
            }
            __syncwarp();
            head_select<true>(sh, NB, H, a.k_h, hb, hs, true, a.idx_h, a.u_h, a.n_u_h, C.lane);
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
        stamp(a, 2);
        const int rc = a.r / 8;
        // u = the segment sums of the pred_a rows, once per CTA into shared
        // memory (after the histogram), then each lane's chunks into registers
        float *us = reinterpret_cast<float *>(shist + NB * kTopkBins);  // [NB][r]
        for (int i = tid; i < NB * a.r; i += kConsumers) {
            const int b = i / a.r, q = i - b * a.r;
            us[i] = sum_segs(a.part1 + (size_t)b * rows1 * nseg + (size_t)(H + q) * nseg, nseg);
        }
        for (int i = tid; i < NB * kTopkBins; i += kConsumers)
            shist[i] = 0;
        ConsumerGroup::sync();
        float ua[kNR][NB][8];
#pragma unroll
        for (int i = 0; i < kNR; ++i) {
            const int c = C.lane + 32 * i;
#pragma unroll
            for (int b = 0; b < NB; ++b)
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    ua[i][b][e] = c < rc ? us[b * a.r + c * 8 + e] : 0.f;
        }
        stamp(a, 3);
        const int j0 = share(a.N, cta, G), j1 = share(a.N, cta + 1, G);
        const int rps = pred2_rows_per_stage(a.r);
        bool wok = true;
        int k = 0;
        for (int j = j0; j < j1; j += rps, ++k) {
            if ((k & 3) == 3)  // keep the consumer warps together (see column_stages)
                ConsumerGroup::sync();
            const unsigned char *st = wok ? cons_acquire(C.R, C.bd) : nullptr;
            if (!st) {
                wok = false;  // same barriers, no data
                continue;
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
    stamp(a, 4);
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
    stamp(a, 5);
    C.arrive(kSwPass);

    // ---- the head union, LN1(x), QKV (CTAs 0 .. G-2)
    const int nuh = C.ok ? C.flag_count(kSwHeads, a.n_u_h, a.max_u_h) : 0;
    if (cta < G - 1) {
        if (C.ok) {
            ActSrc<NB> A;
            A.x = a.x;
            A.ld = d;
            A.coherent = false;
            A.norm = true;
            for (int b = 0; b < NB; ++b) {
                A.mean[b] = mean1[b];
                A.rstd[b] = rstd1[b];
            }
            A.g = g1;
            A.beta = ln ? be1 : nullptr;
            stamp(a, 6);
            const long long U = (long long)3 * nuh * kDH * nseg;
            rowdot_stages(C, share(U, cta, G - 1), share(U, cta + 1, G - 1), nseg, cpr, A,
                          a.partQ, (long long)3 * a.max_u_h * kDH * nseg);
        }
        stamp(a, 7);
        C.arrive(kSwQkv);
        // ---- attention units (batch row, head slot, chunk) over CTAs 0 .. G-2
        if (C.ok && C.wait(kSwQkv, G - 1, 4)) {
            stamp(a, 8);
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
                attn_unit(a, C.uni, b, j, c, h);
            }
        }
        stamp(a, 9);
        C.arrive(kSwAttn);
    } else {
        // the last CTA takes no QKV rows and no attention: it finishes the
        // neuron selection beside them (the flag is raised either way)
        C.arrive(kSwAttn);
        if (C.ok && C.wait(kSwPass, G, 3)) {
            stamp(a, 6);
            neuron_final<ConsumerGroup>(ns, final_smem(C.uni, a.N, misc + kMScr));
            stamp(a, 7);
        }
        ConsumerGroup::sync();
        if (tid == 0) {
            __threadfence();
            st_release_gpu(C.ctl(kSwNeurons), 1);
        }
    }

    // ---- out-projection: coefficients (merged attention records), columns
    const int g = cta / a.gm, mem = cta - g * a.gm;
    const GroupCols gcol = group_cols(d, g, a.ncg);
    const int pps = pieces_per_stage(gcol.ncol);
    float acc[kNJ][NB];
    int nun = 0;
    if (C.ok && C.wait(kSwAttn, G, 5)) {
        stamp(a, 10);
        // the neuron union (published beside QKV) for fc1 and fc2
        nun = C.flag_count(kSwNeurons, a.n_u_n, a.max_u_n);
        const int RO = nuh * kDH;
        const int q0 = share(RO, mem, a.gm), q1 = share(RO, mem + 1, a.gm);
        float *coef = reinterpret_cast<float *>(C.uni);
        // chunk weights of the head slots [j0, j1] this CTA's rows touch
        const int j0 = q0 / kDH, nj = q1 > q0 ? (q1 - 1) / kDH - j0 + 1 : 0;
        float *wgt = coef + (size_t)(q1 - q0) * NB;  // [nj][NB][kMaxAttnChunks]
        for (int i = tid; i < nj * NB; i += kConsumers)
            attn_chunk_weights(a, i % NB, j0 + i / NB, wgt + (size_t)i * kMaxAttnChunks);
        ConsumerGroup::sync();
        for (int i = tid; i < (q1 - q0) * NB; i += kConsumers) {
            const int qq = i / NB, b = i - qq * NB;
            const int q = q0 + qq, j = q / kDH;
            coef[i] = attn_merge(a, b, j, q - j * kDH,
                                 wgt + ((size_t)(j - j0) * NB + b) * kMaxAttnChunks);
        }
        ConsumerGroup::sync();
        stamp(a, 11);
        if (C.ok && column_stages(C, q0, q1, pps, gcol.ncol, coef, acc)) {
            for (int j = 0; j < kNJ; ++j) {
                const int col = tid + j * kConsumers;
                if (col < gcol.ncol)
                    for (int b = 0; b < NB; ++b)
                        a.partO[((size_t)cta * NB + b) * a.cg + col] = acc[j][b];
            }
        }
    }
    stamp(a, 12);
    C.arrive(kSwOproj + g);

    // ---- h1 on this CTA's slice of its group's columns
    if (C.ok && C.wait(kSwOproj + g, a.gm, 6)) {
        stamp(a, 13);
        group_reduce(C, a.partO, a.x, false, static_cast<const __half *>(a.b_o), a.h1);
    }
    stamp(a, 14);
    C.arrive(kSwNorm2);

    // ---- LN2 of the whole h1 (every CTA reads it), fc1
    if (C.ok && C.wait(kSwNorm2, G, 7)) {
        stamp(a, 15);
        ActSrc<NB> A;
        A.x = a.h1;
        A.ld = d;
        A.coherent = true;
        A.norm = true;
        row_stats(C, a.h1, d, true, d, A.mean, A.rstd);
        A.g = g2;
        A.beta = ln ? be2 : nullptr;
        stamp(a, 16);
        const long long U = (long long)nun * nseg;
        rowdot_stages(C, share(U, cta, G), share(U, cta + 1, G), nseg, cpr, A, a.partF,
                      (long long)a.max_u_n * nseg);
    }
    stamp(a, 17);
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
            const float s =
                sum_segs(a.partF + (size_t)b * a.max_u_n * nseg + (size_t)row * nseg, nseg);
            const float bias = (jn >= 0 && jn < a.N) ? __half2float(b1[jn]) : 0.f;
            coef[i] = fmaxf(s + bias, 0.f);
        }
        ConsumerGroup::sync();
        stamp(a, 18);
        if (column_stages(C, i0, i1, pps, gcol.ncol, coef, acc)) {
            for (int j = 0; j < kNJ; ++j) {
                const int col = tid + j * kConsumers;
                if (col < gcol.ncol)
                    for (int b = 0; b < NB; ++b)
                        a.partY[((size_t)cta * NB + b) * a.cg + col] = acc[j][b];
            }
        }
    }
    stamp(a, 19);
    C.arrive(kSwFc2 + g);
    if (C.ok && C.wait(kSwFc2 + g, a.gm, 9)) {
        stamp(a, 20);
        group_reduce(C, a.partY, a.h1, true, static_cast<const __half *>(a.b2), a.y);
    }
    stamp(a, 21);
}

// ---------------------------------------------------------------------------
// Producer: warp 12 walks the CTA's units of every phase in the consumers'
// order.  Lane 0 issues the stages' bulk copies (contiguous units merged into
// one copy) and, a ring's worth further on, L2 prefetches of the units that
// follow (kPfAhead bytes), so that HBM keeps streaming while the consumers
// wait at a phase hand-off for longer than the ring covers.  The other lanes
// share the index loads; every lane runs the same control flow.
enum Phase { kPhPred1 = 0, kPhPred2, kPhQkv, kPhOproj, kPhFc1, kPhFc2, kPhEnd };

DV_DEV const __half *hp(const void *p) { return static_cast<const __half *>(p); }

struct Prod {
    const StreamArgs &a;
    Ring R;
    Bound bd;
    int *uh_s;   // [256] head union
    int *un_s;   // [2][kIdxCache] neuron-union entries of this CTA's fc1 / fc2 rows
    int lane;
    bool ok;
    int cta, g, mem;
    GroupCols gcol;
    bool heads, neurons;  // union known, caches loaded
    int nuh, nun;
    int un_base0, un_cnt0, un_base1, un_cnt1;  // cached neuron-union entries: fc1, fc2 rows
    long long cp_bytes;   // bytes the copy cursor has issued
    long long pf_bytes;   // bytes of the units the prefetch cursor has passed
    int pf_ph;
    int pf_u, pf_u1;      // prefetch cursor: next unit, end of its phase's range (-1: not set)
    int stages;           // stages issued

    // Unit range [*u0, *u1) of phase ph for this CTA.
    DV_DEV void range(int ph, int *u0, int *u1) const
    {
        const int G = a.G, nseg = a.nseg;
        long long U = 0;
        int part = cta, parts = G;
        switch (ph) {
        case kPhPred1: U = (long long)(a.H + a.r) * nseg; break;
        case kPhPred2: {  // row blocks of a stage each
            const int j0 = share(a.N, cta, G), j1 = share(a.N, cta + 1, G);
            const int rps = pred2_rows_per_stage(a.r);
            *u0 = 0;
            *u1 = (j1 - j0 + rps - 1) / rps;
            return;
        }
        case kPhQkv:
            if (cta >= G - 1) {
                *u0 = *u1 = 0;
                return;
            }
            U = (long long)3 * nuh * kDH * nseg;
            parts = G - 1;
            break;
        case kPhOproj: U = (long long)nuh * kDH; part = mem; parts = a.gm; break;
        case kPhFc1: U = (long long)nun * nseg; break;
        case kPhFc2: U = nun; part = mem; parts = a.gm; break;
        default: *u0 = *u1 = 0; return;
        }
        *u0 = share(U, part, parts);
        *u1 = share(U, part + 1, parts);
    }

    // Neuron-union entry i of an mlp phase (which: 0 fc1, 1 fc2): from the
    // cache, else (cached_only) -1, else from global memory.
    DV_DEV int neuron_at(int which, int i, bool cached_only) const
    {
        const int o = i - (which ? un_base1 : un_base0);
        int jn;
        if (o >= 0 && o < (which ? un_cnt1 : un_cnt0))
            jn = un_s[which * kIdxCache + o];
        else if (cached_only)
            return -1;
        else
            jn = __ldcg(a.u_n + i);
        return (jn >= 0 && jn < a.N) ? jn : 0;  // out of range: flagged when the union is loaded
    }

    // Row `row`'s start in a row-dot phase (false: not available to the
    // prefetch cursor without a global load).
    DV_DEV bool row_start(int ph, int row, const __half **p, bool cached_only = false) const
    {
        const int d = a.d, H = a.H;
        switch (ph) {
        case kPhPred1:
            *p = row < H ? hp(a.pred_h) + (size_t)row * d : hp(a.pred_a) + (size_t)(row - H) * d;
            return true;
        case kPhQkv: {
            const int j = row / (3 * kDH), rem = row - j * 3 * kDH;
            const int t = rem / kDH, e = rem - t * kDH;
            *p = hp(a.w_qkv) + (((size_t)t * H + uh_s[j]) * kDH + e) * d;
            return true;
        }
        case kPhFc1: {
            const int jn = neuron_at(0, row, cached_only);
            if (jn < 0)
                return false;
            *p = hp(a.w1) + (size_t)jn * d;
            return true;
        }
        default: return false;
        }
    }

    // Source and size of unit u of phase ph (false: not available to the
    // prefetch cursor without a global load).  Row-dot phases count their
    // units segment-major (the consumers' order).
    DV_DEV bool unit(int ph, int u, const void **src, uint32_t *bytes,
                     bool cached_only = false) const
    {
        const int d = a.d, cpr = d / 8, nseg = a.nseg;
        switch (ph) {
        case kPhPred1:
        case kPhQkv:
        case kPhFc1: {
            int u0, u1, sg = 0, row = -1;
            range(ph, &u0, &u1);
            for (; sg < nseg; ++sg) {  // segment-major: find u's segment and row
                int ra, rb;
                seg_rows(u0, u1, nseg, sg, &ra, &rb);
                const int cnt = max(0, rb - ra + 1);
                if (u < cnt) {
                    row = ra + u;
                    break;
                }
                u -= cnt;
            }
            const __half *p;
            if (row < 0 || !row_start(ph, row, &p, cached_only))
                return false;
            *src = p + (size_t)sg * kSeg * 8;
            *bytes = (uint32_t)seg_chunks(sg, cpr) * 16;
            return true;
        }
        case kPhPred2: {
            const int j0 = share(a.N, cta, a.G), j1 = share(a.N, cta + 1, a.G);
            const int rps = pred2_rows_per_stage(a.r);
            const int j = j0 + u * rps, n = min(rps, j1 - j);
            *src = hp(a.pred_b) + (size_t)j * a.r;
            *bytes = (uint32_t)n * a.r * 2;
            return true;
        }

        case kPhOproj: {
            const int j = u / kDH, e = u - j * kDH;
            *src = hp(a.w_oT) + ((size_t)uh_s[j] * kDH + e) * d + gcol.col0;
            *bytes = (uint32_t)gcol.ncol * 2;
            return true;
        }

        case kPhFc2: {
            const int jn = neuron_at(1, u, cached_only);
            if (jn < 0)
                return false;
            *src = hp(a.w2T) + (size_t)jn * d + gcol.col0;
            *bytes = (uint32_t)gcol.ncol * 2;
            return true;
        }
        default: return false;
        }
    }

    // The head union into shared memory (warp-wide; after its flag).
    DV_DEV void load_heads()
    {
        nuh = min(max(__ldcg(a.n_u_h), 0), a.max_u_h);
        for (int j = lane; j < nuh; j += 32) {
            int h = __ldcg(a.u_h + j);
            if (h < 0 || h >= a.H) {
                set_status(a.ctl, DV_ERR_DEVICE_INDEX);
                h = 0;  // a valid row; the result is flagged
            }
            uh_s[j] = h;
        }
        __syncwarp();
        heads = true;
    }
    // The neuron union entries of this CTA's fc1 and fc2 rows (warp-wide).
    DV_DEV void load_neurons()
    {
        nun = min(max(__ldcg(a.n_u_n), 0), a.max_u_n);
        int u0, u1;
        range(kPhFc1, &u0, &u1);
        un_base0 = u0 / a.nseg;
        un_cnt0 = u1 > u0 ? min((u1 - 1) / a.nseg - u0 / a.nseg + 1, kIdxCache) : 0;
        range(kPhFc2, &u0, &u1);
        un_base1 = u0;
        un_cnt1 = min(u1 - u0, kIdxCache);
        for (int w = 0; w < 2; ++w) {
            const int base = w ? un_base1 : un_base0, cnt = w ? un_cnt1 : un_cnt0;
            for (int q = lane; q < cnt; q += 32) {
                const int jn = __ldcg(a.u_n + base + q);
                if (jn < 0 || jn >= a.N)
                    set_status(a.ctl, DV_ERR_DEVICE_INDEX);
                un_s[w * kIdxCache + q] = jn;
            }
        }
        __syncwarp();
        neurons = true;
    }
    // Blocking: wait for a union's flag, then load it (false: gave up).
    DV_DEV bool ensure(bool need_heads)
    {
        if (need_heads ? heads : neurons)
            return true;
        int good = 1;
        if (lane == 0)
            good = poll_ge(a.ctl + (need_heads ? kSwHeads : kSwNeurons), 1, bd) ? 1 : 0;
        ok = ok && __shfl_sync(0xffffffffu, good, 0) != 0;
        if (!ok)
            return false;
        if (need_heads)
            load_heads();
        else
            load_neurons();
        return true;
    }
    // Non-blocking: load a union if its flag is already up.
    DV_DEV bool try_resolve(bool need_heads)
    {
        if (need_heads ? heads : neurons)
            return true;
        int up = 0;
        if (lane == 0)
            up = ld_acquire_gpu(a.ctl + (need_heads ? kSwHeads : kSwNeurons));
        if (!__shfl_sync(0xffffffffu, up, 0))
            return false;
        if (need_heads)
            load_heads();
        else
            load_neurons();
        return true;
    }

    // Advance the prefetch cursor: units between the ring's end and kPfAhead
    // further are fetched into L2 (once each), 32 at a time, a lane each.
    DV_DEV void prefetch_run(long long ring_bytes)
    {
        if constexpr (kPfAhead == 0)
            return;
        const long long lo = cp_bytes + ring_bytes, hi = lo + kPfAhead;
        bool tried = false;
        while (pf_ph < kPhEnd && pf_bytes < hi) {
            if (pf_ph >= kPhQkv) {
                const bool need_heads = pf_ph < kPhFc1;
                if (!(need_heads ? heads : neurons)) {
                    // an L2 round trip: at most one look per call, every 8th stage
                    if (tried || (stages & 7) != 0 || !try_resolve(need_heads))
                        return;
                    tried = true;
                }
            }
            if (pf_u1 < 0) {  // entering the phase (row-dot units: indices from 0)
                range(pf_ph, &pf_u, &pf_u1);
                if (pf_ph == kPhPred1 || pf_ph == kPhQkv || pf_ph == kPhFc1) {
                    pf_u1 -= pf_u;
                    pf_u = 0;
                }
            }
            if (pf_u >= pf_u1) {
                ++pf_ph;
                pf_u1 = -1;
                continue;
            }
            const void *src = nullptr;
            uint32_t bytes = 0;
            const int u = pf_u + lane;
            if (u < pf_u1 && !unit(pf_ph, u, &src, &bytes, true))
                bytes = 0;  // not cached: skipped
            uint32_t pre = bytes;  // inclusive prefix over the lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, pre, o);
                if (lane >= o)
                    pre += t;
            }
            const long long at = pf_bytes + pre - bytes;
            if (bytes && at >= lo && at < hi)
                prefetch_l2(src, bytes);
            pf_bytes += __shfl_sync(0xffffffffu, pre, 31);
            pf_u = min(pf_u + 32, pf_u1);
        }
    }
};

template <int NB>
DV_DEV void producer(Prod &P)
{
    const StreamArgs &a = P.a;
    const int lane = P.lane, nseg = a.nseg, cpr = a.d / 8;
    const long long ring_bytes = (long long)a.nstages * kStreamStageBytes;
    const int pps = pieces_per_stage(P.gcol.ncol);
    P.prefetch_run(ring_bytes);
    for (int ph = kPhPred1; ph < kPhEnd && P.ok; ++ph) {
        stamp(a, 24 + ph);
        if (ph == kPhQkv && !P.ensure(true))
            break;
        if (ph == kPhFc1 && !P.ensure(false))
            break;
        int u0, u1;
        P.range(ph, &u0, &u1);
        if (ph == kPhPred1 || ph == kPhQkv || ph == kPhFc1) {
            // segment-major: per segment, stages of seg_units rows (lane q: row + q)
            for (int sg = 0; sg < nseg && P.ok; ++sg) {
                int ra, rb;
                seg_rows(u0, u1, nseg, sg, &ra, &rb);
                const int nch = seg_chunks(sg, cpr), ups = seg_units(sg, cpr);
                const uint32_t ub = (uint32_t)nch * 16;
                for (int row = ra; row <= rb && P.ok; row += ups) {
                    const int n = min(ups, rb - row + 1);
                    const __half *p = nullptr;
                    if (lane < n)
                        P.row_start(ph, row + lane, &p);
                    bool good = P.ok;
                    if (lane == 0 && good) {
                        good = mbar_wait(&P.R.empty[P.R.slot()], P.R.par() ^ 1u, P.bd);
                        if (good)
                            mbar_expect_tx(&P.R.full[P.R.slot()], ub * n);
                    }
                    P.ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
                    if (!P.ok)
                        break;
                    if (lane < n)
                        bulk_g2s(P.R.buf() + lane * ub, p + (size_t)sg * kSeg * 8, ub,
                                 &P.R.full[P.R.slot()]);
                    ++P.R.k;
                    ++P.stages;
                    P.cp_bytes += ub * n;
                    P.prefetch_run(ring_bytes);
                }
            }
            continue;
        }
        const int umax = ph == kPhPred2 ? 1 : pps;
        for (int u = u0; u < u1 && P.ok;) {
            // lane q describes unit u + q; the stage takes the first n units
            // whose bytes fit (each unit's copy goes at its prefix offset)
            const void *src = nullptr;
            uint32_t bytes = 0;
            if (lane < umax && u + lane < u1)
                P.unit(ph, u + lane, &src, &bytes);
            uint32_t pre = bytes;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, pre, o);
                if (lane >= o)
                    pre += t;
            }
            const bool take = bytes != 0 && pre <= (uint32_t)kStreamStageBytes;
            const unsigned mask = __ballot_sync(0xffffffffu, take);
            const int n = __popc(mask);  // a prefix of the lanes
            const uint32_t total = __shfl_sync(0xffffffffu, pre, n - 1);
            bool good = P.ok;
            if (lane == 0 && good) {
                good = mbar_wait(&P.R.empty[P.R.slot()], P.R.par() ^ 1u, P.bd);
                if (good)
                    mbar_expect_tx(&P.R.full[P.R.slot()], total);
            }
            P.ok = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
            if (!P.ok)
                break;
            if (take)
                bulk_g2s(P.R.buf() + (pre - bytes), src, bytes, &P.R.full[P.R.slot()]);
            ++P.R.k;
            ++P.stages;
            P.cp_bytes += total;
            u += n;
            P.prefetch_run(ring_bytes);
        }
    }
    stamp(a, 30);
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
        const int cta = (int)blockIdx.x, g = cta / a.gm;
        Prod P{a,
               R,
               bd,
               reinterpret_cast<int *>(smem + kOffIdx),
               reinterpret_cast<int *>(smem + kOffIdx) + 256,
               tid & 31,
               true,
               cta,
               g,
               cta - g * a.gm,
               group_cols(a.d, g, a.ncg),
               false,
               false,
               0,
               0,
               0,
               0,
               0,
               0,
               0,
               0,
               kPhPred1,
               0,
               -1,
               0};
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
    u = std::max(u, (size_t)B * kTopkBins * 4 + (size_t)B * 1024 * 4);  // score histogram + u
    u = std::max(u, sizeof(AttnSmem));                           // attention
    u = std::max(u, (size_t)(2 * kHeadKPL + kHeadTopkMax) * 4);  // head selection
    {  // out-projection coefficients and the chunk weights of the head slots they touch
        const size_t rows = ((size_t)max_u_h * kDH + gm - 1) / gm;
        u = std::max(u, rows * B * 4 + (rows / kDH + 2) * B * kMaxAttnChunks * 4);
    }
    u = std::max(u, (size_t)kStreamMaxCtas * B * 3 * 4);               // norm statistics records
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
    case 13: return F<1, 5>(__VA_ARGS__);                                                     \
    case 14: return F<1, 6>(__VA_ARGS__);                                                     \
    case 17: return F<2, 1>(__VA_ARGS__);                                                     \
    case 18: return F<2, 2>(__VA_ARGS__);                                                     \
    case 19: return F<2, 3>(__VA_ARGS__);                                                     \
    case 20: return F<2, 4>(__VA_ARGS__);                                                     \
    case 21: return F<2, 5>(__VA_ARGS__);                                                     \
    case 22: return F<2, 6>(__VA_ARGS__);                                                     \
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
