// dv_select.cuh -- exact top-k selection of the predictor scores, split so
// that it never sits on the critical path of the layer decode.
//
// The selection rule ("DejaVu Guide: Contextual Sparsity for LLM Inference",
// "1. Mathematical Formulation of Lookahead Predictors": Top-k of the scores;
// the guide's listing returns the kept indices sorted): keep the k largest
// binary32 scores of a row, ties to the lower index, indices ascending; then
// the union over the batch rows.
//
// Scores are compared through order-preserving integer keys (score_key).
//  * Heads (n <= 256): one warp runs a bitwise radix select (head_select).
//  * Neurons: every CTA of the scoring kernel adds its scores to a histogram
//    of the key's top 11 bits.  In a later kernel each CTA reads that
//    histogram, finds the bin b1 holding the k-th largest key, and scans its
//    own slice of the scores (neuron_pass): keys above b1 go straight into
//    the row's bitmap, keys inside b1 go to a candidate list.  One CTA of the
//    following kernel finishes the row (neuron_final): a radix select over
//    the candidates' low 21 bits gives the k-th key T; keys > T are kept and,
//    among keys == T, the lowest indices; the bitmaps are compacted into
//    ascending index lists and their union.
#pragma once

#include "dv_common.cuh"

namespace dv {

constexpr int kHeadTopkMax = 256;   // head select handles n <= 256 (8 keys per lane)
constexpr int kHeadKPL = kHeadTopkMax / 32;
constexpr int kScanBatch = 8;    // 16-byte score loads per thread in flight in neuron_select_cta

// Bitmap words (bits[q] for elements q*32 + lane) of the k largest of
// s[0..n), ties to the lower index.  One warp; n <= kHeadTopkMax.  The scores
// are in global memory (written by other CTAs: read at L2) or, with kShared,
// in this CTA's shared memory.
template <bool kShared = false>
DV_DEV void warp_topk_bits(const float *s, int n, int k, unsigned *bits, int lane)
{
    unsigned key[kHeadKPL];
#pragma unroll
    for (int q = 0; q < kHeadKPL; ++q) {
        const int i = q * 32 + lane;
        key[q] = i < n ? score_key(kShared ? s[i] : ld_cg(s + i)) : 0u;
    }
    unsigned T = 0u;
    for (int bit = 31; bit >= 0; --bit) {
        const unsigned cand = T | (1u << bit);
        unsigned c = 0;
#pragma unroll
        for (int q = 0; q < kHeadKPL; ++q)
            c += (q * 32 + lane < n && key[q] >= cand) ? 1u : 0u;
        if ((int)__reduce_add_sync(0xffffffffu, c) >= k)
            T = cand;
    }
    unsigned gt = 0;
#pragma unroll
    for (int q = 0; q < kHeadKPL; ++q)
        gt += (q * 32 + lane < n && key[q] > T) ? 1u : 0u;
    const int need_eq = k - (int)__reduce_add_sync(0xffffffffu, gt);
    int seen = 0;
#pragma unroll
    for (int q = 0; q < kHeadKPL; ++q) {
        const bool valid = q * 32 + lane < n;
        const bool eq = valid && key[q] == T;
        const unsigned m = __ballot_sync(0xffffffffu, eq);
        const int rank = seen + __popc(m & ((1u << lane) - 1u));
        const bool keep = valid && (key[q] > T || (eq && rank < need_eq));
        const unsigned w = __ballot_sync(0xffffffffu, keep);
        if (lane == 0 && q * 32 < n)
            bits[q] = w;
        seen += __popc(m);
    }
    __syncwarp();
}

// Ascending indices of the set bits of bits[0..W) written to out (one warp);
// returns their number.
DV_DEV int warp_compact_bits(const unsigned *bits, int W, int32_t *out, int lane)
{
    int off = 0;
    for (int q = 0; q < W; ++q) {
        const unsigned b = bits[q];
        if (out && ((b >> lane) & 1u))
            out[off + __popc(b & ((1u << lane) - 1u))] = q * 32 + lane;
        off += __popc(b);
    }
    return off;
}

// Head selection of all B rows by one warp.  The union goes to su[] (shared
// memory, ascending) and its length is returned.  When `write` is set the
// per-row lists, the union and its length are also written to global memory.
// kShared: the scores s_h are in shared memory.
template <bool kShared = false>
DV_DEV int head_select(const float *s_h, int B, int H, int k, unsigned *sbits, int32_t *su,
                       bool write, int32_t *idx_h, int32_t *u_h, int32_t *n_u_h, int lane)
{
    const int W = (H + 31) >> 5;
    unsigned *rowbits = sbits, *ubits = sbits + kHeadKPL;
    if (lane < kHeadKPL)
        ubits[lane] = 0u;
    __syncwarp();
    for (int b = 0; b < B; ++b) {
        warp_topk_bits<kShared>(s_h + (size_t)b * H, H, k, rowbits, lane);
        if (lane < W)
            ubits[lane] |= rowbits[lane];
        __syncwarp();
        if (write)
            warp_compact_bits(rowbits, W, idx_h + (size_t)b * k, lane);
        __syncwarp();
    }
    const int nu = warp_compact_bits(ubits, W, su, lane);
    if (write) {
        warp_compact_bits(ubits, W, u_h, lane);
        if (lane == 0)
            *n_u_h = nu;
    }
    __syncwarp();
    return nu;
}

// Head selection of B rows by all warps of the block, the rows dealt out
// to the warps (warp w selects rows w, w + nw, ...): per-row lists to
// idx_h, the union (ascending) to u_h and its length to n_u_h.  wbits holds
// kHeadKPL words per warp, ubits kHeadKPL words (shared memory).  Every
// thread of the block calls it; barriers inside.
DV_DEV void head_select_block(const float *s_h, int B, int H, int k, unsigned *wbits,
                              unsigned *ubits, int32_t *idx_h, int32_t *u_h, int32_t *n_u_h)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int W = (H + 31) >> 5;
    unsigned *rowbits = wbits + warp * kHeadKPL;
    if ((int)threadIdx.x < kHeadKPL)
        ubits[threadIdx.x] = 0u;
    __syncthreads();
    for (int b = warp; b < B; b += nw) {
        warp_topk_bits(s_h + (size_t)b * H, H, k, rowbits, lane);
        if (lane < W)
            atomicOr(&ubits[lane], rowbits[lane]);
        warp_compact_bits(rowbits, W, idx_h + (size_t)b * k, lane);
        __syncwarp();
    }
    __syncthreads();
    if (warp == 0) {
        const int nu = warp_compact_bits(ubits, W, u_h, lane);
        if (lane == 0)
            *n_u_h = nu;
    }
}

// ---------------------------------------------------------------------------
// Neuron selection (state: NeuronSel in the workspace).

// Block-wide: bin of the krem-th largest key of a histogram of nb bins.
template <class Grp = CtaGroup>
DV_DEV void block_find_bin(const int *hist, int nb, int krem, int *scr)
{
    const int nt = Grp::size(), tid = threadIdx.x;
    const int per = (nb + nt - 1) / nt;
    const int top = nb - 1 - tid * per;
    int c = 0;
    for (int q = 0; q < per; ++q) {
        const int bin = top - q;
        if (bin >= 0)
            c += hist[bin];
    }
    int tot;
    const int before = block_excl_scan<Grp>(c, scr + 4, &tot);
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
    Grp::sync();
}

// The pass of one CTA over bitmap words [w0, w1) of every row (all threads
// of the CTA).  Words are whole: each belongs to exactly one CTA.  hbuf:
// shared [kTopkBins]; scr: shared [48]; sb1: shared [B].
template <class Grp = CtaGroup>
DV_DEV void neuron_pass(const NeuronSel &ns, int w0, int w1, int *sb1, int *hbuf, int *scr)
{
    const int tid = threadIdx.x, nt = Grp::size();
    const int lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int W = (ns.N + 31) >> 5;
    for (int b = 0; b < ns.B; ++b) {
        // the row's first-digit histogram, staged with independent loads
        const int *gh = ns.hist + (size_t)b * kTopkBins;
        for (int i = tid; i < kTopkBins; i += nt)
            hbuf[i] = ld_cg(gh + i);
        Grp::sync();
        block_find_bin<Grp>(hbuf, kTopkBins, ns.k, scr);
        if (tid == 0)
            sb1[b] = scr[0];
    }
    Grp::sync();
    for (int b = 0; b < ns.B; ++b) {
        const unsigned b1 = (unsigned)sb1[b];
        const float *s = ns.s_n + (size_t)b * ns.N;
        for (int wd = w0 + warp; wd < w1; wd += nw) {
            const int i = wd * 32 + lane;
            const bool in = i < ns.N;
            const unsigned key = in ? score_key(ld_cg(s + i)) : 0u;
            const unsigned d = key >> 21;
            const unsigned above = __ballot_sync(0xffffffffu, in && d > b1);
            const unsigned cand = __ballot_sync(0xffffffffu, in && d == b1);
            if (lane == 0)
                ns.rowbits[(size_t)b * W + wd] = above;
            if (cand) {
                int base = 0;
                if (lane == 0)
                    base = atomicAdd(ns.cand_cnt + b, __popc(cand));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (in && d == b1) {
                    const int pos = base + __popc(cand & ((1u << lane) - 1u));
                    if (pos < kTopkCand) {
                        ns.cand_key[(size_t)b * kTopkCand + pos] = key;
                        ns.cand_idx[(size_t)b * kTopkCand + pos] = i;
                    }
                }
            }
        }
    }
}

// Shared-memory layout of neuron_final.
struct FinalSmem {
    int *hist;          // [kTopkBins]
    unsigned *rowbits;  // [W]
    unsigned *ubits;    // [W]
    unsigned *ckey;     // [kTopkCand]
    int *cidx;          // [kTopkCand]
    int *scr;           // [48]
};

__host__ __device__ inline size_t neuron_final_smem_bytes(int N)
{
    const int W = (N + 31) >> 5;
    return ((size_t)kTopkBins + 2 * (size_t)W + 2 * (size_t)kTopkCand) * 4;
}

// Ascending indices of the set bits of bits[0..W), block-wide.
template <class Grp = CtaGroup>
DV_DEV int block_compact_bits(const unsigned *bits, int W, int32_t *out, int *scr)
{
    const int nt = Grp::size(), tid = threadIdx.x;
    const int per = (W + nt - 1) / nt;
    const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
    int cnt = 0;
    for (int w = w0; w < w1; ++w)
        cnt += __popc(bits[w]);
    int tot;
    int pos = block_excl_scan<Grp>(cnt, scr + 4, &tot);
    for (int w = w0; w < w1; ++w) {
        unsigned b = bits[w];
        while (b) {
            const int bit = __ffs(b) - 1;
            out[pos++] = w * 32 + bit;
            b &= b - 1u;
        }
    }
    return tot;
}

// Candidates beyond the capacity (many keys share the k-th key's top 11
// bits): finish exactly with passes over the global scores.  Slow, rare.
template <class Grp = CtaGroup>
DV_DEV void neuron_overflow(const float *s, int N, unsigned prefix, int krem, const FinalSmem &sm)
{
    const int tid = threadIdx.x, nt = Grp::size();
    unsigned pmask = 0xffe00000u;
    const int shifts[2] = {10, 0};
    const int widths[2] = {11, 10};
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = shifts[pass], nbins = 1 << widths[pass];
        for (int i = tid; i < nbins; i += nt)
            sm.hist[i] = 0;
        Grp::sync();
        for (int i = tid; i < N; i += nt) {
            const unsigned key = score_key(ld_cg(s + i));
            if ((key & pmask) == prefix)
                atomicAdd(&sm.hist[(key >> shift) & (unsigned)(nbins - 1)], 1);
        }
        Grp::sync();
        block_find_bin<Grp>(sm.hist, nbins, krem, sm.scr);
        prefix |= (unsigned)sm.scr[0] << shift;
        pmask |= (unsigned)(nbins - 1) << shift;
        krem = sm.scr[1];
        Grp::sync();
    }
    const unsigned T = prefix;
    int seen = 0;
    for (int base = 0; base < N; base += nt) {
        const int i = base + tid;
        const unsigned key = i < N ? score_key(ld_cg(s + i)) : 0u;
        const int eq = (i < N && key == T) ? 1 : 0;
        int tot;
        const int rank = block_excl_scan<Grp>(eq, sm.scr + 4, &tot);
        if (i < N && (key > T || (eq && seen + rank < krem)))
            atomicOr(&sm.rowbits[i >> 5], 1u << (i & 31));
        seen += tot;
    }
    Grp::sync();
}

// Finish row b: sm.rowbits holds the keys above bin b1, sm.ckey / sm.cidx the
// ncand keys inside it (all of them when ncand <= kTopkCand; else the row is
// finished from the global scores).  Selects the krem largest candidates
// (ties to the lower index), adds the row to sm.ubits and writes idx_n[b].
template <class Grp = CtaGroup>
DV_DEV void neuron_row_finish(const NeuronSel &ns, int b, unsigned b1, int krem, int ncand,
                              const FinalSmem &sm)
{
    const int tid = threadIdx.x, nt = Grp::size();
    const int W = (ns.N + 31) >> 5;
    if (ncand > kTopkCand) {
        neuron_overflow<Grp>(ns.s_n + (size_t)b * ns.N, ns.N, b1 << 21, krem, sm);
    } else {
        unsigned prefix = b1 << 21, pmask = 0xffe00000u;
        int kr = krem;
        const int shifts[2] = {10, 0};
        const int widths[2] = {11, 10};
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = shifts[pass], nbins = 1 << widths[pass];
            for (int i = tid; i < nbins; i += nt)
                sm.hist[i] = 0;
            Grp::sync();
            for (int i = tid; i < ncand; i += nt) {
                const unsigned key = sm.ckey[i];
                if ((key & pmask) == prefix)
                    atomicAdd(&sm.hist[(key >> shift) & (unsigned)(nbins - 1)], 1);
            }
            Grp::sync();
            block_find_bin<Grp>(sm.hist, nbins, kr, sm.scr);
            prefix |= (unsigned)sm.scr[0] << shift;
            pmask |= (unsigned)(nbins - 1) << shift;
            kr = sm.scr[1];
            Grp::sync();
        }
        const unsigned T = prefix;
        const int need_eq = kr;
        const int n_eq = sm.hist[T & 1023u];  // candidates equal to T
        for (int i = tid; i < ncand; i += nt) {
            const unsigned key = sm.ckey[i];
            bool keep = key > T;
            if (key == T) {
                if (n_eq == need_eq) {
                    keep = true;
                } else {
                    const int idx = sm.cidx[i];
                    int rank = 0;
                    for (int q = 0; q < ncand; ++q)
                        rank += (sm.ckey[q] == T && sm.cidx[q] < idx);
                    keep = rank < need_eq;
                }
            }
            if (keep) {
                const int idx = sm.cidx[i];
                atomicOr(&sm.rowbits[idx >> 5], 1u << (idx & 31));
            }
        }
        Grp::sync();
    }
    for (int i = tid; i < W; i += nt)
        sm.ubits[i] |= sm.rowbits[i];
    block_compact_bits<Grp>(sm.rowbits, W, ns.idx_n + (size_t)b * ns.k, sm.scr);
}

// Union of the rows (sm.ubits) to u_n / n_u_n.
template <class Grp = CtaGroup>
DV_DEV void neuron_union_out(const NeuronSel &ns, const FinalSmem &sm)
{
    const int W = (ns.N + 31) >> 5;
    Grp::sync();
    const int tot = block_compact_bits<Grp>(sm.ubits, W, ns.u_n, sm.scr);
    if (threadIdx.x == 0)
        *ns.n_u_n = tot;
}

// Bin b1 of the k-th largest key of row b and the rank krem left inside it,
// from the row's global first-digit histogram (staged in sm.hist).
template <class Grp = CtaGroup>
DV_DEV void neuron_row_bin(const NeuronSel &ns, int b, const FinalSmem &sm, unsigned *b1,
                           int *krem)
{
    const int tid = threadIdx.x, nt = Grp::size();
    const int *ghist = ns.hist + (size_t)b * kTopkBins;
    for (int i = tid; i < kTopkBins; i += nt)
        sm.hist[i] = __ldcg(ghist + i);
    Grp::sync();
    block_find_bin<Grp>(sm.hist, kTopkBins, ns.k, sm.scr);
    *b1 = (unsigned)sm.scr[0];
    *krem = sm.scr[1];
    Grp::sync();  // every thread holds b1, krem before scr is reused
}

// Finish the selection of every row from the bitmaps and candidate lists of
// the distributed pass (neuron_pass) and write idx_n, u_n, n_u_n; leave the
// histogram and candidate counts zero.  One whole CTA; smem as FinalSmem.
template <class Grp = CtaGroup>
DV_DEV void neuron_final(const NeuronSel &ns, const FinalSmem &sm)
{
    const int tid = threadIdx.x, nt = Grp::size();
    const int W = (ns.N + 31) >> 5;
    for (int i = tid; i < W; i += nt)
        sm.ubits[i] = 0u;
    for (int b = 0; b < ns.B; ++b) {
        const unsigned *gbits = ns.rowbits + (size_t)b * W;
        for (int i = tid; i < W; i += nt)
            sm.rowbits[i] = __ldcg(gbits + i);
        unsigned b1;
        int krem;
        neuron_row_bin<Grp>(ns, b, sm, &b1, &krem);
        const int ncand = __ldcg(ns.cand_cnt + b);
        if (ncand <= kTopkCand)
            for (int i = tid; i < ncand; i += nt) {
                sm.ckey[i] = __ldcg(ns.cand_key + (size_t)b * kTopkCand + i);
                sm.cidx[i] = __ldcg(ns.cand_idx + (size_t)b * kTopkCand + i);
            }
        neuron_row_finish<Grp>(ns, b, b1, krem, ncand, sm);
        // leave this row's shared state zero for the next call
        int *ghist = ns.hist + (size_t)b * kTopkBins;
        for (int i = tid; i < kTopkBins; i += nt)
            ghist[i] = 0;
        if (tid == 0)
            ns.cand_cnt[b] = 0;
        Grp::sync();
    }
    neuron_union_out<Grp>(ns, sm);
}

// Blocked selection (ns.block > 1: blocks of ns.block contiguous neurons, a
// multiple of 32; "DejaVu Guide ...", "Core Innovation 2", "1. Blocked
// Channel Sparsity"): a block's score is the largest score of its members;
// every row keeps its k / block best blocks, ties to the lower block (a
// bitonic sort of the block keys).  Writes idx_n, u_n, n_u_n and leaves the
// histogram and candidate counts zero.  One whole CTA; smem as FinalSmem
// (cidx holds the block maxima, ckey the sort keys: at most kTopkCand / 2
// blocks).
template <class Grp = CtaGroup>
DV_DEV void select_union_out(const NeuronSel &ns, const FinalSmem &sm, int nparts);

template <class Grp = CtaGroup>
DV_DEV void block_select(const NeuronSel &ns, const FinalSmem &sm, int part = 0, int nparts = 1)
{
    const int tid = threadIdx.x, nt = Grp::size();
    const int W = (ns.N + 31) >> 5, nb = ns.N / ns.block, kb = ns.k / ns.block;
    const int wpb = ns.block >> 5;  // bitmap words per block
    float *bm = reinterpret_cast<float *>(sm.cidx);  // block maxima (<= kTopkCand / 2)
    for (int i = tid; i < W; i += nt)
        sm.ubits[i] = 0u;
    // block maxima: a warp reads 128 consecutive scores per load (a float4
    // per lane, kScanBatch loads in flight) and reduces each block's lanes
    // (ns.block / 4 of them, a power of two up to 32) with shuffles
    const int lanes = ns.block >> 2, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
    const int nch = ns.N >> 7;  // 128-score chunks (ns.N is a multiple of the block, >= 32)
    for (int b = part; b < ns.B; b += nparts) {
        const float4 *s4 = reinterpret_cast<const float4 *>(ns.s_n + (size_t)b * ns.N);
        for (int c0 = warp; c0 < nch; c0 += nw * kScanBatch) {
            float4 v[kScanBatch];
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u) {
                const int c = c0 + u * nw;
                v[u] = c < nch ? __ldcg(s4 + (size_t)c * 32 + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u) {
                const int c = c0 + u * nw;
                float m = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
                for (int off = 1; off < lanes; off <<= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                if (c < nch && (lane & (lanes - 1)) == 0)
                    bm[(c * 128 + lane * 4) / ns.block] = m;
            }
        }
        // a row not a whole number of 128-score chunks: its last blocks one by one
        for (int j = (nch * 128) / ns.block + tid; j < nb; j += nt) {
            const float *p = ns.s_n + (size_t)b * ns.N + (size_t)j * ns.block;
            float m = ld_cg(p);
            for (int i = 1; i < ns.block; ++i)
                m = fmaxf(m, ld_cg(p + i));
            bm[j] = m;
        }
        for (int i = tid; i < W; i += nt)
            sm.rowbits[i] = 0u;
        Grp::sync();
        // the blocks in descending order of (score, then lower index first):
        // a bitonic sort of 64-bit keys (order-preserving score bits above
        // the complemented block index, so every key is distinct), padded
        // with zero keys to a power of two; the first kb are kept
        unsigned long long *key = reinterpret_cast<unsigned long long *>(sm.ckey);
        int np = 1;
        while (np < nb)
            np <<= 1;
        Grp::sync();
        for (int j = tid; j < np; j += nt)
            key[j] = j < nb ? ((unsigned long long)score_key(bm[j]) << 32) |
                                  (unsigned long long)(0xffffffffu - (unsigned)j)
                            : 0ull;
        Grp::sync();
        for (int size = 2; size <= np; size <<= 1)
            for (int stride = size >> 1; stride > 0; stride >>= 1) {
                for (int i = tid; i < (np >> 1); i += nt) {
                    // pair (lo, lo + stride) of the i-th comparator
                    const int lo = ((i / stride) * (stride << 1)) + (i % stride);
                    const int hi = lo + stride;
                    const bool desc = (lo & size) == 0;  // descending runs first
                    const unsigned long long a = key[lo], c = key[hi];
                    if ((a < c) == desc) {
                        key[lo] = c;
                        key[hi] = a;
                    }
                }
                Grp::sync();
            }
        for (int q = tid; q < kb; q += nt) {
            const int j = (int)(0xffffffffu - (unsigned)(key[q] & 0xffffffffull));
            for (int t = 0; t < wpb; ++t)
                sm.rowbits[j * wpb + t] = 0xffffffffu;
        }
        Grp::sync();
        for (int i = tid; i < W; i += nt)
            sm.ubits[i] |= sm.rowbits[i];
        block_compact_bits<Grp>(sm.rowbits, W, ns.idx_n + (size_t)b * ns.k, sm.scr);
        // the scores' histogram is not used here: leave it zero for the next call
        int *ghist = ns.hist + (size_t)b * kTopkBins;
        for (int i = tid; i < kTopkBins; i += nt)
            ghist[i] = 0;
        if (tid == 0)
            ns.cand_cnt[b] = 0;
        Grp::sync();
    }
    select_union_out<Grp>(ns, sm, nparts);
}

// The union of the rows after a selection split over nparts CTAs (part p
// took rows p, p + nparts, ...): each ORs its rows' union into the global
// bitmap ns.gubits, counts itself in *ns.gdone, and the last to arrive
// compacts the bitmap to u_n / n_u_n and clears both for the next call.
// nparts == 1: straight from shared memory.
template <class Grp>
DV_DEV void select_union_out(const NeuronSel &ns, const FinalSmem &sm, int nparts)
{
    if (nparts <= 1) {
        neuron_union_out<Grp>(ns, sm);
        return;
    }
    const int tid = threadIdx.x, nt = Grp::size();
    const int W = (ns.N + 31) >> 5;
    Grp::sync();
    for (int i = tid; i < W; i += nt)
        if (sm.ubits[i])
            atomicOr(ns.gubits + i, sm.ubits[i]);
    __threadfence();
    Grp::sync();
    if (tid == 0)
        sm.scr[45] = atomicAdd(ns.gdone, 1) == nparts - 1;
    Grp::sync();
    if (!sm.scr[45])
        return;
    __threadfence();
    for (int i = tid; i < W; i += nt)
        sm.ubits[i] = __ldcg(ns.gubits + i);
    Grp::sync();
    const int tot = block_compact_bits<Grp>(sm.ubits, W, ns.u_n, sm.scr);
    if (tid == 0)
        *ns.n_u_n = tot;
    for (int i = tid; i < W; i += nt)
        ns.gubits[i] = 0u;
    if (tid == 0)
        *ns.gdone = 0;
}

// The whole neuron selection in one CTA: for every row, the bin of the k-th
// key from the global histogram, one pass over the row's scores into
// shared-memory bitmaps and candidates, then the finish.  Leaves the global
// histogram zero.  smem as FinalSmem.  Each thread reads 4 consecutive
// scores per load (16 bytes when the row is 16-byte aligned) and kScanBatch
// such groups at a time, so few requests carry the row even when the memory
// system is busy.
//
// part / nparts: this CTA takes rows part, part + nparts, ... of the batch;
// the union is finished by select_union_out.
static __device__ __noinline__ void neuron_select_cta(const NeuronSel &ns, const FinalSmem &sm,
                                                      int part = 0, int nparts = 1)
{
    if (ns.block > 1) {
        block_select(ns, sm, part, nparts);
        return;
    }
    const int tid = threadIdx.x, nt = blockDim.x;
    const int W = (ns.N + 31) >> 5;
    const int G = (ns.N + 3) >> 2;  // groups of 4 scores
    const bool vec = (ns.N & 3) == 0;
    for (int i = tid; i < W; i += nt)
        sm.ubits[i] = 0u;
    for (int b = part; b < ns.B; b += nparts) {
        const float *s = ns.s_n + (size_t)b * ns.N;
        // the row's histogram first (one 16-byte load per thread), then the bin
        const int4 *gh4 = reinterpret_cast<const int4 *>(ns.hist + (size_t)b * kTopkBins);
        for (int i = tid; i < kTopkBins / 4; i += nt)
            reinterpret_cast<int4 *>(sm.hist)[i] = __ldcg(gh4 + i);
        for (int i = tid; i < W; i += nt)
            sm.rowbits[i] = 0u;
        if (tid == 0)
            sm.scr[44] = 0;  // candidate count
        __syncthreads();
        block_find_bin(sm.hist, kTopkBins, ns.k, sm.scr);
        const unsigned b1 = (unsigned)sm.scr[0];
        const int krem = sm.scr[1];
        __syncthreads();
        for (int g0 = tid; g0 < G; g0 += nt * kScanBatch) {
            float v[kScanBatch][4];
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u) {
                const int g = g0 + u * nt;
                if (vec) {
                    const float4 t = g < G ? __ldcg(reinterpret_cast<const float4 *>(s) + g)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    v[u][0] = t.x;
                    v[u][1] = t.y;
                    v[u][2] = t.z;
                    v[u][3] = t.w;
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        v[u][q] = 4 * g + q < ns.N ? ld_cg(s + 4 * g + q) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int i = 4 * (g0 + u * nt) + q;
                    if (i >= ns.N)
                        continue;
                    const unsigned key = score_key(v[u][q]);
                    const unsigned d = key >> 21;
                    if (d > b1) {
                        atomicOr(&sm.rowbits[i >> 5], 1u << (i & 31));
                    } else if (d == b1) {
                        const int pos = atomicAdd(&sm.scr[44], 1);
                        if (pos < kTopkCand) {
                            sm.ckey[pos] = key;
                            sm.cidx[pos] = i;
                        }
                    }
                }
            }
        }
        __syncthreads();
        const int ncand = sm.scr[44];
        __syncthreads();
        neuron_row_finish(ns, b, b1, krem, ncand, sm);
        int *ghist = ns.hist + (size_t)b * kTopkBins;
        for (int i = tid; i < kTopkBins; i += nt)
            ghist[i] = 0;
        __syncthreads();
    }
    select_union_out(ns, sm, nparts);
}

DV_DEV FinalSmem final_smem(void *base, int N, int *scr)
{
    const int W = (N + 31) >> 5;
    FinalSmem sm;
    sm.hist = static_cast<int *>(base);
    sm.rowbits = reinterpret_cast<unsigned *>(sm.hist + kTopkBins);
    sm.ubits = sm.rowbits + W;
    sm.ckey = sm.ubits + W;
    sm.cidx = reinterpret_cast<int *>(sm.ckey + kTopkCand);
    sm.scr = scr;
    return sm;
}

}  // namespace dv
