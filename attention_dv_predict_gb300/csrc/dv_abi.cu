// dv_abi.cu -- C entry points of libdv: argument checks, workspace layout and
// the launch sequence of the sparse layer decode.  See include/dv.h.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "dv_internal.h"

using namespace dv;

namespace {

constexpr int kLayerLaunches = 7;
constexpr int kSideFlagWord = 1;  // workspace control word of the side-work flag
constexpr int kSelDoneWord = 2;   // ... CTAs done with their rows of a split neuron selection
constexpr int kSideDoneWord = 3;  // ... side CTAs of the stage-2 predictor done
constexpr int kMaxSelCtas = 8;    // CTAs the fused decode's neuron selection is split over

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t esize(int dtype) { return dtype == DV_F16 ? 2 : 4; }
int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

int batch_pad(int B)
{
    if (B <= 8) {
        int p = 1;
        while (p < B)
            p <<= 1;
        return p;
    }
    return (int)align_up((size_t)B, 8);
}

dv_status check_desc(const dv_layer_desc *D)
{
    if (!D)
        return DV_ERR_INVALID_ARG;
    if (D->d_model <= 0 || D->n_heads <= 0 || D->head_dim <= 0 || D->d_ffn <= 0 ||
        D->pred_rank <= 0 || D->kv_cap <= 0)
        return DV_ERR_INVALID_ARG;
    if (D->dtype != DV_F32 && D->dtype != DV_F16)
        return DV_ERR_INVALID_ARG;
    if (D->norm != DV_LAYERNORM && D->norm != DV_RMSNORM)
        return DV_ERR_INVALID_ARG;
    if (!(D->ln_eps > 0.f) || !std::isfinite(D->ln_eps))
        return DV_ERR_INVALID_ARG;
    const int epc = (int)(16 / esize(D->dtype));
    if (D->d_model % epc || D->pred_rank % epc)
        return DV_ERR_UNSUPPORTED;
    const int dh = D->head_dim;
    const size_t hb = (size_t)dh * esize(D->dtype);
    if ((dh & (dh - 1)) || hb < 16 || hb > 512)
        return DV_ERR_UNSUPPORTED;
    // activations of one row must fit the row-dot kernel's shared memory
    if (rowdot_smem(RK_PRED1, 1, D->d_model) > kSmemCap ||
        rowdot_smem(RK_PRED2, 1, D->pred_rank) > kSmemCap)
        return DV_ERR_UNSUPPORTED;
    // one warp selects the heads; the neuron selection's bitmaps fit one CTA
    if (D->n_heads > 256 || D->d_ffn > (1 << 19))
        return DV_ERR_UNSUPPORTED;
    if ((long long)3 * D->n_heads * dh > (1 << 24) || D->d_ffn > (1 << 24) ||
        (long long)D->kv_cap * dh > (1LL << 31) / 4)
        return DV_ERR_UNSUPPORTED;
    if (D->neuron_block < 0 || D->mlp < DV_MLP_RELU || D->mlp > DV_MLP_SWIGLU)
        return DV_ERR_INVALID_ARG;
    if (D->neuron_block > 1 &&
        (D->neuron_block != 32 && D->neuron_block != 64 && D->neuron_block != 128 ||
         D->d_ffn % D->neuron_block || D->d_ffn / D->neuron_block > kTopkCand / 2))
        return DV_ERR_UNSUPPORTED;
    return DV_OK;
}

// The neuron keep count in whole blocks when the layer selects blocks.
bool k_neurons_ok(const dv_layer_desc &D, int kn)
{
    return kn >= 1 && kn <= D.d_ffn && (D.neuron_block <= 1 || kn % D.neuron_block == 0);
}

dv_status check_weights(const dv_layer_weights *w)
{
    if (!w)
        return DV_ERR_INVALID_ARG;
    const void *p[] = {w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, w->w_oT, w->b_o, w->ln2_g,
                       w->ln2_b, w->w1, w->b1, w->w2T, w->b2, w->pred_h, w->pred_a, w->pred_b};
    for (const void *q : p)
        if (!q || !aligned16(q))
            return DV_ERR_INVALID_ARG;
    return DV_OK;
}

bool ptr_ok(const void *p) { return p && aligned16(p); }

thread_local int t_cuda_error = 0;  // the CUDA error behind this thread's last DV_ERR_CUDA

// e failed: keep it for dv_cuda_error.
bool failed(cudaError_t e)
{
    if (e == cudaSuccess)
        return false;
    t_cuda_error = (int)e;
    return true;
}

dv_status cuda_status(cudaError_t e) { return failed(e) ? DV_ERR_CUDA : DV_OK; }

struct Launch {
    cudaStream_t st;
    int nsm;
    // chain the call's kernels by programmatic dependent launch (see
    // run_attn for the one boundary the tensor-core configuration keeps in
    // stream order)
    bool pdl;
    void *const *events;  // optional trace events
    int n_events;
    int next_event;
    unsigned long long *stamps;  // optional chain timeline [kernels][nsm][kChainStamps]
    int next_kernel;

    // the timeline slots of the next kernel (NULL when not stamping)
    unsigned long long *kernel_stamps()
    {
        return stamps ? stamps + (size_t)(next_kernel++) * nsm * kChainStamps : nullptr;
    }

    dv_status mark()
    {
        if (!events)
            return DV_OK;
        if (next_event >= n_events)
            return DV_ERR_INVALID_ARG;
        cudaEvent_t ev = static_cast<cudaEvent_t>(events[next_event++]);
        return cuda_status(cudaEventRecord(ev, st));
    }
};

dv_status make_launch(void *stream, void *const *events, int n_events, Launch *L)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return DV_ERR_CUDA;
    int nsm = 0;
    if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        nsm <= 0)
        return DV_ERR_CUDA;
    if (nsm * kWarpsPerBlock > kMaxWarps)
        return DV_ERR_UNSUPPORTED;
    L->st = static_cast<cudaStream_t>(stream);
    L->nsm = nsm;
    L->pdl = true;  // see pdl_for
    L->events = events;
    L->n_events = n_events;
    L->next_event = 0;
    L->stamps = nullptr;
    L->next_kernel = 0;
    return DV_OK;
}

template <typename P>
P *at(void *ws, size_t off) { return reinterpret_cast<P *>(static_cast<char *>(ws) + off); }

// ---------------------------------------------------------------------------
// The blocks of the decode step.  Where Launch::pdl is set (every call but
// binary16 ones from kMmaMinBatch batch rows) each launch after the first of
// a call is a programmatic dependent launch (the kernels wait for their
// inputs with griddepcontrol.wait); the first one, and every launch when
// pdl is off, is ordered normally after prior work.

NeuronSel make_neuron_sel(const dv_layer_desc &D, int B, int kn, const dv_selection &sel,
                          void *ws, const WsLayout &L)
{
    NeuronSel ns;
    std::memset(&ns, 0, sizeof(ns));
    ns.s_n = at<float>(ws, L.s_n);
    ns.B = B;
    ns.N = D.d_ffn;
    ns.k = kn;
    ns.hist = at<int>(ws, L.hist);
    ns.rowbits = at<unsigned>(ws, L.nbits);
    ns.cand_key = at<unsigned>(ws, L.cand_key);
    ns.cand_idx = at<int>(ws, L.cand_idx);
    ns.cand_cnt = at<int>(ws, L.cand_cnt);
    ns.idx_n = sel.idx_n;
    ns.u_n = sel.u_n;
    ns.n_u_n = sel.n_u_n;
    ns.status = at<int>(ws, L.ctl);
    ns.block = D.neuron_block > 1 ? D.neuron_block : 0;
    ns.gubits = at<unsigned>(ws, L.sel_ubits);
    ns.gdone = at<int>(ws, L.ctl) + kSelDoneWord;
    return ns;
}

// Binary16 layers use the tensor-core row kernel (QKV, FC1) and column kernel
// (out-projection, fc2) from kMmaMinBatch batch rows on.
// Programmatic dependent launch between the call's kernels: on, except for
// the tensor-core configuration from 8 batch rows, where the chained decode
// measured slower than stream order at OPT-175B (batch 8: 693 against 688 us;
// batch 16: 1315 against 1288 us; batch 4 gains: 400 against 405 us).
bool use_mma(const dv_layer_desc &D, int B);
bool pdl_for(const dv_layer_desc &D, int B) { return !use_mma(D, B) || B < 8; }

bool use_mma(const dv_layer_desc &D, int B)
{
    // SwiGLU layers run on CUDA cores at every batch size
    return D.dtype == DV_F16 && B >= kMmaMinBatch && D.d_model % 32 == 0 &&
           D.mlp == DV_MLP_RELU;
}

// Kernel launches of the fused (chained) decode.
int layer_launches(const dv_layer_desc &, int) { return kLayerLaunches; }

// Row count the tensor-core kernel's partial slots are sized for: the
// largest of QKV, fc1 and the stage-1 predictor.
int mma_rows_max(const dv_layer_desc &D)
{
    const int qkv = 3 * D.n_heads * D.head_dim, p1 = D.n_heads + D.pred_rank;
    const int m = qkv > D.d_ffn ? qkv : D.d_ffn;
    return m > p1 ? m : p1;
}

// The predictor stages run on the tensor-core row kernel too when the
// others do, from 5 batch rows, and the rank is a whole number of 16-byte
// chunks.  Below 5 batch rows the CUDA-core kernels (4 rows per weight pass) were
// faster (OPT-175B, batch 4: 376 against 386 us per decode); from 5 rows
// they take 8 rows a pass and fall behind (batch 8: 604 against 573 us).
bool pred_mma(const dv_layer_desc &D, int B)
{
    return use_mma(D, B) && B >= 5 && D.pred_rank % 8 == 0;
}

// Fills the tensor-core fields of a; returns its dynamic shared memory.
// fixed_rows > 0 (the predictor stages: every row, known on the host): when
// there are fewer 16-row groups than warps, K is cut into more segments so
// that every warp has a (group, segment) to stream, within the partial
// slots the workspace holds.
size_t set_mma(RowArgs &a, const dv_layer_desc &D, void *ws, const WsLayout &L, int nsm,
               int fixed_rows = 0)
{
    int S = 1, ks = 0;
    const int nt = rowdot_mma_tiles(a.B);
    rowdot_mma_plan(a.K, nt, &S, &ks);
    const int groups_max = ceil_div(mma_rows_max(D), 16);
    a.mma_groups = groups_max;
    if (fixed_rows > 0) {
        const int groups = ceil_div(fixed_rows, 16);
        int s_ws = 1, ks_ws = 0;  // the segments the partial slots are sized for
        rowdot_mma_plan(D.d_model, nt, &s_ws, &ks_ws);
        // at most K / 128 segments, several CTAs per segment, and at most
        // kMmaSegMax: the last warp of a group loads its S partials of 8 nt
        // rows (35 segments at OPT-175B, batch 32: a 20 us tail)
        constexpr int kMmaSegMax = 8;
        const int want = std::min(std::min(ceil_div(nsm * kWarpsPerBlock, groups), a.K / 128),
                                  std::min(nsm / 4, kMmaSegMax));
        if (want > S) {
            const int ks2 = ceil_div(ceil_div(a.K, want), 32) * 32;
            const int s2 = ceil_div(a.K, ks2);
            if ((long long)groups * s2 <= (long long)groups_max * s_ws && s2 > S) {
                S = s2;
                ks = ks2;
                a.mma_groups = groups;
            }
        }
    }
    a.mma_seg = S;
    a.mma_ks = ks;
    a.mma_nt = nt;
    a.mma_part = at<float>(ws, L.mma_part);
    a.mma_cnt = at<int>(ws, L.mma_cnt);
    return rowdot_mma_smem(ks, nt);
}

// Row-kernel variant for fc1 on the tensor cores: 0 = mma.sync (default),
// 1 = tcgen05 from 9 batch rows (dv_set_row_kernel).
std::atomic<int> g_row_variant{0};

bool row_tc(const dv_layer_desc &D, int B)
{
    return g_row_variant.load() == 1 && use_mma(D, B) && B > 8 && D.d_model % 64 == 0;
}

// Rows of the partial slots of the tcgen05 kernel: 128-row tiles.
int tc_tiles_max(const dv_layer_desc &D) { return ceil_div(mma_rows_max(D), 128); }

void set_row_tc(RowArgs &a, const dv_layer_desc &D, void *ws, const WsLayout &L)
{
    a.mma_nt = rowdot_mma_tiles(a.B);  // 2 or 4: batch tiles of 16 or 32 rows
    rowdot_tc_plan(a.K, 8 * a.mma_nt, &a.mma_seg, &a.mma_ks);
    a.mma_groups = tc_tiles_max(D);
    a.mma_part = at<float>(ws, L.mma_part);
    a.mma_cnt = at<int>(ws, L.mma_cnt);
}

// PRED1 (head scores, low-rank factor u) and PRED2 (neuron scores +
// first-digit histogram).  pdl_first: launch PRED1 as a programmatic
// dependent of the previous kernel on the stream.  No entry point does: a
// cross-stream event wait before the call is not covered by PRED1's grid
// wait (a lookahead predictor on a second stream then overwrote a selection
// still in use), and the gain measured was within noise.
dv_status run_scores(const dv_layer_desc &D, const dv_layer_weights &w, const float *xp, int B,
                     float *sh_user, float *sn_user, void *ws, const WsLayout &L, Launch &lc,
                     const PredSide *side = nullptr, bool pdl_first = false)
{
    const int d = D.d_model, H = D.n_heads, N = D.d_ffn, r = D.pred_rank;
    int *ctl = at<int>(ws, L.ctl);

    RowArgs a;
    std::memset(&a, 0, sizeof(a));
    int nb = rowdot_nb(B, d, RK_PRED1);
    a.K = d;
    a.geo = rowdot_geometry(d, D.dtype, nb);
    a.max_rows = H + r;
    a.B = B;
    a.x = xp;
    a.x_ld = d;
    a.w0 = w.pred_h;
    a.w1 = w.pred_a;
    a.split_rows = H;
    a.out0 = at<float>(ws, L.s_h);
    a.out1 = at<float>(ws, L.u);
    a.user_scores = sh_user;
    a.part = at<float>(ws, L.part_pred1);
    a.rowcnt = at<int>(ws, L.cnt_pred1);
    a.status = ctl;
    a.stamps = lc.kernel_stamps();
    if (side)
        a.side_flag = ctl + kSideFlagWord;
    dim3 grid(lc.nsm, ceil_div(B, nb));
    dv_status s = lc.mark();
    if (s)
        return s;
    // (the no-allocation scratch has no tensor-core partial slots: CUDA cores)
    const bool mma = pred_mma(D, B) && L.mma_cnt != 0;
    if (mma) {
        const size_t sm = set_mma(a, D, ws, L, lc.nsm, H + r);
        if (failed(launch_rowdot_mma(RK_PRED1, a, dim3(lc.nsm, ceil_div(B, 8 * a.mma_nt)), sm,
                                     lc.st, lc.pdl && pdl_first)))
            return DV_ERR_CUDA;
    } else if (failed(launch_rowdot(RK_PRED1, D.dtype, nb, a, grid, rowdot_smem(RK_PRED1, nb, d),
                                  lc.st, lc.pdl && pdl_first))) {
        return DV_ERR_CUDA;
    }

    RowArgs b2;
    std::memset(&b2, 0, sizeof(b2));
    nb = rowdot_nb(B, r, RK_PRED2);
    b2.K = r;
    b2.geo = rowdot_geometry(r, D.dtype, nb);
    b2.max_rows = N;
    b2.B = B;
    b2.x = at<float>(ws, L.u);
    b2.x_ld = r;
    b2.w0 = w.pred_b;
    b2.out0 = at<float>(ws, L.s_n);
    b2.user_scores = sn_user;
    b2.hist = at<int>(ws, L.hist);
    b2.part = at<float>(ws, L.part_pred1);
    b2.rowcnt = at<int>(ws, L.cnt_pred1);
    b2.status = ctl;
    b2.stamps = lc.kernel_stamps();
    if (side) {
        // the tensor-core kernel splits the side work (norm(x) rows) over up
        // to kMaxSelCtas CTAs: one CTA's L2 bandwidth took ~60 us for 8 rows
        // of 12288 at OPT-175B
        b2.side_cta = mma ? std::min(B, kMaxSelCtas) : 1;
        b2.side = *side;
        b2.side_flag = ctl + kSideFlagWord;
        b2.side_done = ctl + kSideDoneWord;
    }
    grid = dim3(lc.nsm, ceil_div(B, nb));
    if ((s = lc.mark()))
        return s;
    if (mma) {
        const size_t sm = set_mma(b2, D, ws, L, lc.nsm, N);
        if (failed(launch_rowdot_mma(RK_PRED2, b2, dim3(lc.nsm, ceil_div(B, 8 * b2.mma_nt)), sm,
                                     lc.st, lc.pdl)))
            return DV_ERR_CUDA;
    } else if (failed(launch_rowdot(RK_PRED2, D.dtype, nb, b2, grid, rowdot_smem(RK_PRED2, nb, r),
                                  lc.st, lc.pdl))) {
        return DV_ERR_CUDA;
    }
    return DV_OK;
}

// Attention block.  Fused mode (ns != nullptr): the head union and norm(x)
// come from the stage-2 predictor's side CTA, the QKV kernel runs the
// neuron pass after its rows and the attention kernel's CTA 0 finishes the
// neuron selection.  first: this is the call's first launch.
dv_status run_attn(const dv_layer_desc &D, const dv_layer_weights &w, const float *x, int B,
                   const int32_t *u_h, const int32_t *n_u_h, int max_u_h, void *kc, void *vc,
                   int kv_len, float *h1, void *ws, const WsLayout &L, Launch &lc, bool first,
                   const NeuronSel *ns)
{
    const int d = D.d_model, H = D.n_heads, dh = D.head_dim;
    int *ctl = at<int>(ws, L.ctl);

    RowArgs a;
    std::memset(&a, 0, sizeof(a));
    int nb = rowdot_nb(B, d, RK_QKV);
    a.K = d;
    a.geo = rowdot_geometry(d, D.dtype, nb);
    a.max_rows = 3 * max_u_h * dh;
    a.B = B;
    a.n_sel = n_u_h;
    a.max_sel = max_u_h;
    a.sel = u_h;
    a.sel_range = H;
    a.x = x;
    a.x_ld = d;
    a.norm_g = w.ln1_g;
    a.norm_b = w.ln1_b;
    a.norm_kind = D.norm;
    a.eps = D.ln_eps;
    a.w0 = w.w_qkv;
    a.bias = w.b_qkv;
    a.H = H;
    a.dh = dh;
    a.out0 = at<float>(ws, L.q);
    a.kc = kc;
    a.vc = vc;
    a.kv_len = kv_len;
    a.kv_cap = D.kv_cap;
    a.q_scale = (float)(1.0 / std::sqrt((double)dh));
    a.part = at<float>(ws, L.part_qkv);
    a.rowcnt = at<int>(ws, L.cnt_qkv);
    a.status = ctl;
    a.stamps = lc.kernel_stamps();
    size_t smem = rowdot_smem(RK_QKV, nb, d);
    if (ns) {
        // heads and norm(x) come from the stage-2 predictor kernel's side CTA;
        // the last CTA of this kernel selects the neurons
        a.x = at<float>(ws, L.xn);
        a.norm_g = nullptr;
        a.norm_b = nullptr;
        // the last min(B, kMaxSelCtas) CTAs select the neurons, rows split
        // among them (one CTA takes about 7 us per row at N = 49152)
        a.side_cta = B < kMaxSelCtas ? B : kMaxSelCtas;
        a.ns = *ns;
        a.side_flag = ctl + kSideFlagWord;
        const size_t fs = select_final_smem(D.d_ffn);
        if (fs > smem)
            smem = fs;
    }
    dim3 grid(lc.nsm, ceil_div(B, nb));
    dv_status s = lc.mark();
    if (s)
        return s;
    if (use_mma(D, B)) {
        size_t sm = set_mma(a, D, ws, L, lc.nsm);
        if (ns && select_final_smem(D.d_ffn) > sm)
            sm = select_final_smem(D.d_ffn);
        // The stage-2 predictor -> QKV boundary stays in stream order here:
        // with it and the stage-1 -> stage-2 boundary both programmatic, the
        // tensor-core QKV kernel's CTAs ran about 80 us longer (median 90 ->
        // 169 us at OPT-175B, batch 4; the decode 405 -> 498 us), while either
        // boundary alone, or every other boundary, costs nothing (every
        // boundary but this one: 400 us).
        if (failed(launch_rowdot_mma(RK_QKV, a, dim3(lc.nsm, ceil_div(B, 8 * a.mma_nt)), sm,
                                     lc.st, false)))
            return DV_ERR_CUDA;
    } else if (failed(launch_rowdot(RK_QKV, D.dtype, nb, a, grid, smem, lc.st, lc.pdl && !first))) {
        return DV_ERR_CUDA;
    }

    AttnArgs t;
    std::memset(&t, 0, sizeof(t));
    t.B = B;
    t.H = H;
    t.dh = dh;
    t.kv_cap = D.kv_cap;
    t.kv_len = kv_len;
    t.n_sel = n_u_h;
    t.max_sel = max_u_h;
    t.sel = u_h;
    t.q = at<float>(ws, L.q);
    t.kc = kc;
    t.vc = vc;
    const int L1 = kv_len + 1;
    // chunks per (batch row, head): enough CTAs to cover the SMs once
    int chunks = lc.nsm / (B * max_u_h);
    if (chunks < 1)
        chunks = 1;
    if (chunks > L1)
        chunks = L1;
    if (chunks > kMaxAttnChunks)
        chunks = kMaxAttnChunks;
    t.splits = chunks;
    t.part = at<float>(ws, L.attn_part);
    t.status = ctl;
    t.stamps = lc.kernel_stamps();
    if (ns)
        t.side_flag = ctl + kSideFlagWord;
    const int lpk = (int)((size_t)dh * esize(D.dtype) / 16);
    if ((s = lc.mark()))
        return s;
    if (failed(launch_attn(D.dtype, lpk, t, dim3(lc.nsm), lc.st, lc.pdl)))
        return DV_ERR_CUDA;

    ColArgs c;
    std::memset(&c, 0, sizeof(c));
    c.d = d;
    c.B = B;
    c.n_sel = n_u_h;
    c.max_sel = max_u_h;
    c.sel = u_h;
    c.sel_range = H;
    c.dh = dh;
    c.w = w.w_oT;
    c.attn_rec = at<float>(ws, L.attn_part);
    c.attn_C = chunks;
    c.res = x;
    c.bias = w.b_o;
    c.out = h1;
    c.part = at<float>(ws, L.cpart_o);
    c.cnt = at<int>(ws, L.ccnt_o);
    c.status = ctl;
    c.stamps = lc.kernel_stamps();
    nb = colacc_nb(B);
    if ((s = lc.mark()))
        return s;
    if (use_mma(D, B)) {
        const int nt = colacc_mma_tiles(B, CK_OPROJ);
        if (failed(launch_colacc_mma(CK_OPROJ, nt, c, dim3(lc.nsm, ceil_div(B, 8 * nt)), lc.st, lc.pdl)))
            return DV_ERR_CUDA;
    } else if (failed(launch_colacc(CK_OPROJ, D.dtype, nb, c, dim3(lc.nsm, ceil_div(B, nb)), lc.st,
                             lc.pdl))) {
        return DV_ERR_CUDA;
    }
    return DV_OK;
}

dv_status run_mlp(const dv_layer_desc &D, const dv_layer_weights &w, const float *h1, int B,
                  const int32_t *u_n, const int32_t *n_u_n, int max_u_n, float *y, void *ws,
                  const WsLayout &L, Launch &lc, bool first)
{
    const int d = D.d_model, N = D.d_ffn;
    int *ctl = at<int>(ws, L.ctl);

    if (!use_mma(D, B) && mlp_fused_ok(D, B, max_u_n, lc.nsm)) {
        // one pass over the selected fc1 rows and fc2 columns, then the
        // partials' sum
        MlpArgs m;
        std::memset(&m, 0, sizeof(m));
        m.swiglu = D.mlp == DV_MLP_SWIGLU;
        m.d = d;
        m.N = N;
        m.B = B;
        m.sel = u_n;
        m.n_sel = n_u_n;
        m.max_sel = max_u_n;
        m.h1 = h1;
        m.norm_g = w.ln2_g;
        m.norm_b = w.ln2_b;
        m.norm_kind = D.norm;
        m.eps = D.ln_eps;
        m.w1 = w.w1;
        m.b1 = w.b1;
        m.w2T = w.w2T;
        m.part = at<float>(ws, L.mlp_part);
        m.status = ctl;
        m.stamps = lc.kernel_stamps();
        PartSumArgs ps;
        std::memset(&ps, 0, sizeof(ps));
        ps.d = d;
        ps.B = B;
        ps.nparts = lc.nsm;
        ps.res = h1;
        ps.bias = w.b2;
        ps.part = m.part;
        ps.out = y;
        ps.stamps = lc.kernel_stamps();
        ps.stamp_ctas = lc.nsm;  // the timeline has a slot per SM
        dv_status s = lc.mark();
        if (s)
            return s;
        if (failed(launch_mlp(D.dtype, m, lc.nsm, lc.st, lc.pdl && !first)))
            return DV_ERR_CUDA;
        if ((s = lc.mark()))
            return s;
        if (failed(launch_part_sum(D.dtype, ps, lc.st)))
            return DV_ERR_CUDA;
        return DV_OK;
    }

    RowArgs a;
    std::memset(&a, 0, sizeof(a));
    int nb = rowdot_nb(B, d, RK_FC1);
    const int sw = D.mlp == DV_MLP_SWIGLU ? 1 : 0;
    a.swiglu = sw;
    a.K = d;
    a.geo = rowdot_geometry(d, D.dtype, nb);
    a.max_rows = max_u_n << sw;
    a.B = B;
    a.n_sel = n_u_n;
    a.max_sel = max_u_n;
    a.sel = u_n;
    a.sel_range = N;
    a.x = h1;
    a.x_ld = d;
    a.norm_g = w.ln2_g;
    a.norm_b = w.ln2_b;
    a.norm_kind = D.norm;
    a.eps = D.ln_eps;
    a.w0 = w.w1;
    a.bias = w.b1;
    a.out0 = at<float>(ws, L.act);
    a.part = at<float>(ws, L.part_fc1);
    a.rowcnt = at<int>(ws, L.cnt_fc1);
    a.status = ctl;
    a.stamps = lc.kernel_stamps();
    dv_status s = lc.mark();
    if (s)
        return s;
    if (row_tc(D, B)) {  // the tcgen05 fc1 kernel (opt-in, dv_set_row_kernel)
        set_row_tc(a, D, ws, L);
        if (failed(launch_rowdot_tc(a, dim3(lc.nsm, ceil_div(B, 8 * a.mma_nt)), lc.st,
                                    lc.pdl && !first)))
            return DV_ERR_CUDA;
    } else if (use_mma(D, B)) {
        const size_t sm = set_mma(a, D, ws, L, lc.nsm);
        if (failed(launch_rowdot_mma(RK_FC1, a, dim3(lc.nsm, ceil_div(B, 8 * a.mma_nt)), sm, lc.st,
                              lc.pdl && !first)))
            return DV_ERR_CUDA;
    } else if (failed(launch_rowdot(RK_FC1, D.dtype, nb, a, dim3(lc.nsm, ceil_div(B, nb)),
                             rowdot_smem(RK_FC1, nb, d), lc.st, lc.pdl && !first))) {
        return DV_ERR_CUDA;
    }

    ColArgs c;
    std::memset(&c, 0, sizeof(c));
    c.d = d;
    c.B = B;
    c.n_sel = n_u_n;
    c.max_sel = max_u_n;
    c.sel = u_n;
    c.sel_range = N;
    c.dh = 1;
    c.swiglu = sw;
    c.w = w.w2T;
    c.coef = at<float>(ws, L.act);
    c.coef_ld = max_u_n << sw;
    c.res = h1;
    c.bias = w.b2;
    c.out = y;
    c.part = at<float>(ws, L.cpart_2);
    c.cnt = at<int>(ws, L.ccnt_2);
    c.status = ctl;
    c.stamps = lc.kernel_stamps();
    nb = colacc_nb(B);
    if ((s = lc.mark()))
        return s;
    if (use_mma(D, B)) {
        const int nt = colacc_mma_tiles(B, CK_FC2);
        if (failed(launch_colacc_mma(CK_FC2, nt, c, dim3(lc.nsm, ceil_div(B, 8 * nt)), lc.st, lc.pdl)))
            return DV_ERR_CUDA;
    } else if (failed(launch_colacc(CK_FC2, D.dtype, nb, c, dim3(lc.nsm, ceil_div(B, nb)), lc.st,
                             lc.pdl))) {
        return DV_ERR_CUDA;
    }
    return DV_OK;
}

dv_status check_ws(const dv_layer_desc &D, int B, void *ws, size_t ws_bytes, WsLayout *L)
{
    if (!ws_layout(D, B, L))
        return DV_ERR_INVALID_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L->total)
        return DV_ERR_WORKSPACE;
    return DV_OK;
}

bool sel_ok(const dv_selection *sel)
{
    return sel && sel->idx_h && sel->idx_n && sel->u_h && sel->n_u_h && sel->u_n && sel->n_u_n;
}

// The streaming kernel (dv_stream.cu) serves binary16 layers with 128-wide
// heads at batches of 1 and 2 whose shapes fit its tiling: rows of at most
// 6 x 384 chunks (d <= 18432), predictor rank <= 1024, a column-group split
// of the SMs, and one CTA per SM with the shared memory below.  Fills `a`
// (all but the call's pointers) and returns true when it serves.
bool stream_plan(const dv_layer_desc &D, int B, int k_h, int k_n, int kv_len, int G,
                 StreamArgs *a, int *ni, size_t *smem)
{
    if (D.dtype != DV_F16 || D.head_dim != 128 || B < 1 || B > 2 || G < 2 ||
        G > kStreamMaxCtas || D.neuron_block > 1 || D.mlp != DV_MLP_RELU)
        return false;
    const int d = D.d_model, cpr = d / 8;
    const int nseg = ceil_div(cpr, kStreamUnitBytes / 16);
    if (d % 8 || nseg > 6 || D.pred_rank % 8 || D.pred_rank > 1024 || D.n_heads > 256)
        return false;
    int ncg = 0;
    for (int c : {8, 4, 2, 1})
        if (G % c == 0 && 8 * ceil_div(cpr, c) <= 2048 && G / c <= kStreamMaxGroupCtas) {
            ncg = c;
            break;
        }
    if (!ncg)
        return false;
    const int cg = 8 * ceil_div(cpr, ncg), gm = G / ncg;
    const int max_u_h = std::min(D.n_heads, B * k_h), max_u_n = std::min(D.d_ffn, B * k_n);
    int C = (G - 1) / (B * max_u_h);
    C = std::max(1, std::min(C, std::min(kMaxAttnChunks, kv_len + 1)));
    const size_t uni = stream_union_bytes(B, D.d_ffn, max_u_h, max_u_n, cg, gm);
    const size_t fixed = stream_smem_bytes((int)uni, 0);
    if (fixed + 3 * (size_t)kStreamStageBytes > kStreamSmemMax)
        return false;
    const int nst = (int)std::min<size_t>(kStreamMaxStages,
                                          (kStreamSmemMax - fixed) / kStreamStageBytes);
    const size_t sm = stream_smem_bytes((int)uni, nst);
    // one CTA per SM must fit; the answer is kept per device and size
    struct Fit {
        int dev, nb, ni;
        size_t smem;
        int ctas;
    };
    static std::mutex mu;
    static Fit known[32];
    static int n_known = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    int ctas = -1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int i = 0; i < n_known; ++i)
            if (known[i].dev == dev && known[i].nb == B && known[i].ni == nseg &&
                known[i].smem == sm)
                ctas = known[i].ctas;
        if (ctas < 0) {
            ctas = stream_ctas_per_sm(B, nseg, sm);
            if (n_known < 32)
                known[n_known++] = Fit{dev, B, nseg, sm, ctas};
        }
    }
    if (ctas < 1)
        return false;
    std::memset(a, 0, sizeof(*a));
    a->B = B;
    a->d = d;
    a->H = D.n_heads;
    a->dh = D.head_dim;
    a->N = D.d_ffn;
    a->r = D.pred_rank;
    a->k_h = k_h;
    a->k_n = k_n;
    a->max_u_h = max_u_h;
    a->max_u_n = max_u_n;
    a->kv_len = kv_len;
    a->kv_cap = D.kv_cap;
    a->norm_kind = D.norm;
    a->eps = D.ln_eps;
    a->q_scale = (float)(1.0 / std::sqrt((double)D.head_dim));
    a->G = G;
    a->nseg = nseg;
    a->ncg = ncg;
    a->gm = gm;
    a->cg = cg;
    a->attn_C = C;
    a->nstages = nst;
    a->uni_bytes = (int)uni;
    *ni = nseg;
    *smem = sm;
    return true;
}

dv_status stream_launch(const dv_layer_desc &D, const dv_layer_weights &w, const float *x,
                        const float *xp, int B, int k_h, int k_n, void *kc, void *vc, int kv_len,
                        const dv_selection &sel, float *h1, float *y, void *ws, const WsLayout &L,
                        const Launch &lc, bool *served, unsigned long long *stamps = nullptr,
                        int n_stamps = 0)
{
    StreamArgs a;
    int ni = 0;
    size_t smem = 0;
    *served = false;
    if (!stream_plan(D, B, k_h, k_n, kv_len, lc.nsm, &a, &ni, &smem))
        return DV_OK;
    *served = true;
    if (stamps && n_stamps < lc.nsm * kStreamStamps)
        return DV_ERR_INVALID_ARG;
    a.stamps = stamps;
    a.x = x;
    a.x_pred = xp;
    a.ln1_g = w.ln1_g;
    a.ln1_b = w.ln1_b;
    a.w_qkv = w.w_qkv;
    a.b_qkv = w.b_qkv;
    a.w_oT = w.w_oT;
    a.b_o = w.b_o;
    a.ln2_g = w.ln2_g;
    a.ln2_b = w.ln2_b;
    a.w1 = w.w1;
    a.b1 = w.b1;
    a.w2T = w.w2T;
    a.b2 = w.b2;
    a.pred_h = w.pred_h;
    a.pred_a = w.pred_a;
    a.pred_b = w.pred_b;
    a.kc = kc;
    a.vc = vc;
    a.idx_h = sel.idx_h;
    a.idx_n = sel.idx_n;
    a.u_h = sel.u_h;
    a.n_u_h = sel.n_u_h;
    a.u_n = sel.u_n;
    a.n_u_n = sel.n_u_n;
    a.h1 = h1;
    a.y = y;
    a.part1 = at<float>(ws, L.st_part1);
    a.s_h = at<float>(ws, L.s_h);
    a.s_n = at<float>(ws, L.s_n);
    a.partQ = at<float>(ws, L.st_partQ);
    a.attn_rec = at<float>(ws, L.attn_part);
    a.partO = at<float>(ws, L.st_partO);
    a.stats = at<float>(ws, L.st_stats);
    a.partF = at<float>(ws, L.st_partF);
    a.partY = at<float>(ws, L.st_partY);
    a.hist = at<int>(ws, L.hist);
    a.rowbits = at<unsigned>(ws, L.nbits);
    a.cand_key = at<unsigned>(ws, L.cand_key);
    a.cand_idx = at<int>(ws, L.cand_idx);
    a.cand_cnt = at<int>(ws, L.cand_cnt);
    a.ctl = at<int>(ws, L.ctl);
    return cuda_status(launch_stream(B, ni, a, smem, lc.st));
}

dv_status layer_decode_impl(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                            const float *x_pred, int batch, int k_heads, int k_neurons, void *kc,
                            void *vc, int kv_len, const dv_selection *sel, float *h1, float *y,
                            void *ws, size_t ws_bytes, void *const *events, int n_events,
                            void *stream, bool pdl_first, bool persistent = false,
                            unsigned long long *stamps = nullptr, int n_stamps = 0)
{
    dv_status s = check_desc(desc);
    if (s)
        return s;
    if ((s = check_weights(w)))
        return s;
    const dv_layer_desc &D = *desc;
    if (batch < 1 || batch > DV_MAX_BATCH || k_heads < 1 || k_heads > D.n_heads ||
        !k_neurons_ok(D, k_neurons) || kv_len < 0 || kv_len >= D.kv_cap)
        return DV_ERR_INVALID_ARG;
    if (!ptr_ok(x) || (x_pred && !ptr_ok(x_pred)) || !ptr_ok(y) || (h1 && !ptr_ok(h1)) ||
        !ptr_ok(kc) || !ptr_ok(vc) || !sel_ok(sel))
        return DV_ERR_INVALID_ARG;
    WsLayout L;
    if ((s = check_ws(D, batch, ws, ws_bytes, &L)))
        return s;
    Launch lc;
    if ((s = make_launch(stream, events, n_events, &lc)))
        return s;
    lc.pdl = pdl_for(D, batch);
    if (events && n_events < layer_launches(D, batch) + 1)
        return DV_ERR_INVALID_ARG;
    float *h1p = h1 ? h1 : at<float>(ws, L.h1);
    const int max_u_h = batch * k_heads < D.n_heads ? batch * k_heads : D.n_heads;
    const int max_u_n = batch * k_neurons < D.d_ffn ? batch * k_neurons : D.d_ffn;
    const NeuronSel ns = make_neuron_sel(D, batch, k_neurons, *sel, ws, L);
    PredSide side;
    std::memset(&side, 0, sizeof(side));
    side.s_h = at<float>(ws, L.s_h);
    side.H = D.n_heads;
    side.k_h = k_heads;
    side.idx_h = sel->idx_h;
    side.u_h = sel->u_h;
    side.n_u_h = sel->n_u_h;
    side.x = x;
    side.x_ld = D.d_model;
    side.d = D.d_model;
    side.g = w->ln1_g;
    side.beta = w->ln1_b;
    side.norm_kind = D.norm;
    side.eps = D.ln_eps;
    side.xn = at<float>(ws, L.xn);
    if (stamps && !persistent) {
        if ((size_t)n_stamps < (size_t)kLayerLaunches * lc.nsm * kChainStamps)
            return DV_ERR_INVALID_ARG;
        lc.stamps = stamps;
    }
    if (persistent) {  // the streaming kernel, where it serves
        bool served = false;
        s = events ? DV_OK
                   : stream_launch(D, *w, x, x_pred ? x_pred : x, batch, k_heads, k_neurons, kc,
                                   vc, kv_len, *sel, h1p, y, ws, L, lc, &served, stamps, n_stamps);
        if (s)
            return s;
        return served ? DV_OK : DV_ERR_UNSUPPORTED;
    }
    if ((s = run_scores(D, *w, x_pred ? x_pred : x, batch, nullptr, nullptr, ws, L, lc, &side,
                        pdl_first)))
        return s;
    if ((s = run_attn(D, *w, x, batch, sel->u_h, sel->n_u_h, max_u_h, kc, vc, kv_len, h1p, ws, L,
                      lc, false, &ns)))
        return s;
    if ((s = run_mlp(D, *w, h1p, batch, sel->u_n, sel->n_u_n, max_u_n, y, ws, L, lc, false)))
        return s;
    if ((s = lc.mark()))
        return s;
    return DV_OK;
}

}  // namespace

namespace dv {

bool ws_layout(const dv_layer_desc &D, int B, WsLayout *L)
{
    if (check_desc(&D) != DV_OK || B < 1 || B > DV_MAX_BATCH)
        return false;
    const size_t d = D.d_model, H = D.n_heads, dh = D.head_dim, N = D.d_ffn, r = D.pred_rank;
    const size_t bp = (size_t)batch_pad(B);
    const size_t splits = (size_t)kMaxAttnChunks;
    const size_t S = (size_t)ceil_div(D.d_model, 32 * (int)(16 / esize(D.dtype)));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    std::memset(L, 0, sizeof(*L));
    L->ctl = take(64 * 4);
    L->hist = take((size_t)B * kTopkBins * 4);
    L->s_h = take((size_t)B * H * 4);
    L->u = take((size_t)B * r * 4);
    L->s_n = take((size_t)B * N * 4);
    L->q = take((size_t)B * H * dh * 4);
    L->attn_part = take((size_t)B * H * splits * (kAttnRec + dh) * 4);
    L->h1 = take((size_t)B * d * 4);
    L->act = take((size_t)B * N * 2 * 4);  // two values per neuron for SwiGLU
    L->part_pred1 = take(bp * kMaxWarps * 2 * 4);
    L->part_qkv = take(bp * kMaxWarps * 2 * 4);
    L->part_fc1 = take(bp * kMaxWarps * 2 * 4);
    L->cnt_pred1 = take(bp * (H + r > N ? H + r : N) * 4);
    L->cnt_qkv = take(bp * 3 * H * dh * 4);
    L->cnt_fc1 = take(bp * N * 2 * 4);  // two rows per neuron for SwiGLU
    // column kernel: two partial slots per CTA, one column block each, for
    // every batch row of its passes (the tensor-core variant's last pass of
    // 8 nt rows may run past the padded batch)
    const size_t cb_max = (size_t)colacc_block_cols(D.dtype, 1) * 2;  // NB x block columns
    const size_t cnt_t = (size_t)std::max(colacc_mma_tiles(B, CK_OPROJ), colacc_mma_tiles(B, CK_FC2));
    const size_t cbp = std::max(bp, (size_t)ceil_div(B, 8 * (int)cnt_t) * 8 * cnt_t);
    L->cpart_o = take(cbp * (kMaxWarps / kWarpsPerBlock) * 2 * cb_max * 4);
    L->cpart_2 = take(cbp * (kMaxWarps / kWarpsPerBlock) * 2 * cb_max * 4);
    L->ccnt_o = take(bp * S * 4);
    L->ccnt_2 = take(bp * S * 4);
    L->stage_x = take((size_t)B * d * 4);
    L->stage_xp = take((size_t)B * d * 4);
    L->stage_y = take((size_t)B * d * 4);
    L->sel_idx_h = take((size_t)B * H * 4);
    L->sel_idx_n = take((size_t)B * N * 4);
    L->sel_u_h = take(H * 4);
    L->sel_n_u_h = take(4);
    L->sel_u_n = take(N * 4);
    L->sel_n_u_n = take(4);
    L->nbits = take((size_t)B * ((N + 31) / 32) * 4);
    L->sel_ubits = take(((N + 31) / 32) * 4);
    L->cand_key = take((size_t)B * kTopkCand * 4);
    L->cand_idx = take((size_t)B * kTopkCand * 4);
    L->cand_cnt = take((size_t)B * 4);
    L->xn = take((size_t)B * d * 4);
    {  // tensor-core row kernel (binary16, nt batch tiles of 8 per weight pass)
        int S = 1, ks = 0;
        const int nt = rowdot_mma_tiles(B);
        rowdot_mma_plan(D.d_model, nt, &S, &ks);
        const size_t passes = (size_t)ceil_div(B, 8 * nt);
        const size_t groups = (size_t)ceil_div(mma_rows_max(D), 16);
        size_t part = passes * groups * S * 128 * nt * 4;
        if (nt >= 2) {  // or the tcgen05 fc1 kernel's: 128-row tiles x its segments
            int St = 1, kst = 0;
            rowdot_tc_plan(D.d_model, 8 * nt, &St, &kst);
            const size_t tc = passes * (size_t)tc_tiles_max(D) * St * 128 * (8 * nt) * 4;
            part = std::max(part, tc);
        }
        L->mma_part = take(part);
        L->mma_cnt = take(passes * groups * 4);
    }
    {  // streaming kernel (binary16, batches 1-2; sized for either when B <= 2)
        const size_t nseg = (size_t)ceil_div(D.d_model / 8, kStreamUnitBytes / 16);
        const size_t bs = (size_t)(B <= 2 ? B : 0);
        L->st_part1 = take(bs * (H + r) * nseg * 4);
        L->st_partQ = take(bs * 3 * H * dh * nseg * 4);
        L->st_partF = take(bs * N * nseg * 4);
        // G x cg <= gm x (d + 8 ncg), gm <= kStreamMaxGroupCtas, ncg <= 8
        L->st_partO = take(bs * kStreamMaxGroupCtas * (d + 64) * 4);
        L->st_partY = take(bs * kStreamMaxGroupCtas * (d + 64) * 4);
        L->st_stats = take(bs * kStreamMaxCtas * 4 * 4);
        L->mlp_part = take(bs * kPartMaxCtas * d * 4);
    }
    L->total = off;
    L->bpad = (int)bp;
    L->attn_splits_max = (int)splits;
    return true;
}

}  // namespace dv

extern "C" {

// Every launch's own return code is checked where it is made; the entry
// points do not end with cudaGetLastError(), whose per-thread slot the
// process shares with every other user of the same CUDA runtime library (an
// error another component left there is not this call's).  The error behind
// the last DV_ERR_CUDA of this thread is kept in t_cuda_error instead.
dv_status dv_set_row_kernel(int variant)
{
    if (variant != 0 && variant != 1)
        return DV_ERR_INVALID_ARG;
    g_row_variant.store(variant);
    return DV_OK;
}

int dv_cuda_error(void)
{
    const int e = t_cuda_error;
    t_cuda_error = 0;
    return e;
}

const char *dv_status_string(int status)
{
    switch (status) {
    case DV_OK: return "ok";
    case DV_ERR_INVALID_ARG: return "invalid argument";
    case DV_ERR_UNSUPPORTED: return "unsupported shape or type";
    case DV_ERR_CUDA: return "CUDA runtime error";
    case DV_ERR_TIMEOUT: return "device wait timed out";
    case DV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DV_ERR_DEVICE_INDEX: return "a kernel met an index outside its range";
    case DV_ERR_SCRATCH_LIMIT:
        return "shape and batch need more scratch than dv_predict_topk_noalloc holds";
    default: return "unknown status";
    }
}

int dv_abi_version(void) { return DV_ABI_VERSION; }

size_t dv_workspace_size(const dv_layer_desc *desc, int batch)
{
    if (!desc)
        return 0;
    WsLayout L;
    if (!ws_layout(*desc, batch, &L))
        return 0;
    return L.total;
}

int dv_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256)
        return DV_ERR_WORKSPACE;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

int dv_check(void *ws, size_t ws_bytes, void *stream)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256)
        return DV_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (failed(cudaStreamSynchronize(st)))
        return DV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DV_ERR_CUDA;
    if (v != 0 && cudaMemset(ws, 0, sizeof(int)) != cudaSuccess)
        return DV_ERR_CUDA;
    return v;
}

int dv_layer_decode_launches(const dv_layer_desc *desc, int batch)
{
    if (check_desc(desc) != DV_OK || batch < 1 || batch > DV_MAX_BATCH)
        return 0;
    return layer_launches(*desc, batch);
}

int dv_mlp_one_pass(const dv_layer_desc *desc, int batch, int max_u_n)
{
    if (check_desc(desc) != DV_OK || batch < 1 || batch > DV_MAX_BATCH || max_u_n < 1)
        return 0;
    Launch lc;
    if (make_launch(nullptr, nullptr, 0, &lc) != DV_OK)
        return 0;
    return !use_mma(*desc, batch) && mlp_fused_ok(*desc, batch, max_u_n, lc.nsm);
}

int dv_layer_decode_persistent_ok(const dv_layer_desc *desc, int batch)
{
    if (check_desc(desc) != DV_OK || batch < 1 || batch > DV_MAX_BATCH)
        return 0;
    Launch lc;
    StreamArgs a;
    int ni = 0;
    size_t sm = 0;
    return make_launch(nullptr, nullptr, 0, &lc) == DV_OK &&
           stream_plan(*desc, batch, desc->n_heads, desc->d_ffn, desc->kv_cap - 1, lc.nsm, &a,
                       &ni, &sm);
}

int dv_predict_topk(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x_pred,
                    int batch, int k_heads, int k_neurons, const dv_selection *sel,
                    float *scores_h, float *scores_n, void *ws, size_t ws_bytes, void *stream)
{
    dv_status s = check_desc(desc);
    if (s)
        return s;
    if (!w || !ptr_ok(w->pred_h) || !ptr_ok(w->pred_a) || !ptr_ok(w->pred_b))
        return DV_ERR_INVALID_ARG;
    const dv_layer_desc &D = *desc;
    if (batch < 1 || batch > DV_MAX_BATCH || k_heads < 1 || k_heads > D.n_heads ||
        !k_neurons_ok(D, k_neurons) || !ptr_ok(x_pred) || !sel_ok(sel))
        return DV_ERR_INVALID_ARG;
    WsLayout L;
    if ((s = check_ws(D, batch, ws, ws_bytes, &L)))
        return s;
    Launch lc;
    if ((s = make_launch(stream, nullptr, 0, &lc)))
        return s;
    lc.pdl = pdl_for(D, batch);
    if ((s = run_scores(D, *w, x_pred, batch, scores_h, scores_n, ws, L, lc)))
        return s;
    SelectArgs sa;
    std::memset(&sa, 0, sizeof(sa));
    sa.s_h = at<float>(ws, L.s_h);
    sa.H = D.n_heads;
    sa.k_h = k_heads;
    sa.idx_h = sel->idx_h;
    sa.u_h = sel->u_h;
    sa.n_u_h = sel->n_u_h;
    sa.ns = make_neuron_sel(D, batch, k_neurons, *sel, ws, L);
    if (failed(launch_select(sa, lc.nsm, lc.st)))
        return DV_ERR_CUDA;
    return DV_OK;
}

int dv_sparse_attn(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x, int batch,
                   const int32_t *u_h, const int32_t *n_u_h, int max_u_h, void *k_cache,
                   void *v_cache, int kv_len, float *h1, void *ws, size_t ws_bytes, void *stream)
{
    dv_status s = check_desc(desc);
    if (s)
        return s;
    if ((s = check_weights(w)))
        return s;
    const dv_layer_desc &D = *desc;
    if (batch < 1 || batch > DV_MAX_BATCH || max_u_h < 1 || max_u_h > D.n_heads || kv_len < 0 ||
        kv_len >= D.kv_cap || !ptr_ok(x) || !ptr_ok(h1) || !u_h || !n_u_h || !ptr_ok(k_cache) ||
        !ptr_ok(v_cache) || x == h1)
        return DV_ERR_INVALID_ARG;
    WsLayout L;
    if ((s = check_ws(D, batch, ws, ws_bytes, &L)))
        return s;
    Launch lc;
    if ((s = make_launch(stream, nullptr, 0, &lc)))
        return s;
    lc.pdl = pdl_for(D, batch);
    if ((s = run_attn(D, *w, x, batch, u_h, n_u_h, max_u_h, k_cache, v_cache, kv_len, h1, ws, L,
                      lc, true, nullptr)))
        return s;
    return DV_OK;
}

int dv_sparse_mlp(const dv_layer_desc *desc, const dv_layer_weights *w, const float *h1, int batch,
                  const int32_t *u_n, const int32_t *n_u_n, int max_u_n, float *y, void *ws,
                  size_t ws_bytes, void *stream)
{
    dv_status s = check_desc(desc);
    if (s)
        return s;
    if ((s = check_weights(w)))
        return s;
    const dv_layer_desc &D = *desc;
    if (batch < 1 || batch > DV_MAX_BATCH || max_u_n < 1 || max_u_n > D.d_ffn || !ptr_ok(h1) ||
        !ptr_ok(y) || !u_n || !n_u_n || h1 == y)
        return DV_ERR_INVALID_ARG;
    WsLayout L;
    if ((s = check_ws(D, batch, ws, ws_bytes, &L)))
        return s;
    Launch lc;
    if ((s = make_launch(stream, nullptr, 0, &lc)))
        return s;
    lc.pdl = pdl_for(D, batch);
    if ((s = run_mlp(D, *w, h1, batch, u_n, n_u_n, max_u_n, y, ws, L, lc, true)))
        return s;
    return DV_OK;
}

int dv_layer_decode_presel(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                           int batch, const int32_t *u_h, const int32_t *n_u_h, int max_u_h,
                           const int32_t *u_n, const int32_t *n_u_n, int max_u_n, void *k_cache,
                           void *v_cache, int kv_len, float *h1, float *y, void *ws,
                           size_t ws_bytes, void *stream)
{
    dv_status s = check_desc(desc);
    if (s)
        return s;
    if ((s = check_weights(w)))
        return s;
    const dv_layer_desc &D = *desc;
    if (batch < 1 || batch > DV_MAX_BATCH || max_u_h < 1 || max_u_h > D.n_heads || max_u_n < 1 ||
        max_u_n > D.d_ffn || kv_len < 0 || kv_len >= D.kv_cap || !ptr_ok(x) || !ptr_ok(y) ||
        (h1 && !ptr_ok(h1)) || !u_h || !n_u_h || !u_n || !n_u_n || !ptr_ok(k_cache) ||
        !ptr_ok(v_cache) || x == y || x == h1 || (h1 && h1 == y))
        return DV_ERR_INVALID_ARG;
    WsLayout L;
    if ((s = check_ws(D, batch, ws, ws_bytes, &L)))
        return s;
    Launch lc;
    if ((s = make_launch(stream, nullptr, 0, &lc)))
        return s;
    lc.pdl = pdl_for(D, batch);
    float *h1p = h1 ? h1 : at<float>(ws, L.h1);
    if ((s = run_attn(D, *w, x, batch, u_h, n_u_h, max_u_h, k_cache, v_cache, kv_len, h1p, ws, L,
                      lc, true, nullptr)))
        return s;
    if ((s = run_mlp(D, *w, h1p, batch, u_n, n_u_n, max_u_n, y, ws, L, lc, false)))
        return s;
    return DV_OK;
}

int dv_layer_decode(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                    const float *x_pred, int batch, int k_heads, int k_neurons, void *k_cache,
                    void *v_cache, int kv_len, const dv_selection *sel, float *h1, float *y,
                    void *ws, size_t ws_bytes, void *stream)
{
    return layer_decode_impl(desc, w, x, x_pred, batch, k_heads, k_neurons, k_cache, v_cache,
                             kv_len, sel, h1, y, ws, ws_bytes, nullptr, 0, stream, false);
}

int dv_layer_decode_chained(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                            const float *x_pred, int batch, int k_heads, int k_neurons,
                            void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                            float *h1, float *y, void *ws, size_t ws_bytes, void *stream)
{
    return layer_decode_impl(desc, w, x, x_pred, batch, k_heads, k_neurons, k_cache, v_cache,
                             kv_len, sel, h1, y, ws, ws_bytes, nullptr, 0, stream, false);
}

int dv_layer_decode_stamped(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                            const float *x_pred, int batch, int k_heads, int k_neurons,
                            void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                            float *h1, float *y, void *ws, size_t ws_bytes, int persistent,
                            unsigned long long *stamps, int n_stamps, void *stream)
{
    if (!stamps || (reinterpret_cast<uintptr_t>(stamps) & 7u) || n_stamps < 0)
        return DV_ERR_INVALID_ARG;
    return layer_decode_impl(desc, w, x, x_pred, batch, k_heads, k_neurons, k_cache, v_cache,
                             kv_len, sel, h1, y, ws, ws_bytes, nullptr, 0, stream, false,
                             persistent != 0, stamps, n_stamps);
}

int dv_layer_decode_persistent(const dv_layer_desc *desc, const dv_layer_weights *w,
                               const float *x, const float *x_pred, int batch, int k_heads,
                               int k_neurons, void *k_cache, void *v_cache, int kv_len,
                               const dv_selection *sel, float *h1, float *y, void *ws,
                               size_t ws_bytes, void *stream)
{
    return layer_decode_impl(desc, w, x, x_pred, batch, k_heads, k_neurons, k_cache, v_cache,
                             kv_len, sel, h1, y, ws, ws_bytes, nullptr, 0, stream, false, true);
}

int dv_layer_decode_traced(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                           const float *x_pred, int batch, int k_heads, int k_neurons,
                           void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                           float *h1, float *y, void *ws, size_t ws_bytes, void *const *events,
                           int n_events, void *stream)
{
    if (!events)
        return DV_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i)
        if (!events[i])
            return DV_ERR_INVALID_ARG;
    return layer_decode_impl(desc, w, x, x_pred, batch, k_heads, k_neurons, k_cache, v_cache,
                             kv_len, sel, h1, y, ws, ws_bytes, events, n_events, stream, false);
}

int dv_layer_decode_host(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x_host,
                         const float *x_pred_host, int batch, int k_heads, int k_neurons,
                         void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                         float *y_host, void *ws, size_t ws_bytes, void *stream)
{
    dv_status s = check_desc(desc);
    if (s)
        return s;
    if (!x_host || !y_host || batch < 1 || batch > DV_MAX_BATCH)
        return DV_ERR_INVALID_ARG;
    WsLayout L;
    if ((s = check_ws(*desc, batch, ws, ws_bytes, &L)))
        return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)batch * desc->d_model * sizeof(float);
    float *x_dev = at<float>(ws, L.stage_x);
    float *xp_dev = x_pred_host ? at<float>(ws, L.stage_xp) : nullptr;
    float *y_dev = at<float>(ws, L.stage_y);
    if (cudaMemcpyAsync(x_dev, x_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return DV_ERR_CUDA;
    if (xp_dev &&
        cudaMemcpyAsync(xp_dev, x_pred_host, bytes, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return DV_ERR_CUDA;
    dv_selection own;
    if (!sel) {  // keep the selection in the workspace
        own.idx_h = at<int32_t>(ws, L.sel_idx_h);
        own.idx_n = at<int32_t>(ws, L.sel_idx_n);
        own.u_h = at<int32_t>(ws, L.sel_u_h);
        own.n_u_h = at<int32_t>(ws, L.sel_n_u_h);
        own.u_n = at<int32_t>(ws, L.sel_u_n);
        own.n_u_n = at<int32_t>(ws, L.sel_n_u_n);
        sel = &own;
    }
    s = layer_decode_impl(desc, w, x_dev, xp_dev, batch, k_heads, k_neurons, k_cache, v_cache,
                          kv_len, sel, nullptr, y_dev, ws, ws_bytes, nullptr, 0, stream, false);
    if (s)
        return s;
    if (cudaMemcpyAsync(y_host, y_dev, bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return DV_ERR_CUDA;
    return cuda_status(cudaStreamSynchronize(st));
}

int dv_test_hold_wait(void *ws, size_t ws_bytes, int wait_id, int budget_us, void *stream)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < 256)
        return DV_ERR_WORKSPACE;
    if (wait_id < 0 || wait_id > 9 || budget_us < 1)
        return DV_ERR_INVALID_ARG;
    static_assert(kSwHold == kSwBudget + 1, "budget and hold are adjacent control words");
    const int words[2] = {wait_id ? budget_us : 0, wait_id};
    return cuda_status(cudaMemcpyAsync(static_cast<int *>(ws) + kSwBudget, words, sizeof(words),
                                       cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)));
}

int dv_hbm_copy(void *dst, const void *src, size_t bytes, void *stream)
{
    if (!ptr_ok(dst) || !ptr_ok(src) || bytes == 0 || (bytes & 15u))
        return DV_ERR_INVALID_ARG;
    Launch lc;
    dv_status s = make_launch(stream, nullptr, 0, &lc);
    if (s)
        return s;
    return cuda_status(launch_copy(dst, src, bytes / 16, lc.nsm * 4, lc.st));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// dv_predict_topk_noalloc: the predictor and top-k with their scratch in a
// fixed device array of this library instead of a caller workspace.
//
// Some callers cannot hand the library device memory when they predict: a
// serving loop whose memory pool has already given all free HBM to its KV
// cache arena, or code that must not call an allocator at that point because
// cudaMalloc/cudaFree synchronise the device.  This entry point allocates
// nothing: its scratch is a static device array, one per device, whose
// address is looked up once per device.

namespace {

constexpr size_t kNoallocScratch = DV_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratch];

std::mutex g_noalloc_mu;
struct NoallocBase {
    unsigned long long ctx_id;  // unique ID of the context the address belongs to (0: none)
    void *ptr;
};
NoallocBase g_noalloc_base[kMaxDevices];

// Layout inside the scratch.  The fields the kernels require to start at
// zero (status word, first-digit histograms, candidate counters, row
// counters) come first, in [0, *zero_bytes); every other field is written
// before it is read.
size_t noalloc_layout(const dv_layer_desc &D, int B, WsLayout *L, size_t *zero_bytes)
{
    const size_t H = D.n_heads, N = D.d_ffn, r = D.pred_rank;
    const size_t bp = (size_t)batch_pad(B);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    std::memset(L, 0, sizeof(*L));
    L->ctl = take(64 * 4);
    L->hist = take((size_t)B * kTopkBins * 4);
    L->cand_cnt = take((size_t)B * 4);
    L->cnt_pred1 = take(bp * (H + r > N ? H + r : N) * 4);
    *zero_bytes = off;
    L->s_h = take((size_t)B * H * 4);
    L->u = take((size_t)B * r * 4);
    L->s_n = take((size_t)B * N * 4);
    L->part_pred1 = take(bp * kMaxWarps * 2 * 4);
    L->nbits = take((size_t)B * ((N + 31) / 32) * 4);
    L->sel_ubits = take(((N + 31) / 32) * 4);
    L->cand_key = take((size_t)B * kTopkCand * 4);
    L->cand_idx = take((size_t)B * kTopkCand * 4);
    L->total = off;
    L->bpad = (int)bp;
    return off;
}

// Unique ID of the calling thread's current CUDA context (0 if there is none
// or the driver cannot tell).  Context IDs are never reused within a process,
// so a context re-created after cudaDeviceReset gets a new one.  The two
// driver calls are resolved through the runtime, so the library does not link
// the driver library itself.
unsigned long long current_context_id()
{
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the scratch on the current device.  It is looked up with
// the device current the first time the device is used, and again whenever
// the device's context has changed since (after cudaDeviceReset the module is
// loaded anew and the array may move); where the context cannot be
// identified it is looked up on every call.
dv_status noalloc_base(void **out)
{
    int dev = 0;
    if (failed(cudaGetDevice(&dev)))
        return DV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return DV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> guard(g_noalloc_mu);
    NoallocBase &nb = g_noalloc_base[dev];
    const unsigned long long id = current_context_id();
    if (id != 0 && nb.ctx_id == id && nb.ptr) {
        *out = nb.ptr;
        return DV_OK;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
        return DV_ERR_CUDA;
    if (reinterpret_cast<uintptr_t>(p) & 255u)
        return DV_ERR_WORKSPACE;
    nb.ctx_id = current_context_id();  // the lookup may have created the context
    nb.ptr = p;
    *out = p;
    return DV_OK;
}

}  // namespace

extern "C" {

int dv_predict_topk_noalloc(const dv_layer_desc *desc, const dv_layer_weights *w,
                            const float *x_pred, int batch, int k_heads, int k_neurons,
                            const dv_selection *sel, float *scores_h, float *scores_n,
                            void *stream)
{
    dv_status s = check_desc(desc);
    if (s)
        return s;
    if (!w || !ptr_ok(w->pred_h) || !ptr_ok(w->pred_a) || !ptr_ok(w->pred_b))
        return DV_ERR_INVALID_ARG;
    const dv_layer_desc &D = *desc;
    if (batch < 1 || batch > DV_MAX_BATCH || k_heads < 1 || k_heads > D.n_heads ||
        !k_neurons_ok(D, k_neurons) || !ptr_ok(x_pred) || !sel_ok(sel))
        return DV_ERR_INVALID_ARG;
    WsLayout L;
    size_t zero_bytes = 0;
    if (noalloc_layout(D, batch, &L, &zero_bytes) > kNoallocScratch)
        return DV_ERR_SCRATCH_LIMIT;
    void *ws = nullptr;
    if ((s = noalloc_base(&ws)))
        return s;
    Launch lc;
    if ((s = make_launch(stream, nullptr, 0, &lc)))
        return s;
    lc.pdl = pdl_for(D, batch);
    if (cudaMemsetAsync(ws, 0, zero_bytes, lc.st) != cudaSuccess)
        return DV_ERR_CUDA;
    if ((s = run_scores(D, *w, x_pred, batch, scores_h, scores_n, ws, L, lc)))
        return s;
    SelectArgs sa;
    std::memset(&sa, 0, sizeof(sa));
    sa.s_h = at<float>(ws, L.s_h);
    sa.H = D.n_heads;
    sa.k_h = k_heads;
    sa.idx_h = sel->idx_h;
    sa.u_h = sel->u_h;
    sa.n_u_h = sel->n_u_h;
    sa.ns = make_neuron_sel(D, batch, k_neurons, *sel, ws, L);
    if (failed(launch_select(sa, lc.nsm, lc.st)))
        return DV_ERR_CUDA;
    return DV_OK;
}

}  // extern "C"
