// dv_internal.h -- argument blocks, workspace layout and launcher entry
// points shared by the host code and the kernel translation units of libdv.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "dv.h"

namespace dv {

constexpr int kThreads = 512;                    // block size of the GEMV kernels
constexpr int kWarpsPerBlock = kThreads / 32;
constexpr int kTopkBins = 2048;                  // first radix digit: 11 bits
constexpr int kMaxWarps = 8192;                  // bound on grid warps (workspace sizing)
constexpr int kTopkCand = 4096;                  // top-k candidates kept in shared memory
constexpr int kMaxAttnChunks = 64;               // attention chunks per (batch row, head)
constexpr int kAttnRec = 4;                      // floats before o[] in a split record
constexpr size_t kSmemCap = 200 * 1024;          // dynamic shared memory budget
constexpr int kMaxDevices = 64;

// One-time set-up of a kernel per device (its shared-memory opt-in, made
// once so that later launches can be captured in a CUDA graph): run(f) calls
// f() with the current device until it has succeeded once.  First calls from
// several host threads are serialised by a mutex; later calls cost one
// atomic load.
class DeviceOnce {
public:
    template <class F>
    cudaError_t run(F &&f)
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess)
            return e;
        if (dev < 0 || dev >= kMaxDevices)
            return cudaErrorInvalidDevice;
        if (done_[dev].load(std::memory_order_acquire))
            return cudaSuccess;
        std::lock_guard<std::mutex> lock(mu_);
        if (done_[dev].load(std::memory_order_relaxed))
            return cudaSuccess;
        e = f();
        if (e == cudaSuccess)
            done_[dev].store(true, std::memory_order_release);
        return e;
    }

private:
    std::atomic<bool> done_[kMaxDevices] = {};
    std::mutex mu_;
};

enum RowKind { RK_PRED1 = 0, RK_PRED2 = 1, RK_QKV = 2, RK_FC1 = 3 };
enum ColKind { CK_OPROJ = 0, CK_FC2 = 1 };

// ---------------------------------------------------------------------------
// Neuron top-k state shared by the kernels that compute it (workspace).
struct NeuronSel {
    const float *s_n;      // [B][N] scores
    int B, N, k;
    int *hist;             // [B][kTopkBins] first-digit histogram (zero at rest)
    unsigned *rowbits;     // [B][ceil(N/32)] kept-set bitmaps
    unsigned *cand_key;    // [B][kTopkCand]
    int *cand_idx;         // [B][kTopkCand]
    int *cand_cnt;         // [B] (zero at rest)
    int32_t *idx_n;        // [B][k] outputs
    int32_t *u_n, *n_u_n;
    int *status;
    int block;             // > 1: blocks of this many contiguous neurons (block_select)
    unsigned *gubits;      // [ceil(N/32)] union of a selection split over CTAs (zero at rest)
    int *gdone;            // CTAs done with their rows (zero at rest)
};

struct SelectArgs {
    const float *s_h;      // [B][H] head scores
    int H, k_h;
    int32_t *idx_h, *u_h, *n_u_h;
    NeuronSel ns;
};

// ---------------------------------------------------------------------------
// Row-dot kernel: out_row = dot(W[row], xs) over a list of rows, with an
// optional norm of the activations and a per-kind epilogue.
//
// Work geometry (rowdot_geometry): a row has `cpr` 16-byte chunks.  Long rows
// (cpr >= 32*U) are cut into `nsu` units of `ucr` chunks each ("segment
// mode"); short rows are packed `rpu` to a unit, one group of 32/rpu lanes per
// row ("multi-row mode", nsu == 0, ucr == cpr).  Units are dealt to the
// grid's warps in contiguous, balanced ranges.
struct RowGeo {
    int cpr;   // chunks per row
    int ucr;   // chunks of one row handled by one lane group per unit
    int nsu;   // units per row (segment mode), 0 in multi-row mode
    int rpu;   // rows per unit (multi-row mode), 1 in segment mode
    int U;     // chunks in flight per lane (template parameter of the kernel)
};

// Side work of the stage-2 predictor kernel in the fused decode (one CTA):
// head selection and the normalised input of the attention block.
struct PredSide {
    const float *s_h;     // head scores [B][H]
    int H, k_h;
    int32_t *idx_h, *u_h, *n_u_h;
    const float *x;       // layer input [B][x_ld]
    int x_ld, d;
    const void *g, *beta; // norm parameters (dtype of the weights)
    int norm_kind;
    float eps;
    float *xn;            // out: norm(x) [B][d]
};

// Timeline of the chained decode (profiling): kernel k of the call writes,
// for each CTA c of its first batch tile, %globaltimer nanoseconds to
// stamps[(k * CTAs + c) * kChainStamps + i]: i = 0 the CTA starts, 1 its
// inputs are ready (the grid dependency or the side flag passed), 2 it ends;
// slot 3 holds the SM it ran on; 4 .. 7 are points inside a kernel
// (attention: 4 warp 0's first batch of keys consumed, 5 warp 0's keys done,
// 6 the chunk record written; the one-pass MLP: 4 its activations summed).
constexpr int kChainStamps = 8;

// Polls of the side-work flag before the QKV kernel falls back to waiting
// for the whole stage-2 predictor grid.
constexpr int kSideSpin = 20000;

struct RowArgs {
    int swiglu;       // FC1 of a SwiGLU layer: rows 2j, 2j + 1 are slot j's gate and up
    int K;            // row length in elements
    RowGeo geo;
    int B;            // batch rows
    int max_rows;     // host bound on the number of rows
    const int32_t *n_sel;  // device length of the gather list (QKV, FC1)
    int max_sel;      // host bound on *n_sel
    const int32_t *sel;    // gather list (u_h for QKV, u_n for FC1)
    int sel_range;    // valid gathered indices are [0, sel_range)
    const float *x;   // activations [B][x_ld]
    int x_ld;
    const void *norm_g, *norm_b;  // NULL: no norm
    int norm_kind;
    float eps;
    const void *w0, *w1;  // PRED1: pred_h, pred_a; PRED2: pred_b; QKV: w_qkv; FC1: w1
    const void *bias;     // QKV: b_qkv; FC1: b1
    int H, dh, split_rows;
    float *out0, *out1;   // PRED1: s_h, u; PRED2: s_n; QKV: q; FC1: act
    float *user_scores;   // optional copy of the scores (predictor kinds)
    void *kc, *vc;
    int kv_len, kv_cap;
    float q_scale;
    float *part;          // range-boundary partials [tiles][warps][2][NB]
    int *rowcnt;          // segments accounted per row [tiles][max_rows], zero at rest
    int *hist;            // PRED2: first-digit histogram [B][kTopkBins], zero at rest
    // Fused decode only: the last CTA column does side work instead of rows --
    // PRED2: head selection and norm(x) (PredSide); QKV: the whole neuron
    // selection (NeuronSel), after waiting for the stage-2 grid.
    int side_cta;
    PredSide side;
    NeuronSel ns;
    // fused decode: PRED1 clears it, PRED2's side CTA sets it once its results
    // are published; the QKV kernel starts on it instead of the grid dependency
    int *side_flag;
    int *side_done;       // PRED2 with several side CTAs: how many have finished
    // tensor-core variant (k_rowdot_mma): K segments, their length, group
    // partials [tiles][groups][segments][16][8] and arrival counters
    int mma_seg, mma_ks, mma_groups;
    int mma_nt;       // 8-row batch tiles per weight pass (1, 2 or 4)
    float *mma_part;
    int *mma_cnt;
    int *status;
    unsigned long long *stamps;  // optional timeline [CTAs][4] (kChainStamps)
};

// Column-accumulate kernel: out[b][c] = res[b][c] + bias[c]
//                                      + sum_i coef[b][i] * W[row(i)][c].
// FC2 of a SwiGLU layer (swiglu): coef[b][i] = silu(g) u from the pair
// (g, u) = act[b][2i], act[b][2i + 1].
struct ColArgs {
    int swiglu;
    int d;
    int B;
    const int32_t *n_sel;
    int max_sel;
    const int32_t *sel;   // u_h (OPROJ, rows = heads x dh) or u_n (FC2)
    int sel_range;
    int dh;
    const void *w;        // w_oT or w2T
    const float *coef;    // FC2: [B][coef_ld]
    int coef_ld;
    // OPROJ: the attention kernel's chunk records [B][max_sel][attn_C][kAttnRec + dh]
    // (running max, sum of weights, weighted V), merged into the coefficients
    const float *attn_rec;
    int attn_C;
    const float *res;     // [B][d]
    const void *bias;     // [d]
    float *out;           // [B][d]
    float *part;          // block partials [tiles][CTAs][2][NB][block columns]
    int *cnt;             // rows accounted per column block [tiles][blocks], zero at rest
    int *status;
    unsigned long long *stamps;  // optional timeline [CTAs][4] (kChainStamps)
};

// 16-byte chunks per lane of the column kernel (columns per block = 32 * P *
// elements per chunk); fewer for larger batch tiles to bound registers.
template <int NB>
__host__ __device__ constexpr int colacc_chunks() { return NB <= 2 ? 2 : 1; }

// Dynamic shared memory of the column kernel: block partials of the 16 warps
// (CB columns each), then kColStageRows row offsets and coefficients (nb per
// row) and kColMaxCover partial slots.
constexpr int kColStageRows = 1024;
constexpr int kColMaxCover = 512;
__host__ __device__ constexpr size_t colacc_smem_bytes(int cb, int nb)
{
    return (size_t)kWarpsPerBlock * cb * 4 + (size_t)kColStageRows * 8 +
           (size_t)kColStageRows * nb * 4 + (size_t)kColMaxCover * 4;
}

// Split-KV decode attention over the selected heads.
struct AttnArgs {
    int B, H, dh, kv_cap, kv_len;
    const int32_t *n_sel;
    int max_sel;
    const int32_t *sel;
    const float *q;       // [B][max_sel][dh], already scaled
    const void *kc, *vc;  // [B][H][kv_cap][dh]
    int splits;           // chunks per (batch row, head)
    float *part;          // out: chunk records [B][max_sel][splits][kAttnRec + dh]
    const int *side_flag; // fused decode: set once the head union is published
    int *status;
    unsigned long long *stamps;  // optional timeline [CTAs][4] (kChainStamps)
};

// Sparse MLP block as one pass (dv_mlp.cu; batches 1 and 2): CTA c computes
// the activations of its share of the neuron union and accumulates their
// fc2 rows into part[c][b][d]; a second kernel adds the partials, h1 and b2.
struct MlpArgs {
    int swiglu;           // gate and up rows per neuron, act = silu(gate) * up
    int d, N, B;
    const int32_t *sel;   // u_n
    const int32_t *n_sel;
    int max_sel;
    const float *h1;      // [B][d] (the attention block's output)
    const void *norm_g, *norm_b;
    int norm_kind;
    float eps;
    const void *w1, *b1, *w2T;
    float *part;          // [CTAs][B][d]
    int *status;
    unsigned long long *stamps;  // optional timeline
};
constexpr int kMlpMaxRows = 64;   // neurons per CTA
constexpr int kMlpMaxSeg = 8;     // fc1 row segments
bool mlp_fused_ok(const dv_layer_desc &D, int B, int max_u_n, int nsm);
cudaError_t launch_mlp(int dtype, const MlpArgs &a, int grid, cudaStream_t st, bool pdl);

// Sum of the per-CTA partials of a one-pass column accumulation
// (dv_partials.cuh): out[b][col] = res[b][col] + bias[col] + sum_c
// part[c][b][col].
struct PartSumArgs {
    int d, B, nparts;
    const float *res;
    const void *bias;
    const float *part;    // [nparts][B][d]
    float *out;           // [B][d]
    unsigned long long *stamps;
    int stamp_ctas;       // CTAs (first ones) that record a timeline
};
constexpr int kPartMaxCtas = 256;  // CTAs of a one-pass kernel (partials' workspace)
// CTAs per batch row: 64 columns each (192 at d = 12288, so every SM works)
inline int part_sum_groups(int d) { return (d / 4 + 15) / 16; }
cudaError_t launch_part_sum(int dtype, const PartSumArgs &a, cudaStream_t st);

// Dynamic shared memory of the attention kernel: the 16 warps' partial
// outputs of dh floats.
__host__ __device__ constexpr size_t attn_smem_bytes(int dh) { return (size_t)kWarpsPerBlock * dh * 4; }

constexpr int kSelStage = 1024;  // gather indices a row-dot CTA stages in shared memory

// ---------------------------------------------------------------------------
// Workspace layout (byte offsets from the workspace base, 256-byte aligned).
struct WsLayout {
    size_t ctl;       // int[64]: [0] status
    size_t hist;      // int[B][kTopkBins]
    size_t s_h, u, s_n;
    size_t q, attn_part;  // attention chunk records [B][H][splits][kAttnRec + dh]
    size_t h1, act;
    size_t part_pred1, part_qkv, part_fc1;
    size_t cnt_pred1, cnt_qkv, cnt_fc1;
    size_t cpart_o, cpart_2, ccnt_o, ccnt_2;
    size_t stage_x, stage_xp, stage_y;
    size_t sel_idx_h, sel_idx_n, sel_u_h, sel_n_u_h, sel_u_n, sel_n_u_n;
    size_t nbits, cand_key, cand_idx, cand_cnt;  // neuron selection state
    size_t sel_ubits;  // union bitmap of a selection split over CTAs
    size_t xn;  // normalised input of the attention block (fused decode)
    size_t mma_part, mma_cnt;  // tensor-core row kernel: group partials and counters
    // streaming kernel: segment sums of the predictor, QKV and fc1 rows,
    // column partials of the out-projection and fc2, norm statistics
    size_t st_part1, st_partQ, st_partF, st_partO, st_partY, st_stats;
    size_t mlp_part;  // one-pass MLP: per-CTA partials of y
    size_t total;
    int bpad;         // batch rounded up to the largest batch tile (8)
    int attn_splits_max;
};

bool ws_layout(const dv_layer_desc &D, int B, WsLayout *L);

// Launchers (one per kernel family); return the CUDA error of the launch.
cudaError_t launch_rowdot(int kind, int dtype, int nb, const RowArgs &a, dim3 grid, size_t smem,
                          cudaStream_t st, bool pdl);
cudaError_t launch_colacc(int kind, int dtype, int nb, const ColArgs &a, dim3 grid,
                          cudaStream_t st, bool pdl);
cudaError_t launch_attn(int dtype, int lanes_per_key, const AttnArgs &a, dim3 grid,
                        cudaStream_t st, bool pdl);
// Stand-alone selection (dv_predict_topk): head select + neuron pass on `grid`
// CTAs, then the final neuron step on one CTA.
cudaError_t launch_select(const SelectArgs &a, int grid, cudaStream_t st);
size_t select_final_smem(int N);
cudaError_t launch_copy(void *dst, const void *src, size_t n16, int grid, cudaStream_t st);

// Largest-batch tile each kernel family handles per CTA.
int rowdot_nb(int B, int K, int kind);
RowGeo rowdot_geometry(int K, int dtype, int nb);
int colacc_nb(int B);
int colacc_block_cols(int dtype, int nb);
size_t rowdot_smem(int kind, int nb, int K);
// Tensor-core row kernel (binary16 weights, batch tiles of 8; QKV and FC1).
cudaError_t launch_rowdot_mma(int kind, const RowArgs &a, dim3 grid, size_t smem,
                              cudaStream_t st, bool pdl);
void rowdot_mma_plan(int K, int nt, int *S, int *ks);
// tcgen05 variant of the fc1 row kernel (batch tiles of 8 mma_nt = 16 or 32
// rows; mma_groups = the 128-row tile stride of the partial slots).
void rowdot_tc_plan(int K, int bt, int *S, int *ks);
size_t rowdot_tc_smem();
cudaError_t launch_rowdot_tc(const RowArgs &a, dim3 grid, cudaStream_t st, bool pdl);
// Staged activation row stride (halves) of the tensor-core row kernel for K
// segments of ks: 64 bytes modulo 128, so the two 8-row halves of a warp's
// 16-byte fragment reads fall in distinct banks (a stride of 0 modulo 128
// doubles the shared-memory wavefronts).
__host__ __device__ inline int rowdot_mma_ldx(int ks) { return ks + (ks % 64 == 0 ? 32 : 64); }
size_t rowdot_mma_smem(int ks, int nt);
int rowdot_mma_tiles(int B);  // batch tiles per weight pass
constexpr int kMmaMinBatch = 3;  // batches from which binary16 layers use tensor cores
// Tensor-core column kernel (binary16, nt batch tiles of 8 per CTA;
// out-projection, fc2): grid.y = ceil(B / (8 nt)).
int colacc_mma_tiles(int B, int kind);
cudaError_t launch_colacc_mma(int kind, int nt, const ColArgs &a, dim3 grid, cudaStream_t st,
                              bool pdl);
size_t colacc_mma_smem();


// ---------------------------------------------------------------------------
// Streaming layer kernel (dv_stream.cu): the whole decode step as one
// persistent cooperative grid whose producer warp streams every selected
// weight byte into a shared-memory ring (bulk copies) while the consumer warps
// compute; phases hand over through counters in the workspace control words.
constexpr int kStreamStageBytes = 32768;  // one ring stage
constexpr int kStreamMaxStages = 16;
constexpr int kStreamThreads = 416;       // 12 consumer warps + the producer warp
constexpr int kStreamUnitBytes = 6144;    // a row segment: 384 chunks of 16 bytes
constexpr int kStreamStamps = 32;         // phase timeline points per CTA

// Control words of the streaming kernel (int offsets into the workspace's
// control block; all zero at rest).
enum StreamWord {
    kSwPred1 = 16,  // CTAs done with the predictor's first stage
    kSwPred2,       // ... its neuron scores (histogram complete)
    kSwPass,        // ... their share of the neuron selection pass
    kSwQkv,         // ... QKV (all but the last CTA)
    kSwAttn,        // ... attention (all CTAs)
    kSwNorm2,       // ... the out-projection sums of their columns and the norm statistics
    kSwFc1,         // ... fc1
    kSwExit,        // CTAs at the end; the last resets the words
    kSwHeads,       // flag: head selection published
    kSwNeurons,     // flag: neuron selection published
    kSwBudget,      // test hook: wait budget in microseconds (0: the default)
    kSwHold,        // test hook: id of a wait that is made never to complete (0: none)
    kSwOproj = 32,  // [8] per column group: CTAs done with their out-projection partials
    kSwFc2 = 40,    // [8] per column group: ... fc2 partials
    kSwEnd = 48
};

struct StreamArgs {
    int B, d, H, dh, N, r;
    int k_h, k_n, max_u_h, max_u_n;
    int kv_len, kv_cap;
    int norm_kind;
    float eps, q_scale;
    const float *x, *x_pred;
    // binary16 weights (dv_layer_weights order)
    const void *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_oT, *b_o, *ln2_g, *ln2_b, *w1, *b1, *w2T, *b2,
        *pred_h, *pred_a, *pred_b;
    void *kc, *vc;
    int32_t *idx_h, *idx_n, *u_h, *n_u_h, *u_n, *n_u_n;
    float *h1, *y;
    // geometry
    int G;       // CTAs (one per SM)
    int nseg;    // 384-chunk segments of a d-long row
    int ncg;     // column groups of the out-projection and fc2
    int gm;      // CTAs per column group (G / ncg)
    int cg;      // columns of the widest group (groups split the row's 16-byte
                 // chunks into ncg nearly equal runs); stride of the partials
    int attn_C;  // attention chunks per (batch row, head)
    int nstages; // ring stages
    int uni_bytes;  // shared-memory union region (phase scratch)
    // workspace
    float *part1;     // [B][(H + r) nseg] predictor row-segment sums
    float *s_h, *s_n; // [B][H], [B][N] scores
    float *partQ;     // [B][3 max_u_h dh nseg] QKV row-segment sums
    float *attn_rec;  // [B][max_u_h][attn_C][kAttnRec + dh]
    float *partO;     // [G][B][cg] out-projection column partials (a group's own width)
    float *stats;     // [G][B][4] norm statistics of each CTA's columns
    float *partF;     // [B][max_u_n nseg] fc1 row-segment sums
    float *partY;     // [G][B][cg] fc2 column partials
    int *hist;        // [B][kTopkBins]
    unsigned *rowbits, *cand_key;
    int *cand_idx, *cand_cnt;
    int *ctl;         // control block ([0] status)
    unsigned long long *stamps;  // optional phase timeline [G][kStreamStamps] (globaltimer)
};

// The streaming kernel's column partials assume at most this many CTAs per
// column group (workspace sizing).
constexpr int kStreamMaxGroupCtas = 32;
constexpr int kStreamMaxCtas = 512;

// Launch of the streaming kernel for a batch of nb (1 or 2) and ni 384-chunk
// segments per row (1..6); cooperative, `grid` CTAs of kStreamThreads.
cudaError_t launch_stream(int nb, int ni, const StreamArgs &a, size_t smem, cudaStream_t st);
// CTAs of the streaming kernel one SM holds at this shared memory (0 on error).
int stream_ctas_per_sm(int nb, int ni, size_t smem);
// Shared memory of the streaming kernel: fixed part + union + ring, and the
// fixed part alone.
size_t stream_smem_bytes(int uni_bytes, int nstages);
size_t stream_fixed_smem();
// Bytes of the union region (the largest phase scratch) for these sizes.
size_t stream_union_bytes(int B, int N, int max_u_h, int max_u_n, int cg, int gm);
constexpr size_t kStreamSmemMax = 226 * 1024;  // dynamic part (the opt-in limit is 227 KB)

}  // namespace dv
