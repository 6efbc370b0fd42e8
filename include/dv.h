/*
 * dv.h -- C ABI of the contextually sparse (DejaVu) decode step of one
 * transformer layer, for NVIDIA GB300 (sm_103a).
 *
 * The method (DejaVu, "Deja Vu: Contextual Sparsity for Efficient LLMs at
 * Inference Time", abstract; "DejaVu Guide: Contextual Sparsity for LLM
 * Inference", "Core Innovation 1: Asynchronous Lookahead Predictors" and
 * "Core Innovation 2: Hardware-Efficient Dynamic Sparse Matrix Execution"):
 * a cheap predictor scores the layer's attention heads and MLP neurons from
 * an input vector and keeps the top-k of each; the layer then reads from HBM
 * only the selected heads' QKV rows, out-projection rows and KV cache, and
 * the selected neurons' fc1 rows and fc2 rows.  Dense weights stay intact.
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, unless an
 *    entry point says "host".  The library allocates no memory and keeps no
 *    state between calls other than what lives in the caller's workspace.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and returns without synchronising, except where stated.
 *    Index counts stay on the device; no call reads device memory on the
 *    host, so a call can be captured in a CUDA graph.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns DV_ERR_INVALID_ARG (or DV_ERR_UNSUPPORTED for a shape
 *    the kernels do not handle) and launches nothing.  A launch failure
 *    returns DV_ERR_CUDA.  A kernel that meets a bad value at run time (an
 *    index outside its range) skips it and records the first such event in
 *    the workspace status word, which dv_check() reads.
 *  - The workspace (`ws`, `ws_bytes` >= dv_workspace_size()) must be zeroed
 *    once with dv_workspace_init() before its first use; every call leaves
 *    it ready for the next one.  Calls that share a workspace must not run
 *    concurrently.
 *  - Layouts are row-major.  Weight matrices, biases, norm parameters and the
 *    KV cache are stored in `desc.dtype` (binary32 or binary16); activations
 *    are binary32; accumulation is binary32.  Every weight and activation
 *    pointer must be 16-byte aligned.
 *
 * Shapes (d = d_model, H = n_heads, dh = head_dim, N = d_ffn, r = pred_rank,
 * B = batch, kv_cap = KV positions allocated per batch row and head):
 *   ln1_g, ln1_b, ln2_g, ln2_b, b_o, b2   [d]
 *   w_qkv  [3, H, dh, d]   (q, k, v rows of every head)
 *   b_qkv  [3, H, dh]
 *   w_oT   [H, dh, d]      (out-projection transposed: head h's input columns
 *                           are the contiguous rows w_oT[h])
 *   w1     [N, d]          (fc1: neuron j's row is contiguous)
 *   b1     [N]
 *   w2T    [N, d]          (fc2 transposed: neuron j's output column is the
 *                           contiguous row w2T[j])
 *   pred_h [H, d]          (head predictor)
 *   pred_a [r, d], pred_b [N, r]   (low-rank neuron predictor)
 *   k_cache, v_cache [B, H, kv_cap, dh]
 */
#ifndef DV_H
#define DV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DV_ABI_VERSION 2
#define DV_MAX_BATCH 32

typedef enum {
    DV_OK = 0,
    DV_ERR_INVALID_ARG = 1,  /* bad pointer, size, count or alignment */
    DV_ERR_UNSUPPORTED = 2,  /* valid but not handled (e.g. head_dim not a power of two) */
    DV_ERR_CUDA = 3,         /* a CUDA runtime call failed */
    DV_ERR_TIMEOUT = 4,      /* a bounded device-side wait gave up */
    DV_ERR_WORKSPACE = 5,    /* workspace missing, misaligned or too small */
    DV_ERR_DEVICE_INDEX = 6, /* a kernel met an index outside its range (skipped) */
    DV_ERR_SCRATCH_LIMIT = 7 /* dv_predict_topk_noalloc: shape needs more than its scratch */
} dv_status;

typedef enum { DV_F32 = 0, DV_F16 = 1 } dv_dtype;
typedef enum { DV_LAYERNORM = 0, DV_RMSNORM = 1 } dv_norm;
/* MLP of the layer: OPT's fc1, ReLU, fc2 (w1 [N, d], w2T [N, d]) or the
 * LLaMA-style SwiGLU (gate and up rows of neuron j interleaved in w1
 * [N, 2, d], b1 [N, 2]; down-projection columns in w2T [N, d]). */
typedef enum { DV_MLP_RELU = 0, DV_MLP_SWIGLU = 1 } dv_mlp;

/* Shape and storage of one layer. */
typedef struct {
    int32_t d_model;
    int32_t n_heads;
    int32_t head_dim;   /* power of two; head_dim * sizeof(dtype) in [16, 512] */
    int32_t d_ffn;
    int32_t pred_rank;
    int32_t dtype;      /* dv_dtype of weights, biases, norms and KV cache */
    int32_t norm;       /* dv_norm used before attention and before the MLP */
    float ln_eps;
    int32_t kv_cap;     /* KV positions per (batch row, head) */
    /* 0 or 1: neurons are selected one by one.  32, 64 or 128 (dividing
     * d_ffn, at most 2048 blocks): neurons are selected in blocks
     * of that many contiguous channels ("DejaVu Guide ...", "Core Innovation
     * 2", "1. Blocked Channel Sparsity"): a block's score is the largest
     * score of its members, each row keeps its k_neurons / neuron_block best
     * blocks (ties to the lower block), and k_neurons must be a multiple of
     * neuron_block. */
    int32_t neuron_block;
    int32_t mlp;        /* dv_mlp */
} dv_layer_desc;

/* Device pointers to one layer's weights (shapes in the header comment). */
typedef struct {
    const void *ln1_g, *ln1_b;
    const void *w_qkv, *b_qkv;
    const void *w_oT, *b_o;
    const void *ln2_g, *ln2_b;
    const void *w1, *b1;
    const void *w2T, *b2;
    const void *pred_h, *pred_a, *pred_b;
} dv_layer_weights;

/* Device buffers receiving a selection.
 *   idx_h [B, k_heads], idx_n [B, k_neurons]: each row's top-k, ascending;
 *   u_h [min(H, B*k_heads)], u_n [min(N, B*k_neurons)]: union of the rows,
 *   ascending; its length is written to n_u_h[0] / n_u_n[0]. */
typedef struct {
    int32_t *idx_h, *idx_n;
    int32_t *u_h, *n_u_h;
    int32_t *u_n, *n_u_n;
} dv_selection;

/* Static description of a status code (never NULL). */
const char *dv_status_string(int status);

/* The CUDA runtime's error code behind the last DV_ERR_CUDA returned on
 * this host thread (reading it clears it; 0 if none).  Diagnostic. */
int dv_cuda_error(void);

/* DV_ABI_VERSION of the built library. */
int dv_abi_version(void);

/* Row-kernel variant of the fc1 rows on the tensor cores ("DejaVu Guide:
 * Contextual Sparsity for LLM Inference", the pipeline's "Sparse Gather GEMV
 * on Tensor Cores"), process-wide, for calls issued after it returns:
 *   0  mma.sync m16n8k16 kernel (the default);
 *   1  tcgen05.mma kernel (M = 128 gathered rows, accumulator in tensor
 *      memory) for binary16 ReLU layers from 9 batch rows with d_model a
 *      multiple of 64; every other case keeps variant 0.
 * Results agree within the binary32 accumulation error; the ring, segment
 * and partial order differ, so the bits may not.  DV_ERR_INVALID_ARG for
 * another value.  Not thread-safe against calls in flight on other
 * threads. */
dv_status dv_set_row_kernel(int variant);

/* Bytes of workspace the calls below need for this layer shape and batch
 * (sized for the largest possible unions).  0 if desc or batch is invalid. */
size_t dv_workspace_size(const dv_layer_desc *desc, int batch);

/* Zero a workspace on `stream` (one cudaMemsetAsync).  Needed once before a
 * workspace is first used. */
int dv_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream`, then read the workspace status word (device faults
 * recorded by kernels, see DV_ERR_DEVICE_INDEX / DV_ERR_TIMEOUT) and clear
 * it.  Returns DV_OK if nothing was recorded. */
int dv_check(void *ws, size_t ws_bytes, void *stream);

/* Kernel launches one dv_layer_decode call enqueues (the events
 * dv_layer_decode_traced records sit around them).  0 if desc or batch is
 * invalid. */
int dv_layer_decode_launches(const dv_layer_desc *desc, int batch);

/* 1 if dv_sparse_mlp (and the MLP half of dv_layer_decode) with a neuron
 * union of at most max_u_n runs as one pass over the selected fc1 rows and
 * fc2 columns plus a kernel that adds the per-CTA partials of y, on the
 * current device; 0 if it runs as the fc1 and fc2 kernels, or for invalid
 * arguments. */
int dv_mlp_one_pass(const dv_layer_desc *desc, int batch, int max_u_n);



/* 1 if dv_layer_decode_persistent (the streaming kernel) serves this shape
 * and batch on the current device for every k_heads, k_neurons and kv_len,
 * else 0. */
int dv_layer_decode_persistent_ok(const dv_layer_desc *desc, int batch);

/*
 * dv_predict_topk -- the lookahead predictors and top-k selection.
 * ("DejaVu Guide ...", "1. Mathematical Formulation of Lookahead Predictors":
 * head mask = Top-k_head(x . W_pred_attn), neuron mask = Top-k_mlp(x .
 * W_pred_mlp); the guide's listing, DejaVuLookaheadPredictor.forward, returns
 * the kept indices sorted.)
 *   head scores   s_h[b][h] = x_pred[b] . pred_h[h]
 *   neuron scores s_n[b][j] = (x_pred[b] . pred_a^T) . pred_b[j]   (rank r)
 * For every row b: the k_heads / k_neurons largest binary32 scores, ties to
 * the lower index, written ascending to sel->idx_h[b] / sel->idx_n[b]; then
 * the union over rows to sel->u_h / sel->u_n with device counts.
 *   x_pred   [B, d] binary32 device input.
 *   scores_h [B, H], scores_n [B, N]: optional device outputs of the scores
 *            (NULL to skip).
 * Errors: DV_ERR_INVALID_ARG for k outside [1, H] / [1, N], batch outside
 * [1, DV_MAX_BATCH], NULL or misaligned pointers.
 */
int dv_predict_topk(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x_pred,
                    int batch, int k_heads, int k_neurons, const dv_selection *sel,
                    float *scores_h, float *scores_n, void *ws, size_t ws_bytes, void *stream);

/*
 * dv_sparse_attn -- head-pruned attention block with its residual.
 * ("DejaVu Guide ...", "2. Head-Pruned Attention Dispatch": an inactive head's
 * projection weights, output-projection weights and historical KV cache are
 * not read.)  For every row b, with xn = norm(x[b]; ln1_g, ln1_b) and every
 * head h in u_h[0 .. *n_u_h):
 *   q, k, v = xn . w_qkv[{0,1,2}, h]^T + b_qkv[{0,1,2}, h];  q *= 1/sqrt(dh)
 *   k_cache[b, h, kv_len] = k, v_cache[b, h, kv_len] = v  (rounded to dtype)
 *   o_h = softmax(q . K[b, h, 0..kv_len]^T) . V[b, h, 0..kv_len]
 *   h1[b] = x[b] + b_o + sum_h o_h . w_oT[h]
 * Unselected heads' caches (slot kv_len included) are not touched.
 *   x [B, d], h1 [B, d] binary32 device; u_h / n_u_h device, max_u_h = the
 *   length of u_h (upper bound of *n_u_h, <= H); 0 <= kv_len < kv_cap.
 */
int dv_sparse_attn(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x, int batch,
                   const int32_t *u_h, const int32_t *n_u_h, int max_u_h, void *k_cache,
                   void *v_cache, int kv_len, float *h1, void *ws, size_t ws_bytes, void *stream);

/*
 * dv_sparse_mlp -- contextually sparse MLP block with its residual.
 * ("DejaVu Guide ...", listing DejaVuSparseMLP.forward_sparse: gather the
 * selected fc1 rows, activation, gather the matching fc2 columns, project
 * down; DejaVuTransformerLayer.forward: pre-norm and residual add.)  For every
 * row b, with hn = norm(h1[b]; ln2_g, ln2_b) and i < *n_u_n, j = u_n[i]:
 *   a_i = max(0, hn . w1[j] + b1[j])
 *   y[b] = h1[b] + b2 + sum_i a_i * w2T[j]
 *   h1, y [B, d] binary32 device (may not alias); max_u_n = length of u_n.
 */
int dv_sparse_mlp(const dv_layer_desc *desc, const dv_layer_weights *w, const float *h1, int batch,
                  const int32_t *u_n, const int32_t *n_u_n, int max_u_n, float *y, void *ws,
                  size_t ws_bytes, void *stream);

/*
 * dv_layer_decode -- one sparse decode step of one layer: dv_predict_topk on
 * x_pred (x if NULL), then dv_sparse_attn and dv_sparse_mlp over the unions.
 * ("DejaVu Guide ...", listing DejaVuTransformerLayer.forward(x, x_prev,
 * k_heads, k_neurons).)
 *   h1: optional device output [B, d] of the attention block's result
 *       (NULL keeps it in the workspace).
 * Seven kernels (the predictors, QKV, attention, out-projection, fc1, fc2;
 * at batches 1-2 fc1 and fc2 are one pass plus a sum of partials) chained
 * by programmatic dependent launch.  Binary16 layers run QKV, fc1,
 * out-projection and fc2 on tensor cores from 3 batch rows and both
 * predictor stages from 5; there the stage-2 predictor -> QKV boundary is
 * in stream order, and from 8 rows every boundary is.  Serves every shape
 * and batch.
 */
int dv_layer_decode(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                    const float *x_pred, int batch, int k_heads, int k_neurons, void *k_cache,
                    void *v_cache, int kv_len, const dv_selection *sel, float *h1, float *y,
                    void *ws, size_t ws_bytes, void *stream);

/*
 * dv_layer_decode_chained -- the same call as dv_layer_decode (the name
 * states the launch structure for callers that compare the two paths).
 */
int dv_layer_decode_chained(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                            const float *x_pred, int batch, int k_heads, int k_neurons,
                            void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                            float *h1, float *y, void *ws, size_t ws_bytes, void *stream);

/*
 * dv_layer_decode_persistent -- dv_layer_decode as ONE persistent streaming
 * kernel (binary16 layers with 128-wide heads, batches 1 and 2, shapes that
 * fit its tiling: see dv_layer_decode_persistent_ok; DV_ERR_UNSUPPORTED,
 * launching nothing, elsewhere).  A producer warp per SM streams every
 * selected weight row into a shared-memory ring with bulk copies while the
 * other warps compute; the steps hand over through counters in the
 * workspace (bounded waits; DV_ERR_TIMEOUT in the status word if one ran
 * out).  Same selections as the chain; sums in a different order, so the
 * outputs agree to rounding.  Measured slower than the chain at the
 * OPT-175B shape (about 250 against 128 us at batch 1), so not the default.
 * Arguments as dv_layer_decode.
 */
int dv_layer_decode_persistent(const dv_layer_desc *desc, const dv_layer_weights *w,
                               const float *x, const float *x_pred, int batch, int k_heads,
                               int k_neurons, void *k_cache, void *v_cache, int kv_len,
                               const dv_selection *sel, float *h1, float *y, void *ws,
                               size_t ws_bytes, void *stream);

/*
 * dv_layer_decode_stamped -- dv_layer_decode (persistent == 0) or
 * dv_layer_decode_persistent (persistent != 0) that also records a timeline
 * in stamps (device, 8-byte aligned): %globaltimer nanoseconds, G = the
 * device's SM count.  Points a CTA does not reach are left as they were.
 *   persistent == 0: n_stamps >= 7 * G * 8; kernel k of the chain (0 the
 *     first predictor, 1 the second, 2 QKV, 3 attention, 4 out-projection,
 *     5 fc1 or the one-pass MLP, 6 fc2 or the sum of the MLP's partials)
 *     writes for each of its CTAs c (first batch tile)
 *     stamps[(k * G + c) * 8 + i]: i = 0 the CTA starts, 1 its inputs are
 *     ready, 2 it ends, 3 the SM it ran on (%smid); 4 .. 7 points inside a
 *     kernel (attention: 4 warp 0's first batch of keys consumed, 5 warp
 *     0's keys done, 6 the chunk record written; the one-pass MLP: 4 its
 *     activations summed; row kernels: 4 activations staged, 5 rows done,
 *     6 a side CTA's selection done; column kernels: 4 the first
 *     coefficients staged, 5 the last piece consumed, 6 a block's combine
 *     starts; the sum of partials: 4 summed).  Slots a CTA never reaches
 *     keep what an earlier call wrote.
 *   persistent != 0: n_stamps >= 32 G; stamps[c * 32 + i] for CTA c at
 *     fixed points: its consumer warps: 0 start, 1 first predictor stage
 *     done, 2 predictor results complete, 3 neuron scoring starts, 4 done, 5
 *     selection pass done, 6/7 QKV start/done (last CTA: neuron selection
 *     start/done), 8/9 attention start/done, 10/11 out-projection
 *     coefficients start/done, 12 out-projection done, 13/14 h1 slice
 *     start/done, 15 norm statistics complete, 16 fc1 starts, 17 fc1 done,
 *     18 fc2 starts, 19 fc2 done, 20/21 y slice start/done; its producer
 *     warp: 24 + p when it starts issuing the copies of phase p (p = 0
 *     predictor, 1 neuron scorer, 2 QKV, 3 out-projection, 4 fc1, 5 fc2),
 *     30 when it has issued its last copy.  DV_ERR_UNSUPPORTED where the
 *     streaming kernel does not serve.
 * For profiling.
 */
int dv_layer_decode_stamped(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                            const float *x_pred, int batch, int k_heads, int k_neurons,
                            void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                            float *h1, float *y, void *ws, size_t ws_bytes, int persistent,
                            unsigned long long *stamps, int n_stamps, void *stream);

/*
 * dv_layer_decode_presel -- the layer decode on a selection computed earlier:
 * dv_sparse_attn then dv_sparse_mlp in one call (five kernels, chained).
 * ("DejaVu Guide ...", "2. Pipelined Overlap Execution": the lookahead
 * predictor for layer l+1 runs while layer l computes, so by the time layer
 * l+1 starts its head and neuron sets are ready.)
 *   u_h / n_u_h (max_u_h), u_n / n_u_n (max_u_n): device unions, ascending,
 *   as dv_predict_topk writes them; x, y [B, d] binary32 device, distinct;
 *   h1 [B, d] optional output of the attention block (NULL: workspace).
 */
int dv_layer_decode_presel(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                           int batch, const int32_t *u_h, const int32_t *n_u_h, int max_u_h,
                           const int32_t *u_n, const int32_t *n_u_n, int max_u_n, void *k_cache,
                           void *v_cache, int kv_len, float *h1, float *y, void *ws,
                           size_t ws_bytes, void *stream);

/*
 * dv_layer_decode_traced -- dv_layer_decode that also records
 * events[0 .. dv_layer_decode_launches()] (cudaEvent_t handles created by the
 * caller): events[i] just before kernel i, the last one after the last
 * kernel.  For per-kernel timing; the events serialise the kernels.
 */
int dv_layer_decode_traced(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x,
                           const float *x_pred, int batch, int k_heads, int k_neurons,
                           void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                           float *h1, float *y, void *ws, size_t ws_bytes, void *const *events,
                           int n_events, void *stream);

/*
 * dv_layer_decode_host -- dv_layer_decode with HOST activations: copies
 * x_host [B, d] (and x_pred_host, may be NULL) from host memory into the
 * workspace, runs the step, copies y back to y_host [B, d] and synchronises
 * `stream` before returning.  Weights, KV cache and selection stay on the
 * device; `sel` may be NULL to keep the selection in the workspace.  Pinned
 * host memory gives asynchronous copies.
 */
int dv_layer_decode_host(const dv_layer_desc *desc, const dv_layer_weights *w, const float *x_host,
                         const float *x_pred_host, int batch, int k_heads, int k_neurons,
                         void *k_cache, void *v_cache, int kv_len, const dv_selection *sel,
                         float *y_host, void *ws, size_t ws_bytes, void *stream);

/*
 * dv_test_hold_wait -- TEST SUPPORT for the bounded waits of the streaming
 * kernel.  Arms the workspace so that the next streaming decode on it
 * (dv_layer_decode_persistent) gives every device-side wait a budget of `budget_us`
 * microseconds (> 0) and makes its wait number `wait_id` never complete:
 *   1 first predictor stage done      4 QKV done (attention starts)
 *   2 neuron scores done              5 attention done (out-projection)
 *   3 neuron selection pass done      6 out-projection partials of a group
 *   7 h1 and its norm statistics      8 fc1 done    9 fc2 partials of a group
 * That wait runs out: the kernel records DV_ERR_TIMEOUT in the status word
 * (dv_check), skips the rest of its work (outputs undefined), still returns,
 * and disarms the workspace and leaves it ready for the next call.
 * wait_id 0 disarms.  Enqueued on `stream` (a host-to-device copy of two
 * words into the workspace's control block).
 */
int dv_test_hold_wait(void *ws, size_t ws_bytes, int wait_id, int budget_us, void *stream);

/*
 * dv_hbm_copy -- copy `bytes` (a multiple of 16; both pointers 16-byte
 * aligned) from src to dst with a 16-byte-vector streaming kernel.  Used to
 * measure the copy bandwidth that serves as the roofline denominator.
 */
int dv_hbm_copy(void *dst, const void *src, size_t bytes, void *stream);

/*
 * dv_predict_topk_noalloc -- dv_predict_topk without a caller workspace.
 * This entry point is an addition of this library; the DejaVu pages have no
 * counterpart.  It is for callers that cannot provide device memory at the
 * point of prediction: a serving loop whose pool has already given all free
 * HBM to its KV cache, or code that must not call an allocator there because
 * cudaMalloc / cudaFree synchronise the device.  It allocates nothing.
 *
 * Computes exactly what dv_predict_topk computes (same kernels, same
 * arguments apart from the workspace).
 *
 * Scratch: a static device array of DV_NOALLOC_SCRATCH_BYTES inside this
 * library, one per device per process -- the exception to the "no state
 * outside the caller's workspace" convention above.  A shape and batch whose
 * scratch (status word, histograms, row counters, scores, partial sums,
 * bitmaps, candidates) does not fit is rejected with DV_ERR_SCRATCH_LIMIT and
 * nothing is launched; at the OPT-175B shape (N = 49152, r = 1000) the limit
 * is reached above batch 16.
 * Set-up: the first call on a device, with that device current, looks up the
 * scratch's device address (which may load the library's device code); the
 * address is kept per device and looked up again only when the device's CUDA
 * context has changed (for instance after cudaDeviceReset).  Make the first
 * call on a device before any stream capture begins.
 * Zeroing: every call first zeroes, on `stream`, the part of the scratch
 * that the kernels require to start at zero (status word, first-digit
 * histograms, candidate counters, row counters); everything else is written
 * before it is read.
 * Concurrency: calls whose execution overlaps on one device (different
 * streams, or different host threads) share the scratch and race; the
 * results are then wrong.  Serialise them.
 * Device-side status: none of the kernels this entry point runs records a
 * fault -- the predictor kernels read only whole weight rows inside their
 * matrices and the selection kernels take no caller indices -- so there is no
 * status word to read back (the workspace entries' dv_check has nothing to
 * report for this path either).
 */
#define DV_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

int dv_predict_topk_noalloc(const dv_layer_desc *desc, const dv_layer_weights *w,
                            const float *x_pred, int batch, int k_heads, int k_neurons,
                            const dv_selection *sel, float *scores_h, float *scores_n,
                            void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DV_H */
