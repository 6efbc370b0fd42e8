/*
 * dv_oracle.c -- plain, slow CPU oracle for the contextually sparse (DejaVu)
 * decode step of one transformer layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library; neither includes the other.
 *
 * Arithmetic: every product and sum is in IEEE binary64, in plain loops whose
 * order is the order of the definitions below.  Weights are read in the
 * caller's storage type (binary32, or binary16 decoded exactly), so the oracle
 * sees the same weight values as the GPU path.
 *
 * Threads: built plainly, the library is single-threaded and the OpenMP
 * pragmas below are ignored.  Built with -fopenmp (a second library, used only
 * to time the CPU baseline on every host core), the loops over independent
 * output elements -- scores, projected rows, output columns -- are shared out
 * among threads.  Each element is still one thread's plain loop in the same
 * order, so both builds give the same bits.
 *
 * Sources (the DejaVu pages):
 *  [P1-MF]  "DejaVu Guide: Contextual Sparsity for LLM Inference",
 *           "1. Mathematical Formulation of Lookahead Predictors": head mask =
 *           Top-k_head(x . W_pred_attn), neuron mask = Top-k_mlp(x . W_pred_mlp).
 *  [P1-LST] same page, "Step-by-Step Implementation: Building a Contextual
 *           Sparse Layer in PyTorch": the predictor scores with bias-free linear
 *           maps and keeps topk indices; the sparse MLP gathers the selected
 *           fc1 rows, applies the activation, gathers the matching fc2 columns
 *           and projects down; the layer is pre-norm with a residual add.
 *  [P1-HP]  same page, "2. Head-Pruned Attention Dispatch": an inactive head's
 *           projection weights, output-projection weights and historical KV
 *           cache are never read.
 *  [P3-ABS] "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference
 *           Time" (abstract): contextual sparsity = small input-dependent sets
 *           of heads and MLP parameters; a low-cost predictor works on each
 *           layer's input.
 *
 * Readings where the pages are silent or disagree (each is a choice of the
 * plainest form the rest supports):
 *  R1  The neuron predictor is low-rank: s = (x . A^T) . Bm^T, no
 *      nonlinearity, no bias; the head predictor is a dense bias-free map.
 *  R2  Scores are rounded to binary32 before selection, so both sides take
 *      the integer decision in the kernel's precision.  Top-k keeps the k
 *      largest scores, ties to the lower index, and returns indices ascending.
 *      -0.0 and +0.0 are equal scores.
 *  R3  Batch > 1: per-row top-k, then the union; every row computes over the
 *      whole union.
 *  R4  Activation ReLU (OPT), not the listing's GeLU; norm LayerNorm with gain
 *      and bias (OPT), RMSNorm (the listing's norm) as an option.
 *  R5  q, k, v, out-proj, fc1 and fc2 all carry biases (OPT).
 *  R6  q is scaled by 1/sqrt(dh) after its bias.  Attention covers the kv_len
 *      cached positions plus the new one.  Only selected heads append their
 *      new k and v (rounded to the cache's storage type, round-to-nearest-
 *      even); the other heads' slot is left untouched.
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* binary16 <-> binary64 from the IEEE 754 binary16 layout:                  */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.                  */

double dvo_half_to_double(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24); /* subnormal: m * 2^-14 / 2^10 */
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/2^10) * 2^(e-15) */
    }
    return s ? -v : v;
}

/* Round a binary64 value to the nearest binary16, ties to even. */
uint16_t dvo_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0) /* halfway between 65504 and 2^16 rounds to even = inf */
        return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: units of 2^-24; nearbyint rounds ties to even */
        double q = nearbyint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)q); /* q == 1024 is the least normal */
    }
    int e2;
    (void)frexp(a, &e2); /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;      /* a = (1 + m/1024) * 2^E */
    double q = nearbyint(ldexp(a, 10 - E)); /* in [1024, 2048] */
    if (q == 2048.0) {
        q = 1024.0;
        E += 1;
    }
    if (E > 15)
        return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* ------------------------------------------------------------------------ */

typedef struct {
    int d_model, n_heads, head_dim, d_ffn, pred_rank;
    int dtype;  /* 0: binary32 storage, 1: binary16 storage */
    int norm;   /* 0: LayerNorm, 1: RMSNorm */
    double eps;
    int kv_cap; /* KV positions per (batch row, head) */
    int neuron_block; /* 0 or 1: neurons selected one by one; > 1: in blocks */
    int mlp;          /* 0: fc1, ReLU, fc2; 1: SwiGLU (gate, up, down) */
} dvo_desc;

typedef struct {
    const void *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_oT, *b_o, *ln2_g, *ln2_b;
    const void *w1, *b1, *w2T, *b2, *pred_h, *pred_a, *pred_b;
} dvo_weights;

/* element i of a tensor in the layer's storage type, as binary64 */
static double ld(const void *p, int dtype, size_t i)
{
    if (dtype == 0)
        return (double)((const float *)p)[i];
    return dvo_half_to_double(((const uint16_t *)p)[i]);
}

/* store v into a tensor of the layer's storage type (round to nearest even) */
static void st(void *p, int dtype, size_t i, double v)
{
    if (dtype == 0)
        ((float *)p)[i] = (float)v;
    else
        ((uint16_t *)p)[i] = dvo_double_to_half(v);
}

static int desc_ok(const dvo_desc *D)
{
    return D && D->d_model > 0 && D->n_heads > 0 && D->head_dim > 0 && D->d_ffn > 0 &&
           D->pred_rank > 0 && (D->dtype == 0 || D->dtype == 1) &&
           (D->norm == 0 || D->norm == 1) && D->kv_cap > 0 && D->neuron_block >= 0 &&
           (D->neuron_block <= 1 || D->d_ffn % D->neuron_block == 0) &&
           (D->mlp == 0 || D->mlp == 1);
}

/* ------------------------------------------------------------------------ */
/* Norm (pre-norm of the listing's layer; LayerNorm per R4).                 */
/* LayerNorm: mu = mean(x), var = mean((x-mu)^2), out = (x-mu)/sqrt(var+eps)  */
/*            * g + b.   RMSNorm: out = x / sqrt(mean(x^2)+eps) * g.          */
void dvo_norm_row(const dvo_desc *D, const double *x, const void *g, const void *b, double *out)
{
    int d = D->d_model;
    if (D->norm == 0) {
        double mu = 0.0, var = 0.0;
        for (int c = 0; c < d; ++c)
            mu += x[c];
        mu /= d;
        for (int c = 0; c < d; ++c)
            var += (x[c] - mu) * (x[c] - mu);
        var /= d;
        double inv = 1.0 / sqrt(var + D->eps);
        for (int c = 0; c < d; ++c)
            out[c] = (x[c] - mu) * inv * ld(g, D->dtype, c) + ld(b, D->dtype, c);
    } else {
        double ms = 0.0;
        for (int c = 0; c < d; ++c)
            ms += x[c] * x[c];
        ms /= d;
        double inv = 1.0 / sqrt(ms + D->eps);
        for (int c = 0; c < d; ++c)
            out[c] = x[c] * inv * ld(g, D->dtype, c);
    }
}

/* ------------------------------------------------------------------------ */
/* Top-k (R2): the k largest binary32 scores, ties to the lower index,       */
/* returned in ascending index order.                                        */

static const float *g_sort_keys; /* qsort has no context argument */

static int cmp_desc_score_then_index(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    float sa = g_sort_keys[a], sb = g_sort_keys[b];
    if (sa > sb) return -1; /* larger score first; -0.0 == +0.0 here */
    if (sa < sb) return 1;
    return (a < b) ? -1 : (a > b); /* equal scores: lower index first */
}

static int cmp_int_asc(const void *pa, const void *pb)
{
    int a = *(const int *)pa, b = *(const int *)pb;
    return (a > b) - (a < b);
}

int dvo_topk(const float *scores, int n, int k, int32_t *out_idx)
{
    if (!scores || !out_idx || n <= 0 || k < 1 || k > n)
        return 1;
    int *order = (int *)malloc((size_t)n * sizeof(int));
    if (!order)
        return 2;
    for (int i = 0; i < n; ++i)
        order[i] = i;
    g_sort_keys = scores;
    qsort(order, (size_t)n, sizeof(int), cmp_desc_score_then_index);
    qsort(order, (size_t)k, sizeof(int), cmp_int_asc);
    for (int i = 0; i < k; ++i)
        out_idx[i] = order[i];
    free(order);
    return 0;
}

/* Blocked top-k ("DejaVu Guide: Contextual Sparsity for LLM Inference",    */
/* "Core Innovation 2", "1. Blocked Channel Sparsity": neurons are kept in   */
/* contiguous blocks of 32 or 64 channels, and a block holding highly active */
/* neurons is loaded whole).  Reading: a block's score is the largest score  */
/* of its members.  The k / block best blocks are taken as dvo_topk takes    */
/* scores (ties to the lower block); their neurons are returned ascending.   */
int dvo_block_topk(const float *scores, int n, int block, int k, int32_t *out_idx)
{
    if (!scores || !out_idx || block < 1 || n <= 0 || n % block || k < 1 || k > n ||
        k % block)
        return 1;
    const int nb = n / block, kb = k / block;
    float *bs = (float *)malloc((size_t)nb * sizeof(float));
    int32_t *bi = (int32_t *)malloc((size_t)kb * sizeof(int32_t));
    if (!bs || !bi) {
        free(bs);
        free(bi);
        return 2;
    }
    for (int j = 0; j < nb; ++j) {
        float m = scores[(size_t)j * block];
        for (int i = 1; i < block; ++i)
            if (scores[(size_t)j * block + i] > m)
                m = scores[(size_t)j * block + i];
        bs[j] = m;
    }
    int rc = dvo_topk(bs, nb, kb, bi);
    if (!rc)
        for (int q = 0; q < kb; ++q)
            for (int i = 0; i < block; ++i)
                out_idx[(size_t)q * block + i] = bi[q] * block + i;
    free(bs);
    free(bi);
    return rc;
}

/* union of B ascending index rows (each of length k) over [0, n): ascending */
int dvo_union(const int32_t *idx, int B, int k, int n, int32_t *out, int32_t *n_out)
{
    unsigned char *f = (unsigned char *)calloc((size_t)n, 1);
    if (!f)
        return 2;
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < k; ++i) {
            int j = idx[(size_t)b * k + i];
            if (j < 0 || j >= n) {
                free(f);
                return 1;
            }
            f[j] = 1;
        }
    int c = 0;
    for (int j = 0; j < n; ++j)
        if (f[j])
            out[c++] = j;
    *n_out = c;
    free(f);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Predictor ([P1-MF], [P1-LST] DejaVuLookaheadPredictor, R1-R3).            */
/*  head scores   s_h[b][h] = sum_c x_pred[b][c] * W_h[h][c]                 */
/*  low-rank u    u[b][q]   = sum_c x_pred[b][c] * A[q][c]                   */
/*  neuron scores s_n[b][j] = sum_q u[b][q] * Bm[j][q]                       */
/* Scores are returned as binary32 (R2).                                     */
int dvo_predict(const dvo_desc *D, const dvo_weights *W, const float *x_pred, int B,
                int k_h, int k_n, float *s_h, float *s_n, int32_t *idx_h, int32_t *idx_n,
                int32_t *u_h, int32_t *n_u_h, int32_t *u_n, int32_t *n_u_n)
{
    if (!desc_ok(D) || !W || !x_pred || B < 1 || !s_h || !s_n || !idx_h || !idx_n || !u_h ||
        !n_u_h || !u_n || !n_u_n)
        return 1;
    int d = D->d_model, H = D->n_heads, N = D->d_ffn, r = D->pred_rank, t = D->dtype;
    if (k_h < 1 || k_h > H || k_n < 1 || k_n > N)
        return 1;
    double *u = (double *)malloc((size_t)r * sizeof(double));
    if (!u)
        return 2;
    for (int b = 0; b < B; ++b) {
        const float *xb = x_pred + (size_t)b * d;
#pragma omp parallel for schedule(static)
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += (double)xb[c] * ld(W->pred_h, t, (size_t)h * d + c);
            s_h[(size_t)b * H + h] = (float)acc;
        }
#pragma omp parallel for schedule(static)
        for (int q = 0; q < r; ++q) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += (double)xb[c] * ld(W->pred_a, t, (size_t)q * d + c);
            u[q] = acc;
        }
#pragma omp parallel for schedule(static)
        for (int j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int q = 0; q < r; ++q)
                acc += u[q] * ld(W->pred_b, t, (size_t)j * r + q);
            s_n[(size_t)b * N + j] = (float)acc;
        }
        const int blk = D->neuron_block > 1 ? D->neuron_block : 1;
        if (dvo_topk(s_h + (size_t)b * H, H, k_h, idx_h + (size_t)b * k_h) ||
            (blk == 1 ? dvo_topk(s_n + (size_t)b * N, N, k_n, idx_n + (size_t)b * k_n)
                      : dvo_block_topk(s_n + (size_t)b * N, N, blk, k_n,
                                       idx_n + (size_t)b * k_n))) {
            free(u);
            return 2;
        }
    }
    free(u);
    if (dvo_union(idx_h, B, k_h, H, u_h, n_u_h) || dvo_union(idx_n, B, k_n, N, u_n, n_u_n))
        return 2;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Head-sparse attention block ([P1-HP], R5, R6): for every row b             */
/*   xn = norm1(x[b])                                                         */
/*   for each selected head h (in u_h order), t in {q,k,v}, e < dh:            */
/*     val = b_qkv[t][h][e] + sum_c xn[c] * W_qkv[t][h][e][c]                 */
/*   q *= 1/sqrt(dh);  cache[b][h][kv_len][:] = round(k), round(v)             */
/*   s_p = sum_e q[e] * K[b][h][p][e] for p = 0..kv_len (stored values)        */
/*   o[e] = sum_p exp(s_p - max) V[b][h][p][e] / sum_p exp(s_p - max)          */
/*   h1[b][c] = x[b][c] + b_o[c] + sum_{j, e} o_j[e] * W_oT[u_h[j]][e][c]      */
/* attn_o (optional) receives o as [B, n_u_h, dh].                            */
int dvo_sparse_attn(const dvo_desc *D, const dvo_weights *W, const float *x, int B,
                    const int32_t *u_h, int n_u_h, void *k_cache, void *v_cache, int kv_len,
                    double *h1, double *attn_o)
{
    if (!desc_ok(D) || !W || !x || B < 1 || !u_h || n_u_h < 0 || n_u_h > D->n_heads ||
        !k_cache || !v_cache || kv_len < 0 || kv_len >= D->kv_cap || !h1)
        return 1;
    int d = D->d_model, H = D->n_heads, dh = D->head_dim, t = D->dtype, cap = D->kv_cap;
    for (int j = 0; j < n_u_h; ++j)
        if (u_h[j] < 0 || u_h[j] >= H)
            return 1;
    double scale = 1.0 / sqrt((double)dh);
    double *xb = (double *)malloc((size_t)d * sizeof(double));
    double *xn = (double *)malloc((size_t)d * sizeof(double));
    double *q = (double *)malloc((size_t)dh * sizeof(double));
    double *s = (double *)malloc((size_t)(kv_len + 1) * sizeof(double));
    double *o = (double *)malloc(((size_t)n_u_h * dh + 1) * sizeof(double));
    if (!xb || !xn || !q || !s || !o) {
        free(xb); free(xn); free(q); free(s); free(o);
        return 2;
    }
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < d; ++c)
            xb[c] = (double)x[(size_t)b * d + c];
        dvo_norm_row(D, xb, W->ln1_g, W->ln1_b, xn);
        for (int j = 0; j < n_u_h; ++j) {
            int h = u_h[j];
            size_t cache_row0 = ((size_t)b * H + h) * (size_t)cap; /* position 0 */
#pragma omp parallel for collapse(2) schedule(static)
            for (int tt = 0; tt < 3; ++tt) {
                for (int e = 0; e < dh; ++e) {
                    size_t row = ((size_t)tt * H + h) * dh + e;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += xn[c] * ld(W->w_qkv, t, row * d + c);
                    double val = ld(W->b_qkv, t, row) + acc;
                    if (tt == 0)
                        q[e] = val * scale;
                    else
                        st(tt == 1 ? k_cache : v_cache, t,
                           (cache_row0 + (size_t)kv_len) * dh + e, val);
                }
            }
            double m = -INFINITY;
            for (int p = 0; p <= kv_len; ++p) {
                double acc = 0.0;
                for (int e = 0; e < dh; ++e)
                    acc += q[e] * ld(k_cache, t, (cache_row0 + p) * dh + e);
                s[p] = acc;
                if (acc > m)
                    m = acc;
            }
            double den = 0.0;
            for (int p = 0; p <= kv_len; ++p) {
                s[p] = exp(s[p] - m);
                den += s[p];
            }
            for (int e = 0; e < dh; ++e) {
                double acc = 0.0;
                for (int p = 0; p <= kv_len; ++p)
                    acc += s[p] * ld(v_cache, t, (cache_row0 + p) * dh + e);
                o[(size_t)j * dh + e] = acc / den;
            }
        }
        if (attn_o)
            memcpy(attn_o + (size_t)b * n_u_h * dh, o, (size_t)n_u_h * dh * sizeof(double));
#pragma omp parallel for schedule(static)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < n_u_h; ++j)
                for (int e = 0; e < dh; ++e)
                    acc += o[(size_t)j * dh + e] *
                           ld(W->w_oT, t, ((size_t)u_h[j] * dh + e) * d + c);
            h1[(size_t)b * d + c] = xb[c] + ld(W->b_o, t, c) + acc;
        }
    }
    free(xb); free(xn); free(q); free(s); free(o);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Activation of neuron j on the normalised input hn.                        */
/*  ReLU MLP (OPT):  pre = b1[j] + sum_c hn[c] * W1[j][c];  a = max(0, pre)    */
/*  SwiGLU (LLaMA-style; "DejaVu Guide ...", "Mathematical Modeling": three   */
/*  MLP matrices, d_ffn = 8/3 d_model "in SwiGLU"): W1 holds neuron j's gate  */
/*  row W1[j][0] and up row W1[j][1] side by side, b1[j][0..1] their biases:  */
/*    g = b1[j][0] + sum_c hn[c] W1[j][0][c],  u = b1[j][1] + sum_c hn[c] W1[j][1][c] */
/*    a = silu(g) * u,  silu(g) = g / (1 + exp(-g));  pre = g                 */
/* The down projection W2T[j] is used as fc2's.                               */
static double neuron_act(const dvo_desc *D, const dvo_weights *W, const double *hn, size_t j,
                         double *pre)
{
    const int d = D->d_model, t = D->dtype;
    if (D->mlp == 0) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += hn[c] * ld(W->w1, t, j * d + c);
        const double p = ld(W->b1, t, j) + acc;
        *pre = p;
        return p > 0.0 ? p : 0.0;
    }
    double ag = 0.0, au = 0.0;
    for (int c = 0; c < d; ++c) {
        ag += hn[c] * ld(W->w1, t, (2 * j) * d + c);
        au += hn[c] * ld(W->w1, t, (2 * j + 1) * d + c);
    }
    const double g = ld(W->b1, t, 2 * j) + ag, u = ld(W->b1, t, 2 * j + 1) + au;
    *pre = g;
    return g / (1.0 + exp(-g)) * u;
}

/* ------------------------------------------------------------------------ */
/* Sparse MLP block ([P1-LST] DejaVuSparseMLP.forward_sparse, R4, R5):        */
/*   hn = norm2(h1[b]);  a_i = activation of neuron u_n[i] (neuron_act)       */
/*   y[b][c] = h1[b][c] + b2[c] + sum_i a_i * W2T[u_n[i]][c]                   */
/* pre (optional) receives the pre-activations (gate, for SwiGLU) [B, n_u_n]. */
int dvo_sparse_mlp(const dvo_desc *D, const dvo_weights *W, const double *h1, int B,
                   const int32_t *u_n, int n_u_n, double *y, double *pre)
{
    if (!desc_ok(D) || !W || !h1 || B < 1 || !u_n || n_u_n < 0 || n_u_n > D->d_ffn || !y)
        return 1;
    int d = D->d_model, N = D->d_ffn, t = D->dtype;
    for (int i = 0; i < n_u_n; ++i)
        if (u_n[i] < 0 || u_n[i] >= N)
            return 1;
    double *hn = (double *)malloc((size_t)d * sizeof(double));
    double *a = (double *)malloc(((size_t)n_u_n + 1) * sizeof(double));
    if (!hn || !a) {
        free(hn); free(a);
        return 2;
    }
    for (int b = 0; b < B; ++b) {
        const double *hb = h1 + (size_t)b * d;
        dvo_norm_row(D, hb, W->ln2_g, W->ln2_b, hn);
#pragma omp parallel for schedule(static)
        for (int i = 0; i < n_u_n; ++i) {
            double p;
            a[i] = neuron_act(D, W, hn, (size_t)u_n[i], &p);
            if (pre)
                pre[(size_t)b * n_u_n + i] = p;
        }
#pragma omp parallel for schedule(static)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int i = 0; i < n_u_n; ++i)
                acc += a[i] * ld(W->w2T, t, (size_t)u_n[i] * d + c);
            y[(size_t)b * d + c] = hb[c] + ld(W->b2, t, c) + acc;
        }
    }
    free(hn); free(a);
    return 0;
}

/* The sparse layer on a given index set: attention block, then MLP block. */
int dvo_layer(const dvo_desc *D, const dvo_weights *W, const float *x, int B,
              const int32_t *u_h, int n_u_h, const int32_t *u_n, int n_u_n, void *k_cache,
              void *v_cache, int kv_len, double *h1, double *y)
{
    int rc = dvo_sparse_attn(D, W, x, B, u_h, n_u_h, k_cache, v_cache, kv_len, h1, NULL);
    if (rc)
        return rc;
    return dvo_sparse_mlp(D, W, h1, B, u_n, n_u_n, y, NULL);
}

/* ------------------------------------------------------------------------ */
/* Dense layer, written out on its own (no index lists): every head appends  */
/* and attends, every neuron fires (neuron_act).  Loop orders (heads, then    */
/* neurons, ascending) match the sparse functions', so selecting every head   */
/* and neuron must reproduce it bit for bit.  pre (optional): [B, N].         */
int dvo_dense_layer(const dvo_desc *D, const dvo_weights *W, const float *x, int B,
                    void *k_cache, void *v_cache, int kv_len, double *h1, double *y,
                    double *pre)
{
    if (!desc_ok(D) || !W || !x || B < 1 || !k_cache || !v_cache || kv_len < 0 ||
        kv_len >= D->kv_cap || !h1 || !y)
        return 1;
    int d = D->d_model, H = D->n_heads, dh = D->head_dim, N = D->d_ffn, t = D->dtype;
    int cap = D->kv_cap;
    double scale = 1.0 / sqrt((double)dh);
    double *xb = (double *)malloc((size_t)d * sizeof(double));
    double *xn = (double *)malloc((size_t)d * sizeof(double));
    double *q = (double *)malloc((size_t)dh * sizeof(double));
    double *s = (double *)malloc((size_t)(kv_len + 1) * sizeof(double));
    double *o = (double *)malloc((size_t)H * dh * sizeof(double));
    double *a = (double *)malloc((size_t)N * sizeof(double));
    if (!xb || !xn || !q || !s || !o || !a) {
        free(xb); free(xn); free(q); free(s); free(o); free(a);
        return 2;
    }
    for (int b = 0; b < B; ++b) {
        for (int c = 0; c < d; ++c)
            xb[c] = (double)x[(size_t)b * d + c];
        dvo_norm_row(D, xb, W->ln1_g, W->ln1_b, xn);
        for (int h = 0; h < H; ++h) {
            size_t base = ((size_t)b * H + h) * (size_t)cap;
            for (int tt = 0; tt < 3; ++tt)
                for (int e = 0; e < dh; ++e) {
                    size_t row = ((size_t)tt * H + h) * dh + e;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += xn[c] * ld(W->w_qkv, t, row * d + c);
                    double val = ld(W->b_qkv, t, row) + acc;
                    if (tt == 0)
                        q[e] = val * scale;
                    else
                        st(tt == 1 ? k_cache : v_cache, t, (base + (size_t)kv_len) * dh + e, val);
                }
            double m = -INFINITY;
            for (int p = 0; p <= kv_len; ++p) {
                double acc = 0.0;
                for (int e = 0; e < dh; ++e)
                    acc += q[e] * ld(k_cache, t, (base + p) * dh + e);
                s[p] = acc;
                if (acc > m)
                    m = acc;
            }
            double den = 0.0;
            for (int p = 0; p <= kv_len; ++p) {
                s[p] = exp(s[p] - m);
                den += s[p];
            }
            for (int e = 0; e < dh; ++e) {
                double acc = 0.0;
                for (int p = 0; p <= kv_len; ++p)
                    acc += s[p] * ld(v_cache, t, (base + p) * dh + e);
                o[(size_t)h * dh + e] = acc / den;
            }
        }
        double *hb = h1 + (size_t)b * d;
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                for (int e = 0; e < dh; ++e)
                    acc += o[(size_t)h * dh + e] * ld(W->w_oT, t, ((size_t)h * dh + e) * d + c);
            hb[c] = xb[c] + ld(W->b_o, t, c) + acc;
        }
        dvo_norm_row(D, hb, W->ln2_g, W->ln2_b, xn);
        for (int j = 0; j < N; ++j) {
            double p;
            a[j] = neuron_act(D, W, xn, (size_t)j, &p);
            if (pre)
                pre[(size_t)b * N + j] = p;
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j)
                acc += a[j] * ld(W->w2T, t, (size_t)j * d + c);
            y[(size_t)b * d + c] = hb[c] + ld(W->b2, t, c) + acc;
        }
    }
    free(xb); free(xn); free(q); free(s); free(o); free(a);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Full sparse decode of one layer: predict (from x_pred), then the layer on  */
/* the predicted unions.  Index outputs as in dvo_predict.                    */
int dvo_layer_decode(const dvo_desc *D, const dvo_weights *W, const float *x,
                     const float *x_pred, int B, int k_h, int k_n, void *k_cache, void *v_cache,
                     int kv_len, float *s_h, float *s_n, int32_t *idx_h, int32_t *idx_n,
                     int32_t *u_h, int32_t *n_u_h, int32_t *u_n, int32_t *n_u_n, double *h1,
                     double *y)
{
    int rc = dvo_predict(D, W, x_pred ? x_pred : x, B, k_h, k_n, s_h, s_n, idx_h, idx_n, u_h,
                         n_u_h, u_n, n_u_n);
    if (rc)
        return rc;
    return dvo_layer(D, W, x, B, u_h, *n_u_h, u_n, *n_u_n, k_cache, v_cache, kv_len, h1, y);
}

/* ------------------------------------------------------------------------ */
/* Threads used by the OpenMP build (n <= 0: every available core); returns  */
/* the number its loops will use.  The plain build always returns 1.         */
int dvo_set_threads(int n)
{
#ifdef _OPENMP
    if (n <= 0)
        n = omp_get_num_procs();
    omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}
