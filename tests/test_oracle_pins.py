"""Pins of the CPU oracle to facts other than itself (no GPU).

Each pin is chosen so that a plausible slip in the oracle -- a dropped term,
a wrong sign, a transposed operand, an off-by-one position, a wrong gather --
fails at least one test:

* binary16 decode/encode against numpy's IEEE conversions (exhaustive decode);
* norms against closed forms and torch's layer_norm;
* top-k and union against brute-force sorting;
* every projection against one-hot weights, where each output must equal one
  chosen input exactly (catches transposes and index slips);
* attention against closed forms (one position -> v; equal scores -> mean of
  V) and permutation invariance of the cached positions;
* invariants stated for the method: selecting every head and neuron equals the
  dense layer bit for bit; a perfect ReLU mask equals the dense MLP bit for
  bit; unselected rows, heads and KV contribute nothing;
* a dense brute force built from numpy/scipy library routines on the tiny
  shape, and the sparse MLP against the dense MLP under a 0/1 neuron mask
  with the selection from numpy scores and a stable argsort;
* the whole decode step against its parts (predict on x_pred, layer on x).
"""

import math

import numpy as np
import pytest
import torch

import dv_inputs
import oracle

TINY = dv_inputs.CONFIGS["tiny"]


def _tiny_random(dtype="f32", norm_affine=True, B=1, seed=0, kv_len=None, cfg=TINY):
    cfg = cfg.with_(dtype=dtype)
    if kv_len is not None:
        cfg = cfg.with_(kv_len=kv_len)
    w = oracle.numpy_weights(dv_inputs.make_weights(cfg, seed, "cpu", norm_affine=norm_affine))
    kc, vc = dv_inputs.make_kv(cfg, B, seed, "cpu")
    x = dv_inputs.make_x(cfg, B, seed, "cpu").numpy()
    D = oracle.desc_from_config(cfg)
    return cfg, D, w, kc.numpy(), vc.numpy(), x


# --------------------------------------------------------------------------
# binary16 conversions


def test_half_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits], dtype=np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_half_encode_round_to_nearest_even():
    rng = np.random.default_rng(1)
    vals = list(rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000))
    one = 1.0
    vals += [0.0, -0.0, one + 2.0 ** -11, one + 3 * 2.0 ** -11, -(one + 2.0 ** -11),
             2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -24, 2.0 ** -14 - 2.0 ** -25, 65504.0,
             65519.99, 65520.0, -65520.0, 1e300, -1e-300, 2.0 ** -14]
    for v in vals:
        want = np.array([v], np.float64).astype(np.float16).view(np.uint16)[0]
        assert oracle.double_to_half(v) == want, v


# --------------------------------------------------------------------------
# norms


def test_layernorm_alternating_closed_form():
    D = oracle.make_desc(8, 1, 8, 8, 8, 0, 2, norm=0, eps=1e-5)
    a = 3.0
    x = np.array([a, -a] * 4, np.float64)
    out = oracle.norm_row(D, x, np.ones(8, np.float32), np.zeros(8, np.float32))
    want = np.array([1, -1] * 4) * a / math.sqrt(a * a + 1e-5)
    np.testing.assert_allclose(out, want, rtol=1e-15, atol=0)


def test_layernorm_matches_torch_and_applies_gain_bias_per_column():
    rng = np.random.default_rng(2)
    d = 64
    D = oracle.make_desc(d, 1, 8, 8, 8, 0, 2, norm=0, eps=1e-5)
    x = rng.standard_normal(d) * 2 + 0.7
    g = (1 + 0.3 * rng.standard_normal(d)).astype(np.float32)
    b = (0.2 * rng.standard_normal(d)).astype(np.float32)
    out = oracle.norm_row(D, x, g, b)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (d,),
                                         torch.from_numpy(g.astype(np.float64)),
                                         torch.from_numpy(b.astype(np.float64)), eps=1e-5)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_rmsnorm_constant_closed_form():
    d = 16
    D = oracle.make_desc(d, 1, 8, 8, 8, 0, 2, norm=1, eps=1e-5)
    c = -1.5
    g = np.arange(1, d + 1, dtype=np.float32)
    out = oracle.norm_row(D, np.full(d, c), g, np.zeros(d, np.float32))
    np.testing.assert_allclose(out, c / math.sqrt(c * c + 1e-5) * g.astype(np.float64), rtol=1e-15)


# --------------------------------------------------------------------------
# top-k and union


def _brute_topk(s, k):
    s = np.asarray(s, np.float32).astype(np.float64)
    order = np.lexsort((np.arange(s.size), -s))  # score desc, index asc
    return np.sort(order[:k])


@pytest.mark.parametrize("n,k", [(1, 1), (7, 3), (96, 20), (1024, 103), (5000, 250),
                                 (5000, 5000)])
def test_topk_brute_force_with_ties(n, k):
    rng = np.random.default_rng(n + k)
    s = np.round(rng.standard_normal(n) * 4).astype(np.float32) / 4  # many exact ties
    s[rng.integers(0, n, max(1, n // 10))] = -0.0
    s[rng.integers(0, n, max(1, n // 10))] = 0.0
    got = oracle.topk(s, k)
    assert np.array_equal(got, _brute_topk(s, k))
    assert np.all(np.diff(got) > 0)


def test_topk_signed_zero_is_a_tie():
    s = np.array([-0.0, 0.0, -0.0, 0.0], np.float32)
    assert list(oracle.topk(s, 1)) == [0]
    assert list(oracle.topk(s, 3)) == [0, 1, 2]


def test_union_matches_numpy():
    rng = np.random.default_rng(3)
    rows = np.stack([np.sort(rng.choice(500, 40, replace=False)) for _ in range(5)]).astype(np.int32)
    got = oracle.union(rows, 500)
    want = rows[0]
    for r in rows[1:]:
        want = np.union1d(want, r)
    assert np.array_equal(got, want)


# --------------------------------------------------------------------------
# predictor


def _zero_weights(d, H, dh, N, r, dtype=np.float32):
    return {
        "ln1_g": np.ones(d, dtype), "ln1_b": np.zeros(d, dtype),
        "w_qkv": np.zeros((3, H, dh, d), dtype), "b_qkv": np.zeros((3, H, dh), dtype),
        "w_oT": np.zeros((H, dh, d), dtype), "b_o": np.zeros(d, dtype),
        "ln2_g": np.ones(d, dtype), "ln2_b": np.zeros(d, dtype),
        "w1": np.zeros((N, d), dtype), "b1": np.zeros(N, dtype),
        "w2T": np.zeros((N, d), dtype), "b2": np.zeros(d, dtype),
        "pred_h": np.zeros((H, d), dtype), "pred_a": np.zeros((r, d), dtype),
        "pred_b": np.zeros((N, r), dtype),
    }


def test_predictor_one_hot_picks_named_inputs():
    d, H, dh, N, r, B = 32, 6, 8, 40, 12, 2
    rng = np.random.default_rng(4)
    w = _zero_weights(d, H, dh, N, r)
    pi_h = rng.permutation(d)[:H]
    c_h = 2.0 ** rng.integers(-3, 4, H)
    for h in range(H):
        w["pred_h"][h, pi_h[h]] = c_h[h]
    sigma = rng.permutation(d)[:r]
    for q in range(r):
        w["pred_a"][q, sigma[q]] = 1.0
    tau = rng.integers(0, r, N)
    for j in range(N):
        w["pred_b"][j, tau[j]] = 1.0
    D = oracle.make_desc(d, H, dh, N, r, 0, 4)
    x = rng.standard_normal((B, d)).astype(np.float32)
    p = oracle.predict(D, w, x, 2, 7)
    assert np.array_equal(p["s_h"], (x[:, pi_h] * c_h).astype(np.float32))
    assert np.array_equal(p["s_n"], x[:, sigma[tau]])
    for b in range(B):
        assert np.array_equal(p["idx_h"][b], _brute_topk(p["s_h"][b], 2))
        assert np.array_equal(p["idx_n"][b], _brute_topk(p["s_n"][b], 7))


def test_predictor_matches_library_matmul():
    cfg, D, w, _, _, x = _tiny_random(B=3)
    p = oracle.predict(D, w, x, cfg.k_heads, cfg.k_neurons)
    x64 = x.astype(np.float64)
    s_h = x64 @ w["pred_h"].astype(np.float64).T
    s_n = (x64 @ w["pred_a"].astype(np.float64).T) @ w["pred_b"].astype(np.float64).T
    np.testing.assert_allclose(p["s_h"], s_h, rtol=2e-7, atol=1e-9)
    np.testing.assert_allclose(p["s_n"], s_n, rtol=2e-7, atol=1e-9)


def test_predictor_counts_sorted_unions():
    cfg, D, w, _, _, x = _tiny_random(B=5)
    k_h, k_n = cfg.k_heads, cfg.k_neurons
    p = oracle.predict(D, w, x, k_h, k_n)
    for idx, n, k, u in ((p["idx_h"], cfg.n_heads, k_h, p["u_h"]),
                         (p["idx_n"], cfg.d_ffn, k_n, p["u_n"])):
        assert idx.shape == (5, k)
        for row in idx:
            assert np.all(np.diff(row) > 0) and row.min() >= 0 and row.max() < n
        assert np.array_equal(u, np.unique(idx))
        assert k <= u.size <= min(n, 5 * k)


# --------------------------------------------------------------------------
# attention block


def test_qkv_oproj_one_hot_and_single_position_attention():
    d, H, dh, N, r, B = 64, 4, 8, 16, 8, 2
    rng = np.random.default_rng(5)
    w = _zero_weights(d, H, dh, N, r)
    srcs = {}
    for t in range(3):
        for h in range(H):
            src = rng.permutation(d)[:dh]
            srcs[t, h] = src
            for e in range(dh):
                w["w_qkv"][t, h, e, src[e]] = 1.0
    w["b_qkv"][:] = rng.standard_normal((3, H, dh)).astype(np.float32)
    cols = rng.permutation(d)[: H * dh].reshape(H, dh)
    for h in range(H):
        for e in range(dh):
            w["w_oT"][h, e, cols[h, e]] = 1.0
    w["b_o"][:] = rng.standard_normal(d).astype(np.float32)
    D = oracle.make_desc(d, H, dh, N, r, 0, 3)
    x = rng.standard_normal((B, d)).astype(np.float32)
    kc = rng.standard_normal((B, H, 3, dh)).astype(np.float32)
    vc = rng.standard_normal((B, H, 3, dh)).astype(np.float32)
    u_h = np.array([1, 3], np.int32)
    h1, o, kc2, vc2 = oracle.sparse_attn(D, w, x, u_h, kc, vc, kv_len=0)
    for b in range(B):
        xn = oracle.norm_row(D, x[b], w["ln1_g"], w["ln1_b"])
        want_h1 = x[b].astype(np.float64) + w["b_o"]
        for j, h in enumerate(u_h):
            k_new = w["b_qkv"][1, h] + xn[srcs[1, h]]
            v_new = w["b_qkv"][2, h] + xn[srcs[2, h]]
            assert np.array_equal(kc2[b, h, 0], k_new.astype(np.float32))
            assert np.array_equal(vc2[b, h, 0], v_new.astype(np.float32))
            # one position: softmax weight exactly 1, o is the stored v
            assert np.array_equal(o[b, j], vc2[b, h, 0].astype(np.float64))
            want_h1[cols[h]] += o[b, j]
        np.testing.assert_allclose(h1[b], want_h1, rtol=0, atol=1e-15)
        for h in (0, 2):  # unselected heads: cache untouched
            assert np.array_equal(kc2[b, h], kc[b, h]) and np.array_equal(vc2[b, h], vc[b, h])


def test_attention_equal_scores_average_values():
    d, H, dh, N, r, L = 32, 2, 8, 8, 8, 9
    rng = np.random.default_rng(6)
    w = _zero_weights(d, H, dh, N, r)
    c = rng.standard_normal(dh).astype(np.float32)
    w["w_qkv"][0] = rng.standard_normal((H, dh, d)).astype(np.float32)  # q random
    w["b_qkv"][1] = c  # new key = c exactly (k rows are zero)
    w["b_qkv"][2] = rng.standard_normal((H, dh)).astype(np.float32)  # new value = bias
    D = oracle.make_desc(d, H, dh, N, r, 0, L + 1)
    x = rng.standard_normal((1, d)).astype(np.float32)
    kc = np.broadcast_to(c, (1, H, L + 1, dh)).copy()
    vc = rng.standard_normal((1, H, L + 1, dh)).astype(np.float32)
    _, o, _, vc2 = oracle.sparse_attn(D, w, x, np.array([0, 1], np.int32), kc, vc, kv_len=L)
    for h in range(H):
        np.testing.assert_allclose(o[0, h], vc2[0, h, : L + 1].astype(np.float64).mean(0),
                                   rtol=1e-13, atol=1e-15)


def test_attention_invariant_to_cached_position_order():
    cfg, D, w, kc, vc, x = _tiny_random(kv_len=40)
    u_h = np.array([2, 5], np.int32)
    _, o1, _, _ = oracle.sparse_attn(D, w, x, u_h, kc, vc, cfg.kv_len)
    perm = np.random.default_rng(7).permutation(cfg.kv_len)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, :, : cfg.kv_len] = kc[:, :, perm]
    vc2[:, :, : cfg.kv_len] = vc[:, :, perm]
    _, o2, _, _ = oracle.sparse_attn(D, w, x, u_h, kc2, vc2, cfg.kv_len)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    vc3 = vc.copy()  # pairing K[p] with another position's V must change o
    vc3[:, :, : cfg.kv_len] = vc[:, :, perm]
    _, o3, _, _ = oracle.sparse_attn(D, w, x, u_h, kc, vc3, cfg.kv_len)
    assert np.max(np.abs(o3 - o1)) > 1e-3


# --------------------------------------------------------------------------
# MLP block


def test_mlp_one_hot():
    d, H, dh, N, r, B = 48, 2, 8, 30, 8, 2
    rng = np.random.default_rng(8)
    w = _zero_weights(d, H, dh, N, r)
    src = rng.integers(0, d, N)
    for j in range(N):
        w["w1"][j, src[j]] = 1.0
    w["b1"][:] = rng.standard_normal(N).astype(np.float32)
    dst = rng.permutation(d)[:N]
    for j in range(N):
        w["w2T"][j, dst[j]] = 1.0
    w["b2"][:] = rng.standard_normal(d).astype(np.float32)
    D = oracle.make_desc(d, H, dh, N, r, 0, 2)
    h1 = rng.standard_normal((B, d))
    u_n = np.sort(rng.choice(N, 11, replace=False)).astype(np.int32)
    y, pre = oracle.sparse_mlp(D, w, h1, u_n)
    for b in range(B):
        hn = oracle.norm_row(D, h1[b], w["ln2_g"], w["ln2_b"])
        want_pre = w["b1"][u_n] + hn[src[u_n]]
        np.testing.assert_allclose(pre[b], want_pre, rtol=0, atol=1e-15)
        want_y = h1[b] + w["b2"]
        want_y[dst[u_n]] += np.maximum(want_pre, 0.0)
        np.testing.assert_allclose(y[b], want_y, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# invariants of the method


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_selecting_everything_equals_dense_bitwise(dtype):
    cfg, D, w, kc, vc, x = _tiny_random(dtype=dtype, B=2)
    h1d, yd, _, kcd, vcd = oracle.dense_layer(D, w, x, kc, vc, cfg.kv_len)
    h1s, ys, kcs, vcs = oracle.layer(D, w, x, np.arange(cfg.n_heads, dtype=np.int32),
                                     np.arange(cfg.d_ffn, dtype=np.int32), kc, vc, cfg.kv_len)
    assert np.array_equal(h1d, h1s) and np.array_equal(yd, ys)
    assert np.array_equal(kcd, kcs) and np.array_equal(vcd, vcs)


def test_perfect_relu_mask_equals_dense_mlp_bitwise():
    cfg, D, w, kc, vc, x = _tiny_random(B=1)
    w["b1"] = (w["b1"] - 0.5).astype(np.float32)  # many zeros, as in the 6.7B shape
    h1d, yd, pre, _, _ = oracle.dense_layer(D, w, x, kc, vc, cfg.kv_len)
    u_n = np.nonzero(pre[0] > 0)[0].astype(np.int32)
    assert 0 < u_n.size < cfg.d_ffn
    y, _ = oracle.sparse_mlp(D, w, h1d, u_n)
    assert np.array_equal(y, yd)


def test_unselected_rows_heads_and_kv_contribute_nothing():
    cfg, D, w, kc, vc, x = _tiny_random(B=2, dtype="f16")
    rng = np.random.default_rng(9)
    u_h = np.array([1, 6], np.int32)
    u_n = np.sort(rng.choice(cfg.d_ffn, cfg.k_neurons, replace=False)).astype(np.int32)
    h1, y, kc1, vc1 = oracle.layer(D, w, x, u_h, u_n, kc, vc, cfg.kv_len)
    w2 = {k: v.copy() for k, v in w.items()}
    off_h = np.setdiff1d(np.arange(cfg.n_heads), u_h)
    off_n = np.setdiff1d(np.arange(cfg.d_ffn), u_n)

    def noise(shape):
        return rng.standard_normal(shape).astype(np.float16)

    w2["w_qkv"][:, off_h] = noise(w2["w_qkv"][:, off_h].shape)
    w2["b_qkv"][:, off_h] = noise(w2["b_qkv"][:, off_h].shape)
    w2["w_oT"][off_h] = noise(w2["w_oT"][off_h].shape)
    w2["w1"][off_n] = noise(w2["w1"][off_n].shape)
    w2["b1"][off_n] = noise(w2["b1"][off_n].shape)
    w2["w2T"][off_n] = noise(w2["w2T"][off_n].shape)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[:, off_h] = noise(kc2[:, off_h].shape)
    vc2[:, off_h] = noise(vc2[:, off_h].shape)
    h1b, yb, kc3, _ = oracle.layer(D, w2, x, u_h, u_n, kc2, vc2, cfg.kv_len)
    assert np.array_equal(h1, h1b) and np.array_equal(y, yb)
    assert np.array_equal(kc3[:, off_h], kc2[:, off_h])  # their slot is not written


# --------------------------------------------------------------------------
# independent restatements


def _np_layernorm(x, g, b, eps):
    mu = x.mean(-1, keepdims=True)
    var = ((x - mu) ** 2).mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * g + b


@pytest.mark.parametrize("dtype,B", [("f32", 1), ("f16", 3)])
def test_dense_layer_numpy_brute_force(dtype, B):
    from scipy.special import softmax

    cfg, D, w, kc, vc, x = _tiny_random(dtype=dtype, B=B)
    h1o, yo, preo, kco, vco = oracle.dense_layer(D, w, x, kc, vc, cfg.kv_len)
    f = {k: v.astype(np.float64) for k, v in w.items()}
    H, dh, d, L = cfg.n_heads, cfg.head_dim, cfg.d_model, cfg.kv_len
    st = np.float32 if dtype == "f32" else np.float16
    K, V = kc.copy(), vc.copy()
    xb = x.astype(np.float64)
    xn = _np_layernorm(xb, f["ln1_g"], f["ln1_b"], cfg.ln_eps)
    qkv = xn @ f["w_qkv"].reshape(3 * H * dh, d).T + f["b_qkv"].reshape(-1)
    qkv = qkv.reshape(B, 3, H, dh)
    q = qkv[:, 0] / math.sqrt(dh)
    K[:, :, L] = qkv[:, 1].astype(st)
    V[:, :, L] = qkv[:, 2].astype(st)
    Kf, Vf = K[:, :, : L + 1].astype(np.float64), V[:, :, : L + 1].astype(np.float64)
    s = np.einsum("bhe,bhpe->bhp", q, Kf)
    o = np.einsum("bhp,bhpe->bhe", softmax(s, axis=-1), Vf)
    h1 = xb + f["b_o"] + o.reshape(B, H * dh) @ f["w_oT"].reshape(H * dh, d)
    hn = _np_layernorm(h1, f["ln2_g"], f["ln2_b"], cfg.ln_eps)
    pre = hn @ f["w1"].T + f["b1"]
    y = h1 + f["b2"] + np.maximum(pre, 0) @ f["w2T"]
    assert np.array_equal(K, kco) and np.array_equal(V, vco)
    np.testing.assert_allclose(h1o, h1, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(preo, pre, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(yo, y, rtol=1e-11, atol=1e-11)


def _ref_topk_rows(scores, k):
    """Per-row k largest binary32 scores, ties to the lower index, ascending:
    a stable argsort on (-score, index), independent of the oracle's sort."""
    out = []
    for row in np.asarray(scores, np.float32):
        keys = np.where(row == 0.0, np.float32(0.0), row)  # -0 and +0 are equal
        order = np.lexsort((np.arange(row.size), -keys.astype(np.float64)))
        out.append(np.sort(order[:k]))
    return np.array(out, np.int32)


def test_sparse_mlp_equals_masked_dense_mlp():
    """The sparse MLP is the dense MLP with every unselected neuron's
    activation forced to zero (the guide's "Core Innovation 2:
    Hardware-Efficient Dynamic Sparse Matrix Execution": only the selected
    neurons' fc1 rows and fc2 columns take part).  The selection comes from
    the low-rank scores computed here with numpy in binary64 and rounded to
    binary32, top-k by a stable argsort; the MLP is dense numpy with a 0/1
    mask over the union of the rows' sets."""
    cfg, D, w, _, _, x = _tiny_random(B=2)
    f = {k: v.astype(np.float64) for k, v in w.items()}
    xp = x.astype(np.float64)
    s_n = ((xp @ f["pred_a"].T) @ f["pred_b"].T).astype(np.float32)
    s_h = (xp @ f["pred_h"].T).astype(np.float32)
    idx_n = _ref_topk_rows(s_n, cfg.k_neurons)
    idx_h = _ref_topk_rows(s_h, cfg.k_heads)
    p = oracle.predict(D, w, x, cfg.k_heads, cfg.k_neurons)
    assert np.array_equal(p["idx_n"], idx_n) and np.array_equal(p["idx_h"], idx_h)
    u_n = np.union1d(idx_n[0], idx_n[1]).astype(np.int32)
    assert np.array_equal(p["u_n"], u_n)

    rng = np.random.default_rng(10)
    h1 = rng.standard_normal((2, cfg.d_model))
    hn = _np_layernorm(h1, f["ln2_g"], f["ln2_b"], cfg.ln_eps)
    mask = np.zeros(cfg.d_ffn)
    mask[u_n] = 1.0
    act = np.maximum(hn @ f["w1"].T + f["b1"], 0.0) * mask
    y_ref = h1 + f["b2"] + act @ f["w2T"]
    y, _ = oracle.sparse_mlp(D, w, h1, u_n)
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)
    # the mask matters: the dense MLP differs
    y_dense = h1 + f["b2"] + np.maximum(hn @ f["w1"].T + f["b1"], 0.0) @ f["w2T"]
    assert np.max(np.abs(y_dense - y)) > 1e-6


def test_layer_decode_composes_predict_and_layer():
    """The decode step predicts the sets from x_pred and runs the layer on x
    over them (the guide's "Core Innovation 1: Asynchronous Lookahead
    Predictors": a layer's sets come from an earlier input).  x_pred != x
    with different sets, so a swap of the two inputs anywhere in the
    composition changes the result; x_pred = None means x."""
    cfg, D, w, kc, vc, x = _tiny_random(dtype="f16", B=3)
    xp = dv_inputs.make_x(cfg.with_(dtype="f16"), 3, 7, "cpu").numpy()
    p = oracle.predict(D, w, xp, cfg.k_heads, cfg.k_neurons)
    px = oracle.predict(D, w, x, cfg.k_heads, cfg.k_neurons)
    assert not np.array_equal(p["u_n"], px["u_n"])
    kc0, vc0 = kc.copy(), vc.copy()
    r = oracle.layer_decode(D, w, x, cfg.k_heads, cfg.k_neurons, kc, vc, cfg.kv_len, x_pred=xp)
    assert np.array_equal(kc, kc0) and np.array_equal(vc, vc0)  # inputs untouched
    for key in ("s_h", "s_n", "idx_h", "idx_n", "u_h", "u_n"):
        assert np.array_equal(r[key], p[key]), key
    h1, y, kc1, vc1 = oracle.layer(D, w, x, p["u_h"], p["u_n"], kc, vc, cfg.kv_len)
    assert np.array_equal(r["h1"], h1) and np.array_equal(r["y"], y)
    assert np.array_equal(r["k_cache"], kc1) and np.array_equal(r["v_cache"], vc1)
    h1s, _, _, _ = oracle.layer(D, w, xp, p["u_h"], p["u_n"], kc, vc, cfg.kv_len)
    assert not np.array_equal(h1s, h1)  # the layer input is x, not x_pred
    r0 = oracle.layer_decode(D, w, x, cfg.k_heads, cfg.k_neurons, kc, vc, cfg.kv_len)
    r1 = oracle.layer_decode(D, w, x, cfg.k_heads, cfg.k_neurons, kc, vc, cfg.kv_len, x_pred=x)
    for key in ("u_h", "u_n", "h1", "y", "k_cache", "v_cache"):
        assert np.array_equal(r0[key], r1[key]), key
    for key in ("u_h", "u_n"):
        assert np.array_equal(r0[key], px[key]), key


def test_oracle_rejects_bad_arguments():
    cfg, D, w, kc, vc, x = _tiny_random()
    with pytest.raises(ValueError):
        oracle.predict(D, w, x, 0, 5)
    with pytest.raises(ValueError):
        oracle.predict(D, w, x, cfg.n_heads + 1, 5)
    with pytest.raises(ValueError):
        oracle.sparse_attn(D, w, x, np.array([cfg.n_heads], np.int32), kc, vc, cfg.kv_len)
    with pytest.raises(ValueError):
        oracle.sparse_attn(D, w, x, np.array([0], np.int32), kc, vc, cfg.kv_len + 1)
