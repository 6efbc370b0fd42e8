"""Pins of the oracle's LLaMA-style MLP (SwiGLU: the gate and up rows of
neuron j side by side in w1 [N, 2, d], act = silu(gate) * up with
silu(g) = g / (1 + exp(-g)), the down projection transposed in w2T)."""

import math

import numpy as np
import pytest

import dv_inputs
import oracle

LT = dv_inputs.CONFIGS["llama_tiny"]


def _random(dtype="f32", B=2, seed=0, cfg=LT):
    cfg = cfg.with_(dtype=dtype)
    w = oracle.numpy_weights(dv_inputs.make_weights(cfg, seed, "cpu", norm_affine=True))
    kc, vc = dv_inputs.make_kv(cfg, B, seed, "cpu")
    x = dv_inputs.make_x(cfg, B, seed, "cpu").numpy()
    return cfg, oracle.desc_from_config(cfg), w, kc.numpy(), vc.numpy(), x


def test_one_hot_closed_form():
    # RMSNorm of a constant row with unit gain is a constant hn, so neuron j's
    # gate is a_j hn + b_j and its up value c_j hn; y = h1 + silu(g) u e_dst
    d, H, dh, N, r = 16, 2, 8, 5, 8
    D = oracle.make_desc(d, H, dh, N, r, 0, 2, norm=1, mlp=1)
    w = {n: np.zeros(s, np.float32) for n, s in {
        "ln1_g": (d,), "ln1_b": (d,), "w_qkv": (3, H, dh, d), "b_qkv": (3, H, dh),
        "w_oT": (H, dh, d), "b_o": (d,), "ln2_g": (d,), "ln2_b": (d,), "w1": (N, 2, d),
        "b1": (N, 2), "w2T": (N, d), "b2": (d,), "pred_h": (H, d), "pred_a": (r, d),
        "pred_b": (N, r)}.items()}
    w["ln2_g"][:] = 1.0
    gates = [-6.0, -1.0, 0.0, 0.5, 7.0]
    ups = [2.0, -3.0, 5.0, 1.5, -0.25]
    for j in range(N):
        w["w1"][j, 0, j] = gates[j] / 2   # hn = 1 everywhere: the dot gives gates[j] / 2
        w["b1"][j, 0] = gates[j] / 2
        w["w1"][j, 1, j + 5] = ups[j]
        w["w2T"][j, 10 + j] = 1.0
    h1 = np.full((1, d), 3.0)
    y, pre = oracle.sparse_mlp(D, w, h1, np.arange(N, dtype=np.int32))
    hn = 3.0 / math.sqrt(9.0 + 1e-5)  # RMSNorm of the constant row (eps 1e-5)
    for j in range(N):
        # the weights and biases above are exact in binary32
        g = gates[j] / 2 * hn + gates[j] / 2
        u = ups[j] * hn
        act = g / (1.0 + math.exp(-g)) * u
        assert pre[0, j] == pytest.approx(g, abs=1e-15)
        assert y[0, 10 + j] == pytest.approx(3.0 + act, abs=1e-14)
    # silu(0) = 0 exactly: neuron 2's output column is left at h1
    assert y[0, 12] == 3.0


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_dense_mlp_matches_numpy(dtype):
    cfg, D, w, kc, vc, x = _random(dtype=dtype)
    h1, y, pre, _, _ = oracle.dense_layer(D, w, x, kc, vc, cfg.kv_len)
    f = lambda a: np.asarray(a, np.float64)
    for b in range(x.shape[0]):
        hn = f(oracle.norm_row(D, h1[b], w["ln2_g"], w["ln2_b"]))
        gate = f(w["w1"])[:, 0, :] @ hn + f(w["b1"])[:, 0]
        up = f(w["w1"])[:, 1, :] @ hn + f(w["b1"])[:, 1]
        act = gate * (1.0 / (1.0 + np.exp(-gate))) * up
        want = h1[b] + f(w["b2"]) + act @ f(w["w2T"])
        np.testing.assert_allclose(pre[b], gate, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(y[b], want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_selecting_everything_equals_dense_bitwise(dtype):
    cfg, D, w, kc, vc, x = _random(dtype=dtype)
    h1d, yd, _, _, _ = oracle.dense_layer(D, w, x, kc, vc, cfg.kv_len)
    _, ys, _, _ = oracle.layer(D, w, x, np.arange(cfg.n_heads, dtype=np.int32),
                               np.arange(cfg.d_ffn, dtype=np.int32), kc, vc, cfg.kv_len)
    assert np.array_equal(yd, ys)


def test_unselected_neurons_contribute_nothing_and_gate_up_are_one_neuron():
    cfg, D, w, kc, vc, x = _random()
    rng = np.random.default_rng(4)
    u_n = np.sort(rng.choice(cfg.d_ffn, cfg.k_neurons, replace=False)).astype(np.int32)
    h1 = rng.standard_normal((2, cfg.d_model))
    y, _ = oracle.sparse_mlp(D, w, h1, u_n)
    w2 = {k: v.copy() for k, v in w.items()}
    off = np.setdiff1d(np.arange(cfg.d_ffn), u_n)
    for n in ("w1", "b1", "w2T"):
        w2[n][off] = rng.standard_normal(w2[n][off].shape).astype(np.float32)
    y2, _ = oracle.sparse_mlp(D, w2, h1, u_n)
    assert np.array_equal(y, y2)
    # the up row of a selected neuron scales its contribution linearly
    j = u_n[0]
    w3 = {k: v.copy() for k, v in w.items()}
    w3["w1"][j, 1] *= 2
    w3["b1"][j, 1] *= 2
    y3, _ = oracle.sparse_mlp(D, w3, h1, np.array([j], np.int32))
    y1, _ = oracle.sparse_mlp(D, w, h1, np.array([j], np.int32))
    np.testing.assert_allclose(y3 - h1, 2 * (y1 - h1) - (h1 * 0 + w["b2"]), rtol=1e-12,
                               atol=1e-12)
