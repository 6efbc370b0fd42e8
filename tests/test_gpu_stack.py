"""The layer stack with the lookahead predictor on a side stream (GPU).

Each layer is checked against the oracle on the GPU's own predictor input
and index sets: layer l+1's sets must be the top-k of the predictor run on
layer l's input (layer 0: its own input), and its output the oracle layer
on those sets.  The overlapped run must equal the serial run bit for bit.
"""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import dv_inputs  # noqa: E402
import oracle  # noqa: E402
from parity import assert_close, check_topk_rows, MAX_ABS, REL_L2  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mods():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv, stack

    return dv, stack


@pytest.mark.parametrize("name,B,n_layers,fused", [("tiny", 2, 4, False), ("opt6.7b", 1, 3, False),
                                                   ("opt6.7b", 1, 3, True), ("opt6.7b", 2, 2, True),
                                                   ("opt6.7b", 4, 2, False)])
def test_stack_layers_match_oracle(mods, name, B, n_layers, fused):
    dv, stack = mods
    cfg = dv_inputs.CONFIGS[name].with_(batch=B)
    desc = dv.desc_from_config(cfg)
    ws = stack.make_stack_weights(cfg, n_layers, device="cuda", seed0=40)
    layers = stack.layers_from_weights(desc, ws)
    caches = stack.stack_caches(cfg, n_layers, B, device="cuda", seed0=40)
    caches_host = [(kc.cpu().numpy(), vc.cpu().numpy()) for kc, vc in caches]
    x0 = dv_inputs.make_x(cfg, B, seed=7, device="cuda")
    st = stack.LayerStack(desc, layers, B, cfg.k_heads, cfg.k_neurons)
    st.keep_selection = True
    y = st.run(x0, caches, cfg.kv_len, fused=fused)
    xs = [t.cpu().numpy() for t in st.x]
    D = oracle.desc_from_config(cfg)
    for l in range(n_layers):
        wh = {k: v.cpu().numpy() for k, v in ws[l].items()}
        sel = st.kept[l]
        x_pred = xs[max(l - 1, 0)]
        p = oracle.predict(D, wh, x_pred, cfg.k_heads, cfg.k_neurons)
        check_topk_rows(sel["idx_h"].cpu().numpy(), p["idx_h"], p["s_h"], cfg.k_heads, "heads")
        check_topk_rows(sel["idx_n"].cpu().numpy(), p["idx_n"], p["s_n"], cfg.k_neurons, "neurons")
        u_h = sel["u_h"][: int(sel["n_u_h"].item())].cpu().numpy()
        u_n = sel["u_n"][: int(sel["n_u_n"].item())].cpu().numpy()
        assert np.array_equal(u_h, np.unique(sel["idx_h"].cpu().numpy()))
        assert np.array_equal(u_n, np.unique(sel["idx_n"].cpu().numpy()))
        kc, vc = caches_host[l]
        h1, yl, _, _ = oracle.layer(D, wh, xs[l], u_h, u_n, kc, vc, cfg.kv_len)
        assert_close(xs[l + 1], yl, f"layer {l} y", MAX_ABS, REL_L2)
        assert_close(xs[l + 1] - xs[l], yl - xs[l].astype(np.float64), f"layer {l} y - x",
                     MAX_ABS, REL_L2)
    assert np.array_equal(y.cpu().numpy(), xs[-1])


def test_stack_fused_is_deterministic(mods):
    dv, stack = mods
    cfg = dv_inputs.CONFIGS["opt6.7b"].with_(batch=2)
    desc = dv.desc_from_config(cfg)
    ws = stack.make_stack_weights(cfg, 3, device="cuda", seed0=91)
    layers = stack.layers_from_weights(desc, ws)
    x0 = dv_inputs.make_x(cfg, 2, seed=4, device="cuda")
    st = stack.LayerStack(desc, layers, 2, cfg.k_heads, cfg.k_neurons)
    outs = []
    for _ in range(2):
        caches = stack.stack_caches(cfg, 3, 2, device="cuda", seed0=91)
        outs.append(st.run(x0, caches, cfg.kv_len, fused=True))
    assert torch.equal(outs[0], outs[1])


def test_stack_overlap_equals_serial(mods):
    dv, stack = mods
    cfg = dv_inputs.CONFIGS["opt6.7b"].with_(batch=2)
    desc = dv.desc_from_config(cfg)
    ws = stack.make_stack_weights(cfg, 3, device="cuda", seed0=90)
    layers = stack.layers_from_weights(desc, ws)
    x0 = dv_inputs.make_x(cfg, 2, seed=3, device="cuda")
    st = stack.LayerStack(desc, layers, 2, cfg.k_heads, cfg.k_neurons)
    outs = []
    for serial in (False, True, False):
        caches = stack.stack_caches(cfg, 3, 2, device="cuda", seed0=90)
        outs.append(st.run(x0, caches, cfg.kv_len, serial=serial, fused=False))
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
