"""dv_predict_topk_noalloc (scratch in a static device array of the library)
against dv_predict_topk (caller workspace), through the C ABI.

Two calls in a row on different inputs check that each call leaves the
shared scratch ready for the next one.  Kept in its own file, collected last.
"""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import dv_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


def _outputs(sel, sh, sn):
    u_h, u_n = sel.unions()
    return {"idx_h": sel.idx_h.clone(), "idx_n": sel.idx_n.clone(), "u_h": u_h.clone(),
            "u_n": u_n.clone(), "s_h": sh.clone(), "s_n": sn.clone()}


@pytest.mark.parametrize("name,B", [("tiny", 3), ("opt6.7b", 2), ("opt175b", 1)])
def test_noalloc_matches_workspace_entry(dv, name, B):
    cfg = dv_inputs.CONFIGS[name].with_(batch=B)
    dev = torch.device("cuda", 0)
    desc = dv.desc_from_config(cfg)
    layer = dv.Layer(desc, dv_inputs.make_weights(cfg, seed=7, device=dev))
    ws = dv.Workspace(desc, B)
    H, N = cfg.n_heads, cfg.d_ffn
    for call, seed in enumerate((21, 22)):  # two calls in a row, different inputs
        x = dv_inputs.make_x(cfg, B, seed=seed, device=dev)
        sel_ref = dv.SelectionBuffers(desc, B, cfg.k_heads, cfg.k_neurons)
        sh_ref = torch.empty((B, H), device=dev)
        sn_ref = torch.empty((B, N), device=dev)
        dv.dv_predict_topk(layer, x, cfg.k_heads, cfg.k_neurons, sel_ref, ws, sh_ref, sn_ref)
        want = _outputs(sel_ref, sh_ref, sn_ref)

        sel = dv.SelectionBuffers(desc, B, cfg.k_heads, cfg.k_neurons)
        sel.idx_n.fill_(-7)
        sel.n_u_n.fill_(-7)
        sh = torch.full((B, H), float("nan"), device=dev)
        sn = torch.full((B, N), float("nan"), device=dev)
        dv.dv_predict_topk_noalloc(layer, x, cfg.k_heads, cfg.k_neurons, sel, sh, sn)
        got = _outputs(sel, sh, sn)
        torch.cuda.synchronize()

        # the same kernels on the same inputs: the index sets agree exactly and
        # the scores within the parity tolerance (in practice bit for bit)
        for key in ("idx_h", "idx_n", "u_h", "u_n"):
            assert torch.equal(got[key], want[key]), (name, call, key)
        for key in ("s_h", "s_n"):
            err = (got[key] - want[key]).abs().max().item()
            assert err <= 1e-6 * max(1.0, want[key].abs().max().item()), (name, call, key, err)
        assert got["u_n"].numel() >= cfg.k_neurons and got["u_h"].numel() >= cfg.k_heads


def test_noalloc_rejects_shapes_beyond_its_scratch(dv):
    # the 175B shape at batch 32 needs more than the fixed scratch
    cfg = dv_inputs.CONFIGS["opt175b"].with_(batch=32)
    desc = dv.desc_from_config(cfg)
    small = dv_inputs.CONFIGS["tiny"]
    layer_w = dv_inputs.make_weights(small, seed=0, device="cuda")
    x = torch.zeros((32, cfg.d_model), device="cuda")
    sel = dv.SelectionBuffers(desc, 32, cfg.k_heads, cfg.k_neurons)
    with pytest.raises(dv.DvError) as e:
        # weight pointers are only checked for alignment before the size check
        dv.dv_predict_topk_noalloc(dv.Layer(desc, layer_w), x, cfg.k_heads,
                                   cfg.k_neurons, sel)
    assert e.value.status == dv.DV_ERR_SCRATCH_LIMIT
