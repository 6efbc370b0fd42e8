"""dv_predict_topk_noalloc (scratch in a static device array of the library)
against dv_predict_topk (caller workspace), through the C ABI.

Two calls in a row on different inputs check that each call leaves the
shared scratch ready for the next one.  Kept in its own file, collected last.
"""
import os
import sys
from fractions import Fraction

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


# A narrow layer with a very wide MLP (binary32, d = 16, r = 8, N = 2^19):
# the neuron predictor's scores, row counters and bitmaps grow with N and the
# batch, so at batch 2 the scratch needs about 8.3 MiB (more than the fixed
# 8 MiB) while batch 1 needs about 4.2 MiB.  Every buffer is sized for this
# descriptor, so nothing depends on the refusal happening before a launch.
WIDE = dv_inputs.LayerConfig("wide_ffn", 16, 2, 8, 1 << 19, 8, 4, 1, "f32", Fraction(1, 100),
                             k_heads_fixed=1)


def test_noalloc_rejects_shapes_beyond_its_scratch(dv):
    dev = torch.device("cuda", 0)
    desc = dv.desc_from_config(WIDE)
    layer = dv.Layer(desc, dv_inputs.make_weights(WIDE, seed=3, device=dev))
    k_h, k_n = WIDE.k_heads, WIDE.k_neurons

    # batch 2: refused, nothing launched, the buffers untouched
    x2 = dv_inputs.make_x(WIDE, 2, seed=4, device=dev)
    sel2 = dv.SelectionBuffers(desc, 2, k_h, k_n)
    sel2.n_u_n.fill_(-7)
    with pytest.raises(dv.DvError) as e:
        dv.dv_predict_topk_noalloc(layer, x2, k_h, k_n, sel2)
    assert e.value.status == dv.DV_ERR_SCRATCH_LIMIT
    torch.cuda.synchronize()
    assert int(sel2.n_u_n.item()) == -7

    # batch 1 of the same layer fits and equals the workspace entry
    x1 = x2[:1].contiguous()
    ws = dv.Workspace(desc, 1)
    ref = dv.SelectionBuffers(desc, 1, k_h, k_n)
    dv.dv_predict_topk(layer, x1, k_h, k_n, ref, ws)
    sel1 = dv.SelectionBuffers(desc, 1, k_h, k_n)
    dv.dv_predict_topk_noalloc(layer, x1, k_h, k_n, sel1)
    torch.cuda.synchronize()
    assert torch.equal(sel1.idx_n, ref.idx_n) and torch.equal(sel1.idx_h, ref.idx_h)
    assert torch.equal(sel1.unions()[1], ref.unions()[1])
