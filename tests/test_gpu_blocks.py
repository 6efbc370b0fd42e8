"""GPU parity of blocked neuron selection (blocks of contiguous channels,
each scored by its largest member score, k / block best kept per row)
against the CPU oracle: the selection alone (dv_predict_topk and its
no-allocation form) and whole layer decodes."""

import numpy as np
import pytest
import torch

import dv_inputs
import oracle
from parity import check_block_rows, check_layer_parity, make_case, run_gpu_layer

pytestmark = pytest.mark.gpu

CFG = dv_inputs.CONFIGS
# 1024 neurons in 32 blocks of 32
SMALL = dv_inputs.LayerConfig("blk32", 264, 6, 64, 1024, 40, 37, 1, "f16",
                              dv_inputs.Fraction(1, 8), k_heads_fixed=3, neuron_block=32)


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


def _predict(dv, case, noalloc=False):
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    sel = dv.SelectionBuffers(desc, case.B, case.k_h, case.k_n)
    ws = dv.Workspace(desc, case.B)
    x = torch.from_numpy(case.x).cuda()
    if noalloc:
        dv.dv_predict_topk_noalloc(layer, x, case.k_h, case.k_n, sel)
    else:
        dv.dv_predict_topk(layer, x, case.k_h, case.k_n, sel, ws)
    torch.cuda.synchronize()
    if not noalloc:
        assert dv.dv_check(ws) == dv.DV_OK
    u_h, u_n = sel.unions()
    return sel.idx_n.cpu().numpy(), u_n.cpu().numpy()


@pytest.mark.parametrize("B", [1, 3, 8])
@pytest.mark.parametrize("cfg", [SMALL, CFG["tiny"].with_(neuron_block=64)],
                         ids=["f16-blk32", "f32-blk64"])
def test_predict_selects_blocks(dv, cfg, B):
    case = make_case(cfg, B=B, seed=B)
    idx_n, u_n = _predict(dv, case)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    p = oracle.predict(D, case.w_host, case.x, case.k_h, case.k_n)
    check_block_rows(idx_n, p["idx_n"], p["s_n"], cfg.neuron_block, case.k_n, "blocks")
    assert np.array_equal(u_n, np.unique(idx_n))


def test_noalloc_predict_selects_blocks(dv):
    case = make_case(SMALL, B=2, seed=12)
    idx_n, u_n = _predict(dv, case, noalloc=True)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    p = oracle.predict(D, case.w_host, case.x, case.k_h, case.k_n)
    check_block_rows(idx_n, p["idx_n"], p["s_n"], 32, case.k_n, "blocks")


def test_counts_not_in_whole_blocks_are_rejected(dv):
    case = make_case(SMALL, B=1, seed=3)
    with pytest.raises(dv.DvError) as e:
        run_gpu_layer(dv, case.__class__(**{**case.__dict__, "k_n": case.k_n + 1}))
    assert e.value.status == dv.DV_ERR_INVALID_ARG


@pytest.mark.parametrize("B", [1, 2, 4])
def test_small_layer_decode(dv, B):
    case = make_case(SMALL, B=B, seed=20 + B, separate_x_pred=(B == 2))
    check_layer_parity(case, run_gpu_layer(dv, case))


@pytest.mark.parametrize("B", [1, 2])
def test_opt175b_blk64(dv, B):
    case = make_case(CFG["opt175b_blk64"], B=B, gen_device="cuda", norm_affine=False)
    g = run_gpu_layer(dv, case)
    out = check_layer_parity(case, g)
    assert g["u_n"].size % 64 == 0 and g["u_n"].size >= 2496
    print("opt175b blocks of 64, B", B, out)
