"""GPU parity of the persistent layer kernel (dv_layer_decode_persistent:
binary16 weights, 128-wide heads, batch 1-2; one cooperative launch whose
phases wait on counters) and of the seven chained kernels of
dv_layer_decode, each against the CPU oracle and against each other."""

import numpy as np
import pytest
import torch

import dv_inputs
from parity import assert_close, check_layer_parity, make_case, run_gpu_layer

pytestmark = pytest.mark.gpu

CFG = dv_inputs.CONFIGS
# 128-wide heads on a small ragged shape: d and N leave partial column blocks
# and uneven row splits in every phase
RAGGED128 = dv_inputs.LayerConfig("ragged128", 520, 5, 128, 1100, 40, 45, 1, "f16",
                                  dv_inputs.Fraction(9, 100), k_heads_fixed=2)
BOTH = ["dv_layer_decode", "dv_layer_decode_persistent"]


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


def test_where_the_persistent_kernel_serves(dv):
    d175 = dv.desc_from_config(CFG["opt175b"])
    assert dv.dv_layer_decode_persistent_ok(d175, 1)
    assert dv.dv_layer_decode_persistent_ok(d175, 2)
    assert not dv.dv_layer_decode_persistent_ok(d175, 3)
    assert dv.dv_layer_decode_launches(d175, 1) == 7
    # binary32 weights and 64-wide heads are not served; the call says so
    assert not dv.dv_layer_decode_persistent_ok(dv.desc_from_config(CFG["tiny"]), 1)
    ragged64 = RAGGED128.with_(head_dim=64)
    assert not dv.dv_layer_decode_persistent_ok(dv.desc_from_config(ragged64), 1)
    case = make_case(ragged64, B=1, seed=1)
    with pytest.raises(dv.DvError) as e:
        run_gpu_layer(dv, case, entry="dv_layer_decode_persistent")
    assert e.value.status == dv.DV_ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", BOTH)
@pytest.mark.parametrize("B", [1, 2])
def test_ragged_shape(dv, entry, B):
    case = make_case(RAGGED128, B=B, seed=10 + B, separate_x_pred=(B == 2))
    g = run_gpu_layer(dv, case, entry=entry)
    check_layer_parity(case, g)


@pytest.mark.parametrize("entry", BOTH)
def test_opt67b_batch2(dv, entry):
    case = make_case(CFG["opt6.7b"], B=2, gen_device="cuda", norm_affine=True)
    g = run_gpu_layer(dv, case, entry=entry)
    check_layer_parity(case, g)


def test_opt175b_persistent(dv):
    # the chained path at this shape is test_gpu_parity.test_opt175b_full
    case = make_case(CFG["opt175b"], gen_device="cuda", norm_affine=False)
    g = run_gpu_layer(dv, case, entry="dv_layer_decode_persistent")
    check_layer_parity(case, g)


def test_persistent_matches_chained(dv):
    case = make_case(CFG["opt66b"], B=1, gen_device="cuda", norm_affine=True)
    gp = run_gpu_layer(dv, case, entry="dv_layer_decode_persistent")
    gc = run_gpu_layer(dv, case, entry="dv_layer_decode")
    # the selections and the appended KV come from identical arithmetic
    for k in ("idx_h", "idx_n", "u_h", "u_n", "kc", "vc"):
        assert np.array_equal(gp[k], gc[k]), k
    # out-projection partials are grouped over one CTA fewer: equal to rounding
    assert_close(gp["h1"] - case.x, gc["h1"] - case.x, "h1 - x", 1e-5, 1e-5)
    assert_close(gp["y"], gc["y"], "y", 1e-5, 1e-6)


def test_graph_replay_resets_phase_counters(dv):
    case = make_case(RAGGED128, B=1, seed=3)
    ref = run_gpu_layer(dv, case, entry="dv_layer_decode_persistent")
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    sel = dv.SelectionBuffers(desc, case.B, case.k_h, case.k_n)
    ws = dv.Workspace(desc, case.B)
    x = torch.from_numpy(case.x).cuda()
    kc = torch.from_numpy(case.kc).cuda()
    vc = torch.from_numpy(case.vc).cuda()
    y = torch.zeros_like(x)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            for _ in range(5):  # each decode rewrites the same KV slot and y
                dv.dv_layer_decode_persistent(layer, x, case.k_h, case.k_n, kc, vc, case.kv_len, sel, y, ws,
                                   stream=s)
    for _ in range(20):
        y.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert dv.dv_check(ws) == dv.DV_OK
    assert np.array_equal(y.cpu().numpy(), ref["y"])
    # control words: [0] status, [1] side flag (set by the last decode), [8, 16)
    # the phase counters, zero at rest
    off = ws.ptr - ws.buf.data_ptr()
    ctl = ws.buf[off:off + 64 * 4].cpu().numpy().view(np.int32)
    assert ctl[8:16].tolist() == [0] * 8
