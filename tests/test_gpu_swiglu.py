"""GPU parity of the LLaMA-style SwiGLU MLP (RMSNorm; gate and up rows of a
neuron side by side in w1, act = silu(gate) * up, down projection in w2T)
against the CPU oracle: whole layer decodes at batches served by the
one-pass MLP (1, 2) and by the row + column kernels (3 and up), caller-chosen
neuron sets, and the LLaMA-3-70B shape."""

import numpy as np
import pytest
import torch

import dv_inputs
import oracle
from parity import assert_close, check_layer_parity, make_case, run_gpu_layer

pytestmark = pytest.mark.gpu

CFG = dv_inputs.CONFIGS
# binary16, d = 264 (33 chunks: ragged), 704 neurons
SW16 = dv_inputs.LayerConfig("sw16", 264, 6, 64, 704, 40, 37, 1, "f16",
                             dv_inputs.Fraction(1, 4), k_heads_fixed=3, norm="rmsnorm",
                             mlp="swiglu")


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


@pytest.mark.parametrize("B", [1, 2, 3, 5])
@pytest.mark.parametrize("cfg", [CFG["llama_tiny"], SW16], ids=["f32", "f16"])
def test_layer_decode(dv, cfg, B):
    case = make_case(cfg, B=B, seed=40 + B, separate_x_pred=(B == 2))
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    assert dv.dv_mlp_one_pass(desc, B, min(B * case.k_n, cfg.d_ffn)) == (B <= 2)
    check_layer_parity(case, run_gpu_layer(dv, case))


@pytest.mark.parametrize("B", [1, 2, 4])
@pytest.mark.parametrize("n", [1, 153, 704])
def test_caller_neuron_sets(dv, B, n):
    case = make_case(SW16, B=B, seed=n + B)
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    ws = dv.Workspace(desc, case.B)
    u_n = np.sort(np.random.default_rng(n).choice(SW16.d_ffn, n, replace=False)).astype(np.int32)
    h1 = torch.from_numpy(case.x).cuda()
    y = torch.empty_like(h1)
    nun = torch.tensor([n], dtype=torch.int32, device="cuda")
    dv.dv_sparse_mlp(layer, h1, torch.from_numpy(u_n).cuda(), nun, y, ws)
    torch.cuda.synchronize()
    assert dv.dv_check(ws) == dv.DV_OK
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    yo, _ = oracle.sparse_mlp(D, case.w_host, case.x.astype(np.float64), u_n)
    assert_close(y.cpu().numpy() - case.x, yo - case.x, "y - h1")


def test_persistent_kernel_does_not_serve_swiglu(dv):
    assert not dv.dv_layer_decode_persistent_ok(dv.desc_from_config(CFG["llama3_70b"]), 1)


def test_llama3_70b(dv):
    case = make_case(CFG["llama3_70b"], B=1, gen_device="cuda", norm_affine=True)
    g = run_gpu_layer(dv, case)
    out = check_layer_parity(case, g)
    assert g["u_n"].size == 7168 and g["u_h"].size == 13
    print("llama3-70b shape", out)
