"""GPU parity of the one-pass sparse MLP (fc1 rows and fc2 columns of each
CTA's share of the neuron union in one kernel, then the sum of the per-CTA
partials of y) against the CPU oracle, through dv_sparse_mlp."""

import numpy as np
import pytest
import torch

import dv_inputs
import oracle
from parity import assert_close, make_case

pytestmark = pytest.mark.gpu

CFG = dv_inputs.CONFIGS
# d = 264: 33 chunks (one fc1 segment, one fc2 chunk column per thread)
RAGGED = dv_inputs.LayerConfig("ragged", 264, 6, 64, 1000, 40, 37, 2, "f16",
                               dv_inputs.Fraction(77, 1000), k_heads_fixed=3)
# d = 2056: 257 chunks (a second fc1 segment of one chunk)
SEG2 = dv_inputs.LayerConfig("seg2", 2056, 8, 64, 3000, 40, 16, 1, "f16",
                             dv_inputs.Fraction(1, 10), k_heads_fixed=2)


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


def _run(dv, case, u_n, n_used=None):
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    ws = dv.Workspace(desc, case.B)
    h1 = torch.from_numpy(case.x).cuda()
    y = torch.empty_like(h1)
    un = torch.from_numpy(np.asarray(u_n, np.int32)).cuda()
    nun = torch.tensor([len(u_n) if n_used is None else n_used], dtype=torch.int32,
                       device="cuda")
    dv.dv_sparse_mlp(layer, h1, un, nun, y, ws)
    torch.cuda.synchronize()
    assert dv.dv_check(ws) == dv.DV_OK
    return y.cpu().numpy()


def test_where_it_serves(dv):
    d175 = dv.desc_from_config(CFG["opt175b"])
    assert dv.dv_mlp_one_pass(d175, 1, 2458) and dv.dv_mlp_one_pass(d175, 2, 4916)
    assert not dv.dv_mlp_one_pass(d175, 3, 7374)  # tensor-core kernels from 3 rows
    # more neurons per CTA than it stages
    G = torch.cuda.get_device_properties(0).multi_processor_count
    assert not dv.dv_mlp_one_pass(d175, 1, 64 * G + 1)
    assert dv.dv_mlp_one_pass(d175, 1, 64 * G)


@pytest.mark.parametrize("B", [1, 2])
@pytest.mark.parametrize("n", [1, 5, 151, 152, 153, 300, 1000])
def test_union_sizes(dv, B, n):
    # fewer neurons than CTAs leaves CTAs with nothing (their partial is zero);
    # 1000 selects every neuron
    case = make_case(RAGGED, B=B, seed=100 + n)
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    assert dv.dv_mlp_one_pass(desc, B, n)
    rng = np.random.default_rng(n)
    u_n = np.sort(rng.choice(case.cfg.d_ffn, n, replace=False)).astype(np.int32)
    y = _run(dv, case, u_n)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    yo, _ = oracle.sparse_mlp(D, case.w_host, case.x.astype(np.float64), u_n)
    assert_close(y, yo, "y")
    assert_close(y - case.x, yo - case.x, "y - h1")


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_two_segment_rows(dv, norm):
    case = make_case(SEG2.with_(norm=norm), B=1, seed=8)
    rng = np.random.default_rng(3)
    u_n = np.sort(rng.choice(case.cfg.d_ffn, 700, replace=False)).astype(np.int32)
    y = _run(dv, case, u_n)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    yo, _ = oracle.sparse_mlp(D, case.w_host, case.x.astype(np.float64), u_n)
    assert_close(y - case.x, yo - case.x, "y - h1")


def test_device_count_below_buffer_and_determinism(dv):
    case = make_case(RAGGED, B=2, seed=4)
    rng = np.random.default_rng(4)
    u_n = np.sort(rng.choice(case.cfg.d_ffn, 500, replace=False)).astype(np.int32)
    y1 = _run(dv, case, u_n, n_used=333)
    y2 = _run(dv, case, u_n, n_used=333)
    assert np.array_equal(y1, y2)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    yo, _ = oracle.sparse_mlp(D, case.w_host, case.x.astype(np.float64), u_n[:333])
    assert_close(y1 - case.x, yo - case.x, "y - h1")


def test_opt175b_batch2_union(dv):
    cfg = CFG["opt175b"]
    case = make_case(cfg, B=2, gen_device="cuda", norm_affine=True)
    rng = np.random.default_rng(11)
    u_n = np.sort(rng.choice(cfg.d_ffn, 2 * cfg.k_neurons - 300, replace=False)).astype(np.int32)
    y = _run(dv, case, u_n)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    yo, _ = oracle.sparse_mlp(D, case.w_host, case.x.astype(np.float64), u_n)
    assert_close(y - case.x, yo - case.x, "y - h1")
