"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Sizes: the tiny shape and a ragged shape that spans several tiles with
ragged tails run in full; the OPT-6.7B/66B/175B shapes run at their full
sizes in the launch configuration the benchmark times, and the oracle
(plain C, binary64) computes every output for comparison.
"""

import numpy as np
import pytest
import torch

import dv_inputs
import oracle
from parity import (assert_close, check_layer_parity, check_topk_rows, make_case,
                    run_gpu_layer)

pytestmark = pytest.mark.gpu

CFG = dv_inputs.CONFIGS
RAGGED = dv_inputs.LayerConfig("ragged", 264, 6, 64, 1000, 40, 37, 2, "f16",
                               dv_inputs.Fraction(77, 1000), k_heads_fixed=3)


@pytest.fixture(scope="module")
def dv():
    from attention_dv_predict_gb300 import build

    build.build()
    from attention_dv_predict_gb300 import dv as mod

    return mod


def test_tiny_fp32_layer(dv):
    case = make_case(CFG["tiny"])
    g = run_gpu_layer(dv, case)
    out = check_layer_parity(case, g, tight=True)
    assert out["diff_heads"] == 0 and out["diff_neurons"] == 0


@pytest.mark.parametrize("norm", ["layernorm", "rmsnorm"])
def test_tiny_batch3_union_and_norms(dv, norm):
    case = make_case(CFG["tiny"].with_(norm=norm), B=3, separate_x_pred=True)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g, tight=True)
    assert CFG["tiny"].k_neurons <= g["u_n"].size <= 3 * CFG["tiny"].k_neurons


@pytest.mark.parametrize("B", [1, 2, 5])
def test_ragged_fp16_shapes(dv, B):
    case = make_case(RAGGED, B=B, seed=B)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)


def test_select_everything_equals_dense_oracle(dv):
    cfg = CFG["tiny"]
    case = make_case(cfg, B=2, k_h=cfg.n_heads, k_n=cfg.d_ffn)
    g = run_gpu_layer(dv, case)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    h1, y, _, _, _ = oracle.dense_layer(D, case.w_host, case.x, case.kc, case.vc, case.kv_len)
    assert np.array_equal(g["u_h"], np.arange(cfg.n_heads))
    assert np.array_equal(g["u_n"], np.arange(cfg.d_ffn))
    assert_close(g["y"], y, "y", 1e-4, 1e-5)
    assert_close(g["h1"], h1, "h1", 1e-4, 1e-5)


@pytest.mark.parametrize("kv_len", [0, 1, 31, 32, 33])
def test_kv_length_edges(dv, kv_len):
    case = make_case(RAGGED, B=2, kv_len=kv_len, kv_cap=kv_len + 3)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)


def test_k_equals_one(dv):
    case = make_case(RAGGED, B=3, k_h=1, k_n=1)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)


def test_ties_pick_lower_index(dv):
    """Duplicate predictor rows give exactly equal scores: when only one of a
    tied pair is kept, it is the lower index."""
    cfg = CFG["tiny"]
    case = make_case(cfg, B=1, k_h=3, k_n=101)
    for key in ("pred_h", "pred_b"):
        h = case.w_host[key]
        h[1::2] = h[0::2]  # rows 2i and 2i+1 identical -> equal scores
        case.w_dev[key].copy_(torch.from_numpy(h))
    g = run_gpu_layer(dv, case)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    p = oracle.predict(D, case.w_host, case.x, case.k_h, case.k_n)
    for got, want, s, k in ((g["idx_h"], p["idx_h"], p["s_h"], case.k_h),
                            (g["idx_n"], p["idx_n"], p["s_n"], case.k_n)):
        check_topk_rows(got, want, s, k, "ties")
        kept = set(got[0].tolist())
        # k is odd, so at least one pair is split by the boundary
        singles = [i for i in kept if (i ^ 1) not in kept]
        assert singles and all(i % 2 == 0 for i in singles), singles


def test_predict_scores_and_sets(dv):
    case = make_case(RAGGED, B=4, seed=11)
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    sel = dv.SelectionBuffers(desc, case.B, case.k_h, case.k_n)
    ws = dv.Workspace(desc, case.B)
    x = torch.from_numpy(case.x).cuda()
    sh = torch.empty((case.B, case.cfg.n_heads), device="cuda")
    sn = torch.empty((case.B, case.cfg.d_ffn), device="cuda")
    dv.dv_predict_topk(layer, x, case.k_h, case.k_n, sel, ws, sh, sn)
    torch.cuda.synchronize()
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    p = oracle.predict(D, case.w_host, case.x, case.k_h, case.k_n)
    assert_close(sh.cpu().numpy(), p["s_h"], "head scores", 1e-4, 1e-5)
    assert_close(sn.cpu().numpy(), p["s_n"], "neuron scores", 1e-4, 1e-5)
    check_topk_rows(sel.idx_h.cpu().numpy(), p["idx_h"], p["s_h"], case.k_h, "heads")
    check_topk_rows(sel.idx_n.cpu().numpy(), p["idx_n"], p["s_n"], case.k_n, "neurons")


# binary16 from batch 3 on: both predictor stages on the tensor-core row
# kernel; rank 1000 leaves an 8-column last 32-k block in stage 2
PRED_MMA = dv_inputs.LayerConfig("pred_mma", 4096, 6, 128, 3000, 1000, 70, 1, "f16",
                                 dv_inputs.Fraction(1, 10), k_heads_fixed=2)


@pytest.mark.parametrize("B", [3, 11, 32])
def test_predict_tensor_core_path(dv, B):
    case = make_case(PRED_MMA, B=B, seed=40 + B)
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    sel = dv.SelectionBuffers(desc, case.B, case.k_h, case.k_n)
    ws = dv.Workspace(desc, case.B)
    x = torch.from_numpy(case.x).cuda()
    sh = torch.empty((case.B, case.cfg.n_heads), device="cuda")
    sn = torch.empty((case.B, case.cfg.d_ffn), device="cuda")
    for _ in range(2):  # the second call finds the histograms cleared by the first
        dv.dv_predict_topk(layer, x, case.k_h, case.k_n, sel, ws, sh, sn)
    torch.cuda.synchronize()
    assert dv.dv_check(ws) == dv.DV_OK
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    p = oracle.predict(D, case.w_host, case.x, case.k_h, case.k_n)
    eh, en = tensor_core_score_bounds(case.w_host, case.x)
    for got, want, tol, what in ((sh, p["s_h"], eh, "head"), (sn, p["s_n"], en, "neuron")):
        err = np.abs(got.cpu().numpy().astype(np.float64) - want)
        assert np.all(err <= tol), f"{what} scores: worst error / bound {np.max(err / tol):.3f}"
    check_topk_rows(sel.idx_h.cpu().numpy(), p["idx_h"], p["s_h"], case.k_h, "heads")
    check_topk_rows(sel.idx_n.cpu().numpy(), p["idx_n"], p["s_n"], case.k_n, "neurons")


def tensor_core_score_bounds(w, x):
    """Elementwise bounds on the tensor-core predictor scores.  Each stage
    runs 2 ceil(K/16) binary32 MMA accumulations (the activations split into
    binary16 hi and lo parts), each off by at most one binary32 ulp of the
    running sum, which is bounded by sum_k |w_k x_k|; the split leaves a
    residual of 2^-22 relative, and the result is rounded once more:
    c = 2 ceil(K/16) + 4 units of 2^-23 sum |w x|.  Stage 2 also carries
    stage 1's error in u through |Bm|."""
    eps = 2.0 ** -23
    x = np.abs(x.astype(np.float64))
    wh = np.abs(w["pred_h"].astype(np.float64))
    a = w["pred_a"].astype(np.float64)
    bm = np.abs(w["pred_b"].astype(np.float64))
    d, r = a.shape[1], a.shape[0]
    c1 = 2 * -(-d // 16) + 4
    c2 = 2 * -(-r // 16) + 4
    eh = c1 * eps * x @ wh.T
    ua = x @ np.abs(a).T  # bounds |u| and stage 1's running sums
    en = c2 * eps * ua @ bm.T + c1 * eps * ua @ bm.T
    return eh + 1e-12, en + 1e-12


def test_layer_tensor_core_predictor(dv):
    case = make_case(PRED_MMA, B=11, seed=61)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)


def test_blocks_on_caller_index_sets(dv):
    """dv_sparse_attn and dv_sparse_mlp on index sets the caller chooses."""
    case = make_case(RAGGED, B=2, seed=5)
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    ws = dv.Workspace(desc, case.B)
    rng = np.random.default_rng(0)
    u_h = np.sort(rng.choice(case.cfg.n_heads, 4, replace=False)).astype(np.int32)
    u_n = np.sort(rng.choice(case.cfg.d_ffn, 300, replace=False)).astype(np.int32)
    x = torch.from_numpy(case.x).cuda()
    kc = torch.from_numpy(case.kc).cuda()
    vc = torch.from_numpy(case.vc).cuda()
    h1 = torch.empty_like(x)
    y = torch.empty_like(x)
    uh_d = torch.from_numpy(u_h).cuda()
    un_d = torch.from_numpy(u_n).cuda()
    nuh = torch.tensor([u_h.size], dtype=torch.int32, device="cuda")
    nun = torch.tensor([u_n.size], dtype=torch.int32, device="cuda")
    dv.dv_sparse_attn(layer, x, uh_d, nuh, kc, vc, case.kv_len, h1, ws)
    dv.dv_sparse_mlp(layer, h1, un_d, nun, y, ws)
    torch.cuda.synchronize()
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    h1o, _, _, _ = oracle.sparse_attn(D, case.w_host, case.x, u_h, case.kc, case.vc, case.kv_len)
    assert_close(h1.cpu().numpy() - case.x, h1o - case.x, "h1 - x")
    yo, _ = oracle.sparse_mlp(D, case.w_host, h1.cpu().numpy().astype(np.float64), u_n)
    assert_close(y.cpu().numpy(), yo, "y")
    assert_close(y.cpu().numpy() - h1.cpu().numpy(), yo - h1.cpu().numpy(), "y - h1")
    # a device count below the buffer length uses only the prefix
    nun.fill_(100)
    dv.dv_sparse_mlp(layer, h1, un_d, nun, y, ws)
    torch.cuda.synchronize()
    yo2, _ = oracle.sparse_mlp(D, case.w_host, h1.cpu().numpy().astype(np.float64), u_n[:100])
    assert_close(y.cpu().numpy(), yo2, "y (prefix)")


def test_out_of_range_indices_are_skipped_and_reported(dv):
    case = make_case(RAGGED, B=1, seed=6)
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    ws = dv.Workspace(desc, 1)
    h1 = torch.from_numpy(case.x).cuda()
    y = torch.empty_like(h1)
    un = torch.tensor([3, case.cfg.d_ffn + 5, 7], dtype=torch.int32, device="cuda")
    nun = torch.tensor([3], dtype=torch.int32, device="cuda")
    dv.dv_sparse_mlp(layer, h1, un, nun, y, ws)
    assert dv.dv_check(ws) == dv.DV_ERR_DEVICE_INDEX
    assert dv.dv_check(ws) == dv.DV_OK  # reading clears it


def test_deterministic_and_graph_replay(dv):
    case = make_case(RAGGED, B=3, seed=7)
    g1 = run_gpu_layer(dv, case)
    g2 = run_gpu_layer(dv, case)
    assert np.array_equal(g1["y"], g2["y"]) and np.array_equal(g1["idx_n"], g2["idx_n"])
    # capture the whole decode in a CUDA graph and replay it
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
            dv.dv_layer_decode(layer, x, case.k_h, case.k_n, kc, vc, case.kv_len, sel, y, ws,
                               stream=s)
    for _ in range(3):
        y.zero_()
        graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), g1["y"])


def test_host_entry_point_matches_device(dv):
    case = make_case(RAGGED, B=2, seed=8)
    g = run_gpu_layer(dv, case)
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    ws = dv.Workspace(desc, case.B)
    kc = torch.from_numpy(case.kc).cuda()
    vc = torch.from_numpy(case.vc).cuda()
    xh = torch.from_numpy(case.x).pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    dv.dv_layer_decode_host(layer, xh, case.k_h, case.k_n, kc, vc, case.kv_len, yh, ws)
    assert np.array_equal(yh.numpy(), g["y"])


def test_hbm_copy(dv):
    src = torch.randn(1 << 22, device="cuda")
    dst = torch.empty_like(src)
    dv.dv_hbm_copy(dst, src)
    torch.cuda.synchronize()
    assert torch.equal(dst, src)


def test_invalid_arguments_launch_nothing(dv):
    case = make_case(CFG["tiny"])
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    sel = dv.SelectionBuffers(desc, 1, case.k_h, case.k_n)
    ws = dv.Workspace(desc, 1)
    x = torch.from_numpy(case.x).cuda()
    kc = torch.from_numpy(case.kc).cuda()
    vc = torch.from_numpy(case.vc).cuda()
    y = torch.full_like(x, 7.0)
    for kh, kn, L in ((0, 5, 3), (case.cfg.n_heads + 1, 5, 3), (2, 0, 3), (2, 5, case.kv_cap)):
        with pytest.raises(dv.DvError) as e:
            dv.dv_layer_decode(layer, x, kh, kn, kc, vc, L, sel, y, ws)
        assert e.value.status == dv.DV_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_shared_memory_opt_in_per_kernel_variant(dv):
    # a binary32 decode first, then a binary16 one whose stage-2 + QKV kernel
    # needs more than the 48 KB of shared memory a kernel gets without
    # opting in (the neuron selection's buffers at N = 36864): each kernel
    # variant must make its own opt-in
    tiny = make_case(CFG["tiny"], B=1, seed=30)
    check_layer_parity(tiny, run_gpu_layer(dv, tiny))
    wide = dv_inputs.LayerConfig("wideN", 264, 6, 64, 36864, 40, 37, 1, "f16",
                                 dv_inputs.Fraction(1, 20), k_heads_fixed=3)
    case = make_case(wide, B=1, seed=31)
    check_layer_parity(case, run_gpu_layer(dv, case))


# ---------------------------------------------------------------------------
# OPT shapes at full size (inputs generated by torch's device RNG, copied to
# the host for the oracle)


def test_opt67b_full(dv):
    case = make_case(CFG["opt6.7b"], gen_device="cuda", norm_affine=False)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)


@pytest.mark.parametrize("B", [1, 8])
def test_opt66b_full(dv, B):
    case = make_case(CFG["opt66b"], B=B, gen_device="cuda", norm_affine=False)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)
    if B == 8:
        assert CFG["opt66b"].k_neurons < g["u_n"].size <= 8 * CFG["opt66b"].k_neurons


@pytest.mark.parametrize("B", [3, 16, 25, 32])
def test_opt67b_batches_tensor_core_path(dv, B):
    # B >= 3 with binary16 weights runs QKV and fc1 on the tensor-core row
    # kernel: one partial batch tile at B = 3, two tiles per weight pass at
    # B = 16, four (the last one partial at B = 25) at B = 25 and 32
    case = make_case(CFG["opt6.7b"], B=B, gen_device="cuda", norm_affine=True)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)


# d = 4128 leaves a 32-column last block for the tensor-core column kernel
# (512-column blocks); batches 3, 5, 11, 17 and 25 give partial tiles of 8,
# one or two CTA tiles of 16 rows, and row-kernel passes of one, two or four
# batch tiles (four at 17 and 25, the last ones empty or partial)
RAGGED_MMA = dv_inputs.LayerConfig("ragged_mma", 4128, 6, 128, 3000, 64, 70, 1, "f16",
                                   dv_inputs.Fraction(1, 10), k_heads_fixed=2)


@pytest.mark.parametrize("B", [3, 5, 11, 17, 25])
def test_tensor_core_paths_ragged(dv, B):
    case = make_case(RAGGED_MMA, B=B, seed=20 + B)
    g = run_gpu_layer(dv, case)
    check_layer_parity(case, g)


def test_tensor_core_column_kernel_several_stages(dv):
    """fc2 over 18000 caller-chosen neurons at batch 8 and d = 12288: each CTA
    holds > 2048 rows of its column block, so it stages them in two passes."""
    cfg = dv_inputs.LayerConfig("wide_mlp", 12288, 2, 128, 20480, 64, 4, 8, "f16",
                                dv_inputs.Fraction(1, 10), k_heads_fixed=1)
    case = make_case(cfg, B=8, seed=31, gen_device="cuda")
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    ws = dv.Workspace(desc, case.B)
    rng = np.random.default_rng(3)
    u_n = np.sort(rng.choice(cfg.d_ffn, 18000, replace=False)).astype(np.int32)
    h1 = torch.from_numpy(case.x).cuda()
    y = torch.empty_like(h1)
    nun = torch.tensor([u_n.size], dtype=torch.int32, device="cuda")
    dv.dv_sparse_mlp(layer, h1, torch.from_numpy(u_n).cuda(), nun, y, ws)
    torch.cuda.synchronize()
    assert dv.dv_check(ws) == dv.DV_OK
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    yo, _ = oracle.sparse_mlp(D, case.w_host, case.x.astype(np.float64), u_n)
    assert_close(y.cpu().numpy() - case.x, yo - case.x, "y - h1")


def test_opt175b_full(dv):
    case = make_case(CFG["opt175b"], gen_device="cuda", norm_affine=False)
    g = run_gpu_layer(dv, case)
    out = check_layer_parity(case, g)
    assert g["u_n"].size == 2458 and g["u_h"].size == 20
    print("opt175b parity", out)


def _predict_only(dv, case):
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    sel = dv.SelectionBuffers(desc, case.B, case.k_h, case.k_n)
    ws = dv.Workspace(desc, case.B)
    x = torch.from_numpy(case.x).cuda()
    sn = torch.empty((case.B, case.cfg.d_ffn), device="cuda")
    dv.dv_predict_topk(layer, x, case.k_h, case.k_n, sel, ws, None, sn)
    torch.cuda.synchronize()
    assert dv.dv_check(ws) == dv.DV_OK
    return sel, sn


def test_topk_all_scores_equal_takes_lowest_indices(dv):
    """Every score ties (zero predictors): more candidates than the kernel keeps
    in shared memory, so the exact fallback path runs; the k lowest indices win."""
    cfg = dv_inputs.LayerConfig("ties", 264, 6, 64, 9000, 40, 5, 2, "f16",
                                dv_inputs.Fraction(1, 18), k_heads_fixed=4)
    case = make_case(cfg, B=2, seed=12)
    for key in ("pred_h", "pred_b"):
        case.w_host[key][:] = 0
        case.w_dev[key].zero_()
    sel, _ = _predict_only(dv, case)
    k_n, k_h = case.k_n, case.k_h
    assert np.array_equal(sel.idx_n.cpu().numpy(), np.tile(np.arange(k_n), (2, 1)))
    assert np.array_equal(sel.idx_h.cpu().numpy(), np.tile(np.arange(k_h), (2, 1)))
    u_h, u_n = sel.unions()
    assert np.array_equal(u_n.cpu().numpy(), np.arange(k_n))
    assert np.array_equal(u_h.cpu().numpy(), np.arange(k_h))


@pytest.mark.parametrize("N", [1003, 4099])
def test_topk_row_lengths_not_multiple_of_four(dv, N):
    cfg = dv_inputs.LayerConfig("oddN", 264, 6, 64, N, 40, 5, 3, "f16",
                                dv_inputs.Fraction(1, 10), k_heads_fixed=2)
    case = make_case(cfg, B=3, seed=N)
    sel, sn = _predict_only(dv, case)
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    p = oracle.predict(D, case.w_host, case.x, case.k_h, case.k_n)
    assert_close(sn.cpu().numpy(), p["s_n"], "neuron scores", 1e-4, 1e-5)
    check_topk_rows(sel.idx_n.cpu().numpy(), p["idx_n"], p["s_n"], case.k_n, "neurons")
    check_topk_rows(sel.idx_h.cpu().numpy(), p["idx_h"], p["s_h"], case.k_h, "heads")
