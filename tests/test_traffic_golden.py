"""The byte model reproduces the DejaVu guide's worked traffic arithmetic.

Fixture: tests/golden/page_traffic_model.json, values as printed in "DejaVu
Guide: Contextual Sparsity for LLM Inference", "Mathematical Modeling: Memory
Traffic and Speedup Bounds" (LLaMA-3-70B, A100 at 2,039 GB/s).
"""

import json
import os

from attention_dv_predict_gb300 import traffic

GOLD = os.path.join(os.path.dirname(__file__), "golden", "page_traffic_model.json")


def _close(name, got, printed):
    want, tol = printed[name]
    assert abs(got - want) <= tol + 1e-9, (name, got, want)


def test_page_traffic_model_numbers():
    g = json.load(open(GOLD))
    i, p = g["inputs"], g["printed"]
    dense = traffic.page_dense_bytes_per_layer(i["d_model"], i["d_ffn"], i["p_bytes"], i["mlp_mats"])
    sparse = traffic.page_sparse_bytes_per_layer(i["d_model"], i["d_ffn"], i["p_bytes"],
                                                 i["s_attn"], i["s_mlp"], i["mlp_mats"])
    _close("attn_mb_per_layer", dense["attn"] / 1e6, p)
    _close("mlp_mb_per_layer", dense["mlp"] / 1e6, p)
    _close("dense_mb_per_layer", dense["total"] / 1e6, p)
    _close("sparse_attn_mb_per_layer", sparse["attn"] / 1e6, p)
    _close("sparse_mlp_mb_per_layer", sparse["mlp"] / 1e6, p)
    _close("sparse_mb_per_layer", sparse["total"] / 1e6, p)
    d_tok = i["n_layers"] * dense["total"]
    s_tok = i["n_layers"] * sparse["total"]
    _close("dense_gb_per_token", d_tok / 1e9, p)
    _close("sparse_gb_per_token", s_tok / 1e9, p)
    _close("reduction", d_tok / s_tok, p)
    bw = i["b_mem_gbps"] * 1e9
    _close("t_dense_ms", traffic.decode_bound_seconds(d_tok, bw) * 1e3, p)
    _close("t_sparse_stream_ms", traffic.decode_bound_seconds(s_tok, bw) * 1e3, p)
    _close("t_dejavu_ms", traffic.decode_bound_seconds(s_tok, bw, i["t_pred_ms"] / 1e3) * 1e3, p)
    _close("t_stream_example_ms", traffic.decode_bound_seconds(i["stream_example_gb"] * 1e9, bw) * 1e3, p)


def test_opt175b_required_bytes():
    # one OPT-175B-shaped sparse layer decode at B=1: 2458 neurons, 20 heads, KV 2048
    b = traffic.sparse_step_bytes(12288, 96, 128, 49152, 1000, 2, 1, 20, 2458, 2048)
    assert b.predictor == 2 * (96 * 12288 + 1000 * 12288 + 49152 * 1000)
    assert b.qkv + b.oproj == 2 * 4 * 20 * 128 * 12288
    assert b.fc1 + b.fc2 == 2 * 2 * 2458 * 12288
    assert b.kv_read == 2 * 2 * 20 * 2049 * 128
    assert 518.9e6 < b.total < 519.0e6
    kb = traffic.kernel_bytes(12288, 96, 128, 49152, 1000, 2, 1, 20, 2458, 2048, n_parts=152)
    chain = ["pred_stage1", "pred_stage2", "qkv", "attn", "oproj", "fc1", "fc2"]
    assert abs(sum(kb[k] for k in chain) - b.total) < 0.01 * b.total
    # the one-pass MLP reads the same weights as fc1 + fc2; its second kernel
    # reads one partial of y per CTA
    assert abs(kb["mlp"] - (kb["fc1"] + kb["fc2"])) < 0.001 * kb["mlp"]
    assert kb["mlp_reduce"] == 4 * 12288 * (152 + 2) + 2 * 12288
