"""Pins of the oracle's blocked neuron selection ("DejaVu Guide: Contextual
Sparsity for LLM Inference", "Core Innovation 2", "1. Blocked Channel
Sparsity": neurons are kept in contiguous blocks of 32 or 64 channels; a
block holding highly active neurons is loaded whole).  Reading: a block is
scored by the largest score of its members; the k / block best blocks are
kept, ties to the lower block, and their neurons listed ascending."""

import numpy as np
import pytest

import dv_inputs
import oracle


def _brute_block_topk(s, block, k):
    # block maxima, then score descending / block index ascending
    m = np.asarray(s, np.float32).reshape(-1, block).max(axis=1).astype(np.float64)
    order = np.lexsort((np.arange(m.size), -m))[: k // block]
    blocks = np.sort(order)
    return (blocks[:, None] * block + np.arange(block)[None, :]).reshape(-1)


@pytest.mark.parametrize("n,block,k", [(64, 64, 64), (1024, 64, 128), (1024, 32, 96),
                                       (49152, 64, 2496), (4096, 64, 4096), (96, 32, 32)])
def test_brute_force_with_ties(n, block, k):
    rng = np.random.default_rng(n + block + k)
    s = np.round(rng.standard_normal(n) * 2).astype(np.float32) / 2  # many exact ties
    got = oracle.block_topk(s, block, k)
    assert np.array_equal(got, _brute_block_topk(s, block, k))
    assert got.size == k and np.all(np.diff(got) > 0)
    # whole, aligned blocks
    assert np.all(got.reshape(-1, block) == got.reshape(-1, block)[:, :1] +
                  np.arange(block)[None, :])
    assert np.all(got.reshape(-1, block)[:, 0] % block == 0)


@pytest.mark.parametrize("n,k", [(7, 3), (1024, 103), (5000, 250)])
def test_block_of_one_is_plain_topk(n, k):
    s = np.random.default_rng(n).standard_normal(n).astype(np.float32)
    assert np.array_equal(oracle.block_topk(s, 1, k), oracle.topk(s, k))


def test_block_with_the_largest_score_is_kept_and_a_block_of_all_ties_goes_to_the_lower():
    s = np.zeros(256, np.float32)
    s[200] = 5.0                          # block 3 holds the largest score
    s[70] = 1.0                           # block 1 next
    got = oracle.block_topk(s, 64, 128)
    assert np.array_equal(got, np.r_[np.arange(64, 128), np.arange(192, 256)])
    # every block tied at 0: the lowest blocks
    assert np.array_equal(oracle.block_topk(np.zeros(256, np.float32), 64, 128),
                          np.arange(128))


def test_counts_not_in_whole_blocks_are_rejected():
    s = np.zeros(256, np.float32)
    with pytest.raises(ValueError):
        oracle.block_topk(s, 64, 100)     # k not a multiple of the block
    with pytest.raises(ValueError):
        oracle.block_topk(np.zeros(250, np.float32), 64, 64)  # n not a multiple


def test_predict_selects_blocks_of_the_neuron_scores():
    cfg = dv_inputs.CONFIGS["tiny"].with_(neuron_block=64)   # 16 blocks of 64
    assert cfg.k_neurons == 128                              # 103 rounded up to 2 blocks
    B = 3
    D = oracle.desc_from_config(cfg)
    w = {k: v.numpy() for k, v in dv_inputs.make_weights(cfg, 5).items()}
    x = dv_inputs.make_x(cfg, B, 5).numpy()
    p = oracle.predict(D, w, x, cfg.k_heads, cfg.k_neurons)
    for b in range(B):
        assert np.array_equal(p["idx_n"][b], _brute_block_topk(p["s_n"][b], 64, cfg.k_neurons))
    assert np.array_equal(p["u_n"], np.unique(p["idx_n"]))
    # the head selection is unchanged by the neuron blocks
    p1 = oracle.predict(oracle.desc_from_config(cfg.with_(neuron_block=0)), w, x, cfg.k_heads,
                        cfg.k_neurons)
    assert np.array_equal(p["idx_h"], p1["idx_h"]) and np.array_equal(p["s_n"], p1["s_n"])


def test_selecting_every_block_equals_the_dense_layer():
    cfg = dv_inputs.CONFIGS["tiny"].with_(neuron_block=64)
    D = oracle.desc_from_config(cfg)
    w = {k: v.numpy() for k, v in dv_inputs.make_weights(cfg, 6).items()}
    kc, vc = (t.numpy() for t in dv_inputs.make_kv(cfg, 2, 6))
    x = dv_inputs.make_x(cfg, 2, 6).numpy()
    p = oracle.predict(D, w, x, cfg.n_heads, cfg.d_ffn)  # every head, every block
    assert np.array_equal(p["u_n"], np.arange(cfg.d_ffn))
    h1d, yd, _, _, _ = oracle.dense_layer(D, w, x, kc, vc, cfg.kv_len)
    h1s, ys, _, _ = oracle.layer(D, w, x, p["u_h"], p["u_n"], kc, vc, cfg.kv_len)
    assert np.array_equal(yd, ys) and np.array_equal(h1d, h1s)
