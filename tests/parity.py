"""Helpers for the GPU-vs-oracle parity tests.

The CUDA path runs through the C ABI (attention_dv_predict_gb300.dv); the
expected values come from the CPU oracle run on the same seeded inputs.

Acceptance (the method's stated bar for binary16 weights with binary32
accumulation):
* selected index sets equal the oracle's, except entries whose oracle score
  lies within 1e-3 * max(|s_k|, 1e-6) of the oracle's k-th score s_k
  (compared per row, before the union);
* outputs, compared with the oracle run on the validated GPU index set:
  max-abs error <= 2e-2 and relative L2 error <= 1e-3, on y and on the
  residual-free deltas (h1 - x and y - h1), which the N(0, 1) residual would
  otherwise mask.
"""

from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np
import torch

import dv_inputs
import oracle

MAX_ABS = 2e-2
REL_L2 = 1e-3
TIE_REL = 1e-3


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def assert_close(got, want, what, max_abs=MAX_ABS, rel=REL_L2):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    ma = float(np.max(np.abs(got - want))) if got.size else 0.0
    rl = rel_l2(got, want)
    assert ma <= max_abs and rl <= rel, f"{what}: max-abs {ma:.3e} rel-L2 {rl:.3e}"
    return ma, rl


def check_topk_rows(gpu_idx, ora_idx, ora_scores, k, what):
    """Per row: sorted, unique, k entries; differences only inside the tie band."""
    gpu_idx = np.asarray(gpu_idx)
    n_diff = 0
    for b in range(gpu_idx.shape[0]):
        g = gpu_idx[b]
        assert g.size == k and np.all(np.diff(g) > 0), f"{what} row {b}: not sorted/unique"
        s = np.asarray(ora_scores[b], np.float64)
        assert g.min() >= 0 and g.max() < s.size
        sk = np.sort(s)[::-1][k - 1]
        band = TIE_REL * max(abs(sk), 1e-6)
        diff = np.setxor1d(g, ora_idx[b])
        n_diff += diff.size
        bad = diff[np.abs(s[diff] - sk) > band]
        assert bad.size == 0, f"{what} row {b}: {bad.size} selections outside the tie band"
    return n_diff


def check_block_rows(gpu_idx, ora_idx, ora_scores, block, k, what):
    """Blocked selection, per row: k entries forming whole aligned blocks,
    sorted; blocks differing from the oracle's only inside the tie band of
    the block scores (each block's largest member score)."""
    gpu_idx = np.asarray(gpu_idx)
    n_diff = 0
    for b in range(gpu_idx.shape[0]):
        g = gpu_idx[b]
        assert g.size == k and np.all(np.diff(g) > 0), f"{what} row {b}: not sorted/unique"
        gb = g.reshape(-1, block)
        assert np.all(gb[:, 0] % block == 0) and np.all(gb == gb[:, :1] + np.arange(block)), \
            f"{what} row {b}: not whole blocks"
        bs = np.asarray(ora_scores[b], np.float64).reshape(-1, block).max(axis=1)
        kb = k // block
        sk = np.sort(bs)[::-1][kb - 1]
        band = TIE_REL * max(abs(sk), 1e-6)
        diff = np.setxor1d(gb[:, 0] // block, np.asarray(ora_idx[b]).reshape(-1, block)[:, 0] // block)
        n_diff += diff.size
        bad = diff[np.abs(bs[diff] - sk) > band]
        assert bad.size == 0, f"{what} row {b}: {bad.size} blocks outside the tie band"
    return n_diff


@dataclasses.dataclass
class Case:
    cfg: dv_inputs.LayerConfig
    B: int
    k_h: int
    k_n: int
    kv_len: int
    kv_cap: int
    w_host: Dict[str, np.ndarray]
    w_dev: Dict[str, torch.Tensor]
    x: np.ndarray
    x_pred: Optional[np.ndarray]
    kc: np.ndarray
    vc: np.ndarray


def make_case(cfg, B=None, k_h=None, k_n=None, kv_len=None, seed=0, gen_device="cpu",
              norm_affine=True, separate_x_pred=False, kv_cap=None) -> Case:
    """Seeded inputs, generated on `gen_device` (torch RNG), kept on host and device."""
    B = cfg.batch if B is None else B
    kv_len = cfg.kv_len if kv_len is None else kv_len
    cap = kv_len + 1 if kv_cap is None else kv_cap
    c2 = cfg.with_(kv_len=kv_len)
    w = dv_inputs.make_weights(c2, seed, gen_device, norm_affine=norm_affine)
    kc, vc = dv_inputs.make_kv(c2, B, seed, gen_device, kv_cap=cap)
    x = dv_inputs.make_x(c2, B, seed, gen_device)
    xp = dv_inputs.make_x(c2, B, seed, gen_device, family="x_pred") if separate_x_pred else None
    w_dev = {n: t.cuda() for n, t in w.items()}
    w_host = {n: t.cpu().numpy() for n, t in w.items()}
    return Case(c2, B, cfg.k_heads if k_h is None else k_h, cfg.k_neurons if k_n is None else k_n,
                kv_len, cap, w_host, w_dev, x.cpu().numpy(), None if xp is None else xp.cpu().numpy(),
                kc.cpu().numpy(), vc.cpu().numpy())


def run_gpu_layer(dv, case: Case, stream=None, entry="dv_layer_decode"):
    """`entry` (dv_layer_decode or dv_layer_decode_persistent) on the case;
    returns host copies of everything."""
    desc = dv.desc_from_config(case.cfg, case.kv_cap)
    layer = dv.Layer(desc, case.w_dev)
    sel = dv.SelectionBuffers(desc, case.B, case.k_h, case.k_n)
    ws = dv.Workspace(desc, case.B)
    x = torch.from_numpy(case.x).cuda()
    xp = None if case.x_pred is None else torch.from_numpy(case.x_pred).cuda()
    kc = torch.from_numpy(case.kc).cuda()
    vc = torch.from_numpy(case.vc).cuda()
    y = torch.empty_like(x)
    h1 = torch.empty_like(x)
    getattr(dv, entry)(layer, x, case.k_h, case.k_n, kc, vc, case.kv_len, sel, y, ws, x_pred=xp,
                       h1=h1, stream=stream)
    torch.cuda.synchronize()
    assert dv.dv_check(ws) == dv.DV_OK
    u_h, u_n = sel.unions()
    return {
        "y": y.cpu().numpy(), "h1": h1.cpu().numpy(), "idx_h": sel.idx_h.cpu().numpy(),
        "idx_n": sel.idx_n.cpu().numpy(), "u_h": u_h.cpu().numpy(), "u_n": u_n.cpu().numpy(),
        "kc": kc.cpu().numpy(), "vc": vc.cpu().numpy(),
    }


def check_layer_parity(case: Case, g, tight: bool = False):
    """Compare a GPU layer decode with the oracle; returns a summary dict."""
    D = oracle.desc_from_config(case.cfg, case.kv_cap)
    xp = case.x if case.x_pred is None else case.x_pred
    p = oracle.predict(D, case.w_host, xp, case.k_h, case.k_n)
    nd_h = check_topk_rows(g["idx_h"], p["idx_h"], p["s_h"], case.k_h, "heads")
    blk = getattr(case.cfg, "neuron_block", 0)
    if blk > 1:
        nd_n = check_block_rows(g["idx_n"], p["idx_n"], p["s_n"], blk, case.k_n, "neuron blocks")
    else:
        nd_n = check_topk_rows(g["idx_n"], p["idx_n"], p["s_n"], case.k_n, "neurons")
    assert np.array_equal(g["u_h"], np.unique(g["idx_h"]))
    assert np.array_equal(g["u_n"], np.unique(g["idx_n"]))
    # the oracle layer on the (validated) GPU index set
    h1, y, kc, vc = oracle.layer(D, case.w_host, case.x, g["u_h"], g["u_n"], case.kc, case.vc,
                                 case.kv_len)
    mab, rl = (1e-4, 1e-5) if tight else (MAX_ABS, REL_L2)
    out = {"diff_heads": nd_h, "diff_neurons": nd_n}
    out["y"] = assert_close(g["y"], y, "y", mab, rl)
    out["attn_delta"] = assert_close(g["h1"] - case.x, h1 - case.x.astype(np.float64),
                                     "h1 - x", mab, rl)
    out["mlp_delta"] = assert_close(g["y"] - g["h1"], y - h1, "y - h1", mab, rl)
    # KV: selected heads' slot kv_len matches the oracle's rounded values;
    # every other entry is untouched.  An entry is the storage rounding of a
    # length-d binary32 dot product w . xn, whose accumulation error is of
    # order sqrt(d) * 2^-24 * ||w||_2 * max|xn| (taken four times); beyond
    # that the two sides may differ by one storage ulp.
    L = case.kv_len
    sel_h = g["u_h"]
    d = case.cfg.d_model
    wq = case.w_host["w_qkv"]  # [3, H, dh, d]
    xn_max = np.array([np.abs(oracle.norm_row(D, case.x[b], case.w_host["ln1_g"],
                                              case.w_host["ln1_b"])).max() for b in range(case.B)])
    ulp_rel = 2.0 ** -10 if g["kc"].dtype == np.float16 else 2.0 ** -23
    for t, name, gc, oc, ic in ((1, "k", g["kc"], kc, case.kc), (2, "v", g["vc"], vc, case.vc)):
        gs = gc[:, sel_h, L].astype(np.float64)
        os_ = oc[:, sel_h, L].astype(np.float64)
        wnorm = np.stack([np.linalg.norm(wq[t, h].astype(np.float32), axis=-1)
                          for h in sel_h]).astype(np.float64)  # [|U_h|, dh]
        acc = 4.0 * np.sqrt(d) * 2.0 ** -24 * wnorm[None] * xn_max[:, None, None]
        tol = np.maximum(np.abs(os_), np.abs(gs)) * ulp_rel + acc + 1e-30
        bad = np.abs(gs - os_) > tol
        assert not bad.any(), (f"{name} cache slot mismatch at {np.argwhere(bad)[:4].tolist()}: "
                               f"{gs[bad][:4]} vs {os_[bad][:4]} (tol {tol[bad][:4]})")
        mask = np.ones(gc.shape, bool)
        mask[:, sel_h, L] = False
        assert np.array_equal(gc[mask], ic[mask]), f"{name} cache changed outside the new slot"
    return out
