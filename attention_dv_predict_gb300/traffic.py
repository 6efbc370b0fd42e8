"""Memory-traffic model of a decode step (host logic, no GPU).

Two forms:

* the DejaVu guide's own model ("DejaVu Guide: Contextual Sparsity for LLM
  Inference", "Mathematical Modeling: Memory Traffic and Speedup Bounds"):
  dense bytes per layer = [4 d^2 + m d d_ffn] P with m = 3 weight matrices in
  the SwiGLU MLP the guide assumes; sparse bytes scale the attention part by
  the active-head ratio and the MLP part by the active-neuron ratio; a decode
  step is bounded below by bytes / memory bandwidth (+ predictor time);
* the bytes one sparse OPT-style layer decode must move (the roofline
  numerator): both predictors read whole, only the selected heads' QKV rows,
  out-projection rows and KV cache, only the selected neurons' fc1 rows and
  fc2 rows (m = 2 for OPT's ReLU MLP), plus biases, norms, activations and the
  new K/V written back.
"""

from __future__ import annotations

import dataclasses
from typing import Dict


def page_dense_bytes_per_layer(d_model: int, d_ffn: int, p_bytes: int, mlp_mats: int = 3) -> Dict[str, int]:
    attn = 4 * d_model * d_model * p_bytes
    mlp = mlp_mats * d_model * d_ffn * p_bytes
    return {"attn": attn, "mlp": mlp, "total": attn + mlp}


def page_sparse_bytes_per_layer(d_model: int, d_ffn: int, p_bytes: int, s_attn: float,
                                s_mlp: float, mlp_mats: int = 3) -> Dict[str, float]:
    dense = page_dense_bytes_per_layer(d_model, d_ffn, p_bytes, mlp_mats)
    attn = s_attn * dense["attn"]
    mlp = s_mlp * dense["mlp"]
    return {"attn": attn, "mlp": mlp, "total": attn + mlp}


def decode_bound_seconds(bytes_per_token: float, bandwidth_bytes_per_s: float,
                         t_pred_s: float = 0.0) -> float:
    """T_decode >= D / B_mem (+ T_pred)."""
    return bytes_per_token / bandwidth_bytes_per_s + t_pred_s


@dataclasses.dataclass
class StepBytes:
    predictor: int
    qkv: int
    oproj: int
    fc1: int
    fc2: int
    kv_read: int
    small: int

    @property
    def total(self) -> int:
        return (self.predictor + self.qkv + self.oproj + self.fc1 + self.fc2 + self.kv_read
                + self.small)

    def as_dict(self) -> Dict[str, int]:
        d = dataclasses.asdict(self)
        d["total"] = self.total
        return d


def sparse_step_bytes(d_model: int, n_heads: int, head_dim: int, d_ffn: int, pred_rank: int,
                      p_bytes: int, batch: int, n_u_heads: int, n_u_neurons: int,
                      kv_len: int, swiglu: bool = False) -> StepBytes:
    """Algorithmic bytes of one sparse layer decode over the given unions.

    KV is stored in the weight type; attention reads kv_len + 1 positions
    (the cached ones and the new one) per batch row and selected head.
    swiglu: the MLP has three matrices (gate and up in fc1's place, two rows
    and two biases per neuron).
    """
    d, H, dh, N, r, P, B = d_model, n_heads, head_dim, d_ffn, pred_rank, p_bytes, batch
    uh, un = n_u_heads, n_u_neurons
    predictor = P * (H * d + r * d + N * r)
    qkv = P * 3 * uh * dh * d
    oproj = P * uh * dh * d
    m1 = 2 if swiglu else 1
    fc1 = P * m1 * un * d
    fc2 = P * un * d
    kv_read = P * 2 * B * uh * (kv_len + 1) * dh
    biases = P * (3 * uh * dh + m1 * un + 2 * d)
    norms = P * 4 * d
    acts = 4 * B * d * 2          # x in, y out (float32)
    kv_write = P * 2 * B * uh * dh
    return StepBytes(predictor, qkv, oproj, fc1, fc2, kv_read, biases + norms + acts + kv_write)


def dense_step_bytes(d_model: int, n_heads: int, head_dim: int, d_ffn: int, p_bytes: int,
                     batch: int, kv_len: int, swiglu: bool = False) -> int:
    """Bytes of the same layer decoded densely (no predictor, every head and neuron)."""
    b = sparse_step_bytes(d_model, n_heads, head_dim, d_ffn, 0, p_bytes, batch, n_heads, d_ffn,
                          kv_len, swiglu)
    return b.total - b.predictor


def kernel_bytes(d_model: int, n_heads: int, head_dim: int, d_ffn: int, pred_rank: int,
                 p_bytes: int, batch: int, n_u_heads: int, n_u_neurons: int,
                 kv_len: int, n_parts: int = 0) -> Dict[str, int]:
    """Algorithmic bytes per launch of each kernel of the layer decode.

    "mlp" is the one-pass MLP kernel (fc1 and fc2 together); "mlp_reduce"
    the kernel that adds its n_parts per-CTA partials of y (the partials are
    read once, h1 read, y written)."""
    d, H, dh, N, r, P, B = d_model, n_heads, head_dim, d_ffn, pred_rank, p_bytes, batch
    uh, un = n_u_heads, n_u_neurons
    fc1 = P * un * (d + 1) + P * 2 * d + 4 * B * (d + un)
    fc2 = P * un * d + P * d + 4 * B * (2 * d + un)
    pred2 = P * N * r + 4 * B * r + 4 * B * N
    qkv = (P * 3 * uh * dh * (d + 1) + P * 2 * d + 4 * B * d + 4 * B * uh * dh
           + P * 2 * B * uh * dh)
    return {
        "mlp": P * un * (2 * d + 1) + P * 3 * d + 4 * B * 2 * d,
        "mlp_reduce": 4 * B * d * (n_parts + 2) + P * d,
        "pred_stage1": P * (H + r) * d + 4 * B * d + 4 * B * (H + r),
        "pred_stage2": pred2,
        "qkv": qkv,
        "attn": P * 2 * B * uh * (kv_len + 1) * dh + 4 * 2 * B * uh * dh,
        "oproj": P * uh * dh * d + P * d + 4 * B * (2 * d + uh * dh),
        "fc1": fc1,
        "fc2": fc2,
    }
