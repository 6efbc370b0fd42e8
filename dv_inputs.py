"""Seeded synthetic inputs for the contextually sparse (DejaVu) layer decode.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It draws random numbers and lays out tensors; it holds none of
the method's arithmetic (no norm, no projection, no selection).

Workload shapes follow the OPT family the DejaVu pages measure ("Deja Vu: How
Contextual Sparsity Accelerates LLM Inference by 6x", "What Is Contextual
Sparsity?": 96 heads and 49,152 neurons per OPT-175B layer; "DejaVu Guide:
Contextual Sparsity for LLM Inference", "Production Benchmarks": OPT-66B,
OPT-175B).  No trained weights exist here, so every tensor is random:

* every weight matrix and bias ~ N(0, 0.02), cast to the weight dtype
  (round-to-nearest);
* norm gain = 1 and bias = 0, unless ``norm_affine`` asks for gain
  1 + N(0, 0.1) and bias N(0, 0.1) (tests use that to exercise both);
* activations x (and a separate x_pred when asked) ~ N(0, 1), float32;
* KV caches ~ N(0, 1) cast to the KV dtype (= weight dtype);
* OPT-6.7B shape: the fc1 bias is shifted by -0.5 so that a large share of
  ReLU outputs are zero;
* OPT-175B shape: neuron predictor rows are Zipf-skewed: row j of the
  second low-rank factor is scaled by 1 / (1 + pi(j)), pi a random
  permutation of 0..N-1 drawn from seed 0 (exponent 1).

Draw order is fixed: each tensor family has its own generator seeded from
(seed, family), so changing the batch does not change the weights.
"""

from __future__ import annotations

import dataclasses
import math
from fractions import Fraction
from typing import Dict, Optional

import torch

# Tensor families -> generator sub-seed.
_FAMILY = {"weights": 1, "kv": 2, "x": 3, "x_pred": 4, "zipf": 5}

# Order in which the layer's weight tensors are drawn (one weights generator).
WEIGHT_ORDER = (
    "ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_oT", "b_o", "ln2_g", "ln2_b",
    "w1", "b1", "w2T", "b2", "pred_h", "pred_a", "pred_b",
)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape of one decoder layer plus the per-step keep fractions."""

    name: str
    d_model: int
    n_heads: int
    head_dim: int
    d_ffn: int
    pred_rank: int
    kv_len: int
    batch: int
    dtype: str  # "f32" or "f16" (weights, biases, norms and KV cache)
    frac_neurons: Fraction
    frac_heads: Optional[Fraction] = None  # None -> k_heads_fixed
    k_heads_fixed: Optional[int] = None
    fc1_bias_shift: float = 0.0
    zipf_exponent: float = 0.0
    norm: str = "layernorm"
    ln_eps: float = 1e-5
    neuron_block: int = 0  # 0: neurons selected one by one; > 1: contiguous blocks
    mlp: str = "relu"      # "relu" (fc1, ReLU, fc2) or "swiglu" (gate, up, down)

    @property
    def k_neurons(self) -> int:
        # blocked selection keeps whole blocks: the count rounded up to one
        k = keep_count(self.frac_neurons, self.d_ffn)
        if self.neuron_block > 1:
            k = -(-k // self.neuron_block) * self.neuron_block
        return k

    @property
    def k_heads(self) -> int:
        if self.k_heads_fixed is not None:
            return self.k_heads_fixed
        return keep_count(self.frac_heads, self.n_heads)

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


def keep_count(frac: Fraction, count: int) -> int:
    """k = ceil(frac * count), in exact rational arithmetic."""
    v = Fraction(frac) * count
    return max(1, math.ceil(v))


CONFIGS: Dict[str, LayerConfig] = {
    # tiny OPT-style layer, fp32, top-k 10% neurons / 2 heads
    "tiny": LayerConfig("tiny", 256, 8, 32, 1024, 32, 64, 1, "f32",
                        Fraction(1, 10), k_heads_fixed=2),
    # OPT-6.7B shape, keep 10% neurons / 25% heads, fc1 bias shifted -0.5
    "opt6.7b": LayerConfig("opt6.7b", 4096, 32, 128, 16384, 512, 512, 1, "f16",
                           Fraction(1, 10), Fraction(1, 4), fc1_bias_shift=-0.5),
    # OPT-66B shape, keep 5% neurons / 20% heads (batch 1 and 8)
    "opt66b": LayerConfig("opt66b", 9216, 72, 128, 36864, 1000, 1024, 1, "f16",
                          Fraction(1, 20), Fraction(1, 5)),
    # OPT-175B shape, keep 5% neurons (2458) / 20 heads, Zipf-skewed scores
    "opt175b": LayerConfig("opt175b", 12288, 96, 128, 49152, 1000, 2048, 1, "f16",
                           Fraction(1, 20), Fraction(1, 5), zipf_exponent=1.0),
    # LLaMA-style layers (RMSNorm, SwiGLU MLP): a tiny one, and the LLaMA-3-70B
    # shape the guide's traffic arithmetic uses (d 8192, d_ffn 28672, keep 25%
    # of the neurons and 20% of the heads; all 64 heads full width, the
    # grouped KV heads of the real model not modelled)
    "llama_tiny": LayerConfig("llama_tiny", 256, 8, 32, 704, 32, 64, 1, "f32",
                              Fraction(1, 4), k_heads_fixed=2, norm="rmsnorm", mlp="swiglu"),
    "llama3_70b": LayerConfig("llama3_70b", 8192, 64, 128, 28672, 1024, 2048, 1, "f16",
                              Fraction(1, 4), Fraction(1, 5), norm="rmsnorm", mlp="swiglu"),
    # the OPT-175B shape with neurons kept in blocks of 64 contiguous channels
    # (5% of 768 blocks, rounded up: 39 blocks = 2496 neurons)
    "opt175b_blk64": LayerConfig("opt175b_blk64", 12288, 96, 128, 49152, 1000, 2048, 1,
                                 "f16", Fraction(1, 20), Fraction(1, 5), zipf_exponent=1.0,
                                 neuron_block=64),
}

# The 24-layer OPT-175B-shaped stack reuses the opt175b layer shape.
STACK_LAYERS = 24


def _gen(seed: int, family: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1000 + _FAMILY[family])
    return g


def _torch_dtype(name: str):
    return {"f32": torch.float32, "f16": torch.float16}[name]


def _normal(shape, std, g, device, dtype):
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def zipf_row_scale(n: int, exponent: float) -> torch.Tensor:
    """g_j = (1 + pi(j))^-exponent with pi a seed-0 random permutation (CPU)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(_FAMILY["zipf"])
    perm = torch.randperm(n, generator=g)
    return (1.0 + perm.to(torch.float64)) ** (-float(exponent))


def make_weights(cfg: LayerConfig, seed: int = 0, device="cpu",
                 norm_affine: bool = False) -> Dict[str, torch.Tensor]:
    """Random-init weights of one layer, laid out as the C ABI expects.

    Layouts (row-major): w_qkv [3, H, dh, d]; b_qkv [3, H, dh];
    w_oT [H, dh, d] (out-projection, transposed so a head's columns are
    contiguous rows); w1 [N, d]; w2T [N, d] (fc2 transposed); pred_h [H, d];
    pred_a [r, d]; pred_b [N, r]; norms and biases 1-D.  SwiGLU layers
    (cfg.mlp == "swiglu"): w1 [N, 2, d] (neuron j's gate and up rows side by
    side), b1 [N, 2]; w2T is the down projection, transposed.
    """
    d, H, dh, N, r = cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn, cfg.pred_rank
    dt = _torch_dtype(cfg.dtype)
    g = _gen(seed, "weights", device)
    shapes = {
        "ln1_g": (d,), "ln1_b": (d,), "w_qkv": (3, H, dh, d), "b_qkv": (3, H, dh),
        "w_oT": (H, dh, d), "b_o": (d,), "ln2_g": (d,), "ln2_b": (d,),
        "w1": (N, 2, d) if cfg.mlp == "swiglu" else (N, d),
        "b1": (N, 2) if cfg.mlp == "swiglu" else (N,), "w2T": (N, d), "b2": (d,),
        "pred_h": (H, d), "pred_a": (r, d), "pred_b": (N, r),
    }
    out: Dict[str, torch.Tensor] = {}
    for name in WEIGHT_ORDER:
        shape = shapes[name]
        if name in ("ln1_g", "ln2_g"):
            if norm_affine:
                t = torch.randn(shape, generator=g, device=device).mul_(0.1).add_(1.0)
            else:
                t = torch.ones(shape, device=device)
            out[name] = t.to(dt)
        elif name in ("ln1_b", "ln2_b"):
            if norm_affine:
                t = torch.randn(shape, generator=g, device=device).mul_(0.1)
            else:
                t = torch.zeros(shape, device=device)
            out[name] = t.to(dt)
        elif name == "b1" and cfg.fc1_bias_shift != 0.0:
            t = torch.randn(shape, generator=g, device=device).mul_(0.02)
            out[name] = t.add_(cfg.fc1_bias_shift).to(dt)
        elif name == "pred_b" and cfg.zipf_exponent != 0.0:
            t = torch.randn(shape, generator=g, device=device).mul_(0.02)
            scale = zipf_row_scale(N, cfg.zipf_exponent).to(device=device, dtype=torch.float32)
            out[name] = t.mul_(scale[:, None]).to(dt)
        else:
            out[name] = _normal(shape, 0.02, g, device, dt)
    return out


def make_kv(cfg: LayerConfig, batch: int, seed: int = 0, device="cpu",
            kv_cap: Optional[int] = None):
    """KV caches [B, H, kv_cap, dh] ~ N(0, 1); positions >= kv_len are also filled."""
    cap = cfg.kv_len + 1 if kv_cap is None else kv_cap
    dt = _torch_dtype(cfg.dtype)
    g = _gen(seed, "kv", device)
    shape = (batch, cfg.n_heads, cap, cfg.head_dim)
    k = _normal(shape, 1.0, g, device, dt)
    v = _normal(shape, 1.0, g, device, dt)
    return k, v


def make_x(cfg: LayerConfig, batch: int, seed: int = 0, device="cpu",
           family: str = "x") -> torch.Tensor:
    """Layer input (or predictor input) rows ~ N(0, 1), float32 [B, d]."""
    g = _gen(seed, family, device)
    return torch.randn((batch, cfg.d_model), generator=g, device=device, dtype=torch.float32)
