"""ctypes front end of the CPU oracle (``dv_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it.  It never imports the CUDA package and the
CUDA package never imports it; both take their inputs from ``dv_inputs``.

Arrays are numpy.  Weight tensors are passed in their storage type
(float32, or float16 whose bits the C code decodes exactly).  Every function
returns fresh output arrays; KV caches are copied before the oracle appends to
them unless ``inplace=True``.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional

import numpy as np

from . import build as _build

_P = C.c_void_p
_I32P = C.POINTER(C.c_int32)
_F32P = C.POINTER(C.c_float)
_F64P = C.POINTER(C.c_double)

WEIGHT_FIELDS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_oT", "b_o", "ln2_g", "ln2_b",
                 "w1", "b1", "w2T", "b2", "pred_h", "pred_a", "pred_b")


class Desc(C.Structure):
    _fields_ = [("d_model", C.c_int), ("n_heads", C.c_int), ("head_dim", C.c_int),
                ("d_ffn", C.c_int), ("pred_rank", C.c_int), ("dtype", C.c_int),
                ("norm", C.c_int), ("eps", C.c_double), ("kv_cap", C.c_int),
                ("neuron_block", C.c_int), ("mlp", C.c_int)]


class Weights(C.Structure):
    _fields_ = [(n, _P) for n in WEIGHT_FIELDS]


_lib = None
_lib_omp = None


def _load(path: str):
    L = C.CDLL(path)
    L.dvo_half_to_double.argtypes = [C.c_uint16]
    L.dvo_half_to_double.restype = C.c_double
    L.dvo_double_to_half.argtypes = [C.c_double]
    L.dvo_double_to_half.restype = C.c_uint16
    L.dvo_norm_row.argtypes = [C.POINTER(Desc), _F64P, _P, _P, _F64P]
    L.dvo_norm_row.restype = None
    L.dvo_topk.argtypes = [_F32P, C.c_int, C.c_int, _I32P]
    L.dvo_block_topk.argtypes = [_F32P, C.c_int, C.c_int, C.c_int, _I32P]
    L.dvo_union.argtypes = [_I32P, C.c_int, C.c_int, C.c_int, _I32P, _I32P]
    L.dvo_predict.argtypes = [C.POINTER(Desc), C.POINTER(Weights), _F32P, C.c_int, C.c_int,
                              C.c_int, _F32P, _F32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P]
    L.dvo_sparse_attn.argtypes = [C.POINTER(Desc), C.POINTER(Weights), _F32P, C.c_int, _I32P,
                                  C.c_int, _P, _P, C.c_int, _F64P, _F64P]
    L.dvo_sparse_mlp.argtypes = [C.POINTER(Desc), C.POINTER(Weights), _F64P, C.c_int, _I32P,
                                 C.c_int, _F64P, _F64P]
    L.dvo_layer.argtypes = [C.POINTER(Desc), C.POINTER(Weights), _F32P, C.c_int, _I32P, C.c_int,
                            _I32P, C.c_int, _P, _P, C.c_int, _F64P, _F64P]
    L.dvo_dense_layer.argtypes = [C.POINTER(Desc), C.POINTER(Weights), _F32P, C.c_int, _P, _P,
                                  C.c_int, _F64P, _F64P, _F64P]
    L.dvo_layer_decode.argtypes = [C.POINTER(Desc), C.POINTER(Weights), _F32P, _F32P, C.c_int,
                                   C.c_int, C.c_int, _P, _P, C.c_int, _F32P, _F32P, _I32P,
                                   _I32P, _I32P, _I32P, _I32P, _I32P, _F64P, _F64P]
    L.dvo_set_threads.argtypes = [C.c_int]
    L.dvo_set_threads.restype = C.c_int
    for f in ("dvo_topk", "dvo_block_topk", "dvo_union", "dvo_predict", "dvo_sparse_attn", "dvo_sparse_mlp",
              "dvo_layer", "dvo_dense_layer", "dvo_layer_decode"):
        getattr(L, f).restype = C.c_int
    return L


def lib(threads: int = 0):
    """The oracle library.  threads == 0: the plain single-threaded build;
    threads > 0 (or -1 for every host core): the OpenMP build, set to that
    many threads (same results bit for bit)."""
    global _lib, _lib_omp
    if threads == 0:
        if _lib is None:
            _lib = _load(_build.build())
        return _lib
    if _lib_omp is None:
        _build.build()
        path = _build.build_omp()
        if path is None:
            raise RuntimeError("the OpenMP build of the oracle is unavailable on this host")
        _lib_omp = _load(path)
    _lib_omp.dvo_set_threads(int(threads))
    return _lib_omp


def threads_used(threads: int) -> int:
    """Threads the library chosen by ``threads`` runs its loops on."""
    return 1 if threads == 0 else lib(threads).dvo_set_threads(int(threads))


def _ptr(a: np.ndarray, ctype=None):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    p = a.ctypes.data_as(C.c_void_p)
    return C.cast(p, ctype) if ctype is not None else p


def _storage_dtype(dtype: int):
    return np.float32 if dtype == 0 else np.float16


def make_desc(d_model, n_heads, head_dim, d_ffn, pred_rank, dtype, kv_cap,
              norm: int = 0, eps: float = 1e-5, neuron_block: int = 0, mlp: int = 0) -> Desc:
    """dtype: 0 binary32 storage, 1 binary16 storage; norm: 0 LayerNorm, 1 RMSNorm;
    neuron_block: 0/1 neurons one by one, > 1 blocks of that many; mlp: 0 ReLU
    fc1/fc2, 1 SwiGLU."""
    return Desc(d_model, n_heads, head_dim, d_ffn, pred_rank, dtype, norm, eps, kv_cap,
                neuron_block, mlp)


def desc_from_config(cfg, kv_cap: Optional[int] = None) -> Desc:
    """Desc from a ``dv_inputs.LayerConfig`` (read by attribute)."""
    cap = cfg.kv_len + 1 if kv_cap is None else kv_cap
    return make_desc(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn, cfg.pred_rank,
                     0 if cfg.dtype == "f32" else 1, cap,
                     0 if cfg.norm == "layernorm" else 1, cfg.ln_eps,
                     getattr(cfg, "neuron_block", 0), 1 if getattr(cfg, "mlp", "relu") == "swiglu" else 0)


class _W:
    """Keeps the numpy arrays alive while C holds their pointers."""

    def __init__(self, D: Desc, w: Dict[str, np.ndarray]):
        st = _storage_dtype(D.dtype)
        self.arrays = {}
        for n in WEIGHT_FIELDS:
            a = np.ascontiguousarray(w[n])
            if a.dtype != st:
                raise TypeError(f"weight {n} has dtype {a.dtype}, expected {st}")
            self.arrays[n] = a
        self.s = Weights(*[_ptr(self.arrays[n]) for n in WEIGHT_FIELDS])


def _rc(rc, what):
    if rc != 0:
        raise ValueError(f"{what} returned {rc}")


def half_to_double(bits: int) -> float:
    return lib().dvo_half_to_double(int(bits))


def double_to_half(x: float) -> int:
    return int(lib().dvo_double_to_half(float(x)))


def norm_row(D: Desc, x: np.ndarray, g: np.ndarray, b: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(g)
    b = np.ascontiguousarray(b)
    out = np.empty(D.d_model, np.float64)
    lib().dvo_norm_row(C.byref(D), _ptr(x, _F64P), _ptr(g), _ptr(b), _ptr(out, _F64P))
    return out


def topk(scores: np.ndarray, k: int) -> np.ndarray:
    s = np.ascontiguousarray(scores, dtype=np.float32)
    out = np.empty(k, np.int32)
    _rc(lib().dvo_topk(_ptr(s, _F32P), s.size, k, _ptr(out, _I32P)), "dvo_topk")
    return out


def block_topk(scores: np.ndarray, block: int, k: int) -> np.ndarray:
    """The neurons of the k / block best blocks (block score: the largest member score)."""
    s = np.ascontiguousarray(scores, dtype=np.float32)
    out = np.empty(k, np.int32)
    _rc(lib().dvo_block_topk(_ptr(s, _F32P), s.size, block, k, _ptr(out, _I32P)),
        "dvo_block_topk")
    return out


def union(idx: np.ndarray, n: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    B, k = idx.shape
    out = np.empty(max(1, B * k), np.int32)
    cnt = np.zeros(1, np.int32)
    _rc(lib().dvo_union(_ptr(idx, _I32P), B, k, n, _ptr(out, _I32P), _ptr(cnt, _I32P)),
        "dvo_union")
    return out[: int(cnt[0])].copy()


def predict(D: Desc, w: Dict[str, np.ndarray], x_pred: np.ndarray, k_h: int, k_n: int,
            threads: int = 0):
    """Scores (binary32), per-row top-k and unions.  Returns a dict."""
    W = _W(D, w)
    x = np.ascontiguousarray(x_pred, dtype=np.float32)
    B = x.shape[0]
    H, N = D.n_heads, D.d_ffn
    s_h = np.empty((B, H), np.float32)
    s_n = np.empty((B, N), np.float32)
    idx_h = np.empty((B, k_h), np.int32)
    idx_n = np.empty((B, k_n), np.int32)
    u_h = np.empty(H, np.int32)
    u_n = np.empty(N, np.int32)
    nuh = np.zeros(1, np.int32)
    nun = np.zeros(1, np.int32)
    _rc(lib(threads).dvo_predict(C.byref(D), C.byref(W.s), _ptr(x, _F32P), B, k_h, k_n,
                          _ptr(s_h, _F32P), _ptr(s_n, _F32P), _ptr(idx_h, _I32P),
                          _ptr(idx_n, _I32P), _ptr(u_h, _I32P), _ptr(nuh, _I32P),
                          _ptr(u_n, _I32P), _ptr(nun, _I32P)), "dvo_predict")
    return {"s_h": s_h, "s_n": s_n, "idx_h": idx_h, "idx_n": idx_n,
            "u_h": u_h[: int(nuh[0])].copy(), "u_n": u_n[: int(nun[0])].copy()}


def _caches(D, k_cache, v_cache, inplace):
    st = _storage_dtype(D.dtype)
    if inplace:
        assert k_cache.dtype == st and v_cache.dtype == st
        assert k_cache.flags["C_CONTIGUOUS"] and v_cache.flags["C_CONTIGUOUS"]
        return k_cache, v_cache
    return (np.ascontiguousarray(k_cache, dtype=st).copy(),
            np.ascontiguousarray(v_cache, dtype=st).copy())


def sparse_attn(D: Desc, w, x, u_h, k_cache, v_cache, kv_len, inplace=False):
    """h1 (binary64 [B, d]), o ([B, |u_h|, dh]) and the appended caches."""
    W = _W(D, w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    B = x.shape[0]
    u = np.ascontiguousarray(u_h, dtype=np.int32)
    kc, vc = _caches(D, k_cache, v_cache, inplace)
    h1 = np.empty((B, D.d_model), np.float64)
    o = np.empty((B, max(1, u.size), D.head_dim), np.float64)
    _rc(lib().dvo_sparse_attn(C.byref(D), C.byref(W.s), _ptr(x, _F32P), B, _ptr(u, _I32P), u.size,
                              _ptr(kc), _ptr(vc), kv_len, _ptr(h1, _F64P), _ptr(o, _F64P)),
        "dvo_sparse_attn")
    return h1, o[:, : u.size], kc, vc


def sparse_mlp(D: Desc, w, h1, u_n):
    """y (binary64 [B, d]) and fc1 pre-activations ([B, |u_n|])."""
    W = _W(D, w)
    h = np.ascontiguousarray(h1, dtype=np.float64)
    B = h.shape[0]
    u = np.ascontiguousarray(u_n, dtype=np.int32)
    y = np.empty((B, D.d_model), np.float64)
    pre = np.empty((B, max(1, u.size)), np.float64)
    _rc(lib().dvo_sparse_mlp(C.byref(D), C.byref(W.s), _ptr(h, _F64P), B, _ptr(u, _I32P), u.size,
                             _ptr(y, _F64P), _ptr(pre, _F64P)), "dvo_sparse_mlp")
    return y, pre[:, : u.size]


def layer(D: Desc, w, x, u_h, u_n, k_cache, v_cache, kv_len, inplace=False, threads: int = 0):
    """Sparse layer on the given unions: (h1, y, k_cache, v_cache)."""
    W = _W(D, w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    B = x.shape[0]
    uh = np.ascontiguousarray(u_h, dtype=np.int32)
    un = np.ascontiguousarray(u_n, dtype=np.int32)
    kc, vc = _caches(D, k_cache, v_cache, inplace)
    h1 = np.empty((B, D.d_model), np.float64)
    y = np.empty((B, D.d_model), np.float64)
    _rc(lib(threads).dvo_layer(C.byref(D), C.byref(W.s), _ptr(x, _F32P), B, _ptr(uh, _I32P), uh.size,
                        _ptr(un, _I32P), un.size, _ptr(kc), _ptr(vc), kv_len, _ptr(h1, _F64P),
                        _ptr(y, _F64P)), "dvo_layer")
    return h1, y, kc, vc


def dense_layer(D: Desc, w, x, k_cache, v_cache, kv_len, inplace=False):
    """Dense layer: (h1, y, fc1 pre-activations [B, N], k_cache, v_cache)."""
    W = _W(D, w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    B = x.shape[0]
    kc, vc = _caches(D, k_cache, v_cache, inplace)
    h1 = np.empty((B, D.d_model), np.float64)
    y = np.empty((B, D.d_model), np.float64)
    pre = np.empty((B, D.d_ffn), np.float64)
    _rc(lib().dvo_dense_layer(C.byref(D), C.byref(W.s), _ptr(x, _F32P), B, _ptr(kc), _ptr(vc),
                              kv_len, _ptr(h1, _F64P), _ptr(y, _F64P), _ptr(pre, _F64P)),
        "dvo_dense_layer")
    return h1, y, pre, kc, vc


def layer_decode(D: Desc, w, x, k_h, k_n, k_cache, v_cache, kv_len, x_pred=None, inplace=False,
                 threads: int = 0):
    """The whole decode step (``dvo_layer_decode``): predict from x_pred
    (x when None), then the sparse layer on x over the predicted unions.
    Returns the dict of ``predict`` plus h1, y and the appended caches."""
    W = _W(D, w)
    x = np.ascontiguousarray(x, dtype=np.float32)
    B = x.shape[0]
    xp = None if x_pred is None else np.ascontiguousarray(x_pred, dtype=np.float32)
    if xp is not None and xp.shape != x.shape:
        raise ValueError("x_pred must have the shape of x")
    H, N = D.n_heads, D.d_ffn
    kc, vc = _caches(D, k_cache, v_cache, inplace)
    s_h = np.empty((B, H), np.float32)
    s_n = np.empty((B, N), np.float32)
    idx_h = np.empty((B, k_h), np.int32)
    idx_n = np.empty((B, k_n), np.int32)
    u_h = np.empty(H, np.int32)
    u_n = np.empty(N, np.int32)
    nuh = np.zeros(1, np.int32)
    nun = np.zeros(1, np.int32)
    h1 = np.empty((B, D.d_model), np.float64)
    y = np.empty((B, D.d_model), np.float64)
    _rc(lib(threads).dvo_layer_decode(C.byref(D), C.byref(W.s), _ptr(x, _F32P),
                               None if xp is None else _ptr(xp, _F32P), B, k_h, k_n, _ptr(kc),
                               _ptr(vc), kv_len, _ptr(s_h, _F32P), _ptr(s_n, _F32P),
                               _ptr(idx_h, _I32P), _ptr(idx_n, _I32P), _ptr(u_h, _I32P),
                               _ptr(nuh, _I32P), _ptr(u_n, _I32P), _ptr(nun, _I32P),
                               _ptr(h1, _F64P), _ptr(y, _F64P)), "dvo_layer_decode")
    return {"s_h": s_h, "s_n": s_n, "idx_h": idx_h, "idx_n": idx_n,
            "u_h": u_h[: int(nuh[0])].copy(), "u_n": u_n[: int(nun[0])].copy(),
            "h1": h1, "y": y, "k_cache": kc, "v_cache": vc}


def numpy_weights(w_torch: Dict) -> Dict[str, np.ndarray]:
    """torch CPU tensors -> numpy arrays (same storage type)."""
    return {k: v.detach().cpu().contiguous().numpy() for k, v in w_torch.items()}


__all__ = ["Desc", "make_desc", "desc_from_config", "half_to_double", "double_to_half",
           "norm_row", "topk", "union", "predict", "sparse_attn", "sparse_mlp", "layer",
           "dense_layer", "layer_decode", "numpy_weights", "lib", "threads_used"]
