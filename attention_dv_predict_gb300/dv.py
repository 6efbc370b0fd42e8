"""Python binding of libdv.so (include/dv.h): argument marshalling only.

Every computation runs in the library's CUDA kernels.  PyTorch supplies
device memory and streams.  Importing this module fails if the library has
not been built (``python -m attention_dv_predict_gb300.build``); there is no
fallback.
"""

from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m attention_dv_predict_gb300.build` "
        "(the sparse layer decode has no CPU fallback)")

_lib = C.CDLL(LIB_PATH)

DV_OK, DV_ERR_INVALID_ARG, DV_ERR_UNSUPPORTED, DV_ERR_CUDA = 0, 1, 2, 3
DV_ERR_TIMEOUT, DV_ERR_WORKSPACE, DV_ERR_DEVICE_INDEX, DV_ERR_SCRATCH_LIMIT = 4, 5, 6, 7
DV_F32, DV_F16 = 0, 1
DV_LAYERNORM, DV_RMSNORM = 0, 1
DV_MLP_RELU, DV_MLP_SWIGLU = 0, 1
DV_MAX_BATCH = 32

WEIGHT_FIELDS = ("ln1_g", "ln1_b", "w_qkv", "b_qkv", "w_oT", "b_o", "ln2_g", "ln2_b",
                 "w1", "b1", "w2T", "b2", "pred_h", "pred_a", "pred_b")


class LayerDesc(C.Structure):
    _fields_ = [("d_model", C.c_int32), ("n_heads", C.c_int32), ("head_dim", C.c_int32),
                ("d_ffn", C.c_int32), ("pred_rank", C.c_int32), ("dtype", C.c_int32),
                ("norm", C.c_int32), ("ln_eps", C.c_float), ("kv_cap", C.c_int32),
                ("neuron_block", C.c_int32), ("mlp", C.c_int32)]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in WEIGHT_FIELDS]


class Selection(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("idx_h", "idx_n", "u_h", "n_u_h", "u_n", "n_u_n")]


_P = C.c_void_p
_I = C.c_int
_SZ = C.c_size_t
_D = C.POINTER(LayerDesc)
_W = C.POINTER(LayerWeights)
_S = C.POINTER(Selection)

_SIGS = {
    "dv_status_string": ([_I], C.c_char_p),
    "dv_cuda_error": ([], _I),
    "dv_abi_version": ([], _I),
    "dv_set_row_kernel": ([_I], _I),
    "dv_workspace_size": ([_D, _I], _SZ),
    "dv_workspace_init": ([_P, _SZ, _P], _I),
    "dv_check": ([_P, _SZ, _P], _I),
    "dv_layer_decode_launches": ([_D, _I], _I),
    "dv_layer_decode_persistent_ok": ([_D, _I], _I),
    "dv_mlp_one_pass": ([_D, _I, _I], _I),
    "dv_predict_topk": ([_D, _W, _P, _I, _I, _I, _S, _P, _P, _P, _SZ, _P], _I),
    "dv_predict_topk_noalloc": ([_D, _W, _P, _I, _I, _I, _S, _P, _P, _P], _I),
    "dv_sparse_attn": ([_D, _W, _P, _I, _P, _P, _I, _P, _P, _I, _P, _P, _SZ, _P], _I),
    "dv_sparse_mlp": ([_D, _W, _P, _I, _P, _P, _I, _P, _P, _SZ, _P], _I),
    "dv_layer_decode": ([_D, _W, _P, _P, _I, _I, _I, _P, _P, _I, _S, _P, _P, _P, _SZ, _P], _I),
    "dv_layer_decode_persistent": ([_D, _W, _P, _P, _I, _I, _I, _P, _P, _I, _S, _P, _P, _P, _SZ,
                                    _P], _I),
    "dv_layer_decode_chained": ([_D, _W, _P, _P, _I, _I, _I, _P, _P, _I, _S, _P, _P, _P, _SZ,
                                 _P], _I),
    "dv_layer_decode_stamped": ([_D, _W, _P, _P, _I, _I, _I, _P, _P, _I, _S, _P, _P, _P, _SZ,
                                 _I, _P, _I, _P], _I),
    "dv_layer_decode_presel": ([_D, _W, _P, _I, _P, _P, _I, _P, _P, _I, _P, _P, _I, _P, _P, _P,
                                _SZ, _P], _I),
    "dv_layer_decode_traced": ([_D, _W, _P, _P, _I, _I, _I, _P, _P, _I, _S, _P, _P, _P, _SZ,
                                C.POINTER(_P), _I, _P], _I),
    "dv_layer_decode_host": ([_D, _W, _P, _P, _I, _I, _I, _P, _P, _I, _S, _P, _P, _SZ, _P], _I),
    "dv_hbm_copy": ([_P, _P, _SZ, _P], _I),
    "dv_test_hold_wait": ([_P, _SZ, _I, _I, _P], _I),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)


class DvError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        extra = f", cudaError {cuda_error}" if cuda_error else ""
        super().__init__(f"{fn}: {status_string(status)} ({status}{extra})")


def status_string(status: int) -> str:
    return _lib.dv_status_string(int(status)).decode()


def abi_version() -> int:
    return _lib.dv_abi_version()


def _check(fn: str, status: int):
    if status == DV_ERR_CUDA:
        raise DvError(fn, status, int(_lib.dv_cuda_error()))
    if status != DV_OK:
        raise DvError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


# ---------------------------------------------------------------------------


def make_desc(d_model, n_heads, head_dim, d_ffn, pred_rank, dtype, kv_cap,
              norm=DV_LAYERNORM, ln_eps=1e-5, neuron_block=0, mlp=0) -> LayerDesc:
    return LayerDesc(d_model, n_heads, head_dim, d_ffn, pred_rank, dtype, norm, ln_eps, kv_cap,
                     neuron_block, mlp)


def desc_from_config(cfg, kv_cap: Optional[int] = None) -> LayerDesc:
    """LayerDesc from a ``dv_inputs.LayerConfig`` (read by attribute)."""
    cap = cfg.kv_len + 1 if kv_cap is None else kv_cap
    return make_desc(cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.d_ffn, cfg.pred_rank,
                     DV_F32 if cfg.dtype == "f32" else DV_F16, cap,
                     DV_LAYERNORM if cfg.norm == "layernorm" else DV_RMSNORM, cfg.ln_eps,
                     getattr(cfg, "neuron_block", 0),
                     1 if getattr(cfg, "mlp", "relu") == "swiglu" else 0)


class Layer:
    """One layer's device weights plus the C struct pointing at them."""

    def __init__(self, desc: LayerDesc, weights: Dict[str, torch.Tensor]):
        self.desc = desc
        self.weights = {n: weights[n].contiguous() for n in WEIGHT_FIELDS}
        for n, t in self.weights.items():
            if not t.is_cuda:
                raise ValueError(f"weight {n} must be a CUDA tensor")
        self.c = LayerWeights(*[_ptr(self.weights[n]) for n in WEIGHT_FIELDS])


class Workspace:
    """Device workspace sized for (desc, batch), zeroed once."""

    def __init__(self, desc: LayerDesc, batch: int, device=None, stream=None):
        n = workspace_size(desc, batch)
        if n == 0:
            raise DvError("dv_workspace_size", DV_ERR_INVALID_ARG)
        # torch's caching allocator returns 512-byte aligned blocks
        self.buf = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.buf.data_ptr()) % 256
        self.ptr = self.buf.data_ptr() + off
        self.nbytes = n
        _check("dv_workspace_init", _lib.dv_workspace_init(C.c_void_p(self.ptr), n,
                                                            _stream(stream)))

    @property
    def cptr(self):
        return C.c_void_p(self.ptr)


class SelectionBuffers:
    """Device buffers for one selection (per-row top-k and unions)."""

    def __init__(self, desc: LayerDesc, batch: int, k_heads: int, k_neurons: int, device=None):
        dev = device or "cuda"
        H, N = desc.n_heads, desc.d_ffn
        self.batch, self.k_heads, self.k_neurons = batch, k_heads, k_neurons
        self.max_u_h = min(H, batch * k_heads)
        self.max_u_n = min(N, batch * k_neurons)
        self.idx_h = torch.empty((batch, k_heads), dtype=torch.int32, device=dev)
        self.idx_n = torch.empty((batch, k_neurons), dtype=torch.int32, device=dev)
        self.u_h = torch.empty(self.max_u_h, dtype=torch.int32, device=dev)
        self.u_n = torch.empty(self.max_u_n, dtype=torch.int32, device=dev)
        self.n_u_h = torch.zeros(1, dtype=torch.int32, device=dev)
        self.n_u_n = torch.zeros(1, dtype=torch.int32, device=dev)
        self.c = Selection(_ptr(self.idx_h), _ptr(self.idx_n), _ptr(self.u_h), _ptr(self.n_u_h),
                           _ptr(self.u_n), _ptr(self.n_u_n))

    def unions(self):
        """(u_h, u_n) trimmed to their device counts (synchronises)."""
        nh, nn = int(self.n_u_h.item()), int(self.n_u_n.item())
        return self.u_h[:nh], self.u_n[:nn]


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI).


def workspace_size(desc: LayerDesc, batch: int) -> int:
    return int(_lib.dv_workspace_size(C.byref(desc), int(batch)))


def dv_set_row_kernel(variant: int) -> None:
    """0: fc1 rows on mma.sync (default); 1: on tcgen05 (binary16, ReLU, B >= 9)."""
    _check("dv_set_row_kernel", _lib.dv_set_row_kernel(int(variant)))


def dv_check(ws: Workspace, stream=None) -> int:
    return int(_lib.dv_check(ws.cptr, ws.nbytes, _stream(stream)))


def dv_layer_decode_launches(desc: LayerDesc, batch: int) -> int:
    return int(_lib.dv_layer_decode_launches(C.byref(desc), int(batch)))


def dv_mlp_one_pass(desc: LayerDesc, batch: int, max_u_n: int) -> bool:
    """The MLP half runs as one pass plus the partials' sum (two kernels)."""
    return bool(_lib.dv_mlp_one_pass(C.byref(desc), int(batch), int(max_u_n)))


def dv_layer_decode_persistent_ok(desc: LayerDesc, batch: int) -> bool:
    return bool(_lib.dv_layer_decode_persistent_ok(C.byref(desc), int(batch)))


def dv_predict_topk(layer: Layer, x_pred: torch.Tensor, k_heads: int, k_neurons: int,
                    sel: SelectionBuffers, ws: Workspace, scores_h: Optional[torch.Tensor] = None,
                    scores_n: Optional[torch.Tensor] = None, stream=None):
    B = x_pred.shape[0]
    _check("dv_predict_topk", _lib.dv_predict_topk(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x_pred), B, k_heads, k_neurons,
        C.byref(sel.c), _ptr(scores_h), _ptr(scores_n), ws.cptr, ws.nbytes, _stream(stream)))


def dv_predict_topk_noalloc(layer: Layer, x_pred: torch.Tensor, k_heads: int, k_neurons: int,
                            sel: SelectionBuffers, scores_h: Optional[torch.Tensor] = None,
                            scores_n: Optional[torch.Tensor] = None, stream=None):
    B = x_pred.shape[0]
    _check("dv_predict_topk_noalloc", _lib.dv_predict_topk_noalloc(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x_pred), B, k_heads, k_neurons,
        C.byref(sel.c), _ptr(scores_h), _ptr(scores_n), _stream(stream)))


def dv_sparse_attn(layer: Layer, x: torch.Tensor, u_h: torch.Tensor, n_u_h: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int, h1: torch.Tensor,
                   ws: Workspace, max_u_h: Optional[int] = None, stream=None):
    B = x.shape[0]
    m = u_h.numel() if max_u_h is None else max_u_h
    _check("dv_sparse_attn", _lib.dv_sparse_attn(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x), B, _ptr(u_h), _ptr(n_u_h), m,
        _ptr(k_cache), _ptr(v_cache), kv_len, _ptr(h1), ws.cptr, ws.nbytes, _stream(stream)))


def dv_sparse_mlp(layer: Layer, h1: torch.Tensor, u_n: torch.Tensor, n_u_n: torch.Tensor,
                  y: torch.Tensor, ws: Workspace, max_u_n: Optional[int] = None, stream=None):
    B = h1.shape[0]
    m = u_n.numel() if max_u_n is None else max_u_n
    _check("dv_sparse_mlp", _lib.dv_sparse_mlp(
        C.byref(layer.desc), C.byref(layer.c), _ptr(h1), B, _ptr(u_n), _ptr(n_u_n), m, _ptr(y),
        ws.cptr, ws.nbytes, _stream(stream)))


def dv_layer_decode(layer: Layer, x: torch.Tensor, k_heads: int, k_neurons: int,
                    k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int,
                    sel: SelectionBuffers, y: torch.Tensor, ws: Workspace,
                    x_pred: Optional[torch.Tensor] = None, h1: Optional[torch.Tensor] = None,
                    stream=None):
    B = x.shape[0]
    _check("dv_layer_decode", _lib.dv_layer_decode(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x), _ptr(x_pred), B, k_heads, k_neurons,
        _ptr(k_cache), _ptr(v_cache), kv_len, C.byref(sel.c), _ptr(h1), _ptr(y), ws.cptr,
        ws.nbytes, _stream(stream)))


def dv_layer_decode_chained(layer: Layer, x: torch.Tensor, k_heads: int, k_neurons: int,
                            k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int,
                            sel: SelectionBuffers, y: torch.Tensor, ws: Workspace,
                            x_pred: Optional[torch.Tensor] = None,
                            h1: Optional[torch.Tensor] = None, stream=None):
    """dv_layer_decode as the seven chained kernels (every shape and batch)."""
    B = x.shape[0]
    _check("dv_layer_decode_chained", _lib.dv_layer_decode_chained(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x), _ptr(x_pred), B, k_heads, k_neurons,
        _ptr(k_cache), _ptr(v_cache), kv_len, C.byref(sel.c), _ptr(h1), _ptr(y), ws.cptr,
        ws.nbytes, _stream(stream)))


def dv_layer_decode_stamped(layer: Layer, x: torch.Tensor, k_heads: int, k_neurons: int,
                            k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int,
                            sel: SelectionBuffers, y: torch.Tensor, ws: Workspace,
                            stamps: torch.Tensor, x_pred: Optional[torch.Tensor] = None,
                            h1: Optional[torch.Tensor] = None, persistent: bool = False,
                            stream=None):
    """The decode with its timeline in ``stamps`` (int64): [7, SMs, 8] for the
    chain, [SMs, 32] for the persistent streaming kernel."""
    B = x.shape[0]
    _check("dv_layer_decode_stamped", _lib.dv_layer_decode_stamped(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x), _ptr(x_pred), B, k_heads, k_neurons,
        _ptr(k_cache), _ptr(v_cache), kv_len, C.byref(sel.c), _ptr(h1), _ptr(y), ws.cptr,
        ws.nbytes, int(bool(persistent)), _ptr(stamps), stamps.numel(), _stream(stream)))


def dv_layer_decode_persistent(layer: Layer, x: torch.Tensor, k_heads: int, k_neurons: int,
                               k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int,
                               sel: SelectionBuffers, y: torch.Tensor, ws: Workspace,
                               x_pred: Optional[torch.Tensor] = None,
                               h1: Optional[torch.Tensor] = None, stream=None):
    """dv_layer_decode through the streaming kernel only (see dv_layer_decode_persistent_ok)."""
    B = x.shape[0]
    _check("dv_layer_decode_persistent", _lib.dv_layer_decode_persistent(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x), _ptr(x_pred), B, k_heads, k_neurons,
        _ptr(k_cache), _ptr(v_cache), kv_len, C.byref(sel.c), _ptr(h1), _ptr(y), ws.cptr,
        ws.nbytes, _stream(stream)))


def dv_layer_decode_presel(layer: Layer, x: torch.Tensor, sel: SelectionBuffers,
                           k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int,
                           y: torch.Tensor, ws: Workspace, h1: Optional[torch.Tensor] = None,
                           stream=None):
    """Layer decode on the unions already in ``sel`` (e.g. from a lookahead predictor)."""
    B = x.shape[0]
    _check("dv_layer_decode_presel", _lib.dv_layer_decode_presel(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x), B, _ptr(sel.u_h), _ptr(sel.n_u_h),
        sel.max_u_h, _ptr(sel.u_n), _ptr(sel.n_u_n), sel.max_u_n, _ptr(k_cache), _ptr(v_cache),
        kv_len, _ptr(h1), _ptr(y), ws.cptr, ws.nbytes, _stream(stream)))


def dv_layer_decode_traced(layer: Layer, x: torch.Tensor, k_heads: int, k_neurons: int,
                           k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int,
                           sel: SelectionBuffers, y: torch.Tensor, ws: Workspace,
                           events: Sequence[torch.cuda.Event],
                           x_pred: Optional[torch.Tensor] = None,
                           h1: Optional[torch.Tensor] = None, stream=None):
    B = x.shape[0]
    s = stream if stream is not None else torch.cuda.current_stream()
    for e in events:  # torch creates the CUDA event on its first record
        if e.cuda_event == 0:
            e.record(s)
    arr = (C.c_void_p * len(events))(*[C.c_void_p(e.cuda_event) for e in events])
    _check("dv_layer_decode_traced", _lib.dv_layer_decode_traced(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x), _ptr(x_pred), B, k_heads, k_neurons,
        _ptr(k_cache), _ptr(v_cache), kv_len, C.byref(sel.c), _ptr(h1), _ptr(y), ws.cptr,
        ws.nbytes, arr, len(events), _stream(stream)))


def dv_layer_decode_host(layer: Layer, x_host: torch.Tensor, k_heads: int, k_neurons: int,
                         k_cache: torch.Tensor, v_cache: torch.Tensor, kv_len: int,
                         y_host: torch.Tensor, ws: Workspace,
                         sel: Optional[SelectionBuffers] = None,
                         x_pred_host: Optional[torch.Tensor] = None, stream=None):
    """Host activations in and out (pinned CPU tensors give async copies); synchronous."""
    for t in (x_host, y_host) + ((x_pred_host,) if x_pred_host is not None else ()):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.float32:
            raise ValueError("host activations must be contiguous float32 CPU tensors")
    B = x_host.shape[0]
    _check("dv_layer_decode_host", _lib.dv_layer_decode_host(
        C.byref(layer.desc), C.byref(layer.c), _ptr(x_host), _ptr(x_pred_host), B, k_heads,
        k_neurons, _ptr(k_cache), _ptr(v_cache), kv_len,
        C.byref(sel.c) if sel is not None else None, _ptr(y_host), ws.cptr, ws.nbytes,
        _stream(stream)))


def dv_test_hold_wait(ws: Workspace, wait_id: int, budget_us: int, stream=None):
    """Test support: make the next streaming decode's wait `wait_id` run out."""
    _check("dv_test_hold_wait", _lib.dv_test_hold_wait(ws.cptr, ws.nbytes, int(wait_id),
                                                        int(budget_us), _stream(stream)))


def dv_hbm_copy(dst: torch.Tensor, src: torch.Tensor, nbytes: Optional[int] = None, stream=None):
    n = src.numel() * src.element_size() if nbytes is None else nbytes
    _check("dv_hbm_copy", _lib.dv_hbm_copy(_ptr(dst), _ptr(src), n, _stream(stream)))
