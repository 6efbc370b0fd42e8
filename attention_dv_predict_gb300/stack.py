"""A stack of sparse layer decodes with the lookahead predictor on a side stream.

("DejaVu Guide: Contextual Sparsity for LLM Inference", "2. Pipelined Overlap
Execution"; "Core Innovation 1: Asynchronous Lookahead Predictors": while
layer l computes, the predictor for layer l+1 runs on another CUDA stream
from the input of layer l, so layer l+1 starts with its head and neuron sets
ready.)

One token step of an L-layer stack, batch B:

    side:  predict(layer 0, x_0)                      -> sel[0]
    for l = 0 .. L-1:
        main:  wait sel[l];  decode_presel(layer l, x_l, sel[l]) -> x_{l+1}
        side:  wait until x_l is final and layer l-1 is done;
               predict(layer l+1, x_pred = x_l)        -> sel[(l+1) % 2]

Layer 0 predicts from its own input (nothing precedes it).  Selections are
double-buffered: the side stream writes sel[(l+1) % 2] only after layer l-1,
the last reader of that buffer, has finished.  Every kernel runs through the
C ABI (`dv.py`); this module only orders the calls and the events.

`serial=True` runs the same calls on one stream (predict then decode for
each layer), the reference point for the overlap.

`fused=True` runs each layer as one dv_layer_decode call on the main
stream with x_pred = the previous layer's input: the same lookahead sets,
predicted inside the layer's own launch sequence instead of on the side
stream.
"""
from typing import List, Optional, Sequence

import torch

from . import dv


class LayerStack:
    def __init__(self, desc: dv.LayerDesc, layers: Sequence[dv.Layer], batch: int,
                 k_heads: int, k_neurons: int, device=None):
        self.desc = desc
        self.layers = list(layers)
        self.batch = batch
        self.k_heads = k_heads
        self.k_neurons = k_neurons
        dev = torch.device(device or "cuda")
        d = desc.d_model
        n = len(self.layers)
        # x[l] is the input of layer l; x[n] is the stack's output
        self.x = [torch.empty((batch, d), dtype=torch.float32, device=dev) for _ in range(n + 1)]
        self.sel = [dv.SelectionBuffers(desc, batch, k_heads, k_neurons, device=dev)
                    for _ in range(2)]
        self.ws_main = dv.Workspace(desc, batch, device=dev)
        self.ws_pred = dv.Workspace(desc, batch, device=dev)
        self.main = torch.cuda.Stream(device=dev)
        self.side = torch.cuda.Stream(device=dev)
        self._ev_input = [torch.cuda.Event() for _ in range(n + 1)]
        self._ev_pred = [torch.cuda.Event() for _ in range(n)]
        # per-layer selections, kept only when asked (tests)
        self.keep_selection = False
        self.kept: List[dict] = []

    def _predict(self, l: int, x_pred: torch.Tensor, stream):
        dv.dv_predict_topk(self.layers[l], x_pred, self.k_heads, self.k_neurons,
                           self.sel[l % 2], self.ws_pred, stream=stream)

    def _keep(self, l: int, stream):
        if self.keep_selection:
            s = self.sel[l % 2]
            with torch.cuda.stream(stream):
                self.kept.append({"idx_h": s.idx_h.clone(), "idx_n": s.idx_n.clone(),
                                  "u_h": s.u_h.clone(), "n_u_h": s.n_u_h.clone(),
                                  "u_n": s.u_n.clone(), "n_u_n": s.n_u_n.clone()})

    def _enqueue_fused(self, x0, caches, kv_len):
        n = len(self.layers)
        main = self.main
        self.kept = []
        main.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(main):
            self.x[0].copy_(x0)
        for l in range(n):
            kc, vc = caches[l]
            dv.dv_layer_decode(self.layers[l], self.x[l], self.k_heads, self.k_neurons, kc, vc,
                               kv_len, self.sel[l % 2], self.x[l + 1], self.ws_main,
                               x_pred=self.x[max(l - 1, 0)], stream=main)
            self._keep(l, main)
        torch.cuda.current_stream().wait_stream(main)
        return self.x[n]

    def enqueue(self, x0: torch.Tensor, caches: Sequence[Sequence[torch.Tensor]], kv_len: int,
                serial: bool = False, fused: bool = False):
        """Enqueue one token step; the output is ``self.x[-1]`` once ``self.main`` reaches it.

        x0 [B, d] binary32 (any stream that ``self.main`` is ordered after);
        caches[l] = (k_cache, v_cache) of layer l.  fused: one
        dv_layer_decode call per layer (the predictor inside it); else the
        predictor on the side stream (or on the main one, serial) beside
        dv_layer_decode_presel.
        """
        if fused:
            return self._enqueue_fused(x0, caches, kv_len)
        n = len(self.layers)
        main, side = self.main, (self.main if serial else self.side)
        self.kept = []
        main.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(main):
            self.x[0].copy_(x0)
        self._ev_input[0].record(main)
        side.wait_event(self._ev_input[0])
        self._predict(0, self.x[0], side)
        self._ev_pred[0].record(side)
        for l in range(n):
            main.wait_event(self._ev_pred[l])
            self._keep(l, main)
            kc, vc = caches[l]
            dv.dv_layer_decode_presel(self.layers[l], self.x[l], self.sel[l % 2], kc, vc, kv_len,
                                      self.x[l + 1], self.ws_main, stream=main)
            self._ev_input[l + 1].record(main)
            if l + 1 < n:
                # the predictor for layer l+1 reads x_l (final since layer l-1
                # finished) and overwrites the buffer layer l-1 read
                side.wait_event(self._ev_input[l])
                self._predict(l + 1, self.x[l], side)
                self._ev_pred[l + 1].record(side)
        torch.cuda.current_stream().wait_stream(main)
        return self.x[n]

    def run(self, x0: torch.Tensor, caches, kv_len: int, serial: bool = False,
            fused: bool = False) -> torch.Tensor:
        """One token step, synchronised; returns a copy of the stack output."""
        y = self.enqueue(x0, caches, kv_len, serial=serial, fused=fused)
        torch.cuda.synchronize()
        return y.clone()


def make_stack_weights(cfg, n_layers: int, device="cuda", seed0: int = 0):
    """Random-init weights of n_layers layers (layer l drawn with seed seed0 + l)."""
    import dv_inputs

    return [dv_inputs.make_weights(cfg, seed=seed0 + l, device=device) for l in range(n_layers)]


def layers_from_weights(desc: dv.LayerDesc, weights) -> List[dv.Layer]:
    return [dv.Layer(desc, w) for w in weights]


def stack_caches(cfg, n_layers: int, batch: int, device="cuda", seed0: int = 0,
                 kv_cap: Optional[int] = None):
    import dv_inputs

    return [dv_inputs.make_kv(cfg, batch, seed=seed0 + l, device=device, kv_cap=kv_cap)
            for l in range(n_layers)]
