"""A stack of mixed-adapter LoRA projections run as one chained pass (the 8B-class workload:
32 layers x 7 projections, every projection a separate layer object of the C ABI).

Per layer l, with h [T, 4096]:
    q = P_q(h); k = P_k(h); v = P_v(h); o = P_o(q); g = P_gate(o); u = P_up(o); h' = P_down(g)
k, v and u are computed (and kept) but do not feed forward: the projection shapes of an
8B-class block (k/v output 1024, MLP width 14336) do not chain otherwise.  Every row keeps
its adapter slot through the whole stack.

Orchestration only: every projection is one ``set_batch_segments`` + ``lora_forward`` of the
C ABI; k, v and u run on a side stream beside the chain; ``capture`` records the whole pass
(both streams) in one CUDA graph.
"""
from __future__ import annotations

import torch

from . import workloads
from .lora import LoraLayer

# (input, output) buffer names per projection, in execution order
CHAIN = (("h", "q"), ("h", "k"), ("h", "v"), ("q", "o"), ("o", "g"), ("o", "u"), ("g", "h"))


class LoraStack:
    def __init__(self, n_layers: int = 32, T: int = 512, S: int = 100, r: int = 16,
                 seed: int = 1005, device="cuda", fp8_base: bool = False):
        """``fp8_base``: every projection's base product in e4m3 (lora_layer_create_fp8)."""
        self.n_layers, self.T, self.S, self.device = n_layers, T, S, torch.device(device)
        self.h0, ids = workloads.stack_tokens(seed=seed, T=T, S=S, device=self.device)
        self.ids = ids.to(self.device)
        self.layers = []
        for l in range(n_layers):
            row = []
            for p in range(len(workloads.STACK_PROJECTIONS)):
                W, adapters = workloads.stack_projection(l, p, seed=seed, S=S, r=r,
                                                         device=self.device)
                layer = LoraLayer(W, S, r, T, fp8_base=fp8_base)
                for s, (A, B, alpha) in enumerate(adapters):
                    layer.load(s, A, B, alpha)
                torch.cuda.synchronize()
                layer._keep.clear()  # sources copied: release them
                del W, adapters
                row.append(layer)
            self.layers.append(row)
        K = {"h": 4096, "q": 4096, "k": 1024, "v": 1024, "o": 4096, "g": 14336, "u": 14336}
        self.buf = {n: torch.empty(T, k, dtype=torch.bfloat16, device=self.device)
                    for n, k in K.items()}
        self.side = torch.cuda.Stream(device=self.device)
        self.graph = None

    def _run(self, layer, src, dst, stream):
        layer.set_batch(self.ids, stream)
        layer.forward(self.buf[src], self.buf[dst], stream)

    def step(self, stream=None, concurrent=True):
        """One chained pass: h <- h0, then every projection of every layer.

        The projections whose outputs do not feed forward (k, v, u) run on a side stream,
        beside the chain q -> o -> gate -> down on `stream`; events order the buffers they
        share: k and v read this layer's h before down overwrites it, u reads o before the
        next layer's o overwrites it.  The side stream joins `stream` at the end."""
        stream = stream or torch.cuda.current_stream(self.device)
        side = self.side if concurrent else stream  # concurrent=False: one stream, in order
        with torch.cuda.stream(stream):
            self.buf["h"].copy_(self.h0)
        e_h = torch.cuda.Event()
        e_h.record(stream)
        e_u = None
        for row in self.layers:
            p_q, p_k, p_v, p_o, p_g, p_u, p_d = row
            side.wait_event(e_h)                      # this layer's h is written
            self._run(p_k, "h", "k", side)
            self._run(p_v, "h", "v", side)
            e_v = torch.cuda.Event()
            e_v.record(side)
            self._run(p_q, "h", "q", stream)
            if e_u is not None:
                stream.wait_event(e_u)                # the previous layer's u has read o
            self._run(p_o, "q", "o", stream)
            e_o = torch.cuda.Event()
            e_o.record(stream)
            side.wait_event(e_o)
            self._run(p_u, "o", "u", side)
            e_u = torch.cuda.Event()
            e_u.record(side)
            self._run(p_g, "o", "g", stream)
            stream.wait_event(e_v)                    # k and v have read h
            self._run(p_d, "g", "h", stream)
            e_h = torch.cuda.Event()
            e_h.record(stream)
        if e_u is not None:
            stream.wait_event(e_u)
        return self.buf["h"]

    def capture(self, stream):
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=stream):
            self.step(stream)
        return self.graph

    def close(self):
        for row in self.layers:
            for layer in row:
                layer.close()
        self.layers = []
