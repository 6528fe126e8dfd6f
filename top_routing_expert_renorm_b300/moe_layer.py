"""MoELayer: holds a layer's configuration, weights and workspace (torch-owned
device memory) and runs the whole forward through moe_forward."""

import torch

from . import api


class MoELayer:
    """One MoE layer. Tensors (all on one CUDA device, contiguous):
    W_gate [d, E] fp32, gate_bias [E] fp32 or None, w1 [E, N1, d], b1 [E, N1] or None,
    w2 [E, d, F] (not for LINEAR), b2 [E, d] or None, shared = (w1, b1, w2, b2[, s1, s2]) or
    None; with INT8 experts w1 / w2 hold int8 codes and s1 [E, N1] / s2 [E, d] their scales,
    with INT4 experts w1 [E, N1, d/2] / w2 [E, d, F/2] the packed codes (uint8).
    The workspace is sized for up to `max_tokens` tokens per call."""

    def __init__(self, cfg, W_gate, gate_bias, w1, b1=None, w2=None, b2=None, shared=None,
                 s1=None, s2=None):
        import torch
        self.cfg = cfg
        bits = {api.C.MOE_I8: 8, api.C.MOE_I4: 4}.get(cfg.w_dtype)
        if bits and w1.dtype == torch.bfloat16:
            # bf16 weights for an INT8 / INT4 layer: quantise them once (codes + row scales)
            w1, s1, w2, s2 = api.quantize_weights(w1, w2, bits=bits)
            if shared is not None:
                sw1, ss1, sw2, ss2 = api.quantize_weights(shared[0], shared[2], bits=bits)
                shared = (sw1, shared[1], sw2, shared[3], ss1, ss2)
        self._keep = [W_gate, gate_bias, w1, b1, w2, b2, shared, s1, s2]
        self.W_gate, self.gate_bias = W_gate, gate_bias
        self.routed = api.weights(w1, b1, w2, b2, s1, s2)
        self.shared = api.weights(*shared) if shared is not None else None
        self.ws = torch.empty(api.workspace_size(cfg), dtype=torch.uint8, device=w1.device)

    def config(self, T):
        c = api.MoeConfig()
        for f, _ in api.MoeConfig._fields_:
            setattr(c, f, getattr(self.cfg, f))
        c.T = T
        return c

    def capture(self, x, out, stream=None):
        """Record one forward of x -> out (fixed buffers) into a CUDA graph and return it;
        graph.replay() then runs the whole layer with a single launch from the host,
        on torch's current stream. x and out must stay allocated while the graph is used.
        One direct forward runs first so that the library's one-time set-up (device
        attribute queries, kernel attributes) happens outside the capture."""
        import torch
        self(x, out=out, stream=stream)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            self(x, out=out)
        return graph

    def __call__(self, x, out=None, topk_idx=None, topk_w=None, load=None, stream=None):
        T = x.shape[0]
        if T > self.cfg.T:
            raise ValueError(f"{T} tokens exceed the layer's max_tokens {self.cfg.T}")
        out = torch.empty_like(x) if out is None else out
        api.forward(self.config(T), x, self.W_gate, self.gate_bias, self.routed, self.shared,
                    out, self.ws, topk_idx=topk_idx, topk_w=topk_w, load=load, stream=stream)
        return out
