"""Named synthetic workloads: shapes, value distributions and tensor recipes.

Every tensor is a slice of the counter-based generator (tensor ids below), so
the host can regenerate any expert's weights without the device, and the
device can fill tens of GB without a host round trip. Distributions follow
the workload descriptions: x ~ N(0,1); weights ~ N(0, 1/fan_in); for the
decode-sized workload the gate weights are U(-1/sqrt(d), 1/sqrt(d)); for the
Mixtral-shaped workload the gate logits are biased by ln p_e with
p_e proportional to (e+1)^-1.1 (Zipf, s = 1.1) to skew the expert load.
"""

from dataclasses import dataclass, replace
import math

import numpy as np

from .gen import NORMAL, UNIFORM, normal_K, uniform_K, host_fill, dev_fill

# tensor ids of the generator
TID_X, TID_WG, TID_W1, TID_B1, TID_W2, TID_B2 = 1, 2, 4, 5, 6, 7
TID_SW1, TID_SB1, TID_SW2, TID_SB2 = 8, 9, 10, 11

KIND_CODE = {"linear": 0, "gelu": 1, "swiglu": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    kind: str               # "linear" | "gelu" | "swiglu"
    act: str                # "f32" | "bf16"
    cf: float = 0.0         # capacity factor; <= 0: no limit
    add_residual: bool = False
    has_shared: bool = False
    gate_dist: str = "normal"   # "normal" | "uniform" | "zero" (every logit equal) |
                                # "grid" (integers -1, 0, 1: logits tie exactly and often)
    x_dist: str = "normal"      # "normal" | "grid" (integers -1, 0, 1 in the first 16 features,
                                # 0 elsewhere: few distinct logits)
    gate_bias: str = "none"     # "none" | "zipf" | "hot" (+20 on expert 0: one expert takes all)
    expert_bias: bool = False
    int8: bool = False          # weight-only INT8 experts (codes + per-row scales)
    int4: bool = False          # weight-only INT4 experts (packed codes + per-row scales)
    n_group: int = 0            # group-limited routing: expert groups (0 = plain top-k)
    topk_group: int = 0         # groups kept per token
    overflow: str = "drop"      # over-capacity slots: "drop" | "shared" | "reroute"
    seed: int = 0
    note: str = ""

    # ---- shapes -----------------------------------------------------------
    @property
    def N1(self):
        return {"linear": self.d, "gelu": self.F, "swiglu": 2 * self.F}[self.kind]

    @property
    def kind_code(self):
        return KIND_CODE[self.kind]

    @property
    def bf16(self):
        return self.act == "bf16"

    @property
    def w2_per_expert(self):
        return 0 if self.kind == "linear" else self.d * self.F

    def with_(self, **kw):
        return replace(self, **kw)

    # ---- scales -----------------------------------------------------------
    def _wg_dist_K(self):
        if self.gate_dist == "uniform":
            return UNIFORM, uniform_K(1.0 / math.sqrt(self.d))
        return NORMAL, normal_K(1.0 / math.sqrt(self.d))

    def _w1_K(self):
        return normal_K(1.0 / math.sqrt(self.d))

    def _w2_K(self):
        return normal_K(1.0 / math.sqrt(self.F if self.kind != "linear" else self.d))

    # ---- host tensors (numpy; bf16 as uint16 bit patterns) ------------------
    def _grid(self, tid, n):
        """n integers in {-1, 0, 1}: uniform values on (-1.5, 1.5) rounded to the nearest
        integer (exact in fp32 and bf16)."""
        u = host_fill(self.seed, tid, 0, n, UNIFORM, uniform_K(1.5), False)
        return np.clip(np.rint(u), -1.0, 1.0).astype(np.float32)

    def _x_grid(self):
        g = self._grid(TID_X, self.T * self.d).reshape(self.T, self.d)
        g[:, 16:] = 0.0
        if self.bf16:   # integers are exact in bf16: the upper half of the fp32 pattern
            return (g.view(np.uint32) >> 16).astype(np.uint16)
        return g

    def x_host(self, rows=None):
        """All of x [T, d], or the listed rows only."""
        if self.x_dist == "grid":
            g = self._x_grid()
            return g if rows is None else g[np.asarray(rows, dtype=np.int64)]
        if rows is None:
            return host_fill(self.seed, TID_X, 0, self.T * self.d, NORMAL, normal_K(1.0),
                             self.bf16).reshape(self.T, self.d)
        out = [host_fill(self.seed, TID_X, int(t) * self.d, self.d, NORMAL, normal_K(1.0),
                         self.bf16) for t in rows]
        return np.stack(out) if out else np.empty((0, self.d),
                                                   np.uint16 if self.bf16 else np.float32)

    def wg_host(self):
        if self.gate_dist == "zero":
            return np.zeros((self.d, self.E), np.float32)
        if self.gate_dist == "grid":
            return self._grid(TID_WG, self.d * self.E).reshape(self.d, self.E)
        dist, K = self._wg_dist_K()
        return host_fill(self.seed, TID_WG, 0, self.d * self.E, dist, K, False).reshape(self.d, self.E)

    def gate_bias_host(self):
        if self.gate_bias == "none":
            return None
        if self.gate_bias == "hot":
            b = np.zeros(self.E, np.float32)
            b[0] = 20.0
            return b
        p = np.array([(e + 1) ** -1.1 for e in range(self.E)], np.float64)
        p /= p.sum()
        return np.log(p).astype(np.float32)

    def w1_host(self, e, shared=False):
        n = self.N1 * self.d
        tid = TID_SW1 if shared else TID_W1
        off = 0 if shared else e * n
        return host_fill(self.seed, tid, off, n, NORMAL, self._w1_K(), self.bf16).reshape(self.N1, self.d)

    def b1_host(self, e, shared=False):
        if not self.expert_bias:
            return None
        tid = TID_SB1 if shared else TID_B1
        off = 0 if shared else e * self.N1
        return host_fill(self.seed, tid, off, self.N1, NORMAL, self._w1_K(), False)

    def w2_host(self, e, shared=False):
        if self.kind == "linear":
            return None
        n = self.w2_per_expert
        tid = TID_SW2 if shared else TID_W2
        off = 0 if shared else e * n
        return host_fill(self.seed, tid, off, n, NORMAL, self._w2_K(), self.bf16).reshape(self.d, self.F)

    def b2_host(self, e, shared=False):
        if not self.expert_bias or self.kind == "linear":
            return None
        tid = TID_SB2 if shared else TID_B2
        off = 0 if shared else e * self.d
        return host_fill(self.seed, tid, off, self.d, NORMAL, self._w2_K(), False)

    def stacked_host(self):
        """Full stacked expert weights on the host (small workloads only)."""
        def cat(fn):
            parts = [fn(e) for e in range(self.E)]
            return None if parts[0] is None else np.ascontiguousarray(np.stack(parts))
        w = dict(w1=cat(self.w1_host), b1=cat(self.b1_host), w2=cat(self.w2_host),
                 b2=cat(self.b2_host))
        if self.has_shared:
            w["shared"] = (self.w1_host(0, True), self.b1_host(0, True),
                           self.w2_host(0, True), self.b2_host(0, True))
        else:
            w["shared"] = None
        return w

    # ---- device tensors (torch) -----------------------------------------------
    def device_inputs(self, device="cuda"):
        """Every input of the layer as torch tensors on `device`, filled on the GPU."""
        import torch
        adt = torch.bfloat16 if self.bf16 else torch.float32
        emp = lambda *s, dt=adt: torch.empty(*s, dtype=dt, device=device)  # noqa: E731
        if self.x_dist == "grid":   # small tie-test layers: made on the host, uploaded
            xh = self._x_grid()
            x = torch.from_numpy(xh.view(np.int16) if self.bf16 else xh).to(device)
            x = x.view(torch.bfloat16) if self.bf16 else x
        else:
            x = dev_fill(emp(self.T, self.d), self.seed, TID_X, 0, NORMAL, normal_K(1.0))
        if self.gate_dist in ("zero", "grid"):
            wg = torch.from_numpy(self.wg_host()).to(device)
        else:
            dist, K = self._wg_dist_K()
            wg = dev_fill(emp(self.d, self.E, dt=torch.float32), self.seed, TID_WG, 0, dist, K)
        gb = self.gate_bias_host()
        gb = None if gb is None else torch.from_numpy(gb).to(device)
        w1 = dev_fill(emp(self.E, self.N1, self.d), self.seed, TID_W1, 0, NORMAL, self._w1_K())
        b1 = (dev_fill(emp(self.E, self.N1, dt=torch.float32), self.seed, TID_B1, 0, NORMAL,
                       self._w1_K()) if self.expert_bias else None)
        w2 = b2 = None
        if self.kind != "linear":
            w2 = dev_fill(emp(self.E, self.d, self.F), self.seed, TID_W2, 0, NORMAL, self._w2_K())
            if self.expert_bias:
                b2 = dev_fill(emp(self.E, self.d, dt=torch.float32), self.seed, TID_B2, 0,
                              NORMAL, self._w2_K())
        shared = None
        if self.has_shared:
            sw1 = dev_fill(emp(self.N1, self.d), self.seed, TID_SW1, 0, NORMAL, self._w1_K())
            sb1 = (dev_fill(emp(self.N1, dt=torch.float32), self.seed, TID_SB1, 0, NORMAL,
                            self._w1_K()) if self.expert_bias else None)
            sw2 = sb2 = None
            if self.kind != "linear":
                sw2 = dev_fill(emp(self.d, self.F), self.seed, TID_SW2, 0, NORMAL, self._w2_K())
                if self.expert_bias:
                    sb2 = dev_fill(emp(self.d, dt=torch.float32), self.seed, TID_SB2, 0,
                                   NORMAL, self._w2_K())
            shared = (sw1, sb1, sw2, sb2)
        return dict(x=x, wg=wg, gate_bias=gb, w1=w1, b1=b1, w2=w2, b2=b2, shared=shared)

    # ---- algorithmic cost (per forward) ----------------------------------------
    def flops(self, P):
        """Router + routed experts (P kept rows) + shared expert."""
        m = {"linear": 1, "gelu": 2, "swiglu": 3}[self.kind]
        f = self.F if self.kind != "linear" else self.d
        fl = 2.0 * self.T * self.d * self.E + 2.0 * P * m * self.d * f
        if self.has_shared:
            fl += 2.0 * self.T * m * self.d * f
        return fl

    def bytes(self, touched_experts):
        """Weights of touched experts + gate weights + x read + out written (INT8 / INT4
        experts: one / half a byte per weight plus a 4-byte scale per weight row)."""
        es = 2 if self.bf16 else 4
        if self.int8:
            per = (self.N1 * self.d + self.w2_per_expert) + 4 * (self.N1 + self.d)
        elif self.int4:
            per = (self.N1 * self.d + self.w2_per_expert) // 2 + 4 * (self.N1 + self.d)
        else:
            per = (self.N1 * self.d + self.w2_per_expert) * es
        b = touched_experts * per + self.d * self.E * 4 + 2 * self.T * self.d * es
        if self.has_shared:
            b += per
        return float(b)


WORKLOADS = {
    "tiny": Workload("tiny", T=64, d=8, E=4, k=2, F=8, kind="linear", act="f32",
                     expert_bias=True,
                     note="tiny top-2: T=64, d=8, E=4, Linear(8->8)+bias experts, fp32"),
    "switch": Workload("switch", T=8192, d=1024, E=64, k=1, F=4096, kind="gelu", act="bf16",
                       cf=1.25, add_residual=True,
                       note="Switch-style top-1, GELU d->4096->d, capacity 1.25, residual pass-through"),
    "mixtral": Workload("mixtral", T=4096, d=4096, E=8, k=2, F=14336, kind="swiglu", act="bf16",
                        gate_bias="zipf",
                        note="Mixtral-shaped top-2 SwiGLU d=4096, F=14336, Zipf(1.1)-biased gate"),
    "deepseek": Workload("deepseek", T=8192, d=7168, E=256, k=8, F=2048, kind="swiglu",
                         act="bf16", cf=1.0, has_shared=True,
                         note="DeepSeek-V3-shaped: 256 routed + 1 shared SwiGLU experts, top-8, cf 1.0"),
    "deepseek_grouped": Workload("deepseek_grouped", T=8192, d=7168, E=256, k=8, F=2048,
                                 kind="swiglu", act="bf16", cf=1.0, has_shared=True, n_group=8,
                                 topk_group=4,
                                 note="DeepSeek-V3-shaped, group-limited routing: 8 groups, 4 kept"),
    "deepseek_reroute": Workload("deepseek_reroute", T=8192, d=7168, E=256, k=8, F=2048,
                                 kind="swiglu", act="bf16", cf=1.0, has_shared=True,
                                 overflow="reroute",
                                 note="DeepSeek-V3-shaped, cf 1.0, over-capacity slots re-routed"),
    "deepseek_cf125": Workload("deepseek_cf125", T=8192, d=7168, E=256, k=8, F=2048,
                               kind="swiglu", act="bf16", cf=1.25, has_shared=True,
                               note="DeepSeek-V3-shaped, capacity factor 1.25"),
    # per-expert shapes of the DeepSeek-V3-shaped layer with 32 experts and 1024 tokens
    # (256 rows per expert at capacity 1.0): small enough for multi-pass profiler captures
    "deepseek_e32": Workload("deepseek_e32", T=1024, d=7168, E=32, k=8, F=2048, kind="swiglu",
                             act="bf16", cf=1.0, has_shared=True,
                             note="DeepSeek-V3 expert shapes, 32 experts (for profiling)"),
    # the DeepSeek-V3-shaped layer's routing, dispatch, gather and combine (T, d, E, k, the
    # shared expert) with F = 64 (0.7 GB of expert weights): memory-bound kernels at full
    # size within a few GB for multi-pass profiler captures
    "deepseek_memprof": Workload("deepseek_memprof", T=8192, d=7168, E=256, k=8, F=64,
                                 kind="swiglu", act="bf16", cf=1.0, has_shared=True,
                                 note="DeepSeek-V3 routing/dispatch/combine shapes, F = 64 (for profiling)"),
    # weight-only INT8 experts (codes + per-row scales) for the decode-sized layers
    "decode1_i8": Workload("decode1_i8", T=1, d=7168, E=256, k=8, F=2048, kind="swiglu",
                           act="bf16", gate_dist="uniform", int8=True,
                           note="decode, 1 token, INT8 expert weights"),
    "decode8_i8": Workload("decode8_i8", T=8, d=7168, E=256, k=8, F=2048, kind="swiglu",
                           act="bf16", gate_dist="uniform", int8=True,
                           note="decode, 8 tokens, INT8 expert weights"),
    "decode64_i8": Workload("decode64_i8", T=64, d=7168, E=256, k=8, F=2048, kind="swiglu",
                            act="bf16", gate_dist="uniform", int8=True,
                            note="decode, 64 tokens, INT8 expert weights"),
    # decode8_i8's expert shapes with 32 experts: small enough for multi-pass profiler captures
    "decode8_i8_e32": Workload("decode8_i8_e32", T=8, d=7168, E=32, k=8, F=2048, kind="swiglu",
                               act="bf16", gate_dist="uniform", int8=True,
                               note="decode, 8 tokens, INT8 weights, 32 experts (for profiling)"),
    # weight-only INT4 experts (packed codes + per-row scales) for the decode-sized layers
    "decode1_i4": Workload("decode1_i4", T=1, d=7168, E=256, k=8, F=2048, kind="swiglu",
                           act="bf16", gate_dist="uniform", int4=True,
                           note="decode, 1 token, INT4 expert weights"),
    "decode8_i4": Workload("decode8_i4", T=8, d=7168, E=256, k=8, F=2048, kind="swiglu",
                           act="bf16", gate_dist="uniform", int4=True,
                           note="decode, 8 tokens, INT4 expert weights"),
    "decode64_i4": Workload("decode64_i4", T=64, d=7168, E=256, k=8, F=2048, kind="swiglu",
                            act="bf16", gate_dist="uniform", int4=True,
                            note="decode, 64 tokens, INT4 expert weights"),
    "decode8_i4_e32": Workload("decode8_i4_e32", T=8, d=7168, E=32, k=8, F=2048, kind="swiglu",
                               act="bf16", gate_dist="uniform", int4=True,
                               note="decode, 8 tokens, INT4 weights, 32 experts (for profiling)"),
    # the Switch-style layer with quantised experts: INT8 runs the shared-memory widening
    # kernel (many rows per expert), INT4 the weight-streaming one
    "switch_i8": Workload("switch_i8", T=8192, d=1024, E=64, k=1, F=4096, kind="gelu",
                          act="bf16", cf=1.25, add_residual=True, int8=True,
                          note="Switch-style top-1 GELU layer with INT8 expert weights"),
    "switch_i4": Workload("switch_i4", T=8192, d=1024, E=64, k=1, F=4096, kind="gelu",
                          act="bf16", cf=1.25, add_residual=True, int4=True,
                          note="Switch-style top-1 GELU layer with INT4 expert weights"),
    # decode8's expert shapes in bf16 with 32 experts: small enough for multi-pass profiler captures
    "decode8_e32": Workload("decode8_e32", T=8, d=7168, E=32, k=8, F=2048, kind="swiglu",
                            act="bf16", gate_dist="uniform",
                            note="decode, 8 tokens, bf16 weights, 32 experts (for profiling)"),
    "decode1": Workload("decode1", T=1, d=7168, E=256, k=8, F=2048, kind="swiglu", act="bf16",
                        gate_dist="uniform", note="decode, 1 token"),
    "decode8": Workload("decode8", T=8, d=7168, E=256, k=8, F=2048, kind="swiglu", act="bf16",
                        gate_dist="uniform", note="decode, 8 tokens"),
    "decode64": Workload("decode64", T=64, d=7168, E=256, k=8, F=2048, kind="swiglu", act="bf16",
                         gate_dist="uniform", note="decode, 64 tokens"),
}


def get(name):
    return WORKLOADS[name]
