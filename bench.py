#!/usr/bin/env python3
"""MoE-layer forward throughput on B300: tokens/s per layer and roofline fraction.

One step = one whole forward of the layer (route -> dispatch -> expert FFNs ->
combine) over one batch of T synthetic tokens, through the C ABI. Inputs are
seeded synthetic tensors with the workload's shapes and distributions (no
dataset or trained weights are involved). Default workload: the DeepSeek-V3-shaped
layer (T=8192, d=7168, 256 routed + 1 shared SwiGLU experts with F=2048, top-8,
capacity factor 1.0), the largest configuration that fits one GPU. The same run
then reports every other named configuration (device-timed) under "configs".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--no-configs]
  python bench.py --impl reference ...   # the CPU oracle, timed as the reference arm

Prints exactly one JSON line on stdout (rank 0). With N > 1 (torchrun) every rank
runs an independent replica (weak scaling: no collective on the data path); the
reported time is the max over ranks.
"""

import argparse
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
METRIC = "MoE-layer fwd tokens/s on 1 B300; % of bf16 tensor / HBM roofline"
DEFAULT_WORKLOAD = "deepseek"
# every other configuration, reported from the same process (device-timed)
SWEEP = ["tiny", "switch", "mixtral", "deepseek_cf125", "deepseek_grouped", "deepseek_reroute",
         "decode1", "decode8", "decode64", "decode1_i8", "decode8_i8", "decode64_i8",
         "decode1_i4", "decode8_i4", "decode64_i4", "switch_i8", "switch_i4"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--flush-mib", type=int, default=256,
                    help="L2 flush buffer written between timed steps (L2 is 126 MB)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration sweep after the headline workload")
    ap.add_argument("--configs", default=",".join(SWEEP),
                    help="comma-separated workloads of the sweep")
    ap.add_argument("--sweep-steps", type=int, default=10)
    return ap.parse_args(argv)


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return FALLBACK_PEAKS, "fallback"


def host_cpu():
    """CPU model and logical core count of the machine running the oracle."""
    model = platform.processor() or "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return model, os.cpu_count()


# ---------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception as e:   # no nvidia-smi: clocks unknown
            log(f"clock sampling unavailable: {e}")
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                n += 1
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() in ("active", "1"):
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------------------------
# algorithmic cost per kernel
# ---------------------------------------------------------------------------------
def _weight_bytes(wl):
    """(bytes of one expert's W1 incl. row scales, bytes of its W2 incl. row scales)."""
    es = 2 if wl.bf16 else 4
    if wl.int8 or wl.int4:
        per = 1 if wl.int8 else 0.5
        return wl.N1 * wl.d * per + 4 * wl.N1, wl.w2_per_expert * per + 4 * wl.d
    return wl.N1 * wl.d * es, wl.w2_per_expert * es


def _base_name(name):
    # INT8 / INT4-weight kernels and the bf16 weight-streaming kernel: same algorithm
    return re.sub(r"_(q[48]t?|st)_", "_", name)


def kernel_roofline_cost(wl, name, P, touched):
    """(flops, bytes) per STEP of all launches of kernel `name`, counted the way the
    layer's roofline counts them: the FLOPs of the contraction the kernel performs, and
    the layer-level bytes it owns -- the weights of the experts with kept rows that it
    streams, W_gate, x read once, the layer output written once. Implementation buffers
    (permuted rows, hidden activations, expert outputs) are not counted."""
    es = 2 if wl.bf16 else 4
    T, d, F, E = wl.T, wl.d, wl.F, wl.E
    w1b, w2b = _weight_bytes(wl)
    name = _base_name(name)
    if name in ("grouped_gemm_gelu", "grouped_gemm_swiglu"):
        fl = 2.0 * P * d * wl.N1 + (2.0 * T * d * wl.N1 if wl.has_shared else 0.0)
        return fl, touched * w1b + (w1b if wl.has_shared else 0) + T * d * es
    if name in ("grouped_gemm_scale", "grouped_gemm_scale_h16"):
        return 2.0 * P * F * d, touched * w2b
    if name == "grouped_gemm_combine1":
        return 2.0 * P * F * d, touched * w2b + T * d * es
    if name == "grouped_gemm_f32":            # shared expert down projection
        return 2.0 * T * F * d, w2b
    if name == "grouped_gemm_shared_combine":  # shared expert down projection + combine
        return 2.0 * T * F * d, w2b + T * d * es
    if name.startswith("router") or name == "router_splitk":
        return 2.0 * T * d * E, T * d * es + d * E * 4
    if name.startswith("combine"):
        return 0.0, T * d * es
    if name == "linear_expert":
        return 2.0 * P * d * d, touched * d * d * 4 + T * d * es
    return 0.0, 0.0


def kernel_algorithmic_cost(wl, name, P, touched):
    """(flops, bytes) per STEP for all launches of kernel `name`, counting every
    buffer the kernel's algorithm must read or write (including implementation
    buffers: hidden activations, expert outputs); a finer figure than the roofline
    cost, kept to explain measured traffic."""
    es = 2 if wl.bf16 else 4
    T, d, F, E = wl.T, wl.d, wl.F, wl.E
    w1b, w2b = _weight_bytes(wl)
    name = _base_name(name)
    if name in ("grouped_gemm_gelu", "grouped_gemm_swiglu"):
        fl = 2.0 * P * d * wl.N1
        by = touched * w1b + P * d * 2 + P * F * 2
        if wl.has_shared:
            fl += 2.0 * T * d * wl.N1
            by += w1b + T * d * 2 + T * F * 2
        return fl, by
    if name == "grouped_gemm_scale":
        return 2.0 * P * F * d, touched * w2b + P * F * 2 + P * d * 4
    if name == "grouped_gemm_scale_h16":   # expert-output rows as fp16 + a byte per 32 values
        return 2.0 * P * F * d, touched * w2b + P * F * 2 + P * d * 2 + P * d // 32
    if name == "grouped_gemm_combine1":   # top-1 down projection writing the layer output
        return 2.0 * P * F * d, (touched * w2b + P * F * 2 + P * d * es
                                 + (P * d * es if wl.add_residual else 0))
    if name == "grouped_gemm_f32":        # shared expert down projection
        return 2.0 * T * F * d, w2b + T * F * 2 + T * d * 4
    if name.startswith("router_logits") or name == "router_splitk":
        return 2.0 * T * d * E, T * d * es + d * E * 4 + T * E * 4
    if name == "router_gemm_tc":          # algorithmic: the fp32 gate GEMM it computes
        return 2.0 * T * d * E, T * d * es + 3 * d * E * 2 + T * 3 * E * 4
    if name == "router_gemm_topk":        # gate GEMM + top-k in its epilogue
        return 2.0 * T * d * E, T * d * es + 3 * d * E * 2 + T * wl.k * 8
    if name == "gate_split":
        return 0.0, d * E * 4 + 3 * d * E * 2
    if name == "topk_renorm":
        return 0.0, T * E * 4 + T * wl.k * 8
    if name.startswith("combine"):
        shared = T * d * 4 if wl.has_shared else 0
        routed = P * d * 2 + P * d // 32 if name == "combine_h16" else P * d * 4
        return 0.0, routed + shared + T * d * es * (2 if wl.add_residual else 1) + T * wl.k * 4
    if name == "gather_rows":
        return 0.0, 2.0 * P * d * es + P * 4
    if name == "linear_expert":
        return 2.0 * P * d * d, E * d * d * 4 + P * d * 8
    return 0.0, 0.0


KERNEL_FILES = {
    "grouped_gemm_q8t": ["grouped_gemm_q8t.cuh", "grouped_gemm_q8.cuh", "grouped_gemm.cuh",
                         "common.cuh"],
    "grouped_gemm_q4t": ["grouped_gemm_q8t.cuh", "grouped_gemm_q8.cuh", "grouped_gemm.cuh",
                         "common.cuh"],
    "grouped_gemm_q8": ["grouped_gemm_q8.cuh", "grouped_gemm.cuh", "common.cuh"],
    "grouped_gemm_st": ["grouped_gemm_q8t.cuh", "grouped_gemm_q8.cuh", "grouped_gemm.cuh",
                        "common.cuh"],
    "grouped_gemm": ["grouped_gemm.cuh", "common.cuh"],
    "router_gemm_tc": ["grouped_gemm.cuh", "common.cuh"],
    "router_gemm_topk": ["grouped_gemm.cuh", "common.cuh"],
    "splitk_reduce": ["grouped_gemm.cuh", "common.cuh"],
    "gate_split": ["router.cuh", "common.cuh"],
    "router": ["router.cuh", "common.cuh"],
    "topk": ["router.cuh", "common.cuh"],
    "dispatch": ["dispatch.cuh", "common.cuh"],
    "gather": ["dispatch.cuh", "common.cuh"],
    "combine": ["combine.cuh", "common.cuh"],
    "linear": ["combine.cuh", "common.cuh"],
}


def kernel_sources_hash(kernel):
    """Hash of the source files that define `kernel` (by name prefix)."""
    files = next((v for k, v in KERNEL_FILES.items() if kernel.startswith(k)), None)
    if files is None:
        return None
    h = hashlib.sha256()
    for fn in files:
        with open(os.path.join(ROOT, "top_routing_expert_renorm_b300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """Per-launch DRAM bytes (read + write) from a committed ncu summary, if that
    summary was taken on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}__{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_sources_sha") != kernel_sources_hash(kernel):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def roofline_of(wl, name, launches, ms, steps, P, touched, peaks, peak_src):
    """The roofline object of kernel `name` from its per-step algorithmic cost and its
    measured CUDA-event time (ms summed over `steps` steps)."""
    fl, by = kernel_roofline_cost(wl, name, P, touched)
    t_step_s = ms / steps / 1000.0
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks["bf16_tflops"])
    if fl / (tflops * 1e12) > by / (hbm * 1e9):
        roof = {"bound": "tensor", "achieved": fl / t_step_s / 1e12, "peak": tflops,
                "unit": "TFLOP/s"}
        sus = float(peaks.get("bf16_tflops_sustained", tflops))
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["frac_of_sustained"] = roof["achieved"] / sus
    else:
        roof = {"bound": "hbm", "achieved": by / t_step_s / 1e9, "peak": hbm, "unit": "GB/s"}
        roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = recorded_traffic(name, wl.name)
    roof["kernel"] = name
    roof["launches_per_step"] = launches / steps
    roof["ms_per_step"] = ms / steps
    roof["peak_source"] = (f"{peak_src} ("
                           f"{'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'}"
                           f"; {'bf16 burst' if roof['bound'] == 'tensor' else 'copy bandwidth'})")
    roof["algorithmic_bytes_per_step"] = by
    roof["algorithmic_flops_per_step"] = fl
    fi, bi = kernel_algorithmic_cost(wl, name, P, touched)
    roof["impl_bytes_per_step"] = bi
    return roof


def layer_roofline(wl, P, touched, step_ms, peaks):
    """Roofline time of the whole layer (slower of its FLOPs at the tensor peak and its
    bytes at the copy bandwidth) over the measured step time."""
    fl, by = wl.flops(P), wl.bytes(touched)
    t_fl = fl / (float(peaks["bf16_tflops"]) * 1e12)
    t_by = by / (float(peaks["hbm_gbs"]) * 1e9)
    return {"frac": max(t_fl, t_by) / (step_ms / 1000.0), "bound": "tensor" if t_fl > t_by else "hbm",
            "roofline_ms": 1000.0 * max(t_fl, t_by), "flops": fl, "bytes": by}


# ---------------------------------------------------------------------------------
# CPU baseline (the oracle, as it stands, single-threaded)
# ---------------------------------------------------------------------------------
def cpu_oracle_sample(wl, route_budget_s, ffn_budget_s, seed=0):
    """Time the oracle on a bounded sample of the workload: gate logits + top-k +
    dispatch for seeded tokens until `route_budget_s` is spent (all T tokens if they fit;
    the dispatch then ranks that sample's assignments at the layer's capacity), and the
    expert FFNs + combine of further seeded tokens until `ffn_budget_s` is spent (at least
    one). Expert weights are regenerated outside the timed parts. Returns
    (tokens_per_s, seconds_timed, description)."""
    import numpy as np
    import oracle as orc
    rng = np.random.default_rng(seed)
    order = rng.permutation(wl.T)
    Wg, gb = wl.wg_host(), wl.gate_bias_host()
    cap = orc.capacity(np.float32(wl.cf), wl.T, wl.k, wl.E)
    # ---- routing + dispatch on a token sample (chunks until the budget is spent) ----
    chunk = max(1, min(wl.T, 512, int(3e7 / (wl.d * wl.E))))   # first chunk: well under 1 s
    S_r, t_route, Ls = 0, 0.0, []
    while S_r < wl.T and (S_r == 0 or t_route < route_budget_s):
        rows = np.sort(order[S_r:S_r + chunk])
        xr = wl.x_host(rows)
        t0 = time.perf_counter()
        L = orc.gate_logits(xr, Wg, gb)
        t_route += time.perf_counter() - t0
        Ls.append(L)
        S_r += len(rows)
        if t_route > 0 and S_r < wl.T and S_r == len(rows):   # size later chunks to the rate
            chunk = max(1, int(S_r * 0.25 * route_budget_s / t_route))
    L = np.concatenate(Ls)
    t0 = time.perf_counter()
    idx, w = orc.topk_renorm(L, wl.k, wl.n_group, wl.topk_group)
    if wl.overflow == "reroute":
        cand = orc.rank_candidates(L, wl.k, wl.k, wl.n_group, wl.topk_group)
        counts, offsets, pt, ps, sd, idx2 = orc.dispatch_reroute(idx, cand, wl.E, cap)
    else:
        counts, offsets, pt, ps, sd = orc.dispatch(idx, wl.E, cap)
        idx2 = idx
    t_route += time.perf_counter() - t0

    # ---- expert FFNs + combine, one token at a time until the budget is spent ----
    def expert_fn(e, shared=False):
        w1, b1, w2, b2 = (wl.w1_host(e, shared), wl.b1_host(e, shared), wl.w2_host(e, shared),
                          wl.b2_host(e, shared))
        if wl.int8:
            q1, s1 = orc.quantize_rows_i8(w1)
            q2, s2 = orc.quantize_rows_i8(w2)
            return lambda xr: orc.expert_row_q8(wl.kind_code, xr, q1, s1, b1, q2, s2, b2, wl.d, wl.F)
        if wl.int4:
            p1, s1 = orc.quantize_rows_i4(w1)
            p2, s2 = orc.quantize_rows_i4(w2)
            q1, q2 = orc.unpack_i4(p1), orc.unpack_i4(p2)
            return lambda xr: orc.expert_row_q8(wl.kind_code, xr, q1, s1, b1, q2, s2, b2, wl.d, wl.F)
        return lambda xr: orc.expert_row(wl.kind_code, xr, w1, b1, w2, b2, wl.d, wl.F)

    shared = expert_fn(0, True) if wl.has_shared else None
    cache = {}
    S_f, t_ffn = 0, 0.0
    while S_f < S_r and (S_f == 0 or t_ffn < ffn_budget_s):
        i = S_f
        t = int(order[i])
        xr = np.ascontiguousarray(wl.x_host([t])[0])
        kept = (sd[i] >= 0).astype(np.int32)
        need = [int(idx2[i, j]) for j in range(wl.k) if kept[j]]
        if len(cache) > 16:
            cache.clear()
        for e in need:
            if e not in cache:
                cache[e] = expert_fn(e)
        t0 = time.perf_counter()
        ys = np.zeros((wl.k, wl.d))
        for j in range(wl.k):
            if kept[j]:
                ys[j] = cache[int(idx2[i, j])](xr)
        ysh = shared(xr) if shared else None
        orc.combine_row(xr, wl.add_residual, w[i], kept, ys, ysh,
                        orc.BF16 if wl.bf16 else orc.F32,
                        overflow_to_shared=wl.overflow == "shared")
        t_ffn += time.perf_counter() - t0
        S_f += 1
    per_token = t_route / S_r + t_ffn / S_f
    part = f"all {wl.T}" if S_r == wl.T else f"a seeded sample of {S_r} of the {wl.T}"
    desc = (f"gate logits + top-k + dispatch of {part} tokens ({t_route:.2f} s; the dispatch at the "
            f"layer's capacity {cap}) + expert FFNs and combine of {S_f} of those tokens "
            f"({t_ffn:.2f} s); tokens/s = 1/(t_route/{S_r} + t_ffn/{S_f}); single-threaded")
    return 1.0 / per_token, t_route + t_ffn, desc


# ---------------------------------------------------------------------------------
# reference arm: the oracle timed as the reference implementation
# ---------------------------------------------------------------------------------
L2_BYTES = 126 * 10 ** 6


def streams_past_l2(wl):
    """True when one forward streams at least four times the L2 (126 MB) through it -- the
    expert weights of the experts that can hold rows, W_gate, x and out -- so that the
    weights a step reads are not left in L2 by the step before it; the timed steps then
    run back to back. Otherwise a buffer larger than L2 is written between steps."""
    return wl.bytes(min(wl.E, wl.T * wl.k)) >= 4 * L2_BYTES


def l2_policy(wl, flush_mib):
    if streams_past_l2(wl):
        return (f"not flushed: each forward streams {wl.bytes(min(wl.E, wl.T * wl.k)) / 1e9:.2f} GB, "
                "over 4x the 126 MB L2")
    return f"flushed between timed steps ({flush_mib} MiB write)"


def workload_config(wl, world, flush_mib):
    """`config` of the line: the workload only, identical on both arms."""
    return {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "top_k": wl.k, "F": wl.F,
            "kind": wl.kind, "capacity_factor": wl.cf, "shared_expert": wl.has_shared,
            "residual": wl.add_residual,
            "expert_groups": [wl.n_group, wl.topk_group] if wl.n_group else None,
            "expert_weights": ("int8 codes + fp32 row scales" if wl.int8 else
                               "int4 codes (2 per byte) + fp32 row scales" if wl.int4 else "bf16"),
            "overflow": wl.overflow,
            "l2": l2_policy(wl, flush_mib),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    vals = []
    descs = None
    for i in range(args.warmup + args.steps):
        v, secs, desc = cpu_oracle_sample(wl, 1.0, 1.0, seed=i)
        if i >= args.warmup:
            vals.append((v, secs))
            descs = desc
    total_tokens = sum(v * s for v, s in vals)   # token-equivalents processed
    total_s = sum(s for _, s in vals)
    value = total_tokens / total_s
    model, ncpu = host_cpu()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total_s / max(1, len(vals)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, int(os.environ.get("WORLD_SIZE", "1")), args.flush_mib),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": descs, "host_cpu": model, "host_nproc": ncpu},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------
def max_over_ranks(ms, world, device):
    """The job's time is the slowest replica's: MAX all-reduce over the ranks (a no-op on
    one rank). `device` is where the process group's backend keeps its tensors."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(T, steps, world, total_ms):
    """Whole-job throughput: every replica processes T tokens per step (weak scaling)."""
    return T * steps * world / (total_ms / 1000.0)


def build_layer(wl, dev):
    """Device inputs and the MoELayer of workload `wl` (bf16 originals of quantised
    experts are released once the layer holds their codes)."""
    import torch
    import top_routing_expert_renorm_b300 as moe
    inp = wl.device_inputs(dev)
    cfg = moe.config_for(wl)
    layer = moe.MoELayer(cfg, inp["wg"], inp["gate_bias"], inp["w1"], inp["b1"], inp["w2"],
                         inp["b2"], inp["shared"])
    if wl.int8 or wl.int4:
        inp["w1"] = inp["w2"] = inp["shared"] = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return inp, cfg, layer


def measure(wl, layer, x, steps, warmup, flush, world, dev, clocks=None, barrier=None):
    """Device-timed forwards: `warmup` untimed, then `steps` timed (CUDA events on the
    launch stream around each step; L2 flushed before each unless a forward streams
    several times the L2, see streams_past_l2), then the same steps again with an event
    pair around every launch for the per-kernel breakdown."""
    import numpy as np
    import torch
    import top_routing_expert_renorm_b300 as moe
    stream = torch.cuda.current_stream()
    out = torch.empty_like(x)
    load = torch.empty(wl.E, dtype=torch.int32, device=dev)

    do_flush = not streams_past_l2(wl)

    def step():
        layer(x, out=out, load=load)

    for _ in range(max(warmup, 3)):
        step()
    torch.cuda.synchronize()
    st = moe.last_device_status()
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after warm-up: {moe.status_string(st)}")
    ld = load.cpu().numpy()
    cap = moe.capacity(layer.cfg)
    P = int(np.minimum(ld, cap).sum())
    touched = int((np.minimum(ld, cap) > 0).sum())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    n_launch0 = moe.kernel_launch_count()
    for i in range(steps):
        if do_flush:
            flush.zero_()                  # L2 flush between timed steps (not timed)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    n_launch = moe.kernel_launch_count() - n_launch0
    # Per-kernel durations: the same steps again with an event pair around every launch
    # (events between launches serialise kernels that may otherwise overlap their
    # neighbours' start and end, so this pass is not the timed one).
    moe.profile_begin()
    for i in range(steps):
        if do_flush:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    kstats = moe.profile_end()
    if barrier:
        barrier()
    clk = clocks.stop() if clocks else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    st = moe.last_device_status()
    if st != 0:
        raise RuntimeError(f"{wl.name}: device status after timing: {moe.status_string(st)}")
    return dict(total_ms=total_ms, step_ms=step_ms, kstats=kstats, P=P, touched=touched,
                n_launch=n_launch, clocks=clk, out=out)


def dominant(kstats, wl):
    """The kernel with the most time per step among those with a roofline cost."""
    ranked = sorted(kstats.items(), key=lambda kv: -kv[1][1])
    for name, (launches, ms) in ranked:
        fl, by = kernel_roofline_cost(wl, name, 1, 1)
        if fl > 0 or by > 0:
            return name, launches, ms
    name, (launches, ms) = ranked[0]
    return name, launches, ms


def sweep(args, dev, flush, peaks, peak_src):
    """Every configuration of the sweep, device-timed in this process."""
    import torch
    from synth import get
    res = {}
    for name in [n for n in args.configs.split(",") if n and n != args.workload]:
        try:
            wl = get(name)
            inp, cfg, layer = build_layer(wl, dev)
            m = measure(wl, layer, inp["x"], args.sweep_steps, 3, flush, 1, dev)
            K = args.sweep_steps
            dname, dl, dms = dominant(m["kstats"], wl)
            roof = roofline_of(wl, dname, dl, dms, K, m["P"], m["touched"], peaks, peak_src)
            lay = layer_roofline(wl, m["P"], m["touched"], m["total_ms"] / K, peaks)
            res[name] = {
                "tokens_per_s": job_tokens_per_s(wl.T, K, 1, m["total_ms"]),
                "ms_per_step": m["total_ms"] / K,
                "layer_roofline_frac": lay["frac"], "layer_bound": lay["bound"],
                "kept_rows_P": m["P"], "touched_experts": m["touched"],
                "dominant_kernel": dname, "dominant_bound": roof["bound"],
                "dominant_achieved": roof["achieved"], "dominant_unit": roof["unit"],
                "dominant_frac": roof["frac"],
                "launches_per_step": m["n_launch"] / K,
                "kernels_ms_per_step": {k: v[1] / K for k, v in
                                        sorted(m["kstats"].items(), key=lambda kv: -kv[1][1])},
            }
            del inp, layer, m
        except Exception as e:   # a failed configuration must not hide the headline line
            res[name] = {"error": f"{type(e).__name__}: {e}"}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    import __graft_entry__
    __graft_entry__.build()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    flush = torch.empty(args.flush_mib * 2 ** 20 // 4, dtype=torch.float32, device=dev)
    peaks, peak_src = load_peaks()

    inp, cfg, layer = build_layer(wl, dev)
    x = inp["x"]
    K = args.steps
    m = measure(wl, layer, x, K, args.warmup, flush, world, dev,
                clocks=ClockSampler(torch.cuda.current_device()),
                barrier=(dist.barrier if world > 1 else None))
    total_ms, kstats, P, touched = m["total_ms"], m["kstats"], m["P"], m["touched"]
    value = job_tokens_per_s(wl.T, K, world, total_ms)
    dname, dlaunch, dms = dominant(kstats, wl)
    roof = roofline_of(wl, dname, dlaunch, dms, K, P, touched, peaks, peak_src)
    lay = layer_roofline(wl, P, touched, total_ms / K, peaks)
    out = m["out"]
    n_launch, clk = m["n_launch"], m["clocks"]

    # ---- end to end through the public API with host buffers ----
    # Every step copies its input x from pinned host memory and its output back to pinned
    # host memory. Copies run on their own streams with double-buffered device tensors,
    # so step i+1's upload and step i-1's download overlap step i's forward. The timed
    # region runs from before the first upload to after the last download. The weights a
    # step streams are larger than L2, so no flush is inserted here.
    e2e = None
    if not args.no_e2e:
        xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        xh.copy_(x)
        oh = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
        xd = [torch.empty_like(x) for _ in range(2)]
        od = [torch.empty_like(out) for _ in range(2)]
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        # the forward of each buffer pair, captured once into a CUDA graph (one host-side
        # launch per step: the public MoELayer.capture API for fixed-shape serving)
        graphs = [layer.capture(xd[b], od[b]) for b in range(2)]

        def pipelined(n):
            ev = lambda: torch.cuda.Event()  # noqa: E731
            h2d, fw, d2h = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
            for i in range(n):
                b = i % 2
                with torch.cuda.stream(up):
                    if i >= 2:
                        up.wait_event(fw[i - 2])          # xd[b] was read by step i-2
                    xd[b].copy_(xh, non_blocking=True)
                    h2d[i].record(up)
                stream.wait_event(h2d[i])
                if i >= 2:
                    stream.wait_event(d2h[i - 2])         # od[b] was downloaded by step i-2
                graphs[b].replay()
                fw[i].record(stream)
                with torch.cuda.stream(down):
                    down.wait_event(fw[i])
                    oh[b].copy_(od[b], non_blocking=True)
                    d2h[i].record(down)

        pipelined(max(args.warmup, 3))
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(up)
        pipelined(K)
        t1.record(down)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
        nb = x.numel() * x.element_size()
        e2e = {"value": job_tokens_per_s(wl.T, K, world, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": nb, "d2h_bytes_per_step": out.numel() * out.element_size(),
               "overlap": "uploads/downloads on their own streams, double-buffered",
               "launch": "MoELayer.capture CUDA graph per buffer pair, replayed every step"}
        del graphs, xd, od, xh, oh
    del inp, layer, x, out, m
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    configs = None
    if rank == 0 and world == 1 and not args.no_configs:
        configs = sweep(args, dev, flush, peaks, peak_src)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, secs, desc = cpu_oracle_sample(wl, 4.0, 8.0)
        model, ncpu = host_cpu()
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": desc, "seconds": secs, "host_cpu": model, "host_nproc": ncpu}

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.bf16 else "f32",
        "data": "synthetic (seeded counter-based generator; random-init weights)",
        "config": workload_config(wl, world, args.flush_mib),
        "run": {"kept_rows_P": P, "touched_experts": touched},
        "roofline": roof,
        "layer_roofline_frac": lay["frac"],
        "layer_roofline": lay,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "clocks": clk,
        "kernels_ms_per_step": {k: v[1] / K for k, v in sorted(kstats.items(),
                                                                key=lambda kv: -kv[1][1])},
        "configs": configs,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    from synth import get
    wl = get(args.workload)
    if args.impl == "reference":
        return run_reference(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
