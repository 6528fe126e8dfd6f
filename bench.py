#!/usr/bin/env python3
"""MoE-layer forward throughput on B300: tokens/s per layer and roofline fraction.

One step = one whole forward of the layer (route -> dispatch -> expert FFNs ->
combine) over one batch of T synthetic tokens, through the C ABI. Inputs are
seeded synthetic tensors with the workload's shapes and distributions (no
dataset or trained weights are involved). Default workload: the Switch-style
top-1 layer (T=8192, d=1024, E=64, GELU d->4096->d, capacity factor 1.25).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed as the reference arm

Prints exactly one JSON line on stdout (rank 0). With N > 1 (torchrun) every rank
runs an independent replica (weak scaling: no collective on the data path); the
reported time is the max over ranks.
"""

import argparse
import hashlib
import json
import os
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


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="switch")
    ap.add_argument("--flush-mib", type=int, default=256,
                    help="L2 flush buffer written between timed steps (L2 is 126 MB)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return FALLBACK_PEAKS, "fallback"


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
# algorithmic cost per kernel (for the roofline object)
# ---------------------------------------------------------------------------------
def kernel_algorithmic_cost(wl, name, P, touched):
    """(flops, bytes) per STEP for all launches of kernel `name`, from the
    algorithm's sizes (not from measured traffic)."""
    es = 2 if wl.bf16 else 4
    T, d, F, E = wl.T, wl.d, wl.F, wl.E
    N1 = wl.N1
    name = re.sub(r"_q[48]t?_", "_", name)  # INT8 / INT4-weight kernels: same algorithm
    quant = wl.int8 or wl.int4
    we = 1 if wl.int8 else (0.5 if wl.int4 else 2)   # bytes per expert weight
    sc1 = 4 * N1 if quant else 0           # per-row scales of one expert
    sc2 = 4 * d if quant else 0
    up = {"grouped_gemm_gelu", "grouped_gemm_swiglu"}
    if name in up:
        fl = 2.0 * P * d * N1
        by = touched * (N1 * d * we + sc1) + P * d * 2 + P * F * 2
        if wl.has_shared:
            fl += 2.0 * T * d * N1
            by += N1 * d * we + sc1 + T * d * 2 + T * F * 2
        return fl, by
    if name == "grouped_gemm_scale":
        return 2.0 * P * F * d, touched * (d * F * we + sc2) + P * F * 2 + P * d * 4
    if name == "grouped_gemm_combine1":   # top-1 down projection writing the layer output
        return 2.0 * P * F * d, (touched * (d * F * we + sc2) + P * F * 2 + P * d * es
                                 + (P * d * es if wl.add_residual else 0))
    if name == "grouped_gemm_f32":        # shared expert down projection
        return 2.0 * T * F * d, d * F * we + sc2 + T * F * 2 + T * d * 4
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
        rows = P + (T if wl.has_shared else 0)
        return 0.0, rows * d * 4 + T * d * es * (2 if wl.add_residual else 1) + T * wl.k * 4
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


# ---------------------------------------------------------------------------------
# CPU baseline (the oracle, as it stands, single-threaded)
# ---------------------------------------------------------------------------------
def cpu_oracle_sample(wl, sample_tokens, seed=0):
    """Time the oracle on a bounded sample: full routing + dispatch over all T tokens,
    expert FFNs + combine for `sample_tokens` seeded tokens. Returns
    (tokens_per_s, seconds_total, description)."""
    import numpy as np
    import oracle as orc
    rng = np.random.default_rng(seed)
    S = min(sample_tokens, wl.T)
    rows = np.sort(rng.choice(wl.T, size=S, replace=False))
    x = wl.x_host()
    Wg, gb = wl.wg_host(), wl.gate_bias_host()
    t0 = time.perf_counter()
    L = orc.gate_logits(x, Wg, gb)
    idx, w = orc.topk_renorm(L, wl.k, wl.n_group, wl.topk_group)
    cap = orc.capacity(np.float32(wl.cf), wl.T, wl.k, wl.E)
    if wl.overflow == "reroute":
        cand = orc.rank_candidates(L, wl.k, wl.k, wl.n_group, wl.topk_group)
        counts, offsets, pt, ps, sd, idx = orc.dispatch_reroute(idx, cand, wl.E, cap)
    else:
        counts, offsets, pt, ps, sd = orc.dispatch(idx, wl.E, cap)
    t_route = time.perf_counter() - t0
    need = sorted({int(idx[t, j]) for t in rows for j in range(wl.k) if sd[t, j] >= 0})

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
    Wc = {e: expert_fn(e) for e in need}
    shared = expert_fn(0, True) if wl.has_shared else None
    t0 = time.perf_counter()
    for t in rows:
        xr = np.ascontiguousarray(x[t])
        ys = np.zeros((wl.k, wl.d))
        kept = (sd[t] >= 0).astype(np.int32)
        for j in range(wl.k):
            if kept[j]:
                ys[j] = Wc[int(idx[t, j])](xr)
        ysh = shared(xr) if shared else None
        orc.combine_row(xr, wl.add_residual, w[t], kept, ys, ysh,
                        orc.BF16 if wl.bf16 else orc.F32,
                        overflow_to_shared=wl.overflow == "shared")
    t_ffn = time.perf_counter() - t0
    per_token = t_route / wl.T + t_ffn / S
    desc = (f"routing+dispatch of all {wl.T} tokens ({t_route:.2f} s) + expert FFN and "
            f"combine of {S} seeded tokens ({t_ffn:.2f} s); tokens/s = 1/(t_route/T + t_ffn/S)")
    return 1.0 / per_token, t_route + t_ffn, desc


def default_sample(wl):
    """Sample size giving roughly 2-5 s of single-core oracle work per run."""
    m = {"linear": 1, "gelu": 2, "swiglu": 3}[wl.kind]
    per_row = 2.0 * m * wl.d * (wl.F if wl.kind != "linear" else wl.d) * (
        wl.k + (1 if wl.has_shared else 0))
    return int(max(1, min(wl.T, 3e9 / per_row)))


# ---------------------------------------------------------------------------------
# reference arm: the oracle timed as the reference implementation
# ---------------------------------------------------------------------------------
def workload_config(wl, world):
    """The workload part of `config`, the same on both arms."""
    return {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "top_k": wl.k, "F": wl.F,
            "kind": wl.kind, "capacity_factor": wl.cf, "shared_expert": wl.has_shared,
            "residual": wl.add_residual,
            "expert_groups": [wl.n_group, wl.topk_group] if wl.n_group else None,
            "expert_weights": ("int8 codes + fp32 row scales" if wl.int8 else
                               "int4 codes (2 per byte) + fp32 row scales" if wl.int4 else "bf16"),
            "overflow": wl.overflow,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_reference(args, wl):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    S = max(1, default_sample(wl) // 2)
    vals = []
    descs = None
    for i in range(args.warmup + args.steps):
        v, secs, desc = cpu_oracle_sample(wl, S, seed=i)
        if i >= args.warmup:
            vals.append((v, secs))
            descs = desc
    total_tokens = sum(v * s for v, s in vals)   # token-equivalents processed
    total_s = sum(s for _, s in vals)
    value = total_tokens / total_s
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total_s / max(1, len(vals)), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, int(os.environ.get("WORLD_SIZE", "1"))),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": descs},
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


def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    import numpy as np
    import __graft_entry__
    __graft_entry__.build()
    import top_routing_expert_renorm_b300 as moe

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()

    inp = wl.device_inputs(dev)
    cfg = moe.config_for(wl)
    layer = moe.MoELayer(cfg, inp["wg"], inp["gate_bias"], inp["w1"], inp["b1"], inp["w2"],
                         inp["b2"], inp["shared"])
    if wl.int8 or wl.int4:
        # the layer holds the INT8 / INT4 codes; the bf16 originals are no longer needed
        inp["w1"] = inp["w2"] = inp["shared"] = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    x = inp["x"]
    out = torch.empty_like(x)
    load = torch.empty(wl.E, dtype=torch.int32, device=dev)
    flush = torch.empty(args.flush_mib * 2 ** 20 // 4, dtype=torch.float32, device=dev)

    def step():
        layer(x, out=out, load=load)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    st = moe.last_device_status()
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {moe.status_string(st)}")
    ld = load.cpu().numpy()
    cap = moe.capacity(cfg)
    P = int(np.minimum(ld, cap).sum())
    touched = int((np.minimum(ld, cap) > 0).sum())

    # ---- timed region ----
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n_launch0 = moe.kernel_launch_count()
    for i in range(K):
        flush.zero_()                      # L2 flush between timed steps (not timed)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    n_launch = moe.kernel_launch_count() - n_launch0
    # Per-kernel durations: the same K steps again with an event pair around every
    # launch (events between launches serialise kernels that may otherwise overlap
    # their neighbours' start and end, so this pass is not the timed one).
    moe.profile_begin()
    for i in range(K):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    kstats = moe.profile_end()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    st = moe.last_device_status()
    if st != 0:
        raise RuntimeError(f"device status after timing: {moe.status_string(st)}")
    value = job_tokens_per_s(wl.T, K, world, total_ms)

    # ---- roofline of the dominant kernel ----
    peaks, peak_src = load_peaks()
    dom = max(kstats.items(), key=lambda kv: kv[1][1])
    dname, (dlaunch, dms) = dom
    fl, by = kernel_algorithmic_cost(wl, dname, P, touched)
    t_step_s = dms / K / 1000.0
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks["bf16_tflops"])
    if fl / (tflops * 1e12) > by / (hbm * 1e9):
        roof = {"bound": "tensor", "achieved": fl / t_step_s / 1e12, "peak": tflops,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": by / t_step_s / 1e9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    tr = recorded_traffic(dname, wl.name)
    roof["traffic"] = tr
    roof["kernel"] = dname
    roof["launches_per_step"] = dlaunch / K
    roof["peak_source"] = f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
    roof["algorithmic_bytes_per_step"] = by
    roof["algorithmic_flops_per_step"] = fl
    # whole-layer roofline (slower of FLOPs at tensor peak and bytes at HBM peak)
    lay_fl = wl.flops(P)
    lay_by = wl.bytes(touched)
    layer_roof_s = max(lay_fl / (tflops * 1e12), lay_by / (hbm * 1e9))
    layer_frac = layer_roof_s / (total_ms / K / 1000.0)

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

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, secs, desc = cpu_oracle_sample(wl, default_sample(wl))
        cpu = {"value": v, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": desc, "seconds": secs}

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
        "config": {**workload_config(wl, world),
                   "l2": f"flushed between steps ({args.flush_mib} MiB write)",
                   "kept_rows_P": P, "touched_experts": touched},
        "roofline": roof,
        "layer_roofline_frac": layer_frac,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "clocks": clk,
        "kernels_ms_per_step": {k: v[1] / K for k, v in sorted(kstats.items(),
                                                                key=lambda kv: -kv[1][1])},
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
