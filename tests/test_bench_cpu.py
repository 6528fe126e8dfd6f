"""The benchmark's cost accounting (CPU only): the algorithmic FLOPs and bytes behind every
roofline fraction, checked against totals worked out by hand from the layer's shapes.

Per forward: FLOPs = 2*T*d*E (gate GEMM) + 2*P*m*d*F (kept rows through the experts; m = 2
for GELU, 3 for SwiGLU) + the shared expert on all T tokens; bytes = weights of the experts
that received a kept row + W_gate (fp32) + x read + out written."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from synth import get  # noqa: E402


@pytest.mark.parametrize("name,P,touched,flops,nbytes", [
    # T=8192, d=1024, E=64, k=1, GELU F=4096: 1.07e9 router + 1.374e11 experts;
    # 64 * 2 * 4096 * 1024 * 2 B of weights + 256 KiB W_gate + 2 * 16 MiB of x / out
    ("switch", 8192, 64, 1.385e11, 1.108e9),
    # T=4096, d=4096, E=8, k=2, SwiGLU F=14336, no capacity: P = T * k
    ("mixtral", 8192, 8, 2.887e12, 2.886e9),
    # T=8192, d=7168, E=256 (+1 shared), k=8, SwiGLU F=2048, all experts touched
    ("deepseek", 65536, 256, 6.524e12, 2.288e10),
])
def test_layer_totals(name, P, touched, flops, nbytes):
    wl = get(name)
    assert wl.flops(P) == pytest.approx(flops, rel=1e-3)
    assert wl.bytes(touched) == pytest.approx(nbytes, rel=1e-3)


@pytest.mark.parametrize("touched,nbytes", [(8, 0.712e9), (57.4, 5.07e9), (222.4, 19.6e9)])
def test_decode_bytes_at_expected_touched_experts(touched, nbytes):
    # decode, T in {1, 8, 64}: expected distinct experts 8, 57.4 and 222.4 of 256
    assert get("decode8").bytes(touched) == pytest.approx(nbytes, rel=3e-3)


def test_quantised_weight_bytes():
    bf, i8, i4 = get("decode8"), get("decode8_i8"), get("decode8_i4")
    n_w = bf.N1 * bf.d + bf.d * bf.F               # weights of one expert
    scales = 4 * (bf.N1 + bf.d)                    # one fp32 scale per weight row
    assert bf.bytes(1) - bf.bytes(0) == 2 * n_w
    assert i8.bytes(1) - i8.bytes(0) == n_w + scales
    assert i4.bytes(1) - i4.bytes(0) == n_w // 2 + scales
    assert i4.bytes(0) == i8.bytes(0) == bf.bytes(0)   # W_gate, x, out do not change


@pytest.mark.parametrize("name", ["switch", "mixtral", "deepseek", "decode64"])
def test_kernel_costs_add_up_to_the_layer_flops(name):
    wl = get(name)
    P, touched = wl.T * wl.k, min(wl.E, wl.T * wl.k)
    up = "grouped_gemm_gelu" if wl.kind == "gelu" else "grouped_gemm_swiglu"
    down = "grouped_gemm_combine1" if (wl.k == 1 and not wl.has_shared) else "grouped_gemm_scale"
    fl = sum(bench.kernel_algorithmic_cost(wl, n, P, touched)[0]
             for n in ("router_gemm_topk", up, down))
    if wl.has_shared:
        fl += bench.kernel_algorithmic_cost(wl, "grouped_gemm_f32", P, touched)[0]
    assert fl == pytest.approx(wl.flops(P), rel=1e-12)


@pytest.mark.parametrize("quant,bytes_per_weight", [("q8t", 1.0), ("q4t", 0.5)])
def test_quantised_kernels_count_their_code_bytes(quant, bytes_per_weight):
    bf = get("decode64")
    wq = get("decode64_i8" if quant == "q8t" else "decode64_i4")
    P, touched = 512, 222
    for kind, rows in (("swiglu", bf.N1 * bf.d), ("scale", bf.d * bf.F)):
        fl_b, by_b = bench.kernel_algorithmic_cost(bf, f"grouped_gemm_{kind}", P, touched)
        fl_q, by_q = bench.kernel_algorithmic_cost(wq, f"grouped_gemm_{quant}_{kind}", P, touched)
        scales = 4 * (bf.N1 if kind == "swiglu" else bf.d)
        assert fl_q == fl_b
        assert by_q == pytest.approx(by_b - touched * rows * (2 - bytes_per_weight) + touched * scales)


def test_roofline_bytes_follow_the_layer_terms():
    # Switch-style top-1 GELU layer: the up projection owns W1 of the 64 touched experts
    # (64 * 4096 * 1024 * 2 B = 536.9 MB) and the read of x (8192 * 1024 * 2 B = 16.8 MB);
    # hidden activations are an implementation buffer and are not counted
    wl = get("switch")
    fl, by = bench.kernel_roofline_cost(wl, "grouped_gemm_gelu", 8184, 64)
    assert by == 64 * 4096 * 1024 * 2 + 8192 * 1024 * 2
    assert fl == 2.0 * 8184 * 1024 * 4096
    # the fused top-1 down projection also writes the layer output once
    _, by_d = bench.kernel_roofline_cost(wl, "grouped_gemm_combine1", 8184, 64)
    assert by_d == 64 * 1024 * 4096 * 2 + 8192 * 1024 * 2


@pytest.mark.parametrize("name", ["switch", "deepseek", "mixtral", "decode64_i4"])
def test_roofline_terms_of_the_kernels_add_up_to_the_layer(name):
    # weights + W_gate + x + out over router, up, down (and combine) = the layer's bytes,
    # except that the router and the up projection each must read x once
    wl = get(name)
    P, touched = wl.T * wl.k, min(wl.E, wl.T * wl.k)
    up = "grouped_gemm_gelu" if wl.kind == "gelu" else "grouped_gemm_swiglu"
    fused = wl.k == 1 and not wl.has_shared
    names = ["router_gemm_topk", up, "grouped_gemm_combine1" if fused else "grouped_gemm_scale"]
    if wl.has_shared:
        names.append("grouped_gemm_f32")
    if not fused:
        names.append("combine_bf16")
    by = sum(bench.kernel_roofline_cost(wl, n, P, touched)[1] for n in names)
    fl = sum(bench.kernel_roofline_cost(wl, n, P, touched)[0] for n in names)
    es = 2 if wl.bf16 else 4
    assert by - wl.T * wl.d * es == pytest.approx(wl.bytes(touched), rel=1e-12)
    assert fl == pytest.approx(wl.flops(P), rel=1e-12)


def test_compact_expert_rows_cost_the_same_roofline_and_fewer_bytes():
    # the down projection and combine that keep expert-output rows as fp16 with one scale
    # byte per 32 values own the same layer-level terms; their algorithmic traffic drops by
    # P * d * (4 - 2 - 1/32) bytes each
    wl = get("deepseek")
    P, touched = wl.T * wl.k, wl.E
    for a, b in (("grouped_gemm_scale", "grouped_gemm_scale_h16"), ("combine_bf16", "combine_h16")):
        assert bench.kernel_roofline_cost(wl, a, P, touched) == bench.kernel_roofline_cost(wl, b, P, touched)
        fa, ba = bench.kernel_algorithmic_cost(wl, a, P, touched)
        fb, bb = bench.kernel_algorithmic_cost(wl, b, P, touched)
        assert fa == fb and ba - bb == P * wl.d * 2 - P * wl.d // 32


def test_weight_streaming_kernels_cost_like_their_algorithm():
    # the bf16 weight-streaming kernel (decode) and the INT8 / INT4 ones are costed as the
    # projection they compute; their source hash covers the weight-streaming kernel's files
    wl = get("decode8")
    P, touched = 64, 61
    for name in ("grouped_gemm_st_swiglu", "grouped_gemm_st_scale"):
        base = name.replace("_st_", "_")
        assert bench._base_name(name) == base
        assert bench.kernel_roofline_cost(wl, name, P, touched) == bench.kernel_roofline_cost(wl, base, P, touched)
        assert bench.kernel_algorithmic_cost(wl, name, P, touched) == bench.kernel_algorithmic_cost(wl, base, P, touched)
    assert "grouped_gemm_q8t.cuh" in next(v for k, v in bench.KERNEL_FILES.items()
                                           if "grouped_gemm_st_swiglu".startswith(k))
    assert bench.kernel_sources_hash("grouped_gemm_st_swiglu") != bench.kernel_sources_hash("grouped_gemm_swiglu")


def test_l2_is_flushed_unless_a_forward_streams_several_times_the_l2():
    # the tiny layer and the small quantised decode layers fit (or nearly fit) in the
    # 126 MB L2: a buffer larger than L2 is written between their timed steps; layers
    # streaming over 4x the L2 per forward run back to back, and config says which
    assert not bench.streams_past_l2(get("tiny"))
    assert "flushed" in bench.workload_config(get("tiny"), 1, 256)["l2"]
    assert not bench.streams_past_l2(get("decode1_i4"))
    for n in ("deepseek", "switch", "mixtral", "decode1", "decode64"):
        wl = get(n)
        assert bench.streams_past_l2(wl)
        assert wl.bytes(min(wl.E, wl.T * wl.k)) >= 4 * 126e6
        assert bench.workload_config(wl, 1, 256)["l2"].startswith("not flushed")


def test_both_arms_report_the_same_config():
    wl = get("deepseek")
    a = bench.workload_config(wl, 1, 256)
    b = bench.workload_config(wl, 1, 256)
    assert a == b and a["workload"] == "deepseek" and "l2" in a
    for k in ("kept_rows_P", "touched_experts"):     # run-derived values stay out of config
        assert k not in a


def test_default_workload_is_the_largest_single_gpu_layer():
    args = bench.parse([])
    assert args.workload == "deepseek"
    assert get(args.workload).flops(get(args.workload).T * get(args.workload).k) == max(
        get(n).flops(get(n).T * get(n).k) for n in bench.SWEEP + ["deepseek"])


def test_cpu_oracle_sample_is_bounded_and_positive():
    v, secs, desc = bench.cpu_oracle_sample(get("tiny"), 0.5, 0.5)
    assert v > 0 and secs < 5
    assert "all 64 tokens" in desc
