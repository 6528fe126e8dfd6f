"""C-ABI library on a machine without a GPU: it loads, exports every declared
symbol, and its host-only logic and argument validation behave as documented.
No call here launches a kernel."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle as orc
from top_routing_expert_renorm_b300 import _capi as C
from top_routing_expert_renorm_b300 import api
from top_routing_expert_renorm_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return C.load()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_no_kernel_launched_on_cpu(lib):
    assert api.kernel_launch_count() == 0


@pytest.mark.parametrize("T,k,E,cf", [(8192, 1, 64, 1.25), (8192, 8, 256, 1.0),
                                      (8192, 8, 256, 1.25), (64, 2, 4, 0.625), (100, 3, 7, 0.0),
                                      (10, 1, 3, 1.0), (10, 2, 4, 100.0), (10, 1, 3, 1e-9),
                                      (4096, 2, 8, -1.0), (1, 8, 256, 1.0)])
def test_capacity_matches_oracle(lib, T, k, E, cf):
    cfg = api.make_config(T, 64, E, k, 64, cf, "gelu", True)
    assert api.capacity(cfg) == orc.capacity(np.float32(cf), T, k, E)


def test_load_report_matches_oracle(lib, golden):
    g = golden("eplb_adv12.json")
    assign, dev, imb = api.load_report(np.array(g["loads"], np.int32), g["devices"])
    assert assign.tolist() == g["lpt_assignment"]
    assert dev.tolist() == g["lpt_device_load"]
    assert round(imb, 3) == g["imbalance_3dp"]
    rng = np.random.default_rng(0)
    for _ in range(20):
        E, D = int(rng.integers(1, 40)), int(rng.integers(1, 9))
        loads = rng.integers(0, 100, E).astype(np.int32)
        a, dv, im = api.load_report(loads, D)
        r = orc.load_report(loads, D)
        assert a.tolist() == r["assign"].tolist() and dv.tolist() == r["dev_load"].tolist()
        assert im == r["imbalance"]


def test_workspace_and_rows(lib):
    cfg = api.make_config(8192, 7168, 256, 8, 2048, 1.0, "swiglu", True, has_shared=True)
    ws = api.workspace_size(cfg)
    assert api.max_rows(cfg) == 8192 * 8
    # x_perm + H (routed rows, then room for the shared expert's when the forward runs it as
    # an extra group) + y (routed + shared rows) + the staged path's shared H + the router's
    # partial logits (three bf16 terms of 256 experts) dominate
    P = 8192 * 8
    big = (P * 7168 * 2 + (P + 8192) * 2048 * 2 + (P + 8192) * 7168 * 4 + 8192 * 2048 * 2
           + 3 * 256 * 8192 * 4)
    assert ws >= big
    assert ws < 1.01 * (big + 64 * 2 ** 20)


@pytest.mark.parametrize("bad", [
    dict(top_k=0), dict(top_k=5, E=4), dict(E=0), dict(E=1025), dict(d=12), dict(d=4),
    dict(T=-1), dict(top_k=33, E=64), dict(F=96), dict(F=0), dict(d=72),
    dict(T=2 ** 28, top_k=8), dict(capacity_factor=float("nan")), dict(kind=7),
    dict(act_dtype=3), dict(has_shared=2), dict(add_residual=-1),
    # group-limited routing: groups must divide E, keep 1..n_group groups, hold k experts
    dict(n_group=3, topk_group=1), dict(n_group=2, topk_group=0), dict(n_group=2, topk_group=3),
    dict(n_group=64, topk_group=1, E=64), dict(n_group=4, topk_group=1, top_k=2),
    dict(n_group=-1, topk_group=1),
    # weight dtype: the activation dtype or INT8 codes (GELU / SwiGLU experts only)
    dict(w_dtype=5), dict(w_dtype=-1),
    dict(w_dtype=C.MOE_I8, kind=C.MOE_EXPERT_LINEAR, act_dtype=C.MOE_F32),
    # overflow policy: 0..2; the dropped weight can only go to a shared expert that exists
    dict(overflow=3), dict(overflow=-1), dict(overflow=C.MOE_OVERFLOW_SHARED)])
def test_invalid_configs_rejected(lib, bad):
    base = dict(T=64, d=128, E=4, top_k=2, F=128, capacity_factor=0.0, act_dtype=C.MOE_BF16,
                kind=C.MOE_EXPERT_GELU, has_shared=0, add_residual=0)
    base.update(bad)
    cfg = C.MoeConfig(**base)
    assert api.workspace_size(cfg) == 0
    assert api.capacity(cfg) == -1
    fake = ctypes.c_void_p(1 << 20)
    st = lib.moe_route(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, fake, None)
    assert st in (C.MOE_ERR_INVALID_ARG, C.MOE_ERR_UNSUPPORTED)


def test_grouped_routing_configs_accepted(lib):
    for n_group, topk_group, E, k in ((2, 1, 4, 2), (4, 2, 4, 2), (8, 4, 256, 8), (32, 1, 32, 1)):
        cfg = api.make_config(64, 128, E, k, 128, 0.0, "gelu", True, n_group=n_group,
                              topk_group=topk_group)
        assert api.workspace_size(cfg) > 0


def test_int8_weights_need_scales(lib):
    cfg = api.make_config(64, 128, 4, 2, 128, 0.0, "swiglu", True, int8_weights=True)
    assert cfg.w_dtype == C.MOE_I8 and api.workspace_size(cfg) > 0
    ok = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 4)
    r = ctypes.byref(cfg)
    ws = 1 << 40
    w = C.MoeExpertWeights(w1=ok, b1=None, w2=ok, b2=None, s1=ok, s2=None)
    assert lib.moe_forward(r, ok, ok, None, ctypes.byref(w), None, ok, None, None, None, ok,
                           ws, None) == C.MOE_ERR_INVALID_ARG
    w = C.MoeExpertWeights(w1=ok, b1=None, w2=ok, b2=None, s1=ok, s2=bad)
    assert lib.moe_forward(r, ok, ok, None, ctypes.byref(w), None, ok, None, None, None, ok,
                           ws, None) == C.MOE_ERR_MISALIGNED
    # the quantiser's own argument checks (no launch)
    assert lib.moe_quantize_i8(ok, 4, 12, ok, ok, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_i8(ok, -1, 64, ok, ok, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_i8(None, 4, 64, ok, ok, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_i8(ok, 4, 64, bad, ok, None) == C.MOE_ERR_MISALIGNED
    assert lib.moe_quantize_i8(ok, 0, 64, ok, ok, None) == C.MOE_OK


def test_int4_weights_need_scales(lib):
    cfg = api.make_config(64, 128, 4, 2, 128, 0.0, "gelu", True, int4_weights=True)
    assert cfg.w_dtype == C.MOE_I4 and api.workspace_size(cfg) > 0
    lin = api.make_config(64, 8, 4, 2, 0, 0.0, "linear", False, int4_weights=True)
    assert api.workspace_size(lin) == 0                     # INT4 is for GELU / SwiGLU experts
    with pytest.raises(ValueError):
        api.make_config(64, 128, 4, 2, 128, int8_weights=True, int4_weights=True)
    ok = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 4)
    r = ctypes.byref(cfg)
    w = C.MoeExpertWeights(w1=ok, b1=None, w2=ok, b2=None, s1=None, s2=ok)
    assert lib.moe_forward(r, ok, ok, None, ctypes.byref(w), None, ok, None, None, None, ok,
                           1 << 40, None) == C.MOE_ERR_INVALID_ARG
    # the quantiser's own argument checks (no launch): a row of 32 codes is 16 bytes
    assert lib.moe_quantize_i4(ok, 4, 48, ok, ok, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_i4(ok, 4, 16, ok, ok, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_i4(ok, -1, 64, ok, ok, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_i4(ok, 4, 64, ok, None, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_quantize_i4(ok, 4, 64, bad, ok, None) == C.MOE_ERR_MISALIGNED
    assert lib.moe_quantize_i4(ok, 0, 64, ok, ok, None) == C.MOE_OK


def test_overflow_policies(lib):
    for ov in ("drop", "shared", "reroute"):
        cfg = api.make_config(64, 128, 8, 2, 128, 1.0, "swiglu", True, has_shared=True,
                              overflow=ov)
        assert api.workspace_size(cfg) > 0
    # re-routing keeps candidates and proposals in the workspace
    base = api.make_config(300, 128, 8, 2, 128, 1.0, "swiglu", True)
    rr = api.make_config(300, 128, 8, 2, 128, 1.0, "swiglu", True, overflow="reroute")
    assert api.workspace_size(rr) >= api.workspace_size(base) + 2 * 300 * 2 * 4
    ok = ctypes.c_void_p(1 << 20)
    # moe_dispatch_noalloc has no workspace to read the candidates from
    assert lib.moe_dispatch_noalloc(ctypes.byref(rr), ok, ok, ok, ok, ok, ok, ok, ok, None,
                                    None) == C.MOE_ERR_UNSUPPORTED
    # the shared-overflow combine needs the routing weights
    sh = api.make_config(64, 128, 8, 2, 128, 1.0, "swiglu", True, has_shared=True,
                         overflow="shared")
    # (cfg, x, y, topk_w, slot_dest, out, stream)
    assert lib.moe_combine(ctypes.byref(sh), ok, ok, None, ok, ok, None) == C.MOE_ERR_INVALID_ARG


def test_unsupported_dtype_kind_pairs(lib):
    for kind, dt in [(C.MOE_EXPERT_LINEAR, C.MOE_BF16), (C.MOE_EXPERT_GELU, C.MOE_F32),
                     (C.MOE_EXPERT_SWIGLU, C.MOE_F32)]:
        cfg = C.MoeConfig(T=8, d=64, E=2, top_k=1, F=64, capacity_factor=0.0, act_dtype=dt,
                          kind=kind, has_shared=0, add_residual=0)
        fake = ctypes.c_void_p(1 << 20)
        assert lib.moe_route(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, fake,
                             None) == C.MOE_ERR_UNSUPPORTED


def test_misaligned_and_missing_pointers(lib):
    cfg = api.make_config(64, 128, 4, 2, 128, 0.0, "gelu", True)
    ok = ctypes.c_void_p(1 << 20)
    bad = ctypes.c_void_p((1 << 20) + 8)
    r = ctypes.byref(cfg)
    assert lib.moe_route(r, bad, ok, None, ok, ok, ok, ok, None) == C.MOE_ERR_MISALIGNED
    assert lib.moe_route(r, None, ok, None, ok, ok, ok, ok, None) == C.MOE_ERR_INVALID_ARG
    assert lib.moe_route(r, ok, ok, None, None, ok, ok, None, None) == C.MOE_ERR_WORKSPACE
    assert lib.moe_combine(r, ok, ok, None, ok, bad, None) == C.MOE_ERR_MISALIGNED
    w = C.MoeExpertWeights(w1=ok, b1=None, w2=None, b2=None)   # GELU needs w2
    assert lib.moe_forward(r, ok, ok, None, ctypes.byref(w), None, ok, None, None, None, ok,
                           1 << 40, None) == C.MOE_ERR_INVALID_ARG
    w = C.MoeExpertWeights(w1=ok, b1=None, w2=ok, b2=None)
    assert lib.moe_forward(r, ok, ok, None, ctypes.byref(w), None, ok, None, None, None, ok,
                           16, None) == C.MOE_ERR_WORKSPACE
    assert lib.moe_grouped_gemm(ok, 10, ok, 2, 96, 64, ok, ok, ok, None) == C.MOE_ERR_INVALID_ARG


def test_zero_tokens_is_a_noop(lib):
    cfg = api.make_config(0, 128, 4, 2, 128, 0.0, "gelu", True)
    r = ctypes.byref(cfg)
    assert lib.moe_route(r, None, None, None, None, None, None, None, None) == C.MOE_OK
    assert lib.moe_combine(r, None, None, None, None, None, None) == C.MOE_OK
    assert api.kernel_launch_count() == 0


def test_status_strings(lib):
    for s in range(8):
        assert api.status_string(s) and api.status_string(s) != "unknown status"
