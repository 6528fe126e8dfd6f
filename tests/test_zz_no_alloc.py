"""moe_dispatch_noalloc: dispatch for callers that cannot allocate device memory.

Some callers of this library cannot call cudaMalloc when they run the layer — for
example a plugin hosted by a framework that owns every device buffer and gives
the plugin no allocator, or a latency-critical loop that must not take
cudaMalloc's implicit device synchronisation. For them moe_dispatch_noalloc keeps
its scratch tables in a fixed static device array inside the library instead of
a caller workspace. This file checks, through the C ABI, that it produces exactly
what moe_dispatch produces, on several calls in a row (the array keeps the last
call's contents, so later calls must not depend on it). The file name sorts last
so that a run stopping at the first failure has already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import top_routing_expert_renorm_b300 as moe
from top_routing_expert_renorm_b300 import _capi as C
from synth import Workload

pytestmark = pytest.mark.gpu


def _buffers(wl, dev="cuda"):
    T, k, E, d = wl.T, wl.k, wl.E, wl.d
    i32 = dict(dtype=torch.int32, device=dev)
    dt = torch.bfloat16 if wl.bf16 else torch.float32
    return dict(load=torch.full((E,), -1, **i32), counts=torch.full((E,), -1, **i32),
                offsets=torch.full((E + 1,), -1, **i32),
                perm_token=torch.full((T * k,), -1, **i32),
                perm_slot=torch.full((T * k,), -1, **i32),
                slot_dest=torch.full((T, k), -9, **i32),
                x_perm=torch.zeros(T * k, d, dtype=dt, device=dev))


def _route(wl):
    inp = wl.device_inputs("cuda")
    cfg = moe.config_for(wl)
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, wl.k, dtype=torch.float32, device="cuda")
    moe.route(cfg, inp["x"], inp["wg"], inp["gate_bias"], None, idx, w, ws)
    return cfg, inp["x"], idx, ws


def _same(a, b, P):
    for key in ("load", "counts", "offsets", "slot_dest"):
        assert torch.equal(a[key], b[key]), key
    for key in ("perm_token", "perm_slot", "x_perm"):
        assert torch.equal(a[key][:P], b[key][:P]), key


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_noalloc_dispatch_matches_workspace_dispatch_on_consecutive_calls():
    cases = [
        Workload("na_a", T=1000, d=128, E=4, k=1, F=128, kind="gelu", act="bf16", cf=1.25),
        Workload("na_b", T=3000, d=256, E=64, k=8, F=128, kind="swiglu", act="bf16", cf=1.0,
                 gate_bias="zipf"),
        Workload("na_c", T=96, d=16, E=5, k=2, F=16, kind="linear", act="f32", cf=0.75),
        # more assignments and experts than one CTA dispatches: the per-chunk count and
        # rank-base tables live in the static array
        Workload("na_d", T=9000, d=64, E=512, k=8, F=64, kind="gelu", act="bf16", cf=1.0),
    ]
    routed = [(_route(wl), wl) for wl in cases]
    # a, b, c, then a again: each call runs over what the previous one left behind
    for (cfg, x, idx, ws), wl in routed + routed[:1]:
        ref = _buffers(wl)
        moe.dispatch(cfg, idx, x, ref["load"], ref["counts"], ref["offsets"], ref["perm_token"],
                     ref["perm_slot"], ref["slot_dest"], ref["x_perm"], ws)
        got = _buffers(wl)
        moe.dispatch_noalloc(cfg, idx, x, got["load"], got["counts"], got["offsets"],
                             got["perm_token"], got["perm_slot"], got["slot_dest"], got["x_perm"])
        assert moe.last_device_status() == 0
        P = int(ref["offsets"][-1].item())
        assert P > 0
        _same(got, ref, P)


def test_noalloc_dispatch_rejects_problems_beyond_its_array():
    cfg = moe.make_config(T=40000, d=64, E=1024, top_k=1, F=64, kind="gelu")
    fn = C.load().moe_dispatch_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(C.MoeConfig)] + [ctypes.c_void_p] * 10
    p = ctypes.c_void_p(1 << 20)
    n0 = moe.kernel_launch_count()
    st = fn(ctypes.byref(cfg), p, None, p, p, p, p, p, p, None, None)
    assert st == C.MOE_ERR_WORKSPACE
    assert moe.kernel_launch_count() == n0       # rejected before any launch


@pytest.mark.parametrize("T,accepted", [(32768, True), (32769, False)])
def test_noalloc_dispatch_limit_is_exact(T, accepted):
    # E = 1024: ceil(T/256) * E fits the array for T = 32768 (128 chunks) and not for one
    # token more (129 chunks)
    E = 1024
    cfg = moe.make_config(T=T, d=64, E=E, top_k=1, F=64, kind="gelu")
    g = torch.Generator(device="cpu").manual_seed(T)
    idx = torch.randint(0, E, (T, 1), dtype=torch.int32, generator=g).cuda()
    wl = Workload("na_lim", T=T, d=64, E=E, k=1, F=64, kind="gelu", act="bf16")
    got = _buffers(wl)
    if not accepted:
        with pytest.raises(moe.MoeError) as e:
            moe.dispatch_noalloc(cfg, idx, None, got["load"], got["counts"], got["offsets"],
                                 got["perm_token"], got["perm_slot"], got["slot_dest"], None)
        assert e.value.status == C.MOE_ERR_WORKSPACE
        return
    ws = torch.empty(moe.workspace_size(cfg), dtype=torch.uint8, device="cuda")
    ref = _buffers(wl)
    moe.dispatch(cfg, idx, None, ref["load"], ref["counts"], ref["offsets"], ref["perm_token"],
                 ref["perm_slot"], ref["slot_dest"], None, ws)
    moe.dispatch_noalloc(cfg, idx, None, got["load"], got["counts"], got["offsets"],
                         got["perm_token"], got["perm_slot"], got["slot_dest"], None)
    assert moe.last_device_status() == 0
    P = int(ref["offsets"][-1].item())
    assert P == T
    for key in ("load", "counts", "offsets", "slot_dest"):
        assert torch.equal(got[key], ref[key]), key
    for key in ("perm_token", "perm_slot"):
        assert torch.equal(got[key][:P], ref[key][:P]), key
