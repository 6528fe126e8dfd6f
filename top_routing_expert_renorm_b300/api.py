"""Python binding of the MoE layer C ABI: argument marshalling only.

Every step of the layer runs in libmoe.so's CUDA kernels. torch is used for
device memory and streams: tensors are passed by data pointer, the stream is
torch's current stream unless one is given.
"""

import ctypes

from . import _capi as C
from ._capi import MoeConfig, MoeExpertWeights


class MoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = C.load().moe_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def _check(status, where):
    if status != C.MOE_OK:
        raise MoeError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_contiguous():
        raise ValueError("tensors passed to the MoE library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


OVERFLOW = {"drop": C.MOE_OVERFLOW_DROP, "shared": C.MOE_OVERFLOW_SHARED,
            "reroute": C.MOE_OVERFLOW_REROUTE}


def make_config(T, d, E, top_k, F=0, capacity_factor=0.0, kind="gelu", bf16=True,
                has_shared=False, add_residual=False, n_group=0, topk_group=0, int8_weights=False,
                overflow="drop", int4_weights=False, y_fp32=False):
    """overflow: "drop", "shared" (dropped weight to the shared expert) or "reroute".
    int8_weights / int4_weights: weight-only INT8 / INT4 experts (codes + row scales).
    y_fp32: forward() keeps fp32 expert-output rows instead of fp16 with a power-of-two
    scale per 32 columns."""
    if int8_weights and int4_weights:
        raise ValueError("int8_weights and int4_weights exclude each other")
    kinds = {"linear": C.MOE_EXPERT_LINEAR, "gelu": C.MOE_EXPERT_GELU,
             "swiglu": C.MOE_EXPERT_SWIGLU}
    return MoeConfig(T=T, d=d, E=E, top_k=top_k, F=F, capacity_factor=capacity_factor,
                     act_dtype=C.MOE_BF16 if bf16 else C.MOE_F32, kind=kinds[kind],
                     has_shared=int(bool(has_shared)), add_residual=int(bool(add_residual)),
                     n_group=n_group, topk_group=topk_group,
                     w_dtype=C.MOE_I8 if int8_weights else (C.MOE_I4 if int4_weights else 0),
                     overflow=OVERFLOW[overflow], y_fp32=int(bool(y_fp32)))


def config_for(workload, T=None):
    """MoeConfig of a synth.Workload (optionally with another token count)."""
    return make_config(T if T is not None else workload.T, workload.d, workload.E, workload.k,
                       workload.F if workload.kind != "linear" else 0, workload.cf,
                       workload.kind, workload.bf16, workload.has_shared, workload.add_residual,
                       workload.n_group, workload.topk_group, workload.int8,
                       workload.overflow, workload.int4)


def weights(w1, b1=None, w2=None, b2=None, s1=None, s2=None):
    """Expert weights; for INT8 / INT4 experts w1 / w2 are the codes and s1 / s2 their
    per-row fp32 scales (see quantize_i8, quantize_i4)."""
    return MoeExpertWeights(w1=_ptr(w1), b1=_ptr(b1), w2=_ptr(w2), b2=_ptr(b2), s1=_ptr(s1),
                            s2=_ptr(s2))


def quantize_weights(w1, w2, stream=None, bits=8):
    """INT8 (bits=8) or packed INT4 (bits=4) codes and per-row scales of stacked bf16 expert
    weights: (q1, s1, q2, s2)."""
    import torch
    out = []
    for w in (w1, w2):
        s = torch.empty(w.shape[:-1], dtype=torch.float32, device=w.device)
        if bits == 8:
            q = torch.empty(w.shape, dtype=torch.int8, device=w.device)
            quantize_i8(w, q, s, stream)
        elif bits == 4:
            q = torch.empty(w.shape[:-1] + (w.shape[-1] // 2,), dtype=torch.uint8, device=w.device)
            quantize_i4(w, q, s, stream)
        else:
            raise ValueError("bits must be 8 or 4")
        out += [q, s]
    return tuple(out)


def quantize_i4(w, q, scale, stream=None):
    """Per-row absmax INT4 codes of a bf16 tensor (rows = all but the last axis, a multiple
    of 32 wide) into the uint8 tensor q (last axis halved: column 2j in the low nibble of
    byte j) and the fp32 tensor scale (one value per row)."""
    cols = w.shape[-1]
    _check(C.load().moe_quantize_i4(_ptr(w), w.numel() // cols, cols, _ptr(q), _ptr(scale),
                                    _stream(stream)), "moe_quantize_i4")


def quantize_i8(w, q, scale, stream=None):
    """Per-row absmax INT8 codes of a bf16 tensor (rows = all but the last axis) into the
    int8 tensor q (same shape) and the fp32 tensor scale (one value per row)."""
    cols = w.shape[-1]
    _check(C.load().moe_quantize_i8(_ptr(w), w.numel() // cols, cols, _ptr(q), _ptr(scale),
                                    _stream(stream)), "moe_quantize_i8")


def workspace_size(cfg):
    return int(C.load().moe_workspace_size(ctypes.byref(cfg)))


def max_rows(cfg):
    return int(C.load().moe_max_rows(ctypes.byref(cfg)))


def capacity(cfg):
    return int(C.load().moe_capacity(ctypes.byref(cfg)))


def route(cfg, x, W_gate, gate_bias, logits, topk_idx, topk_w, ws=None, stream=None):
    _check(C.load().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(W_gate), _ptr(gate_bias),
                              _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(ws),
                              _stream(stream)), "moe_route")


def dispatch(cfg, topk_idx, x, load, counts, offsets, perm_token, perm_slot, slot_dest,
             x_perm, ws, stream=None):
    _check(C.load().moe_dispatch(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(load),
                                 _ptr(counts), _ptr(offsets), _ptr(perm_token), _ptr(perm_slot),
                                 _ptr(slot_dest), _ptr(x_perm), _ptr(ws), _stream(stream)),
           "moe_dispatch")


def expert_ffn(cfg, x_perm, offsets, routed, shared, x, topk_w, perm_token, perm_slot, y, ws,
               stream=None):
    _check(C.load().moe_expert_ffn(ctypes.byref(cfg), _ptr(x_perm), _ptr(offsets),
                                   ctypes.byref(routed),
                                   ctypes.byref(shared) if shared is not None else None,
                                   _ptr(x), _ptr(topk_w), _ptr(perm_token), _ptr(perm_slot),
                                   _ptr(y), _ptr(ws), _stream(stream)), "moe_expert_ffn")


def combine(cfg, x, y, slot_dest, out, topk_w=None, stream=None):
    """topk_w is read when the layer sends overflow weight to the shared expert."""
    _check(C.load().moe_combine(ctypes.byref(cfg), _ptr(x), _ptr(y), _ptr(topk_w),
                                _ptr(slot_dest), _ptr(out), _stream(stream)), "moe_combine")


def forward(cfg, x, W_gate, gate_bias, routed, shared, out, ws, topk_idx=None, topk_w=None,
            load=None, stream=None):
    nbytes = ws.numel() * ws.element_size()
    _check(C.load().moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(W_gate), _ptr(gate_bias),
                                ctypes.byref(routed),
                                ctypes.byref(shared) if shared is not None else None,
                                _ptr(out), _ptr(topk_idx), _ptr(topk_w), _ptr(load), _ptr(ws),
                                nbytes, _stream(stream)), "moe_forward")


def grouped_gemm(A, B, row_offsets, D, ws, stream=None):
    """D[r] = A[r] @ B[g].T for the rows r of group g (bf16 in, fp32 out)."""
    G, N, K = B.shape
    _check(C.load().moe_grouped_gemm(_ptr(A), A.shape[0], _ptr(B), G, N, K, _ptr(row_offsets),
                                     _ptr(D), _ptr(ws), _stream(stream)), "moe_grouped_gemm")


def grouped_gemm_ws_size(G):
    return int(C.load().moe_grouped_gemm_ws_size(G))


def load_report(load_host, D):
    """Host-only LPT report; load_host is a numpy int32 array. Returns (assign, dev_load, imb)."""
    import numpy as np
    load_host = np.ascontiguousarray(load_host, np.int32)
    E = load_host.shape[0]
    assign = np.empty(E, np.int32)
    dev = np.empty(D, np.int64)
    imb = ctypes.c_double()
    _check(C.load().moe_load_report(ctypes.c_void_p(load_host.ctypes.data), E, D,
                                    ctypes.c_void_p(assign.ctypes.data),
                                    ctypes.c_void_p(dev.ctypes.data), ctypes.byref(imb)),
           "moe_load_report")
    return assign, dev, imb.value


def last_device_status(stream=None):
    return int(C.load().moe_last_device_status(_stream(stream)))


def status_string(status):
    return C.load().moe_status_string(status).decode()


def profile_begin():
    _check(C.load().moe_profile_begin(), "moe_profile_begin")


def profile_end(max_stats=64):
    arr = (C.MoeKernelStat * max_stats)()
    n = C.load().moe_profile_end(arr, max_stats)
    if n < 0:
        raise MoeError(C.MOE_ERR_CUDA, "moe_profile_end")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms))
            for i in range(min(n, max_stats))}


def kernel_launch_count():
    return int(C.load().moe_kernel_launch_count())


def selftest_wait_timeout(budget_cycles, stream=None):
    _check(C.load().moe_selftest_wait_timeout(int(budget_cycles), _stream(stream)),
           "moe_selftest_wait_timeout")


def dispatch_noalloc(cfg, topk_idx, x, load, counts, offsets, perm_token, perm_slot, slot_dest,
                     x_perm, stream=None):
    """moe_dispatch without a workspace (scratch in the library's static device array)."""
    fn = C.load().moe_dispatch_noalloc
    fn.restype = ctypes.c_int32
    fn.argtypes = [ctypes.POINTER(MoeConfig)] + [ctypes.c_void_p] * 10
    _check(fn(ctypes.byref(cfg), _ptr(topk_idx), _ptr(x), _ptr(load), _ptr(counts),
              _ptr(offsets), _ptr(perm_token), _ptr(perm_slot), _ptr(slot_dest), _ptr(x_perm),
              _stream(stream)), "moe_dispatch_noalloc")
