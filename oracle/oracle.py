"""ctypes wrappers around liboracle.so (numpy in, numpy out).

Test infrastructure only: see the header of oracle.cpp for the passages each
function follows and the readings taken where the pages are silent.
Dtype codes: 0 = fp32, 1 = bf16 (bf16 arrays are numpy uint16 bit patterns).
Expert kinds: 0 = LINEAR, 1 = GELU, 2 = SWIGLU.
"""

import ctypes
import numpy as np

from .build import build

F32, BF16 = 0, 1
LINEAR, GELU, SWIGLU = 0, 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        vp, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        L.oracle_bf16_round.restype = ctypes.c_uint16
        L.oracle_bf16_round.argtypes = [dbl]
        L.oracle_gelu.restype = dbl
        L.oracle_gelu.argtypes = [dbl]
        L.oracle_silu.restype = dbl
        L.oracle_silu.argtypes = [dbl]
        L.oracle_gate_logits.restype = None
        L.oracle_gate_logits.argtypes = [vp, i32, vp, vp, i32, i32, i32, vp, i32, vp]
        L.oracle_topk_renorm.restype = None
        L.oracle_topk_renorm.argtypes = [vp, i32, i32, i32, vp, vp]
        L.oracle_topk_renorm_grouped.restype = None
        L.oracle_topk_renorm_grouped.argtypes = [vp, i32, i32, i32, i32, i32, vp, vp]
        L.oracle_load.restype = None
        L.oracle_load.argtypes = [vp, i32, i32, i32, vp]
        L.oracle_capacity.restype = ctypes.c_int32
        L.oracle_capacity.argtypes = [dbl, i32, i32, i32]
        L.oracle_dispatch.restype = None
        L.oracle_dispatch.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
        L.oracle_rank_candidates.restype = None
        L.oracle_rank_candidates.argtypes = [vp, i32, i32, i32, i32, i32, i32, vp]
        L.oracle_dispatch_reroute.restype = None
        L.oracle_dispatch_reroute.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.oracle_expert_row.restype = None
        L.oracle_expert_row.argtypes = [i32, vp, i32, vp, vp, vp, vp, i32, i32, i32, vp]
        L.oracle_quantize_rows_i8.restype = None
        L.oracle_quantize_rows_i8.argtypes = [vp, ctypes.c_longlong, i32, vp, vp]
        L.oracle_quantize_rows_i4.restype = None
        L.oracle_quantize_rows_i4.argtypes = [vp, ctypes.c_longlong, i32, vp, vp]
        L.oracle_unpack_i4.restype = None
        L.oracle_unpack_i4.argtypes = [vp, ctypes.c_longlong, i32, vp]
        L.oracle_expert_row_q8.restype = None
        L.oracle_expert_row_q8.argtypes = [i32, vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, vp]
        L.oracle_combine_row.restype = None
        L.oracle_combine_row.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, i32]
        L.oracle_combine_row_ovf.restype = None
        L.oracle_combine_row_ovf.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, i32, vp, i32]
        L.oracle_forward.restype = None
        L.oracle_forward.argtypes = ([i32, i32, i32, i32, i32, i32, dbl, i32,
                                      vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      i32] + [vp] * 10 + [i32])
        L.oracle_load_report.restype = None
        L.oracle_load_report.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp, vp]
        _lib = L
    return _lib


def _p(a):
    """Pointer to a C-contiguous numpy array (or NULL for None)."""
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _dt(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"unsupported dtype {a.dtype}")


def bf16_round(v: float) -> int:
    """Round a real to bf16 (nearest, ties to even); returns the 16-bit pattern."""
    return int(lib().oracle_bf16_round(float(v)))


def gelu(a: float) -> float:
    return float(lib().oracle_gelu(float(a)))


def silu(a: float) -> float:
    return float(lib().oracle_silu(float(a)))


def gate_logits(x, Wg, bias=None, rows=None):
    """Gate logits [T or len(rows), E] in fp32 from double accumulation."""
    T, d = x.shape
    E = Wg.shape[1]
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n = T if rows_a is None else len(rows_a)
    out = np.empty((n, E), np.float32)
    Wg = np.ascontiguousarray(Wg, np.float32)
    b = None if bias is None else np.ascontiguousarray(bias, np.float32)
    lib().oracle_gate_logits(_p(x), _dt(x), _p(Wg), _p(b), T, d, E, _p(rows_a), n, _p(out))
    return out


def topk_renorm(logits, k, n_group=0, topk_group=0):
    """Top-k expert ids (logit desc, id asc) and renormalised weights, [T, k] each.
    With n_group > 0 the selection is group-limited: only the experts of the topk_group
    groups with the best expert logit are candidates."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    if n_group > 0:
        lib().oracle_topk_renorm_grouped(_p(logits), T, E, k, n_group, topk_group, _p(idx),
                                         _p(w))
    else:
        lib().oracle_topk_renorm(_p(logits), T, E, k, _p(idx), _p(w))
    return idx, w


def load(idx, E):
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    out = np.empty(E, np.int32)
    lib().oracle_load(_p(idx), T, k, E, _p(out))
    return out


def capacity(cf, T, k, E):
    return int(lib().oracle_capacity(float(cf), T, k, E))


def dispatch(idx, E, cap):
    """Returns counts[E], offsets[E+1], perm_token[P], perm_slot[P], slot_dest[T,k]."""
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    pt = np.full(T * k, -1, np.int32)
    ps = np.full(T * k, -1, np.int32)
    sd = np.empty((T, k), np.int32)
    lib().oracle_dispatch(_p(idx), T, k, E, int(cap), _p(counts), _p(offsets), _p(pt), _p(ps), _p(sd))
    P = int(offsets[E])
    return counts, offsets, pt[:P].copy(), ps[:P].copy(), sd


def expert_row(kind, x_row, w1, b1, w2, b2, d, F):
    """One token through one expert; returns y[d] in float64 (unrounded)."""
    y = np.empty(d, np.float64)
    x_row = np.ascontiguousarray(x_row)
    wdt = _dt(w1)
    lib().oracle_expert_row(kind, _p(x_row), _dt(x_row), _p(w1), _p(b1), _p(w2), _p(b2),
                            wdt, d, F, _p(y))
    return y


def combine_row(x_row, add_residual, w, kept, ys_k, ys_shared, out_dtype,
                overflow_to_shared=False):
    """One token's output; with overflow_to_shared the dropped slots' weights are added to
    the shared expert's weight (1 + sum of dropped w)."""
    x_row = np.ascontiguousarray(x_row)
    d = x_row.shape[0]
    k = len(w)
    w = np.ascontiguousarray(w, np.float32)
    kept = np.ascontiguousarray(kept, np.int32)
    ys_k = np.ascontiguousarray(ys_k, np.float64)
    ysh = None if ys_shared is None else np.ascontiguousarray(ys_shared, np.float64)
    out = np.empty(d, np.float32 if out_dtype == F32 else np.uint16)
    lib().oracle_combine_row_ovf(_p(x_row), _dt(x_row), int(add_residual), d, k, _p(w), _p(kept),
                                 _p(ys_k), _p(ysh), int(bool(overflow_to_shared)), _p(out),
                                 out_dtype)
    return out


def rank_candidates(logits, k, m, n_group=0, topk_group=0):
    """[T, m] experts at ranking positions k .. k+m-1 of each token (-1 past the end);
    with n_group > 0 only the experts of the chosen groups are ranked."""
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    cand = np.empty((T, m), np.int32)
    lib().oracle_rank_candidates(_p(logits), T, E, k, n_group, topk_group, m, _p(cand))
    return cand


def dispatch_reroute(idx, cand, E, cap):
    """Dispatch with one re-routing round. cand [T, k] are each token's next-ranked
    experts. Returns counts, offsets, perm_token[P], perm_slot[P], slot_dest[T,k] and
    route_idx[T,k] (the expert that processes each slot)."""
    idx = np.ascontiguousarray(idx, np.int32)
    cand = np.ascontiguousarray(cand, np.int32)
    T, k = idx.shape
    assert cand.shape == (T, k)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    pt = np.full(T * k, -1, np.int32)
    ps = np.full(T * k, -1, np.int32)
    sd = np.empty((T, k), np.int32)
    ri = np.empty((T, k), np.int32)
    lib().oracle_dispatch_reroute(_p(idx), _p(cand), T, k, E, int(cap), _p(counts), _p(offsets),
                                  _p(pt), _p(ps), _p(sd), _p(ri))
    P = int(offsets[E])
    return counts, offsets, pt[:P].copy(), ps[:P].copy(), sd, ri


def forward(kind, x, Wg, gate_bias, w1, b1, w2, b2, k, F, cf=0.0, add_residual=False,
            shared=None, overflow=0):
    """Whole-layer forward for host-resident inputs. Returns a dict of every output.

    shared: None or (sw1, sb1, sw2, sb2) for one always-on expert of the same kind.
    overflow: 0 drop, 1 dropped weight to the shared expert, 2 one re-routing round
    (idx then holds the expert that processes each slot).
    """
    T, d = x.shape
    E = Wg.shape[1]
    xdt = _dt(x)
    wdt = _dt(w1)
    out = np.empty((T, d), x.dtype)
    logits = np.empty((T, E), np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    ld = np.empty(E, np.int32)
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    pt = np.full(T * k, -1, np.int32)
    ps = np.full(T * k, -1, np.int32)
    sd = np.empty((T, k), np.int32)
    sw1, sb1, sw2, sb2 = shared if shared is not None else (None, None, None, None)
    lib().oracle_forward(kind, T, d, E, k, F, float(cf), int(bool(add_residual)),
                         _p(x), xdt, _p(np.ascontiguousarray(Wg, np.float32)), _p(gate_bias),
                         _p(w1), _p(b1), _p(w2), _p(b2), _p(sw1), _p(sb1), _p(sw2), _p(sb2),
                         wdt, _p(out), _p(logits), _p(idx), _p(w), _p(ld), _p(counts),
                         _p(offsets), _p(pt), _p(ps), _p(sd), int(overflow))
    P = int(offsets[E])
    return dict(out=out, logits=logits, idx=idx, w=w, load=ld, counts=counts,
                offsets=offsets, perm_token=pt[:P].copy(), perm_slot=ps[:P].copy(),
                slot_dest=sd)


def load_report(load_arr, D):
    """LPT placement report: dict(assign, dev_load, naive_load, imbalance, var_lpt, var_naive)."""
    load_arr = np.ascontiguousarray(load_arr, np.int32)
    E = load_arr.shape[0]
    assign = np.empty(E, np.int32)
    dev = np.empty(D, np.int64)
    naive = np.empty(D, np.int64)
    imb = ctypes.c_double()
    vl = ctypes.c_double()
    vn = ctypes.c_double()
    lib().oracle_load_report(_p(load_arr), E, D, _p(assign), _p(dev), _p(naive),
                             ctypes.byref(imb), ctypes.byref(vl), ctypes.byref(vn))
    return dict(assign=assign, dev_load=dev, naive_load=naive, imbalance=imb.value,
                var_lpt=vl.value, var_naive=vn.value)


def quantize_rows_i8(w_bf16):
    """Per-row absmax INT8 codes [rows, cols] int8 and fp32 scales [rows] of a bf16 matrix
    (uint16 bit patterns, any leading shape; rows = all but the last axis)."""
    w = np.ascontiguousarray(w_bf16, np.uint16)
    cols = w.shape[-1]
    rows = w.size // cols
    q = np.empty(w.shape, np.int8)
    s = np.empty(w.shape[:-1], np.float32)
    lib().oracle_quantize_rows_i8(_p(w), rows, cols, _p(q), _p(s))
    return q, s


def quantize_rows_i4(w_bf16):
    """Per-row absmax INT4 codes, packed two per byte ([..., cols / 2] uint8: column 2j in
    the low nibble of byte j, 2j+1 in the high one), and fp32 scales [rows]."""
    w = np.ascontiguousarray(w_bf16, np.uint16)
    cols = w.shape[-1]
    assert cols % 2 == 0
    rows = w.size // cols
    packed = np.empty(w.shape[:-1] + (cols // 2,), np.uint8)
    s = np.empty(w.shape[:-1], np.float32)
    lib().oracle_quantize_rows_i4(_p(w), rows, cols, _p(packed), _p(s))
    return packed, s


def unpack_i4(packed):
    """int8 codes [..., 2 * bytes] of a packed INT4 matrix."""
    pk = np.ascontiguousarray(packed, np.uint8)
    cols = 2 * pk.shape[-1]
    rows = pk.size // pk.shape[-1]
    q = np.empty(pk.shape[:-1] + (cols,), np.int8)
    lib().oracle_unpack_i4(_p(pk), rows, cols, _p(q))
    return q


def expert_row_q8(kind, x_row, q1, s1, b1, q2, s2, b2, d, F):
    """One token through one GELU / SWIGLU expert with INT8 weights (dequantised s*q)."""
    x_row = np.ascontiguousarray(x_row)
    xd = BF16 if x_row.dtype == np.uint16 else F32
    y = np.empty(d, np.float64)
    lib().oracle_expert_row_q8(kind, _p(x_row), xd, _p(np.ascontiguousarray(q1, np.int8)),
                               _p(np.ascontiguousarray(s1, np.float32)), _p(b1),
                               _p(np.ascontiguousarray(q2, np.int8)),
                               _p(np.ascontiguousarray(s2, np.float32)), _p(b2), d, F, _p(y))
    return y
