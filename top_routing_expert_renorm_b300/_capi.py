"""ctypes declarations of libmoe.so (the C ABI in include/moe.h).

Loading fails loudly when the library is missing: there is no fallback path.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe.so")

# moe_status
MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_WORKSPACE = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_DEVICE_INDEX = 7

# moe_dtype / moe_expert_kind
MOE_F32, MOE_BF16, MOE_I8, MOE_I4 = 0, 1, 2, 3
MOE_EXPERT_LINEAR, MOE_EXPERT_GELU, MOE_EXPERT_SWIGLU = 0, 1, 2
MOE_OVERFLOW_DROP, MOE_OVERFLOW_SHARED, MOE_OVERFLOW_REROUTE = 0, 1, 2


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("F", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("act_dtype", ctypes.c_int32),
                ("kind", ctypes.c_int32), ("has_shared", ctypes.c_int32),
                ("add_residual", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("w_dtype", ctypes.c_int32),
                ("overflow", ctypes.c_int32), ("y_fp32", ctypes.c_int32)]


class MoeExpertWeights(ctypes.Structure):
    _fields_ = [("w1", ctypes.c_void_p), ("b1", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("b2", ctypes.c_void_p), ("s1", ctypes.c_void_p), ("s2", ctypes.c_void_p)]


class MoeKernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


_lib = None


def load():
    """Load libmoe.so once (it must have been built: see build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmoe.so is not built ({LIB_PATH}); run "
                           "`python -m top_routing_expert_renorm_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    cfgp = ctypes.POINTER(MoeConfig)
    wp = ctypes.POINTER(MoeExpertWeights)
    sig = {
        "moe_workspace_size": (sz, [cfgp]),
        "moe_max_rows": (i64, [cfgp]),
        "moe_capacity": (i32, [cfgp]),
        "moe_route": (i32, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "moe_dispatch": (i32, [cfgp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "moe_expert_ffn": (i32, [cfgp, vp, vp, wp, wp, vp, vp, vp, vp, vp, vp, vp]),
        "moe_combine": (i32, [cfgp, vp, vp, vp, vp, vp, vp]),
        "moe_forward": (i32, [cfgp, vp, vp, vp, wp, wp, vp, vp, vp, vp, vp, sz, vp]),
        "moe_grouped_gemm_ws_size": (sz, [i32]),
        "moe_grouped_gemm": (i32, [vp, i64, vp, i32, i32, i32, vp, vp, vp, vp]),
        "moe_load_report": (i32, [vp, i32, i32, vp, vp, vp]),
        "moe_quantize_i8": (i32, [vp, i64, i32, vp, vp, vp]),
        "moe_quantize_i4": (i32, [vp, i64, i32, vp, vp, vp]),
        "moe_last_device_status": (i32, [vp]),
        "moe_status_string": (ctypes.c_char_p, [i32]),
        "moe_profile_begin": (i32, []),
        "moe_profile_end": (i32, [ctypes.POINTER(MoeKernelStat), i32]),
        "moe_kernel_launch_count": (ctypes.c_uint64, []),
        "moe_selftest_wait_timeout": (i32, [i64, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L
