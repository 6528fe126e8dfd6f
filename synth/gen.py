"""Host and device fills of the counter-based generator (see synth_host.c)."""

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SRC = os.path.join(HERE, "synth_host.c")
HOST_LIB = os.path.join(HERE, "libsynth_host.so")
DEV_SRC = os.path.join(HERE, "synth_dev.cu")
DEV_LIB = os.path.join(HERE, "libsynth_dev.so")

NORMAL, UNIFORM = 0, 1
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _stale(lib, src):
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


def build_host(force=False):
    if force or _stale(HOST_LIB, HOST_SRC):
        tmp = HOST_LIB + ".tmp"
        subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-o", tmp,
                        HOST_SRC], check=True)
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_dev(force=False):
    if force or _stale(DEV_LIB, DEV_SRC):
        tmp = DEV_LIB + ".tmp"
        subprocess.run([NVCC, "-O3", "-std=c++17", *ARCH, "-Xcompiler", "-fPIC", "-shared",
                        "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
                        "-o", tmp, DEV_SRC], check=True)
        os.replace(tmp, DEV_LIB)
    return DEV_LIB


_host = None
_dev = None


def _host_lib():
    global _host
    if _host is None:
        L = ctypes.CDLL(build_host())
        u64, vp, i32, f32 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        for name in ("synth_fill_f32", "synth_fill_bf16"):
            fn = getattr(L, name)
            fn.restype = None
            fn.argtypes = [u64, u64, u64, u64, i32, f32, vp]
        _host = L
    return _host


def _dev_lib():
    global _dev
    if _dev is None:
        L = ctypes.CDLL(build_dev())
        u64, vp, i32, f32 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.synth_dev_fill.restype = ctypes.c_int
        L.synth_dev_fill.argtypes = [u64, u64, u64, u64, i32, f32, i32, vp, vp]
        _dev = L
    return _dev


def normal_K(std):
    """fp32 scale turning the centred Irwin-Hall integer into an N(0, std^2)-like draw."""
    return float(np.float32(std * np.sqrt(3.0) / 131072.0))


def uniform_K(halfwidth):
    """fp32 scale turning the odd 24-bit integer into U(-halfwidth, halfwidth)."""
    return float(np.float32(halfwidth / float(1 << 23)))


def host_fill(seed, tid, offset, count, dist, K, bf16):
    """numpy array of `count` elements (float32, or uint16 bf16 bit patterns)."""
    L = _host_lib()
    if bf16:
        out = np.empty(count, np.uint16)
        L.synth_fill_bf16(seed, tid, offset, count, dist, K, ctypes.c_void_p(out.ctypes.data))
    else:
        out = np.empty(count, np.float32)
        L.synth_fill_f32(seed, tid, offset, count, dist, K, ctypes.c_void_p(out.ctypes.data))
    return out


def dev_fill(tensor, seed, tid, offset, dist, K, stream=None):
    """Fill a contiguous CUDA tensor (torch.float32 or torch.bfloat16) in place."""
    import torch
    assert tensor.is_cuda and tensor.is_contiguous()
    bf16 = tensor.dtype == torch.bfloat16
    assert bf16 or tensor.dtype == torch.float32
    s = stream if stream is not None else torch.cuda.current_stream()
    rc = _dev_lib().synth_dev_fill(seed, tid, offset, tensor.numel(), dist, K, int(bf16),
                                   ctypes.c_void_p(tensor.data_ptr()),
                                   ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise RuntimeError(f"synth_dev_fill failed with CUDA error {rc}")
    return tensor
