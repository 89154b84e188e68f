"""Seeded synthetic inputs shared by the oracle (host) and the GPU tests/bench (device).

Nothing here computes any part of the Llama block.  It draws the numbers that
both sides are fed: weights ~ N(0, 0.02), activations and cache ~ N(0, 1),
gains ~ N(1, 0.1) or ones.  The host library (``synth_host.c``) and the device
library (``synth_dev.cu``) implement one counter-based definition, documented at
the top of ``synth_host.c``, so a tensor drawn on the GPU equals, bit for bit,
the same tensor drawn on the host.  The "normal" draws are an Irwin-Hall sum of
twelve uniforms: mean 0, variance 1, bounded at +-6.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_HOST_SO = os.path.join(_DIR, "libsynth_host.so")
_DEV_SO = os.path.join(_DIR, "libsynth_dev.so")
_lock = threading.Lock()
_host = None
_dev = None

F32, BF16 = 0, 1

# Tensor ids inside one seed.  A layer's tensors use LAYER_STRIDE * layer + id.
TID_X = 1
TID_ATTN_G = 2
TID_WQ = 3
TID_WK = 4
TID_WV = 5
TID_WO = 6
TID_FFN_G = 7
TID_WGATE = 8
TID_WUP = 9
TID_WDOWN = 10
TID_KCACHE = 11
TID_VCACHE = 12
TID_FINAL_G = 13
TID_WLM = 14
TID_EMBED = 15     # token embedding table [vocab, d_model]
TID_LOGITS = 16    # stand-alone logits for the next-token choice
LAYER_STRIDE = 32


def host_build_cmd():
    return ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
            "-o", _HOST_SO, os.path.join(_DIR, "synth_host.c")]


def dev_build_cmd(nvcc="nvcc"):
    return [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
            "-Xcompiler", "-fPIC", "-shared", "-o", _DEV_SO, os.path.join(_DIR, "synth_dev.cu")]


def build_host():
    subprocess.check_call(host_build_cmd())


def build_dev():
    subprocess.check_call(dev_build_cmd())


def _stale(so, src):
    return (not os.path.exists(so)) or os.path.getmtime(so) < os.path.getmtime(src)


def _load_host():
    global _host
    with _lock:
        if _host is None:
            if _stale(_HOST_SO, os.path.join(_DIR, "synth_host.c")):
                build_host()
            lib = ctypes.CDLL(_HOST_SO)
            i64, u64, dbl, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
            lib.synth_fill_f32.argtypes = [vp, i64, u64, u64, i64, dbl, dbl]
            lib.synth_fill_bf16.argtypes = [vp, i64, u64, u64, i64, dbl, dbl]
            lib.synth_fill_f64_as.argtypes = [vp, ctypes.c_int, i64, u64, u64, i64, dbl, dbl]
            _host = lib
    return _host


def _load_dev():
    global _dev
    with _lock:
        if _dev is None:
            if not os.path.exists(_DEV_SO):
                raise RuntimeError(f"{_DEV_SO} is missing: run __graft_entry__.build() first")
            lib = ctypes.CDLL(_DEV_SO)
            lib.synth_fill_device.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                              ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                              ctypes.c_double, ctypes.c_double, ctypes.c_void_p]
            lib.synth_fill_device.restype = ctypes.c_int
            _dev = lib
    return _dev


def host_f64(dtype: int, shape, seed: int, tid: int, mean: float, std: float, offset: int = 0):
    """Draws widened exactly to fp64 after rounding to the stored dtype (F32 or BF16)."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float64)
    _load_host().synth_fill_f64_as(out.ctypes.data, int(dtype), n, seed, tid, int(offset),
                                   float(mean), float(std))
    return out.reshape(shape)


def host_bits(dtype: int, shape, seed: int, tid: int, mean: float, std: float, offset: int = 0):
    """Stored representation: float32 array, or uint16 array of bf16 bits."""
    n = int(np.prod(shape)) if len(shape) else 1
    lib = _load_host()
    if dtype == F32:
        out = np.empty(n, dtype=np.float32)
        lib.synth_fill_f32(out.ctypes.data, n, seed, tid, int(offset), float(mean), float(std))
    else:
        out = np.empty(n, dtype=np.uint16)
        lib.synth_fill_bf16(out.ctypes.data, n, seed, tid, int(offset), float(mean), float(std))
    return out.reshape(shape)


def device_fill(ptr: int, dtype: int, n: int, seed: int, tid: int, mean: float, std: float,
                offset: int = 0, stream: int = 0):
    """Fill n elements at device pointer ptr (asynchronous on stream)."""
    rc = _load_dev().synth_fill_device(ctypes.c_void_p(ptr), int(dtype), int(n), seed, tid,
                                       int(offset), float(mean), float(std), ctypes.c_void_p(stream))
    if rc != 0:
        raise RuntimeError(f"synth_fill_device failed with cudaError {rc}")


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
