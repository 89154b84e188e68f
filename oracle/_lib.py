"""Build and load the C++ oracle library (liboracle.so): g++, OpenMP, plain fp64 loops.

TEST INFRASTRUCTURE ONLY: the tests, the build entry point's smoke check and the benchmark's
oracle legs load it.  The library is rebuilt here whenever a source is newer than it (g++ is on
every machine that runs the tests), so a fresh checkout needs no separate build step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

DIR = os.path.dirname(os.path.abspath(__file__))
SO = os.path.join(DIR, "liboracle.so")
SOURCES = ["llama_oracle.cpp", "e4m3.cpp", "sampling.cpp"]
HEADER = "llama_oracle.h"
_lock = threading.Lock()
_lib = None


def build_cmd(out: str = SO, extra=(), src_dir: str = DIR):
    # -ffp-contract=off: every product and sum rounds as written (no fused multiply-add), the same
    # arithmetic on x86 and Arm; no -ffast-math; the OpenMP runtime spreads independent outputs.
    return ["g++", "-std=c++17", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", *extra,
            "-o", out, *[os.path.join(src_dir, s) for s in SOURCES]]


def build() -> str:
    tmp = f"{SO}.{os.getpid()}.tmp"
    subprocess.check_call(build_cmd(tmp))
    os.replace(tmp, SO)
    return SO


def _stale() -> bool:
    if not os.path.exists(SO):
        return True
    t = os.path.getmtime(SO)
    return any(os.path.getmtime(os.path.join(DIR, s)) > t for s in SOURCES + [HEADER])


class LayerC(ctypes.Structure):
    _fields_ = [("attn_norm_g", ctypes.c_void_p), ("wq", ctypes.c_void_p), ("wk", ctypes.c_void_p),
                ("wv", ctypes.c_void_p), ("wo", ctypes.c_void_p), ("ffn_norm_g", ctypes.c_void_p),
                ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("k_past", ctypes.c_void_p), ("v_past", ctypes.c_void_p), ("past_stride", ctypes.c_int64),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p)]


class DimsC(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("S", ctypes.c_int64), ("d_model", ctypes.c_int64),
                ("n_q", ctypes.c_int64), ("n_kv", ctypes.c_int64), ("head_dim", ctypes.c_int64),
                ("d_ff", ctypes.c_int64), ("theta_base", ctypes.c_double), ("eps", ctypes.c_double)]


WeightsC = ctypes.c_void_p * 9   # the nine pointers of oracle_block_weights, in declaration order
LAYER_FN = ctypes.CFUNCTYPE(ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(LayerC))


def load(path: str):
    """A build of the oracle at path, with its signatures declared."""
    L = ctypes.CDLL(path)
    i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    sig = {
        "oracle_threads": (i32, []),
        "oracle_rmsnorm": (i32, [vp, i64, i64, vp, dbl, vp]),
        "oracle_silu": (i32, [vp, i64, vp]),
        "oracle_swiglu_ffn": (i32, [vp, i64, i64, i64, vp, vp, vp, vp]),
        "oracle_ffn_dim_floor": (i64, [i64, i64]),
        "oracle_ffn_dim_ceil": (i64, [i64, i64]),
        "oracle_rope_theta": (i32, [i64, dbl, vp]),
        "oracle_rope": (i32, [vp, i64, i64, i64, vp, dbl, vp]),
        "oracle_kv_head_of": (i64, [i64, i64, i64]),
        "oracle_causal_probs": (i32, [vp, i64, vp, i64, i64, vp, vp]),
        "oracle_gqa_attention": (i32, [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp, vp]),
        "oracle_project_kv": (i32, [ctypes.POINTER(DimsC), vp, vp, i64, vp, vp]),
        "oracle_block_forward": (i32, [ctypes.POINTER(DimsC), vp, vp, i64, vp, vp, i64, vp, i64, vp, vp,
                                       vp, vp, vp]),
        "oracle_block_rows": (i32, [ctypes.POINTER(DimsC), vp, vp, i64, vp, vp, i64, vp, i64, vp]),
        "oracle_stack_decode_step": (i32, [ctypes.POINTER(DimsC), i64, LAYER_FN, vp, vp, i64, vp, vp,
                                           i64, vp]),
        "oracle_block_param_count": (i64, [i64, i64, i64, i64, i64]),
        "oracle_model_param_count": (i64, [i64, i64, i64, i64, i64, i64, i64, i32]),
        "oracle_kv_bytes_per_token": (i64, [i64, i64, i64, i64]),
        "oracle_e4m3_decode": (i32, [vp, i64, vp]),
        "oracle_e4m3_encode": (i32, [vp, i64, vp]),
        "oracle_kv_quantize": (i32, [vp, i64, i64, i64, vp, vp]),
        "oracle_kv_dequantize": (i32, [vp, i64, i64, i64, vp, vp]),
        "oracle_embed": (i32, [vp, i64, i64, vp, i64, vp]),
        "oracle_order_desc": (i32, [vp, i64, vp]),
        "oracle_argmax": (i64, [vp, i64]),
        "oracle_kept_set": (i32, [vp, i64, dbl, i64, dbl, vp, vp]),
        "oracle_sample": (i64, [vp, i64, dbl, i64, dbl, dbl]),
        "oracle_sample_margins": (i32, [vp, i64, dbl, i64, dbl, dbl, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    return L


def lib():
    """The loaded library (built first when a source is newer than it)."""
    global _lib
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = load(SO)
    return _lib


def check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"{what}: the oracle refused its arguments")
