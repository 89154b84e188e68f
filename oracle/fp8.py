"""Python face of the C++ oracle's 8-bit KV cache format (``e4m3.cpp``): OCP E4M3 codes with one
fp32 scale per (layer, K or V, KV head).

TEST INFRASTRUCTURE ONLY (the same rule as llama_oracle.py).  The readings taken where the pages
give no 8-bit format are stated in ``e4m3.cpp``: E4M3 as OCP defines it, x ~= code * s, the
quotient x / s taken in fp32 and rounded to the nearest code (ties to the even code), saturating at
+-448; attention reads the decoded values, the new token's own K/V included.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from ._lib import check, lib


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def e4m3_decode(code) -> np.ndarray:
    """Value of each E4M3 code (uint8 array) as fp64."""
    c = np.ascontiguousarray(code, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    check(lib().oracle_e4m3_decode(_p(c), c.size, _p(out)), "e4m3_decode")
    return out


def e4m3_encode(q) -> np.ndarray:
    """Nearest E4M3 code to each value of q (ties to the even code), saturating at +-448."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    out = np.empty(q.shape, dtype=np.uint8)
    check(lib().oracle_e4m3_encode(_p(q), q.size, _p(out)), "e4m3_encode")
    return out


def _heads(x, scale):
    s = np.ascontiguousarray(np.asarray(scale).reshape(-1), dtype=np.float32)
    n_kv, hd = x.shape[-2], x.shape[-1]
    assert s.shape == (n_kv,), (s.shape, n_kv)
    return s, x.size // (n_kv * hd) if n_kv * hd else 0, n_kv, hd


def quantize(x, scale) -> np.ndarray:
    """Codes of x [..., n_kv, hd] with one scale per KV head (scale [n_kv]), quotient in fp32."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    s, n, n_kv, hd = _heads(x, scale)
    out = np.empty(x.shape, dtype=np.uint8)
    check(lib().oracle_kv_quantize(_p(x), n, n_kv, hd, _p(s), _p(out)), "kv_quantize")
    return out


def dequantize(code, scale) -> np.ndarray:
    """code * s in fp64 for codes [..., n_kv, hd] and scale [n_kv]."""
    c = np.ascontiguousarray(code, dtype=np.uint8)
    s, n, n_kv, hd = _heads(c, scale)
    out = np.empty(c.shape, dtype=np.float64)
    check(lib().oracle_kv_dequantize(_p(c), n, n_kv, hd, _p(s), _p(out)), "kv_dequantize")
    return out


@dataclass
class KVStore:
    """An 8-bit cache's per-head scales for K and V; block_forward / stack_decode_step replace the
    new tokens' K and V by the values the cache stores.  Calling it applies that map directly."""
    k_scale: np.ndarray
    v_scale: np.ndarray

    def __call__(self, k_new, v_new):
        return (dequantize(quantize(k_new, self.k_scale), self.k_scale),
                dequantize(quantize(v_new, self.v_scale), self.v_scale))


def kv_quant_fn(k_scale, v_scale) -> KVStore:
    """The store of an 8-bit cache with these per-head scales."""
    return KVStore(np.asarray(k_scale, dtype=np.float32), np.asarray(v_scale, dtype=np.float32))
