"""Python face of the C++ oracle of the steps either side of the decode stack (``sampling.cpp``):
the embedding lookup, and the choice of the next token from the LM head's logits.

TEST INFRASTRUCTURE ONLY (the same rule as llama_oracle.py).  "LLaMA-3 8B ...", section 三 (the
embedding is a row lookup) and section 十 (argmax, or a draw shaped by temperature, top-k and
top-p).  The readings taken where the page gives no formulas are listed in ``llama_oracle.h``:
T divides the logits (T <= 0: argmax); ranking by logit with ties to the lower id; top-k keeps
the first k; top-p, after top-k, keeps the shortest prefix reaching p of the top-k mass; the draw
is inverse CDF over the kept tokens in increasing id with a caller-supplied uniform u.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import check, lib


def _z(z):
    z = np.ascontiguousarray(np.asarray(z).reshape(-1), dtype=np.float64)
    return z, ctypes.c_void_p(z.ctypes.data), z.shape[0]


def embed(table, tokens) -> np.ndarray:
    """x[b] = E[token_b]: row token_b of the [vocab, d_model] table."""
    t = np.ascontiguousarray(table, dtype=np.float64)
    ids = np.ascontiguousarray(np.asarray(tokens).reshape(-1), dtype=np.int64)
    out = np.empty((ids.shape[0], t.shape[1]))
    check(lib().oracle_embed(t.ctypes.data, t.shape[0], t.shape[1], ids.ctypes.data, ids.shape[0],
                             out.ctypes.data), "embed")
    return out


def order_desc(z) -> np.ndarray:
    """Token ids ranked by logit, larger first, ties by the lower id."""
    z, pz, V = _z(z)
    ids = np.empty(V, dtype=np.int64)
    check(lib().oracle_order_desc(pz, V, ids.ctypes.data), "order_desc")
    return ids


def argmax(z) -> int:
    """The most probable token (the lowest id among equal maxima)."""
    z, pz, V = _z(z)
    return int(lib().oracle_argmax(pz, V))


def kept_set(z, temperature: float, top_k: int, top_p: float) -> np.ndarray:
    """The candidate tokens after top-k and top-p, in ranked order."""
    z, pz, V = _z(z)
    ids = np.empty(V, dtype=np.int64)
    n = ctypes.c_int64(0)
    check(lib().oracle_kept_set(pz, V, float(temperature), int(top_k), float(top_p), ids.ctypes.data,
                                ctypes.byref(n)), "kept_set")
    return ids[:n.value].copy()


def sample(z, temperature: float, top_k: int, top_p: float, u: float) -> int:
    """One draw from softmax(z / T) restricted to the kept set, by inverse CDF in token-id order."""
    z, pz, V = _z(z)
    return int(lib().oracle_sample(pz, V, float(temperature), int(top_k), float(top_p), float(u)))


def sample_margins(z, temperature: float, top_k: int, top_p: float, u: float):
    """(relative gap of the top-p cut to its target, relative gap of u * kept mass to the nearest
    cumulative boundary); inf where the rule does not apply.  An fp32 implementation that agrees
    with this oracle up to rounding can choose differently only where one of these is of the
    order of its rounding error."""
    z, pz, V = _z(z)
    m = np.empty(2)
    check(lib().oracle_sample_margins(pz, V, float(temperature), int(top_k), float(top_p), float(u),
                                      m.ctypes.data), "sample_margins")
    return float(m[0]), float(m[1])
