"""Python face of the fp64 C++ oracle of the Llama decoder block forward (prefill and decode).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` may import this module.  The library in
``llama_decoder_block_fwd_gb300`` never calls it and shares no code with it; both sides only
share the seeded input generator in ``synth/``.

The arithmetic lives in ``llama_oracle.cpp`` (plain double-precision loops, OpenMP over
independent outputs; its header ``llama_oracle.h`` lists the pages, sections and readings each
function follows).  This module only checks shapes, lays arrays out as contiguous float64 and
passes pointers.

Parity pins for each function are in tests/test_oracle_pins.py.  No page prints a block output;
the whole block is pinned against an independent formulation from library routines (attention,
RMSNorm and SiLU routines of torch in float64, RoPE as complex multiplication) in
tests/test_oracle_block_library.py, and the stack by composition and by the same formulation.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from ._lib import LAYER_FN, DimsC, WeightsC, check, lib

_WEIGHT_FIELDS = ("attn_norm_g", "wq", "wk", "wv", "wo", "ffn_norm_g", "w_gate", "w_up", "w_down")


@dataclass(frozen=True)
class Dims:
    """The shared shape record: (B, S, d_model, n_q, n_kv, head_dim, d_ff, theta_base, eps)."""
    B: int
    S: int
    d_model: int
    n_q: int
    n_kv: int
    head_dim: int
    d_ff: int
    theta_base: float
    eps: float

    @property
    def r(self) -> int:
        return self.n_q // self.n_kv


@dataclass
class BlockWeights:
    """[out, in] matrices and [d_model] gains (any float dtype; passed as float64)."""
    attn_norm_g: np.ndarray
    wq: np.ndarray       # [n_q*hd, d]
    wk: np.ndarray       # [n_kv*hd, d]
    wv: np.ndarray       # [n_kv*hd, d]
    wo: np.ndarray       # [d, n_q*hd]
    ffn_norm_g: np.ndarray
    w_gate: np.ndarray   # [d_ff, d]
    w_up: np.ndarray     # [d_ff, d]
    w_down: np.ndarray   # [d, d_ff]


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def threads() -> int:
    """OpenMP threads the oracle's parallel loops use."""
    return int(lib().oracle_threads())


# ---------------------------------------------------------------------------------------- RMSNorm
def rmsnorm(x, g, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2 over the last axis) + eps) * g."""
    x = _f64(x)
    g = _f64(g)
    d = x.shape[-1]
    assert g.shape == (d,), (g.shape, d)
    y = np.empty_like(x)
    check(lib().oracle_rmsnorm(_p(x), x.size // d if d else 0, d, _p(g), float(eps), _p(y)), "rmsnorm")
    return y


# ---------------------------------------------------------------------------------------- SwiGLU
def silu(z) -> np.ndarray:
    """SiLU(z) = z / (1 + e^-z), elementwise."""
    z = _f64(z)
    out = np.empty_like(z)
    check(lib().oracle_silu(_p(z), z.size, _p(out)), "silu")
    return out


def swiglu_ffn(x, w_gate, w_up, w_down) -> np.ndarray:
    """W_down (SiLU(W_gate x) * W_up x) over the last axis of x; weights stored [out, in]."""
    x, wg, wu, wd = _f64(x), _f64(w_gate), _f64(w_up), _f64(w_down)
    d = x.shape[-1]
    dff = wg.shape[0]
    assert wg.shape == (dff, d) and wu.shape == (dff, d) and wd.shape == (d, dff)
    y = np.empty_like(x)
    check(lib().oracle_swiglu_ffn(_p(x), x.size // d, d, dff, _p(wg), _p(wu), _p(wd), _p(y)), "swiglu_ffn")
    return y


def ffn_dim_floor(d: int, multiple_of: int = 256) -> int:
    """floor(8d / (3 * multiple_of)) * multiple_of, the rule as printed."""
    return int(lib().oracle_ffn_dim_floor(d, multiple_of))


def ffn_dim_ceil(d: int, multiple_of: int = 256) -> int:
    """8d/3 rounded up to a multiple of multiple_of."""
    return int(lib().oracle_ffn_dim_ceil(d, multiple_of))


# ---------------------------------------------------------------------------------------- RoPE
def rope_theta(head_dim: int, theta_base: float) -> np.ndarray:
    """theta_k = theta_base^(-2k / head_dim), k = 0 .. head_dim/2 - 1."""
    out = np.empty(head_dim // 2, dtype=np.float64)
    check(lib().oracle_rope_theta(head_dim, float(theta_base), _p(out)), "rope_theta")
    return out


def rope(x, positions, theta_base: float) -> np.ndarray:
    """Rotate each interleaved pair (x_2k, x_2k+1) of x [..., T, H, hd] by positions[t] * theta_k."""
    x = _f64(x)
    pos = _f64(np.asarray(positions).reshape(-1))
    T, H, hd = x.shape[-3:]
    assert pos.shape == (T,), (pos.shape, T)
    y = np.empty_like(x)
    xs, ys = x.reshape(-1, T, H, hd), y.reshape(-1, T, H, hd)
    for i in range(xs.shape[0]):
        xi, yi = np.ascontiguousarray(xs[i]), np.empty((T, H, hd))
        check(lib().oracle_rope(_p(xi), T, H, hd, _p(pos), float(theta_base), _p(yi)), "rope")
        ys[i] = yi
    return y


# ---------------------------------------------------------------------------------------- attention
def kv_head_of(h: int, n_q: int, n_kv: int) -> int:
    """Query head h reads KV head floor(h / r), r = n_q / n_kv."""
    return int(lib().oracle_kv_head_of(h, n_q, n_kv))


def causal_probs(q, k, q_pos) -> np.ndarray:
    """Softmax over keys of q.k / sqrt(hd) with key j visible to a query at position m iff j <= m.

    q: [Sq, hd] (one head), k: [Tk, hd] (its KV head), q_pos: [Sq] absolute positions."""
    q, k = _f64(q), _f64(k)
    pos = _f64(np.asarray(q_pos).reshape(-1))
    Sq, hd = q.shape
    Tk = k.shape[0]
    assert k.shape == (Tk, hd) and pos.shape == (Sq,)
    p = np.empty((Sq, Tk))
    check(lib().oracle_causal_probs(_p(q), Sq, _p(k), Tk, hd, _p(pos), _p(p)), "causal_probs")
    return p


def gqa_attention(q, k, v, pos0: int = 0, q_rows=None) -> np.ndarray:
    """softmax(Q K~^T / sqrt(hd) + M_causal) V~ with K~, V~ the KV heads repeated r times.

    q: [B, Sq, n_q, hd] post-RoPE queries; k, v: [B, Tk, n_kv, hd] keys and values for positions
    0..Tk-1.  Query row s sits at position pos0 + s, or pos0 + q_rows[s].  Returns o [B, Sq, n_q, hd]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Sq, n_q, hd = q.shape
    Tk, n_kv = k.shape[1], k.shape[2]
    assert k.shape == (B, Tk, n_kv, hd) and v.shape == k.shape
    rows = np.arange(Sq) if q_rows is None else np.asarray(q_rows).reshape(-1)
    pos = _f64(pos0 + rows)
    o = np.empty_like(q)
    check(lib().oracle_gqa_attention(_p(q), _p(k), _p(v), B, Sq, Tk, n_q, n_kv, hd, _p(pos), _p(o)),
          "gqa_attention")
    return o


# ---------------------------------------------------------------------------------------- the block
def _dims_c(dims: Dims, B: int, S: int) -> DimsC:
    return DimsC(B, S, dims.d_model, dims.n_q, dims.n_kv, dims.head_dim, dims.d_ff, float(dims.theta_base),
                 float(dims.eps))


def _weights_c(w: BlockWeights, dims: Dims):
    """(pointer array, the float64 arrays it points into) after checking every shape."""
    d, hq, hkv, dff = dims.d_model, dims.n_q * dims.head_dim, dims.n_kv * dims.head_dim, dims.d_ff
    want = {"attn_norm_g": (d,), "wq": (hq, d), "wk": (hkv, d), "wv": (hkv, d), "wo": (d, hq),
            "ffn_norm_g": (d,), "w_gate": (dff, d), "w_up": (dff, d), "w_down": (d, dff)}
    arrs = []
    for name in _WEIGHT_FIELDS:
        a = _f64(getattr(w, name))
        assert a.shape == want[name], (name, a.shape, want[name])
        arrs.append(a)
    return WeightsC(*[a.ctypes.data for a in arrs]), arrs


def project_kv(x, w: BlockWeights, dims: Dims, pos0: int = 0):
    """Post-RoPE K and V of every token: u = RMSNorm(x); k = RoPE(u W_K^T); v = u W_V^T."""
    x = _f64(x)
    B, S, d = x.shape
    wc, keep = _weights_c(w, dims)
    k = np.empty((B, S, dims.n_kv, dims.head_dim))
    v = np.empty_like(k)
    dc = _dims_c(dims, B, S)
    check(lib().oracle_project_kv(ctypes.byref(dc), wc, _p(x), int(pos0), _p(k), _p(v)), "project_kv")
    return k, v


def _scales(kv_store):
    if kv_store is None:
        return None, None
    return (np.ascontiguousarray(kv_store.k_scale, dtype=np.float32),
            np.ascontiguousarray(kv_store.v_scale, dtype=np.float32))


def block_forward(x, w: BlockWeights, dims: Dims, pos0: int = 0, k_past=None, v_past=None, rows=None,
                  kv_store=None):
    """h = x + Attn(RMSNorm(x)); y = h + FFN(RMSNorm(h)).

    x: [B, S, d] for positions pos0 .. pos0+S-1.  k_past/v_past: [B, >= pos0, n_kv, hd] keys and
    values already cached for positions 0..pos0-1 (None when pos0 == 0).  When rows is given, K
    and V are still computed for every token, but the query side (and the output) only for those
    token rows.  kv_store (``fp8.kv_quant_fn``), if given, turns the new K/V into the values an
    8-bit cache stores, and attention reads those.  Returns (y [B, len(rows) or S, d],
    k_new, v_new [B, S, n_kv, hd])."""
    x = _f64(x)
    B, S, d = x.shape
    wc, keep = _weights_c(w, dims)
    n_kv, hd = dims.n_kv, dims.head_dim
    stride = 0
    kp = vp = None
    if pos0 > 0:
        kp, vp = _f64(k_past), _f64(v_past)
        assert kp.shape[0] == B and kp.shape[1] >= pos0 and kp.shape[2:] == (n_kv, hd) and vp.shape == kp.shape
        stride = kp.shape[1]
    sel = None if rows is None else np.ascontiguousarray(np.asarray(rows).reshape(-1), dtype=np.int64)
    R = S if sel is None else sel.shape[0]
    ks, vs = _scales(kv_store)
    y = np.empty((B, R, d))
    k_new = np.empty((B, S, n_kv, hd))
    v_new = np.empty_like(k_new)
    dc = _dims_c(dims, B, S)
    check(lib().oracle_block_forward(ctypes.byref(dc), wc, _p(x), int(pos0), _p(kp), _p(vp), stride, _p(sel), R,
                                     _p(ks), _p(vs), _p(y), _p(k_new), _p(v_new)), "block_forward")
    return y, k_new, v_new


def block_rows(x, w: BlockWeights, dims: Dims, k_all, v_all, rows, pos0: int = 0) -> np.ndarray:
    """The query side of block_forward alone for the listed rows of x [B, S, d], given the keys
    and values of positions 0..Tk-1 (k_all, v_all [B, Tk, n_kv, hd])."""
    x, ka, va = _f64(x), _f64(k_all), _f64(v_all)
    B, S, d = x.shape
    wc, keep = _weights_c(w, dims)
    sel = np.ascontiguousarray(np.asarray(rows).reshape(-1), dtype=np.int64)
    assert ka.shape[0] == B and ka.shape[2:] == (dims.n_kv, dims.head_dim) and va.shape == ka.shape
    y = np.empty((B, sel.shape[0], d))
    dc = _dims_c(dims, B, S)
    check(lib().oracle_block_rows(ctypes.byref(dc), wc, _p(x), int(pos0), _p(ka), _p(va), ka.shape[1], _p(sel),
                                  sel.shape[0], _p(y)), "block_rows")
    return y


# ---------------------------------------------------------------------------------------- the stack
def stack_decode_step(x_emb, layer_weights, n_layers: int, dims: Dims, t_cache: int, kv_cache, final_g, w_lm,
                      kv_store=None) -> np.ndarray:
    """One new token per sequence through n_layers blocks, then RMSNorm and the untied LM head.

    x_emb: [B, d] embedding rows of the new tokens (position t_cache).  layer_weights(l) returns
    the BlockWeights of layer l; kv_cache(l) returns (k, v) [B, >= t_cache, n_kv, hd] holding
    positions 0..t_cache-1; kv_store(l), if given, returns layer l's 8-bit store
    (``fp8.kv_quant_fn``).  The residual stream stays in fp64 across layers.  Each layer's arrays
    are fetched when the stack reaches it and released at the next.  Returns logits [B, vocab]."""
    x = _f64(x_emb)
    B, d = x.shape
    fg, wlm = _f64(final_g), _f64(w_lm)
    vocab = wlm.shape[0]
    assert fg.shape == (d,) and wlm.shape == (vocab, d)
    n_kv, hd = dims.n_kv, dims.head_dim
    held = {}
    errors = []

    def layer(ctx, l, out):
        try:
            held.clear()
            wc, arrs = _weights_c(layer_weights(int(l)), dims)
            k, v = kv_cache(int(l))
            k, v = _f64(k), _f64(v)
            assert k.shape[0] == B and k.shape[1] >= t_cache and k.shape[2:] == (n_kv, hd) and v.shape == k.shape
            ks, vs = _scales(None if kv_store is None else kv_store(int(l)))
            held.update(arrs=arrs, k=k, v=v, ks=ks, vs=vs)
            o = out.contents
            for name, a in zip(_WEIGHT_FIELDS, arrs):
                setattr(o, name, a.ctypes.data)
            o.k_past, o.v_past, o.past_stride = k.ctypes.data, v.ctypes.data, k.shape[1]
            o.k_scale = None if ks is None else ks.ctypes.data
            o.v_scale = None if vs is None else vs.ctypes.data
            return 0
        except Exception as e:  # reported after the call returns
            errors.append(e)
            return 1

    cb = LAYER_FN(layer)
    logits = np.empty((B, vocab))
    dc = _dims_c(dims, B, 1)
    rc = lib().oracle_stack_decode_step(ctypes.byref(dc), int(n_layers), cb, None, _p(x), int(t_cache), _p(fg),
                                        _p(wlm), vocab, _p(logits))
    held.clear()
    if errors:
        raise errors[0]
    check(rc, "stack_decode_step")
    return logits


# ---------------------------------------------------------------------------------------- sizes
def block_param_count(d: int, n_q: int, n_kv: int, hd: int, d_ff: int) -> int:
    """W_Q + W_K + W_V + W_O + three FFN matrices + two RMSNorm gains."""
    return int(lib().oracle_block_param_count(d, n_q, n_kv, hd, d_ff))


def model_param_count(n_layers: int, d: int, n_q: int, n_kv: int, hd: int, d_ff: int, vocab: int,
                      tied: bool = False) -> int:
    """Blocks + embedding + (untied) LM head + final RMSNorm gain."""
    return int(lib().oracle_model_param_count(n_layers, d, n_q, n_kv, hd, d_ff, vocab, int(tied)))


def kv_bytes_per_token(n_layers: int, n_kv: int, hd: int, bytes_per_elem: int) -> int:
    """K and V for every layer: 2 * n_kv * hd elements per layer."""
    return int(lib().oracle_kv_bytes_per_token(n_layers, n_kv, hd, bytes_per_elem))
