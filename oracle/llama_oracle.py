"""fp64 CPU oracle for the Llama decoder block forward (prefill and KV-cache decode).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The library in ``llama_decoder_block_fwd_gb300`` never calls it and
shares no code with it; both sides only share the seeded input generator in
``synth/``.

Every function is the plain definition written out in float64, in the order
the pages state it, with numpy's matmul as the only library primitive.  There
is no tiling, no fusion and no online softmax.

Sources (page title, section):
  [P1] "Llama Architecture: RMSNorm, SwiGLU, RoPE, GQA, and PyTorch
       Implementation" (ailinkdeeptech.com/research/llama):
       Mathematical Foundations 1 (RMSNorm), 2 (SwiGLU), 3 (RoPE), 4 (GQA and
       KV cache scaling); Production PyTorch Implementation, Steps 1-2.
  [P2] "RMSNorm" study note (ai-engineer-exhaustive, LLaMA): "How it works".
  [P3] "LLaMA-3 8B 现代 LLM 架构、计算规模与能耗" (ienjoy.github.io/llama3-8b.html):
       sections 四 (one block), 4.1-4.7 (8Q/2KV toy), 五 (SwiGLU), 六 (parameter
       counts), 七 (KV cache), 九 (decode), 十 (final norm and LM head).
  [P4] "LLaMA Architecture > Model Architecture" (mbrenndoerfer.com):
       "The Transformer Block" (block equations), "Key Architectural Choices".

Readings taken where the pages are silent or disagree:
  * eps sits inside the square root (P2 "How it works", P4, P1 Step 1 code);
    P1 section 1's displayed equation puts it outside.
  * RoPE frequency theta_k = theta_base^(-2k/head_dim), interleaved pairs
    (x_2k, x_2k+1), rotation by +m*theta_k as in P1 section 3's matrix.
  * Positions are 0-based absolute positions; a query at position m sees keys
    0..m (causal, bottom-right aligned when a cache precedes the new tokens).
  * Query head h reads KV head floor(h / r), r = n_q / n_kv (P1 section 4
    repeat_interleave, P3 4.4 g(h) = floor(h/4)).
  * Softmax scale 1/sqrt(head_dim) (P1 section 4, P3 4.5).
  * Weights are stored [out, in] (nn.Linear, P1 section 2), so y = x W^T.
  * No intermediate rounding: the oracle is exact fp64 arithmetic on the
    (already rounded) stored inputs.

Parity pins for each function are in tests/test_oracle_pins.py.  No page prints
a block output; the whole block is pinned against an independent formulation from
library routines (attention, RMSNorm and SiLU routines of torch in float64, RoPE as
complex multiplication) in tests/test_oracle_block_library.py, and the stack by
composition (a stack is the chain of its blocks).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


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


# ----------------------------------------------------------------------------------------
# RMSNorm  [P1 section 1; P2 "How it works"; P4 "Key Architectural Choices"]
# ----------------------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2 over the feature axis) + eps) * g, reduced over the last axis only."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


# ----------------------------------------------------------------------------------------
# SwiGLU  [P1 section 2; P3 section 五; P4 "Key Architectural Choices"]
# ----------------------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + e^-z)."""
    return z / (1.0 + np.exp(-z))


def swiglu_ffn(x: np.ndarray, w_gate: np.ndarray, w_up: np.ndarray, w_down: np.ndarray) -> np.ndarray:
    """W_down (SiLU(W_gate x) * W_up x), no biases; weights stored [out, in]."""
    gate = x @ w_gate.T
    up = x @ w_up.T
    return (silu(gate) * up) @ w_down.T


def ffn_dim_floor(d: int, multiple_of: int = 256) -> int:
    """The d_ff rule as P1 section 2 prints it: floor(8d / (3 * multiple_of)) * multiple_of."""
    return (8 * d) // (3 * multiple_of) * multiple_of


def ffn_dim_ceil(d: int, multiple_of: int = 256) -> int:
    """8d/3 rounded UP to a multiple: the rule that reproduces P4's LLaMA-1 table."""
    return -(-(8 * d) // (3 * multiple_of)) * multiple_of


# ----------------------------------------------------------------------------------------
# RoPE  [P1 section 3; P3 section 四.3]
# ----------------------------------------------------------------------------------------
def rope_theta(head_dim: int, theta_base: float) -> np.ndarray:
    """theta_k = theta_base^(-2k / head_dim), k = 0 .. head_dim/2 - 1."""
    k = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta_base), -2.0 * k / head_dim)


def rope(x: np.ndarray, positions: np.ndarray, theta_base: float) -> np.ndarray:
    """Rotate each interleaved pair (x_2k, x_2k+1) by angle m * theta_k.

    x: [..., T, H, head_dim]; positions: [T] absolute positions m.
    (x_2k, x_2k+1) -> (x_2k cos - x_2k+1 sin, x_2k sin + x_2k+1 cos).
    """
    hd = x.shape[-1]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_theta(hd, theta_base)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape), dtype=np.float64)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


# ----------------------------------------------------------------------------------------
# Causal grouped-query attention  [P1 section 4; P3 4.4-4.6 and section 四.4]
# ----------------------------------------------------------------------------------------
def kv_head_of(h: int, n_q: int, n_kv: int) -> int:
    """Query head h reads KV head floor(h / r), r = n_q / n_kv."""
    return h // (n_q // n_kv)


def causal_probs(q: np.ndarray, k: np.ndarray, q_pos: np.ndarray) -> np.ndarray:
    """Softmax over keys of q.k / sqrt(hd), key j visible to a query at position m iff j <= m.

    q: [Sq, hd] (one head), k: [Tk, hd] (its KV head), q_pos: [Sq] absolute positions.
    The row max is subtracted before exponentiating (an exact identity of softmax).
    """
    hd = q.shape[-1]
    scores = (q @ k.T) / math.sqrt(hd)
    visible = np.arange(k.shape[0])[None, :] <= np.asarray(q_pos)[:, None]
    scores = np.where(visible, scores, -np.inf)
    mx = np.max(scores, axis=-1, keepdims=True)
    e = np.exp(scores - mx)
    return e / np.sum(e, axis=-1, keepdims=True)


def gqa_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, pos0: int = 0,
                  q_rows: np.ndarray | None = None) -> np.ndarray:
    """softmax(Q K~^T / sqrt(hd) + M_causal) V~ with K~, V~ the KV heads repeated r times.

    q: [B, Sq, n_q, hd] post-RoPE queries; k, v: [B, Tk, n_kv, hd] post-RoPE keys and values
    for absolute positions 0..Tk-1.  Query row s sits at position pos0 + s, or at
    pos0 + q_rows[s] when only some rows of the sequence are given.
    Returns o: [B, Sq, n_q, hd].
    """
    B, Sq, n_q, hd = q.shape
    n_kv = k.shape[2]
    rows = np.arange(Sq) if q_rows is None else np.asarray(q_rows)
    q_pos = pos0 + rows
    o = np.empty_like(q, dtype=np.float64)
    for b in range(B):
        for h in range(n_q):
            g = kv_head_of(h, n_q, n_kv)
            p = causal_probs(q[b, :, h, :], k[b, :, g, :], q_pos)
            o[b, :, h, :] = p @ v[b, :, g, :]
    return o


# ----------------------------------------------------------------------------------------
# One decoder block  [P1 Step 2 LlamaTransformerBlock; P3 sections 四-五; P4 block equations]
# ----------------------------------------------------------------------------------------
@dataclass
class BlockWeights:
    """[out, in] matrices and [d_model] gains, fp64."""
    attn_norm_g: np.ndarray
    wq: np.ndarray       # [n_q*hd, d]
    wk: np.ndarray       # [n_kv*hd, d]
    wv: np.ndarray       # [n_kv*hd, d]
    wo: np.ndarray       # [d, n_q*hd]
    ffn_norm_g: np.ndarray
    w_gate: np.ndarray   # [d_ff, d]
    w_up: np.ndarray     # [d_ff, d]
    w_down: np.ndarray   # [d, d_ff]


def project_kv(x: np.ndarray, w: BlockWeights, dims: Dims, pos0: int = 0):
    """Post-RoPE K and V of every token: u = RMSNorm(x); k = RoPE(u W_K^T); v = u W_V^T."""
    B, S, _ = x.shape
    u = rmsnorm(x, w.attn_norm_g, dims.eps)
    pos = pos0 + np.arange(S)
    k = rope((u @ w.wk.T).reshape(B, S, dims.n_kv, dims.head_dim), pos, dims.theta_base)
    v = (u @ w.wv.T).reshape(B, S, dims.n_kv, dims.head_dim)
    return k, v


def block_forward(x: np.ndarray, w: BlockWeights, dims: Dims, pos0: int = 0,
                  k_past: np.ndarray | None = None, v_past: np.ndarray | None = None,
                  rows: np.ndarray | None = None, kv_store=None):
    """h = x + Attn(RMSNorm(x)); y = h + FFN(RMSNorm(h)).

    x: [B, S, d] for positions pos0 .. pos0+S-1.  k_past/v_past: [B, pos0, n_kv, hd] keys and
    values already cached for positions 0..pos0-1 (None when pos0 == 0).  When rows is given,
    K and V are still computed for every token, but the query side (and the output) only for
    those token rows.  kv_store, if given, maps (k_new, v_new) to the values the cache holds
    (an 8-bit cache encodes them); attention then reads those.  Returns (y [B, len(rows) or S, d],
    k_new, v_new [B, S, n_kv, hd]).
    """
    B, S, d = x.shape
    k_new, v_new = project_kv(x, w, dims, pos0)
    if kv_store is not None:
        k_new, v_new = kv_store(k_new, v_new)
    if pos0 > 0:
        k_all = np.concatenate([k_past[:, :pos0], k_new], axis=1)
        v_all = np.concatenate([v_past[:, :pos0], v_new], axis=1)
    else:
        k_all, v_all = k_new, v_new
    sel = np.arange(S) if rows is None else np.asarray(rows)
    xs = x[:, sel, :]
    u = rmsnorm(xs, w.attn_norm_g, dims.eps)
    q = rope((u @ w.wq.T).reshape(B, len(sel), dims.n_q, dims.head_dim), pos0 + sel, dims.theta_base)
    o = gqa_attention(q, k_all, v_all, pos0, q_rows=sel)
    h = xs + o.reshape(B, len(sel), dims.n_q * dims.head_dim) @ w.wo.T
    y = h + swiglu_ffn(rmsnorm(h, w.ffn_norm_g, dims.eps), w.w_gate, w.w_up, w.w_down)
    return y, k_new, v_new


# ----------------------------------------------------------------------------------------
# Stack decode step  [P3 section 二 data flow, section 九 decode, section 十 head]
# ----------------------------------------------------------------------------------------
def stack_decode_step(x_emb: np.ndarray, layer_weights, n_layers: int, dims: Dims, t_cache: int,
                      kv_cache, final_g: np.ndarray, w_lm: np.ndarray, kv_store=None) -> np.ndarray:
    """One new token per sequence through n_layers blocks, then RMSNorm and the untied LM head.

    x_emb: [B, d] embedding rows of the new tokens (position t_cache).  layer_weights(l) returns
    the BlockWeights of layer l; kv_cache(l) returns (k, v) [B, >=t_cache, n_kv, hd] holding
    positions 0..t_cache-1.  kv_store(l), if given, returns layer l's map from the new token's
    K/V to the values the cache holds.  The residual stream stays in fp64 across layers.
    Returns logits [B, vocab].
    """
    x = x_emb[:, None, :].astype(np.float64)
    for l in range(n_layers):
        k_past, v_past = kv_cache(l)
        x, _, _ = block_forward(x, layer_weights(l), dims, pos0=t_cache,
                                k_past=k_past, v_past=v_past,
                                kv_store=None if kv_store is None else kv_store(l))
    z = rmsnorm(x[:, 0, :], final_g, dims.eps)
    return z @ w_lm.T


# ----------------------------------------------------------------------------------------
# Sizes  [P3 sections 六 and 七]
# ----------------------------------------------------------------------------------------
def block_param_count(d: int, n_q: int, n_kv: int, hd: int, d_ff: int) -> int:
    """W_Q + W_K + W_V + W_O + three FFN matrices + two RMSNorm gains."""
    return d * n_q * hd + 2 * d * n_kv * hd + n_q * hd * d + 3 * d * d_ff + 2 * d


def model_param_count(n_layers: int, d: int, n_q: int, n_kv: int, hd: int, d_ff: int,
                      vocab: int, tied: bool = False) -> int:
    """Blocks + embedding + (untied) LM head + final RMSNorm gain."""
    emb = vocab * d
    return n_layers * block_param_count(d, n_q, n_kv, hd, d_ff) + emb + (0 if tied else emb) + d


def kv_bytes_per_token(n_layers: int, n_kv: int, hd: int, bytes_per_elem: int) -> int:
    """K and V for every layer: 2 * n_kv * hd elements per layer."""
    return n_layers * 2 * n_kv * hd * bytes_per_elem
